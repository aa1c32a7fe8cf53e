// Paged MQA logits of grouped query rows on the Blackwell tensor cores,
// fused with the first pass of the top-k selection.
//
// score[r][t] = sum_h w[r][h] * ReLU(q_h . k_t)   (page "cutedsl.dsa.index",
// module docstring; page "amd.ops.fp4_indexer", score_paged).
//
// Work unit: a tile of 128 keys (two 64-token cache pages from the block table)
// against a segment of up to 4 query rows of one request (N = 32 * rows MMA
// columns), so the keys a request's rows share are read from HBM once.
// Keys sit on the MMA's M dimension, heads x rows on N:
//   D[128 keys][32 * rows] = K[128 x 128] . Q[32 * rows x 128]^T   (FP32 in TMEM)
//
// Warp roles of the persistent CTA (one per SM):
//   warp 0     planner: resolves 32 tiles' segments and block-table pages at a
//              time, loads each segment's query rows (TMA), tags each ring
//              stage (8 stages of 16 KB for FP8, 16 of 8 KB for packed MXFP4)
//              and hands the tile's page ids to its copy warp.
//   warps 1-2  tcgen05 issuers of alternate tiles: scale factors into TMEM,
//              the tile's MMAs (FP8: 4 with K = 32; MXFP4: 2 with K = 64) into
//              one of three TMEM accumulators.
//   warps 3-10 epilogue, two groups of four: tcgen05.ld of the accumulator
//              (thread = key), ReLU-weighted head sum, FP32 key scale, logits
//              store, and a shared-memory histogram of the scores for the
//              top-k pass.
//   warps 11-14  copy warps: warp 11 + c issues every TMA copy (both pages'
//              codes and scales) of the tiles at positions c, c + 4, ...  One
//              copy-issuing thread moves about one page per few hundred
//              nanoseconds whatever the page size, so four of them keep the
//              HBM gather going.
//
// Formats: FP8 uses kind::f8f6f4 (E4M3 x E4M3) and multiplies the per-key
// FP32 scale in the epilogue.  FP8-MX uses kind::mxf8f6f4 with one UE8M0 key
// scale per 32 columns (scale byte kk in instruction kk).  MXFP4 keeps its codes packed and uses
// kind::mxf4 (K = 64, two UE8M0 scales per row from TMEM, scale bytes 2m and
// 2m + 1 in instruction m).  Token-major pages are 64 rows of 64 bytes, which
// one TMA box lands in the 64-byte-swizzled K-major layout; as packed stages
// take half the shared memory, that format runs a 16-stage ring.  Row-group
// pages place each column group's 64 x 16 bytes together: one TMA box per
// group lands as 8 unswizzled core matrices, the two pages' boxes of a group
// side by side.
#include "host.h"
#include "scan.cuh"

namespace dsa {

constexpr int kStages = 8;                    // ring stages of 16 KB (FP8 codes)
constexpr int kMaxStages = 16;                // ring stages of 8 KB (packed MXFP4, either placement)
constexpr int kTileRows = 128;
constexpr int kTileBytes = kTileRows * 128;   // codes of 128 keys in shared memory
constexpr int kPageSmem = 64 * 128;           // one FP8 page's codes in shared memory
// Transaction bytes of one TMA copy: an MXFP4 page's codes 4096, an MXFP4
// query row 2048 (packed, as in shared memory).
constexpr uint32_t kFp8PageTx = 64 * 128, kFp4PageTx = 64 * 64;
constexpr uint32_t kFp8QRowTx = kQRowBytes;
// Row-group MXFP4 in shared memory: a tile's column group g at g * 2048 (the
// two pages' 1024-byte boxes in key order); query chunk c (16 bytes = 32
// columns of every head) at c * 2048, query row r's 32 heads at + r * 512.
constexpr int kRgTileGroup = 2 * kRgGroupBytes;
constexpr int kRgQChunk = 2048;
constexpr int kSegRows = 4;                   // most query rows per segment (min(4, 128 / heads))
// Raw query scale bytes staged per row: 32 heads x 4 (token-major MXFP4) or
// the row's 4 x 64 row-group slots.
constexpr int kQsfRow = 128, kQsfRowRg = 4 * kRgQuerySlots;
// A segment's queries: rows x heads x 128 B (FP8, 32 heads) or 64 B (MXFP4);
// heads x segment rows <= 128 (the MMA's N), so one buffer holds 16 KB at most.
constexpr int kQBufBytes = kSegRows * kQRowBytes;
// Two epilogue groups of four warps (one per TMEM lane quarter) drain
// alternate tiles, so two accumulators are read out at once.
constexpr int kEpiGroups = 2;
constexpr int kEpiWarps = 4 * kEpiGroups;
// Two MMA-issuing warps: warp 1 + w issues the tiles of sequence positions
// w, w + 2, ... (so it alone uses ring stages of that parity), which epilogue
// group w drains.
constexpr int kMmaWarps = 2;
constexpr int kFirstEpiWarp = 1 + kMmaWarps;
// Copy warps: warp kFirstCopyWarp + c issues every copy (both pages' codes and
// scales) of the tiles at sequence positions c, c + kCopyWarps, ...  A
// thread that issues TMA copies moves about one page per few hundred
// nanoseconds whatever the page size, so the copy rate an SM needs takes
// several issuing threads.
constexpr int kFirstCopyWarp = kFirstEpiWarp + kEpiWarps;
constexpr int kCopyWarps = 4;
constexpr int kScoreThreads = 32 * (kFirstCopyWarp + kCopyWarps);
// Page ids handed from warp 0 to the copy warps: a ring of kPageRing entries
// {first page, second page} (>= 0 page, kNoPage none, kEndMark end of sequence).
constexpr int kPageRing = 64, kNoPage = -1, kEndMark = -2;
// The planner stays at most kLead positions ahead of the copy warps (the
// ring entry it overwrites, kPageRing positions back, is older still).
constexpr int kLead = 56;
static_assert(kLead < kPageRing, "the ring holds the planner's lead");
static_assert(kStages % kCopyWarps == 0 && kMaxStages % kCopyWarps == 0, "copy warp c owns the stages of its residue");
static_assert(kMmaWarps == kEpiGroups && kStages % kMmaWarps == 0 && kMaxStages % kMmaWarps == 0,
              "issuer w owns stages and group w");
constexpr int kAcc = 3;                       // TMEM accumulators in flight (MMA latency is hidden behind 2)
constexpr int kPlanSmemSegs = 4096;           // segments whose tile prefix the plan keeps on chip
// Tile assignment: every CTA owns one contiguous range of tiles (segment
// locality), the ranges splitting the tiles' estimated cost evenly.

constexpr int OFF_TILES = 0;
constexpr int OFF_QBUF = OFF_TILES + kStages * kTileBytes;
constexpr int OFF_RAWSC = OFF_QBUF + 2 * kQBufBytes;   // key scales per stage
constexpr int OFF_SFA = OFF_RAWSC + kMaxStages * 512;
constexpr int OFF_QSF = OFF_SFA + kMaxStages * 512;
constexpr int kQsfBytes = 4 * kQsfRowRg;                 // raw query scales of a buffer's rows
constexpr int OFF_SFB = OFF_QSF + 2 * kQsfBytes;
constexpr int OFF_KS = OFF_SFB + 2 * kMmaWarps * 512;   // query scale atoms per (buffer, issuer)
constexpr int OFF_W = OFF_KS + kAcc * 128 * 4;            // float[kEpiWarps][4 rows][32 heads]: w per warp
// Score histogram of each epilogue group for its current segment: 4 rows x
// 2048 bins of 16-bit counts, two per word; added to the rows' histograms in
// global memory when the segment changes and at least every kHistFlushTiles
// tiles (so that no count passes 2^16 - 1).
constexpr int kHistFlushTiles = 256;
constexpr int OFF_HIST = OFF_W + kEpiWarps * 128 * 4;   // per warp: segment rows x heads <= 128 weights
constexpr int kGroupHistWords = kSegRows * kHistBins / 2;
// int4[kMaxStages]: {tile in segment, segment, segment ordinal in this CTA's sequence}
// int4[2 * kMaxStages]: per stage {tile in segment, segment, segment ordinal, 0}, {first row, rows, 0, 0}
constexpr int OFF_SINFO = OFF_HIST + kEpiGroups * kGroupHistWords * 4;
// int4[kAcc]: {tile in segment, segment, first row, rows} per accumulator
constexpr int OFF_AINFO = OFF_SINFO + kMaxStages * 32;
constexpr int OFF_PRING = OFF_AINFO + kAcc * 16;   // int4[2 * kPageRing]
constexpr int OFF_BAR = OFF_PRING + kPageRing * 32;
// full, empty, qfull, tfull (per accumulator and epilogue group), done.  A
// group's accumulator barrier is used by the sequence positions it, it + 6, ...
// of that group alone: one barrier per accumulator, filled by both issuers,
// could show a group a phase of the other group's fill (the two issuers'
// MMAs complete in no common order) and its parity wait would take it.
constexpr int kNumBars = 2 * kMaxStages + 2 + kAcc * kEpiGroups + 1;
// TMEM address, abort flag, released[kAcc] at +16, page ring published at +32,
// consumed[kCopyWarps] (entries each copy warp has taken) at +48, then
// armed[kCopyWarps] (positions each copy warp has passed the free-stage wait for)
constexpr int OFF_MISC = OFF_BAR + kNumBars * 8;
constexpr int kScoreSmem = OFF_MISC + 48 + 8 * kCopyWarps + 1024;   // + slack to align the base to 1024
static_assert(kScoreSmem <= 227 * 1024, "scoring CTA exceeds the shared memory of an SM");

// TMEM columns: kAcc accumulators of up to 128 columns, then scale factors.
constexpr uint32_t TM_ACC = 0;
constexpr uint32_t TM_SFA = kAcc * 128;              // kMaxStages x 4 columns
constexpr uint32_t TM_SFB = TM_SFA + 4 * kMaxStages; // (2 buffers x kMmaWarps) x 4 columns
constexpr uint32_t TM_COLS = 512;

// Compile-time traits of a cache format: each (format, heads) pair is its own
// kernel, so a kernel holds only its own format's code (a smaller instruction
// footprint for its fifteen warps of five roles).  Ring geometry: packed MXFP4
// tiles (either placement) take half the shared memory of FP8 ones, so twice
// as many are in flight.  Stage counts are powers of two: position it uses
// stage it & (n - 1) in its (it >> lg)-th round (no division on the per-tile paths).
static_assert(kStages == 1 << 3 && kMaxStages == 1 << 4, "stage counts as their log2 below");
static_assert(kMaxStages * (kTileBytes / 2) == kStages * kTileBytes, "both rings fill the tile area");
template <int F>
struct FmtT {
    static constexpr bool fp4 = F == DSA_FMT_MXFP4 || F == DSA_FMT_MXFP4_RG;
    static constexpr bool rg = F == DSA_FMT_MXFP4_RG;
    static constexpr bool fp8mx = F == DSA_FMT_FP8_MX;
    static constexpr bool key_scale = F == DSA_FMT_FP8;   // FP32 key scale applied in the epilogue
    static constexpr int lg = fp4 ? 4 : 3;
    static constexpr int stage_bytes = fp4 ? kTileBytes / 2 : kTileBytes;
};

struct ScoreArgs {
    int fmt;
    int num_pages;
    const int32_t* block_table;
    int64_t bt_stride;
    const uint8_t* q_rows;
    const __nv_bfloat16* w;
    const int4* segs;
    const int* seg_prefix;
    const int* eff_end;
    const int4* cta;
    float* logits;
    int64_t ld;
    int hist_k;          // rows whose bound exceeds hist_k get a histogram; -1: none
    unsigned* hist;
    int32_t* status;
    int heads;                 // query heads: 32, or (MXFP4 queries of quantize_queries) 16 or 64
    const uint8_t* q_scales;   // MXFP4 query scales of row r at q_scales + r * qs_stride
    int64_t qs_stride;
    int qs_group_major;        // scale of block g of head h at g * 64 + h (else at h * 4 + g)
    int64_t w_stride;          // BF16 head weights of row r at w + r * w_stride
    int rows;                  // query rows of the call
};

// Segment s with prefix[s] <= t < prefix[s + 1] (prefix[S] > t).
__device__ __forceinline__ int find_segment(const int* prefix, int S, int t) {
    int lo = 0, hi = S;   // answer in [0, S)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= t) lo = mid; else hi = mid;
    }
    return lo;
}

// ----------------------------------------------------------------- plan
// One CTA: validates request starts and row bounds, splits requests into
// segments of up to 4 rows and lays their 128-key tiles out in one index space.
constexpr int kPlanThreads = 256;
// A tile's estimated cost: kTileCostBase + kCostRow * its segment's rows.
constexpr int kTileCostBase = 3;
constexpr int kCostRow = 2;
constexpr int kPlanSmemRows = 4096;   // row bounds the plan keeps on chip

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const int32_t* __restrict__ starts,
                                                            const int32_t* __restrict__ row_ends, int R, int rows,
                                                            int max_keys, int* __restrict__ info,
                                                            int4* __restrict__ segs, int* __restrict__ seg_prefix,
                                                            int* __restrict__ eff_end, int4* __restrict__ cta, int G,
                                                            int seg_rows, int32_t* status) {
    // The scoring CTAs (persistent, one per SM, most of its registers) are let
    // in only once the work before this kernel has finished, so that they do
    // not crowd out a still-running predecessor; their prologue then overlaps
    // this kernel.
    pdl_wait();
    pdl_launch_dependents();
    __shared__ int warp_tmp[64];
    __shared__ int chunk_total, chunk_wtotal;
    __shared__ int sp[kPlanSmemSegs + 1];   // tiles per segment, then the tile prefix (when the segments fit)
    __shared__ int se[kPlanSmemRows];       // row bounds (when the rows fit)
    __shared__ unsigned char sn[kPlanSmemSegs];   // rows per segment (when the segments fit)
    __shared__ int bnd[kMaxScoreCtas + 1];        // first tile of every scoring CTA
    const bool rows_fit = rows <= kPlanSmemRows;
    // The first chunk's request starts and all row bounds are loaded together.
    int a0 = 0, b0 = 0;
    if (threadIdx.x < R) {
        a0 = starts[threadIdx.x];
        b0 = starts[threadIdx.x + 1];
    }
    if (rows_fit)
        for (int r = threadIdx.x; r < rows; r += blockDim.x) se[r] = row_ends[r];
    for (int r = threadIdx.x; r < rows; r += blockDim.x) eff_end[r] = 0;   // rows outside every request keep 0
    __syncthreads();
    int carry = 0;
    bool bad = false;
    for (int base = 0; base < R; base += blockDim.x) {
        const int q = base + threadIdx.x;
        int s0 = 0, s1 = 0;
        if (q < R) {
            const int a = base == 0 ? a0 : starts[q], b = base == 0 ? b0 : starts[q + 1];
            if (a < 0 || b < a || b > rows) bad = true;
            s0 = min(max(a, 0), rows);
            s1 = min(max(b, s0), rows);
        }
        const int nseg = (s1 - s0 + seg_rows - 1) / seg_rows;
        const int inc = block_inclusive_scan(nseg, warp_tmp, &chunk_total);
        const int sbase = carry + inc - nseg;
        for (int i = 0; i < nseg; ++i) {
            if (sbase + i > rows) { bad = true; break; }   // overlapping requests: capacity is rows + 1
            const int row0 = s0 + i * seg_rows;
            const int nr = min(seg_rows, s1 - row0);
            int maxend = 0;
            for (int r = row0; r < row0 + nr; ++r) {
                int e = rows_fit ? se[r] : row_ends[r];
                if (e > max_keys) { bad = true; e = max_keys; }
                e = max(e, 0);
                eff_end[r] = e;
                maxend = max(maxend, e);
            }
            segs[sbase + i] = make_int4(q, row0, nr, maxend);
            if (sbase + i < kPlanSmemSegs) {
                sp[sbase + i] = (maxend + kTileRows - 1) / kTileRows;
                sn[sbase + i] = static_cast<unsigned char>(nr);
            }
        }
        carry += chunk_total;
        __syncthreads();
    }
    if (bad && status) atomicOr(status, DSA_STATUS_BAD_GEOMETRY);
    const int S = min(carry, rows + 1);
    // Tile prefix and, when the segments fit on chip, the prefix of the tiles'
    // estimated cost (kTileCostBase + kCostRow x the segment's rows per tile; `se` is free now).
    const bool weighted = S <= kPlanSmemSegs && S <= kPlanSmemRows;
    carry = 0;
    int wcarry = 0;
    for (int base = 0; base < S; base += blockDim.x) {
        const int i = base + threadIdx.x;
        int tiles = 0, cost = 0;
        if (i < S) {
            tiles = i < kPlanSmemSegs ? sp[i] : (segs[i].w + kTileRows - 1) / kTileRows;
            if (weighted) cost = tiles * (kTileCostBase + kCostRow * sn[i]);
        }
        int inc = tiles, winc = cost;   // both prefixes with one set of barriers
        block_inclusive_scan2(inc, winc, warp_tmp, &chunk_total, &chunk_wtotal);
        if (i < S) {
            seg_prefix[i] = carry + inc - tiles;
            if (i < kPlanSmemSegs) sp[i] = carry + inc - tiles;   // this thread's own entry
            if (weighted) se[i] = wcarry + winc - cost;
        }
        carry += chunk_total;
        wcarry += chunk_wtotal;
        __syncthreads();
    }
    const int T = carry;
    if (threadIdx.x == 0) {
        seg_prefix[S] = T;
        if (S <= kPlanSmemSegs) sp[S] = T;
        if (weighted) se[S] = wcarry;
        info[0] = S;
        info[1] = T;
    }
    __syncthreads();
    // Static tile range and first segment of every scoring CTA, so that a CTA
    // starts from one load instead of a search through global memory.  The
    // ranges split the estimated cost evenly, else the tiles.  A tile of a
    // segment of n rows costs kTileCostBase + kCostRow n: its copy and MMA, then
    // n rows of epilogue.  (3, 2) is the pair that timed best on GB300 over
    // decode steps mixing segments of 1 to 4 rows; the ratio matters, and it
    // leaves a 4-row tile at 11/5 of a 1-row one.
    const bool wfit = static_cast<int64_t>(T) * (kTileCostBase + kCostRow * kSegRows) < 0x7FFFFFFF;   // int prefix holds
    // floor(c * X / G) in 32 bits: c * (X / G) + c * (X % G) / G, exact for
    // c <= G <= kMaxScoreCtas (c * (X % G) < 2^20) and X < 2^31.
    auto share = [&](int c, int X) { return c * (X / G) + (c * (X % G)) / G; };
    auto tile_at = [&](int c) -> int {   // first tile of CTA c
        if (!weighted || !wfit || wcarry == 0) return share(c, T);
        const int B = share(c, wcarry);
        int lo = 0, hi = S;   // the last segment with se[lo] <= B
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (se[mid] <= B) lo = mid; else hi = mid;
        }
        const int per = kTileCostBase + kCostRow * sn[lo];
        return min(sp[lo + 1], sp[lo] + (B - se[lo]) / per);
    };
    // every boundary once (CTA c's range is [bnd[c], bnd[c + 1]))
    for (int c = threadIdx.x; c <= G; c += blockDim.x) bnd[c] = c == 0 ? 0 : (c == G ? T : tile_at(c));
    __syncthreads();
    for (int c = threadIdx.x; c < G; c += blockDim.x) {
        const int t0 = bnd[c];
        const int t1 = bnd[c + 1];
        int seg = -1;
        if (S <= kPlanSmemSegs && S > 0) {
            int lo = 0, hi = S;
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (sp[mid] <= t0) lo = mid; else hi = mid;
            }
            seg = lo;
        }
        cta[c] = make_int4(t0, t1, seg, S);
    }
}

// ----------------------------------------------------------------- roles
// Per-tile load plan resolved by one lane of the producer warp.
struct TilePlan {
    int seg;   // segment of the tile
    int j;     // tile index within the segment
    int pid0;  // physical page of keys 0..63 (-1: none)
    int pid1;  // physical page of keys 64..127 (-1: none)
    int row0;  // the segment's first query row
    int nrows; // the segment's rows
};

// Plans of the tiles base + lane (lanes below n; the others get no pages) of
// one warp, whose tiles lie in segments seg, seg + 1, ...: lane k loads the
// tile prefix and record of segment seg + k (one round trip for the warp),
// every lane finds its tile's segment among those 32 by a search over
// shuffled registers, then loads its two block-table entries.  Tiles past
// segment seg + 31 (batches crossing more than 31 segments) search the global
// prefix instead.
__device__ __forceinline__ TilePlan plan_batch(const ScoreArgs& p, int base, int n, int seg, int S) {
    const int lane = threadIdx.x & 31;
    const int t = base + lane;
    const int sk = min(seg + lane, S);
    const int q = p.seg_prefix[sk];                                  // first tile of segment seg + lane
    const int4 rec = sk < S ? p.segs[sk] : make_int4(0, 0, 0, 0);
    int cnt = 0;   // the last k <= 31 with prefix[seg + k] <= t (prefix sorted, prefix[seg] <= t)
#pragma unroll
    for (int step = 16; step >= 1; step >>= 1) {
        const int v = __shfl_sync(0xFFFFFFFFu, q, cnt + step);
        if (cnt + step <= 31 && v <= t) cnt += step;
    }
    TilePlan tp{-1, 0, -1, -1, 0, 0};
    int first = __shfl_sync(0xFFFFFFFFu, q, cnt);
    int4 si;
    si.x = __shfl_sync(0xFFFFFFFFu, rec.x, cnt);
    si.y = __shfl_sync(0xFFFFFFFFu, rec.y, cnt);
    si.z = __shfl_sync(0xFFFFFFFFu, rec.z, cnt);
    si.w = __shfl_sync(0xFFFFFFFFu, rec.w, cnt);
    int sg = seg + cnt;
    if (lane >= n) return tp;
    if (cnt == 31 && sg + 1 < S && p.seg_prefix[sg + 1] <= t) {
        int lo = sg + 1, hi = S;   // the tile lies past the 32 segments loaded above
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (p.seg_prefix[mid] <= t) lo = mid; else hi = mid;
        }
        sg = lo;
        first = p.seg_prefix[sg];
        si = p.segs[sg];
    }
    tp.seg = sg;
    tp.row0 = si.y;
    tp.nrows = si.z;
    const int j = t - first;
    tp.j = j;
    const int npages = (si.w + kPage - 1) / kPage;
    const int32_t* row = p.block_table + static_cast<int64_t>(si.x) * p.bt_stride;
    bool bad = false;
    if (2 * j < npages) {
        const int v = row[2 * j];
        if (v >= 0 && v < p.num_pages) tp.pid0 = v; else bad = true;
    }
    if (2 * j + 1 < npages) {
        const int v = row[2 * j + 1];
        if (v >= 0 && v < p.num_pages) tp.pid1 = v; else bad = true;
    }
    if (bad && p.status) atomicOr(p.status, DSA_STATUS_BAD_PAGE);
    return tp;
}

// Bounded wait until a release counter reaches `need` (wrap-safe compare);
// same give-up rules as mbar_wait.
__device__ __forceinline__ bool count_wait(const uint32_t* c, uint32_t need, volatile int* abort, int32_t* status) {
    if (static_cast<int>(smem_ld_acquire(c) - need) >= 0) return true;
    const unsigned long long t0 = globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (static_cast<int>(smem_ld_acquire(c) - need) >= 0) return true;
        if ((i & 31) == 0) {
            if (*abort) return false;
            if (globaltimer() - t0 > kWaitLimitNs) {
                *abort = 1;
                if (status) atomicOr(status, DSA_STATUS_TIMEOUT);
                return false;
            }
        }
    }
}

// Copies the codes of page h (0 or 1) of a tile, id pid, into stage s (FP8:
// one 128-byte-swizzled box; MXFP4: one 64-byte-swizzled box; row-group: one
// box per column group, group g at g * 2048 + h * 1024).  Key pages are read
// once per step, so they are loaded with an evict-first L2 policy: the step's
// logits, histograms and block tables stay in L2 for the kernels after it.
__device__ __forceinline__ void issue_codes(const CUtensorMap* kmap, uint8_t* smem, uint64_t* bar, int s,
                                            int stage_bytes, bool fp4, bool rg, int h, int pid, uint64_t pol) {
    uint8_t* dst = smem + OFF_TILES + s * stage_bytes;
    if (rg) {
#pragma unroll
        for (int g = 0; g < 4; ++g)
            tma_load_4d_hint(dst + g * kRgTileGroup + h * kRgGroupBytes, kmap, 0, 0, g, pid, bar, pol);
    } else {
        tma_load_3d_hint(dst + h * (fp4 ? kFp4KeyBytes : kPageSmem), kmap, 0, 0, pid, bar, pol);
    }
}
// Copies the 256 scale bytes of page h of a tile into stage s.
__device__ __forceinline__ void issue_scales(const CUtensorMap* smap, uint8_t* smem, uint64_t* bar, int s, int h,
                                             int pid, uint64_t pol) {
    tma_load_2d_hint(smem + OFF_RAWSC + s * 512 + h * 256, smap, 0, pid, bar, pol);
}

// Warp 0 lays out this CTA's sequence of tiles (positions 0, 1, ...): each
// position's ring entry {first page, second page, tile in segment, segment},
// {segment ordinal} is written by lane 0, and a batch of entries is made
// visible to the copy warps with one release.  On a segment change it loads
// the segment's query rows into query buffer (ordinal & 1).
//
// Query buffer b holds the segments of ordinals b, b + 2, ...  Before it is
// refilled, the MMAs of the segment it held must be done: every issuer's last
// tile of that segment has released its ring stage (an issuer's MMAs complete
// in order).  The planner runs ahead of the stages (up to the ring's length),
// so a release is recognised either on the stage's empty barrier (the phase
// of that position's use) or, once the stage has been taken again, by the
// copy warp that owns the position kStages later having passed its wait for
// it (armed counts; kStages is a multiple of the copy warps).
template <int F, int H>
struct Producer {
    using T = FmtT<F>;
    static constexpr bool fp4 = T::fp4;            // MXFP4 codes (either placement): transaction sizes
    static constexpr bool rg = T::rg;              // row-group placement: packed boxes per column group
    static constexpr int lg = T::lg;               // log2 of the ring's stage count
    static constexpr int stage_bytes = T::stage_bytes;   // shared memory of a stage's codes
    const CUtensorMap* kmap;
    const CUtensorMap* smap;
    const CUtensorMap* qmap;
    uint8_t* smem;
    uint64_t* full;
    uint64_t* empty;
    uint64_t* qfull;
    volatile int* abort;
    int4* page_ring;     // per position: {first page, second page, tile in segment, segment}, {ordinal, first row, rows}
    uint32_t* published; // entries made visible (release)
    const uint32_t* consumed;   // [kCopyWarps]: entries each copy warp has taken (acquire)
    const uint32_t* armed;      // [kCopyWarps]: positions each copy warp has passed the free-stage wait for
    int cur = -1, i_seg = 0, it = 0, pub = 0;

    // Makes the entries written so far visible to the copy warps.
    __device__ __forceinline__ void flush() {
        if (it > pub) {
            smem_add_release(published, static_cast<uint32_t>(it - pub));
            pub = it;
        }
    }
    // Room for position it: the copy warps have taken position it - kLead and
    // the ring entry it overwrites, it - kPageRing.
    __device__ __forceinline__ bool taken(const ScoreArgs& p, int old) {
        if (old < 0) return true;
        if (static_cast<int>(smem_ld_acquire(consumed + (old % kCopyWarps)) - (old / kCopyWarps + 1)) >= 0)
            return true;
        flush();   // the copy warps must see the pending entries to make room
        return count_wait(consumed + (old % kCopyWarps), static_cast<uint32_t>(old / kCopyWarps + 1), abort,
                          p.status);
    }
    __device__ __forceinline__ bool room(const ScoreArgs& p) {
        return taken(p, it - kLead) && taken(p, it - kPageRing);
    }
    // Bounded wait for the release of position l's stage use (its MMAs are done).
    // The stage's empty barrier completes one phase per use; its parity names
    // l's phase only while the stage is in l's use: after the copy warp owning
    // l has taken the stage for l (armed covers l) and before it takes it again
    // for l + stages (armed covers that, and l's release came before).
    __device__ __forceinline__ bool released(const ScoreArgs& p, int l) {
        const int stages = 1 << lg;
        const int c = l % kCopyWarps;
        const uint32_t started = static_cast<uint32_t>((l - c) / kCopyWarps + 1);
        const uint32_t need = static_cast<uint32_t>((l + stages - c) / kCopyWarps + 1);
        uint64_t* bar = empty + (l & (stages - 1));
        const uint32_t parity = (l >> lg) & 1;
        const unsigned long long t0 = globaltimer();
        for (uint32_t i = 0;; ++i) {
            const uint32_t a = smem_ld_acquire(armed + c);
            if (static_cast<int>(a - need) >= 0) return true;
            if (static_cast<int>(a - started) >= 0 && mbar_test_wait(bar, parity)) return true;
            if ((i & 63) == 63) {
                if (*abort) return false;
                if (globaltimer() - t0 > kWaitLimitNs) {
                    *abort = 1;
                    if (p.status) atomicOr(p.status, DSA_STATUS_TIMEOUT);
                    return false;
                }
            }
        }
    }
    int last00 = -1, last01 = -1, last10 = -1, last11 = -1;   // last tile of query buffer b for issuer w

    __device__ __forceinline__ int last_tile(int b, int w) const {
        return b ? (w ? last11 : last10) : (w ? last01 : last00);
    }
    __device__ __forceinline__ void set_last_tile(int b, int w, int v) {
        if (b) {
            if (w) last11 = v; else last10 = v;
        } else {
            if (w) last01 = v; else last00 = v;
        }
    }

    // Lane 0: writes position it's entry (loading the segment's queries first
    // when the segment changes); the entry becomes visible at the next flush.
    __device__ __forceinline__ bool add(const ScoreArgs& p, int sg, int j, int p0, int p1, int row0, int nrows) {
        if (sg != cur) {
            cur = sg;
            const int2 si = make_int2(row0, nrows);
            const int qb = i_seg & 1;
            flush();   // the tiles before the change can be copied while this waits
            for (int w = 0; w < kMmaWarps; ++w) {
                const int l = last_tile(qb, w);
                if (l >= 0 && !released(p, l)) return false;
                set_last_tile(qb, w, -1);
            }
            const uint32_t qsf = p.qs_group_major ? kQsfRowRg : kQsfRow;
            const uint32_t qrow = fp4 ? 64u * H : kFp8QRowTx;   // packed MXFP4: heads x 64 B
            const uint32_t bytes = si.y * (fp4 ? qrow + qsf : qrow);
            mbar_arrive_expect_tx(qfull + qb, bytes);
            uint8_t* qdst = smem + OFF_QBUF + qb * kQBufBytes;
            for (int r = 0; r < si.y; ++r) {
                if (rg) {
                    // packed: 16-byte column chunk c of every head at c * 2048 + (r * heads + h) * 16
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        tma_load_3d(qdst + c * kRgQChunk + r * 16 * H, qmap, 16 * c, 0, si.x + r, qfull + qb);
                } else {
                    // FP8 rows of 4096 bytes, packed MXFP4 rows of heads x 64 B
                    tma_load_3d(qdst + r * qrow, qmap, 0, 0, si.x + r, qfull + qb);
                }
                if (fp4)
                    bulk_load(smem + OFF_QSF + qb * kQsfBytes + r * qsf,
                              p.q_scales + static_cast<int64_t>(si.x + r) * p.qs_stride, qsf, qfull + qb);
            }
            ++i_seg;
        }
        if (!room(p)) return false;
        set_last_tile((i_seg - 1) & 1, it % kMmaWarps, it);
        // the copy warp writes the stage's tag and arms its full barrier for the
        // tile's bytes (a tile without valid pages: scores of its keys are unspecified)
        page_ring[2 * (it & (kPageRing - 1))] = make_int4(p0 >= 0 ? p0 : kNoPage, p1 >= 0 ? p1 : kNoPage, j, sg);
        page_ring[2 * (it & (kPageRing - 1)) + 1] = make_int4(i_seg - 1, row0, nrows, 0);
        ++it;
        if (it - pub >= kCopyWarps) flush();   // one release per kCopyWarps entries
        return true;
    }

    // End of this CTA's sequence: one stage tagged -1, with no copies, per copy
    // warp (each copy warp stops at its end mark; each issuer at the first one
    // of its positions).
    static_assert(kCopyWarps >= kMmaWarps, "every issuer meets an end tag");
    __device__ __forceinline__ bool finish(const ScoreArgs& p) {
        for (int w = 0; w < kCopyWarps; ++w) {
            if (!room(p)) return false;
            page_ring[2 * (it & (kPageRing - 1))] = make_int4(kEndMark, kEndMark, -1, -1);
            page_ring[2 * (it & (kPageRing - 1)) + 1] = make_int4(-1, 0, 0, 0);
            ++it;
        }
        flush();
        return true;
    }
};

// Warp 0.  Its 32 lanes resolve the segments and block-table entries of 32
// tiles at once (the next batch's loads are in flight while lane 0 issues the
// current batch's tiles), so block-table latency is paid once per batch.
template <int F, int H>
__device__ __forceinline__ void producer_role(Producer<F, H>& pr, const ScoreArgs& p, int t0, int t1, int seg,
                                              int S) {
    const int lane = threadIdx.x & 31;
    bool ok = true;
    if (t0 < t1) {
        TilePlan nxt = plan_batch(p, t0, min(32, t1 - t0), seg, S);
        for (int base = t0; base < t1 && ok; base += 32) {
            const TilePlan mine = nxt;
            const int last = min(31, t1 - 1 - base);
            const int seg_end = __shfl_sync(0xFFFFFFFFu, mine.seg, last);
            if (base + 32 < t1) nxt = plan_batch(p, base + 32, min(32, t1 - base - 32), seg_end, S);
            for (int i = 0; i <= last && ok; ++i) {
                const int sg = __shfl_sync(0xFFFFFFFFu, mine.seg, i);
                const int j = __shfl_sync(0xFFFFFFFFu, mine.j, i);
                const int p0 = __shfl_sync(0xFFFFFFFFu, mine.pid0, i);
                const int p1 = __shfl_sync(0xFFFFFFFFu, mine.pid1, i);
                const int r0 = __shfl_sync(0xFFFFFFFFu, mine.row0, i);
                const int nr = __shfl_sync(0xFFFFFFFFu, mine.nrows, i);
                if (lane == 0) ok = pr.add(p, sg, j, p0, p1, r0, nr);
                ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            }
            if (lane == 0) pr.flush();   // one release per batch
        }
    }
    if (lane == 0) {
        if (ok) pr.finish(p);
        // Drain: the query rows this warp loaded must have landed before the CTA
        // exits (no later load reuses a buffer, so the last phases are unambiguous).
        const int i_seg = pr.i_seg;
        const unsigned long long deadline = globaltimer() + kWaitLimitNs;
        bool drained = true;
        for (int i = max(0, i_seg - 2); i < i_seg && drained; ++i)
            drained = mbar_drain(pr.qfull + (i & 1), (i >> 1) & 1, deadline, p.status);
    }
    __syncwarp();
}

// Copy warp c (warp kFirstCopyWarp + c).  Follows warp 0's positions c, c +
// kCopyWarps, ... through the page ring: waits for the position's stage to be
// free (and counts that in armed[c]), writes the stage's tag, and copies the
// tile's two pages (codes and scales) into it, arming the stage's full
// barrier for those bytes.  Its stages are its own (the ring's stage count is
// a multiple of the copy warps), so on the way out it drains the copies of its
// last uses of them without ambiguity.
template <int F>
__device__ __forceinline__ void copy_role(const ScoreArgs& p, const CUtensorMap* kmap, const CUtensorMap* smap,
                                          uint8_t* smem, uint64_t* full, uint64_t* empty, const uint32_t* published,
                                          uint32_t* consumed, uint32_t* armed, volatile int* abort, int c) {
    if ((threadIdx.x & 31) != 0) return;
    constexpr bool fp4 = FmtT<F>::fp4, rg = FmtT<F>::rg;
    constexpr int lg = FmtT<F>::lg, stage_bytes = FmtT<F>::stage_bytes;
    const uint32_t page_tx = (fp4 ? kFp4PageTx : kFp8PageTx) + 256u;
    const uint64_t pol = l2_evict_first_policy();
    const int4* ring = reinterpret_cast<const int4*>(smem + OFF_PRING);
    int4* sinfo = reinterpret_cast<int4*>(smem + OFF_SINFO);
    int last_j = -1;   // the last position whose full barrier this warp arrived on
    for (int j = c;; j += kCopyWarps) {
        if (!count_wait(published, static_cast<uint32_t>(j + 1), abort, p.status)) break;
        const int4 v = ring[2 * (j & (kPageRing - 1))];
        const int4 vs = ring[2 * (j & (kPageRing - 1)) + 1];   // {ordinal, first row, rows}
        smem_add_release(consumed + c, 1u);
        const int s = j & ((1 << lg) - 1);
        if (!mbar_wait(empty + s, ((j >> lg) & 1) ^ 1, abort, p.status)) break;
        smem_add_release(armed + c, 1u);   // position j - stages is released
        // the stage's tag: {tile in segment, segment, segment ordinal}; -1 ends an issuer's sequence
        sinfo[2 * s] = v.x == kEndMark ? make_int4(-1, -1, -1, 0) : make_int4(v.z, v.w, vs.x, 0);
        sinfo[2 * s + 1] = make_int4(vs.y, vs.z, 0, 0);
        if (v.x == kEndMark) {
            mbar_arrive(full + s);
            last_j = j;
            break;
        }
        const uint32_t bytes = (v.x >= 0 ? page_tx : 0u) + (v.y >= 0 ? page_tx : 0u);
        if (bytes) {
            mbar_arrive_expect_tx(full + s, bytes);
            if (v.x >= 0) {
                issue_codes(kmap, smem, full + s, s, stage_bytes, fp4, rg, 0, v.x, pol);
                issue_scales(smap, smem, full + s, s, 0, v.x, pol);
            }
            if (v.y >= 0) {
                issue_codes(kmap, smem, full + s, s, stage_bytes, fp4, rg, 1, v.y, pol);
                issue_scales(smap, smem, full + s, s, 1, v.y, pol);
            }
        } else {
            mbar_arrive(full + s);
        }
        last_j = j;
    }
    // every copy issued must have landed before the CTA exits
    const unsigned long long deadline = globaltimer() + kWaitLimitNs;
    for (int jj = last_j; jj >= 0 && jj > last_j - (1 << lg); jj -= kCopyWarps)
        if (!mbar_drain(full + (jj & ((1 << lg) - 1)), (jj >> lg) & 1, deadline, p.status)) break;
}

// Warps 1 .. kMmaWarps.  Issuer w follows the stage tags of sequence
// positions w, w + kMmaWarps, ...; hands each accumulator's tag to the
// epilogue (its end-of-sequence tag as the last one).  An accumulator is
// used by both issuers in turn, so its release is a count (four epilogue
// warps per use) rather than an mbarrier phase, which an issuer running
// ahead could mistake for a later one.
template <int F, int H>
__device__ __forceinline__ void mma_role(const ScoreArgs& p, uint8_t* smem, uint32_t tmem, uint64_t* full,
                                         uint64_t* empty, uint64_t* qfull, uint64_t* tfull, const uint32_t* released,
                                         uint64_t* done_bar, volatile int* abort) {
    const int lane = threadIdx.x & 31;
    const int w = (threadIdx.x >> 5) - 1;
    // FP8 keys with an FP32 scale take the plain FP8 MMA and the key scale in
    // the epilogue.  FP8-MX keys carry four UE8M0 bytes, byte b the scale of
    // columns 32b..32b+31: the block-scaled FP8 MMA applies byte kk in its
    // instruction kk (K = 32), the query's scales being 1 (its scale is folded
    // into the head weights).  MXFP4 uses the block-scaled FP4 MMA.
    constexpr bool key_scale = FmtT<F>::key_scale;
    constexpr bool fp8mx = FmtT<F>::fp8mx;
    constexpr bool block_scaled = !key_scale;
    constexpr bool rg = FmtT<F>::rg;
    constexpr int lg = FmtT<F>::lg;
    constexpr int stage_bytes = FmtT<F>::stage_bytes;
    const int4* sinfo = reinterpret_cast<const int4*>(smem + OFF_SINFO);
    int4* ainfo = reinterpret_cast<int4*>(smem + OFF_AINFO);
    int cur = -1, qb = 0, nrows = 0;
    for (int it = w;; it += kMmaWarps) {
        const int s = it & ((1 << lg) - 1);
        const int a = it % kAcc;
        const uint32_t need = 4u * static_cast<uint32_t>(it / kAcc);   // releases of its earlier uses
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(full + s, (it >> lg) & 1, abort, p.status))) break;
        const int4 tag = sinfo[2 * s];
        const int4 rowinfo = sinfo[2 * s + 1];   // the segment's {first row, rows}
        if (tag.y < 0) {
            // this issuer's epilogue group takes the end tag
            if (!__all_sync(0xFFFFFFFFu, count_wait(released + a, need, abort, p.status))) break;
            if (lane == 0) {
                ainfo[a] = make_int4(tag.x, tag.y, 0, 0);
                mbar_arrive(tfull + a * kEpiGroups + w);
                mbar_arrive(tfull + a * kEpiGroups + w);
            }
            __syncwarp();
            break;
        }
        if (tag.z != cur) {
            cur = tag.z;
            nrows = rowinfo.y;
            qb = cur & 1;
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(qfull + qb, (cur >> 1) & 1, abort, p.status))) break;
            if (block_scaled) {
                // Query block scales: line L of the atom holds the words of MMA
                // rows L, 32 + L, 64 + L, 96 + L (row n = r * heads + h: head h of query row r).
                const uint8_t* raw = smem + OFF_QSF + qb * kQsfBytes;
                // the word of MMA row n: head-major rows hold it as is; group-major
                // rows hold block g's byte at g * 64 + head; FP8 queries are unscaled (2^0)
                auto word = [&](int n) -> uint32_t {
                    const int r = n / H, h = n - r * H;
                    if (r >= nrows || fp8mx) return 0x7F7F7F7Fu;
                    if (!p.qs_group_major) return reinterpret_cast<const uint32_t*>(raw + r * kQsfRow)[h];
                    const uint8_t* b = raw + r * kQsfRowRg + h;
                    return static_cast<uint32_t>(b[0]) | (static_cast<uint32_t>(b[kRgQuerySlots]) << 8) |
                           (static_cast<uint32_t>(b[2 * kRgQuerySlots]) << 16) |
                           (static_cast<uint32_t>(b[3 * kRgQuerySlots]) << 24);
                };
                uint8_t* atom = smem + OFF_SFB + (qb * kMmaWarps + w) * 512;
                uint4 line;
                line.x = word(lane);
                line.y = word(32 + lane);
                line.z = word(64 + lane);
                line.w = word(96 + lane);
                reinterpret_cast<uint4*>(atom)[lane] = line;
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0)
                    tc_cp_32x128b_warpx4(tmem + TM_SFB + (qb * kMmaWarps + w) * 4, desc_rows16(smem_u32(atom)));
            }
        }
        if (!__all_sync(0xFFFFFFFFu, count_wait(released + a, need, abort, p.status))) break;
        tc_fence_after();
        const uint32_t* rs = reinterpret_cast<const uint32_t*>(smem + OFF_RAWSC + s * 512);
        uint32_t w0, w1, w2, w3;
        if (rg) {
            // page h's scale bytes are [group][64 keys]: gather key t's four into one word
            const uint8_t* rb = smem + OFF_RAWSC + s * 512;
            auto word = [&](int t) {
                const uint8_t* b = rb + (t >> 6) * 256 + (t & 63);
                return static_cast<uint32_t>(b[0]) | (static_cast<uint32_t>(b[64]) << 8) |
                       (static_cast<uint32_t>(b[128]) << 16) | (static_cast<uint32_t>(b[192]) << 24);
            };
            w0 = word(lane);
            w1 = word(32 + lane);
            w2 = word(64 + lane);
            w3 = word(96 + lane);
        } else {
            w0 = rs[lane];
            w1 = rs[32 + lane];
            w2 = rs[64 + lane];
            w3 = rs[96 + lane];
        }
        if (key_scale) {
            float* ks = reinterpret_cast<float*>(smem + OFF_KS + a * 512);
            ks[lane] = __uint_as_float(w0);
            ks[32 + lane] = __uint_as_float(w1);
            ks[64 + lane] = __uint_as_float(w2);
            ks[96 + lane] = __uint_as_float(w3);
        } else {
            reinterpret_cast<uint4*>(smem + OFF_SFA + s * 512)[lane] = make_uint4(w0, w1, w2, w3);
            fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) {
            const uint32_t d = tmem + TM_ACC + a * 128;
            const uint32_t ka = smem_u32(smem + OFF_TILES + s * stage_bytes);
            const uint32_t kb = smem_u32(smem + OFF_QBUF + qb * kQBufBytes);
            const uint32_t n = static_cast<uint32_t>(H * nrows);
            if (key_scale) {
                const uint64_t ad = desc_sw128(ka), bd = desc_sw128(kb);
                const uint32_t id = idesc_f8f6f4(kMmaE4M3, kMmaE4M3, 128, n);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) tc_mma_f8f6f4(d, ad + 2 * kk, bd + 2 * kk, id, kk > 0);
            } else if (fp8mx) {
                const uint32_t sfa = tmem + TM_SFA + s * 4;
                tc_cp_32x128b_warpx4(sfa, desc_rows16(smem_u32(smem + OFF_SFA + s * 512)));
                const uint32_t sfb = tmem + TM_SFB + (qb * kMmaWarps + w) * 4;
                const uint64_t ad = desc_sw128(ka), bd = desc_sw128(kb);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_mxf8(d, ad + 2 * kk, bd + 2 * kk, idesc_mx(kMmaE4M3, kMmaE4M3, 128, n, kk, kk), sfa, sfb,
                                kk > 0);
            } else if (rg) {
                const uint32_t sfa = tmem + TM_SFA + s * 4;
                tc_cp_32x128b_warpx4(sfa, desc_rows16(smem_u32(smem + OFF_SFA + s * 512)));
                const uint32_t sfb = tmem + TM_SFB + (qb * kMmaWarps + w) * 4;
#pragma unroll
                for (int m = 0; m < 2; ++m)
                    tc_mma_mxf4(d, desc_kmajor_plain(ka + 2 * m * kRgTileGroup, kRgTileGroup, 128),
                                desc_kmajor_plain(kb + 2 * m * kRgQChunk, kRgQChunk, 128),
                                idesc_mx(kMmaMxf4E2M1, kMmaMxf4E2M1, 128, n, 2 * m, 2 * m), sfa, sfb, m > 0);
            } else {
                // token-major: 64-byte rows (128 E2M1 per key or head); instruction m reads
                // the row's bytes 32m .. 32m + 31
                const uint32_t sfa = tmem + TM_SFA + s * 4;
                tc_cp_32x128b_warpx4(sfa, desc_rows16(smem_u32(smem + OFF_SFA + s * 512)));
                const uint32_t sfb = tmem + TM_SFB + (qb * kMmaWarps + w) * 4;
                const uint64_t ad = desc_sw64(ka), bd = desc_sw64(kb);
#pragma unroll
                for (int m = 0; m < 2; ++m)
                    tc_mma_mxf4(d, ad + 2 * m, bd + 2 * m, idesc_mx(kMmaMxf4E2M1, kMmaMxf4E2M1, 128, n, 2 * m, 2 * m),
                                sfa, sfb, m > 0);
            }
            ainfo[a] = make_int4(tag.x, tag.y, rowinfo.x, rowinfo.y);
            tc_commit(empty + s);
            tc_commit(tfull + a * kEpiGroups + w);
            mbar_arrive(tfull + a * kEpiGroups + w);   // releases the key scales and the tag written above
        }
        __syncwarp();
    }
    if (lane == 0) {
        tc_commit(done_bar);
        mbar_drain(done_bar, 0, globaltimer() + kWaitLimitNs, p.status);
    }
    __syncwarp();
}

// Scores of one query row for the 32 keys of this warp (one per lane) from
// the H head columns v of its accumulator: sum_h w_h * max(acc_h, 0), four
// partial sums by head mod 4, combined as ((s0 + s1) + (s2 + s3)).  The ReLU
// is an integer max on the FP32 bits (negative values, -0 included, have the
// sign bit set and are negative as signed integers); the multiply-adds run two
// at a time (fma.rn.f32x2, each lane rounded as fmaf).
template <int H>
__device__ __forceinline__ float head_sum(const uint32_t* v, const float* wr, float ksm) {
    unsigned long long s01 = 0ull, s23 = 0ull;   // (s0, s1), (s2, s3) as f32x2, +0.0
#pragma unroll
    for (int h4 = 0; h4 < H / 4; ++h4) {
        const float4 w4 = reinterpret_cast<const float4*>(wr)[h4];
        const int r0 = max(static_cast<int>(v[4 * h4 + 0]), 0), r1 = max(static_cast<int>(v[4 * h4 + 1]), 0);
        const int r2 = max(static_cast<int>(v[4 * h4 + 2]), 0), r3 = max(static_cast<int>(v[4 * h4 + 3]), 0);
        asm("{\n\t.reg .b64 a, b;\n\tmov.b64 a, {%1, %2};\n\tmov.b64 b, {%3, %4};\n\t"
            "fma.rn.f32x2 %0, a, b, %0;\n\t}"
            : "+l"(s01)
            : "f"(w4.x), "f"(w4.y), "r"(r0), "r"(r1));
        asm("{\n\t.reg .b64 a, b;\n\tmov.b64 a, {%1, %2};\n\tmov.b64 b, {%3, %4};\n\t"
            "fma.rn.f32x2 %0, a, b, %0;\n\t}"
            : "+l"(s23)
            : "f"(w4.z), "f"(w4.w), "r"(r2), "r"(r3));
    }
    const float s0 = __uint_as_float(static_cast<uint32_t>(s01)), s1 = __uint_as_float(static_cast<uint32_t>(s01 >> 32));
    const float s2 = __uint_as_float(static_cast<uint32_t>(s23)), s3 = __uint_as_float(static_cast<uint32_t>(s23 >> 32));
    return ((s0 + s1) + (s2 + s3)) * ksm;
}

// Logit store and histogram count of one row's 32 scores (one per lane);
// hrow is the row's part of the group's shared histogram.
__device__ __forceinline__ void emit_row(const ScoreArgs& p, int row, int tpos, float sc, int end, bool hist_on,
                                         uint32_t* hrow) {
    const bool valid = tpos < end;
    if (valid) p.logits[static_cast<int64_t>(row) * p.ld + tpos] = sc;
    if (valid && hist_on) {
        const uint32_t bin = hist_bin(sc);
        atomicAdd(hrow + (bin >> 1), 1u << ((bin & 1u) << 4));
    }
}

// Named barrier over the 128 threads of epilogue group g, returning the OR of `pred`.
__device__ __forceinline__ bool group_sync_any(int g, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(1 + g)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void group_sync(int g) { asm volatile("bar.sync %0, 128;" ::"r"(1 + g) : "memory"); }

// Adds the group's shared histogram of segment rows row0 .. row0 + nrows
// (those whose bit is set in hist_m) to the rows' global histograms and
// clears it.  e: thread index within the group.
__device__ __forceinline__ void flush_group_hist(const ScoreArgs& p, uint32_t* gh, int g, int row0, int nrows,
                                                 unsigned hist_m, int e) {
    group_sync(g);
    for (int r = 0; r < nrows; ++r) {
        if (!((hist_m >> r) & 1u)) continue;
        uint32_t* hr = gh + r * (kHistBins / 2);
        unsigned* dst = p.hist + static_cast<int64_t>(row0 + r) * kHistBins;
        // One 64-bit add per word updates both of its bins (2w in the low half,
        // 2w + 1 in the high one): a row's count stays below 2^31, so the low
        // bin never carries into its neighbour.
        unsigned long long* dst2 = reinterpret_cast<unsigned long long*>(dst);
        for (int w = e; w < kHistBins / 2; w += 128) {
            const uint32_t c = hr[w];
            if (c) {
                atomicAdd(dst2 + w, (static_cast<unsigned long long>(c >> 16) << 32) | (c & 0xFFFFu));
                hr[w] = 0u;
            }
        }
    }
    group_sync(g);
}

// Warps kFirstEpiWarp .. + kEpiWarps.  Group g drains the accumulators of
// sequence positions g, g + kEpiGroups, ...; every warp works on its own
// (per-warp head weights, row bounds in registers, one release count per tile).
// H query heads: row r of a segment owns accumulator columns r * H .. r * H + H - 1.
template <int F, int H>
__device__ __forceinline__ void epilogue_role(const ScoreArgs& p, uint8_t* smem, uint32_t tmem, uint64_t* tfull,
                                              uint32_t* released, volatile int* abort) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int group = (warp - kFirstEpiWarp) >> 2;
    const int quarter = warp & 3;            // TMEM lanes this warp may access
    const int m = quarter * 32 + lane;       // key of the tile this thread owns
    float* wsm = reinterpret_cast<float*>(smem + OFF_W) + (warp - kFirstEpiWarp) * 128;
    const int4* ainfo = reinterpret_cast<const int4*>(smem + OFF_AINFO);
    constexpr bool f32scale = FmtT<F>::key_scale;   // FP32 key scale (FP8-MX scales act inside the MMA)
    const uint32_t tbase = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + TM_ACC;
    uint32_t* gh = reinterpret_cast<uint32_t*>(smem + OFF_HIST) + group * kGroupHistWords;
    const int e = threadIdx.x - 32 * kFirstEpiWarp - group * 128;   // thread index within the group
    int cur = -1, row0 = 0, nrows = 0, seg_tiles = 0;
    int end_l = 0;        // lane r < nrows: bound of row row0 + r
    unsigned hist_m = 0;  // bit r: row r gets a histogram
    // the next segment's weights (element lane + 32 i of its rows x H) and bounds, loaded ahead
    constexpr int kPfRows = H > 32 ? 128 / H : kSegRows;
    constexpr int kPfPerLane = kPfRows * H / 32;
    int pf_row0 = -1, pf_end = 0;
    float pf_w[kPfPerLane];
#pragma unroll
    for (int i = 0; i < kPfPerLane; ++i) pf_w[i] = 0.0f;
    bool aborted = false;
    for (int it = group;; it += kEpiGroups) {
        const int a = it % kAcc;
        // One decision for the group's four warps: all stop if any wait gave up
        // (they share the histogram and its flush barriers).
        const bool ok = mbar_wait(tfull + a * kEpiGroups + group, (it / (kAcc * kEpiGroups)) & 1, abort, p.status);
        if (group_sync_any(group, !ok)) {
            aborted = true;
            break;
        }
        tc_fence_after();
        const int4 tag = ainfo[a];   // {tile in segment, segment, first row, rows}; segment -1 ends the sequence
        if (tag.y < 0) break;
        if (tag.y != cur || seg_tiles == kHistFlushTiles) {
            if (cur >= 0 && hist_m) flush_group_hist(p, gh, group, row0, nrows, hist_m, e);
            seg_tiles = 0;
        }
        ++seg_tiles;
        if (tag.y != cur) {
            cur = tag.y;
            row0 = tag.z;
            nrows = tag.w;
            if (pf_row0 == row0) {   // prefetched at the previous segment change
#pragma unroll
                for (int i = 0; i < kPfPerLane; ++i)
                    if (lane + 32 * i < nrows * H) wsm[lane + 32 * i] = pf_w[i];
                end_l = lane < nrows ? pf_end : 0;
            } else {
                for (int i = lane; i < nrows * H; i += 32)
                    wsm[i] = __bfloat162float(p.w[static_cast<int64_t>(row0 + i / H) * p.w_stride + i % H]);
                end_l = lane < nrows ? p.eff_end[row0 + lane] : 0;
            }
            hist_m = __ballot_sync(0xFFFFFFFFu, lane < nrows && p.hist_k >= 0 && end_l > p.hist_k);
            __syncwarp();
            // Segments lie in row order, so the next one most likely starts at row
            // row0 + nrows: its weights and bounds are loaded now and used at the
            // next change (the loads complete while the tiles in between are drained).
            pf_row0 = row0 + nrows;
#pragma unroll
            for (int i = 0; i < kPfPerLane; ++i) {
                const int r = pf_row0 + (lane + 32 * i) / H;
                pf_w[i] = r < p.rows ? __bfloat162float(p.w[static_cast<int64_t>(r) * p.w_stride + (lane + 32 * i) % H])
                                     : 0.0f;
            }
            pf_end = (lane < kPfRows && pf_row0 + lane < p.rows) ? p.eff_end[pf_row0 + lane] : 0;
        }
        const float ksm = f32scale ? reinterpret_cast<const float*>(smem + OFF_KS + a * 512)[m] : 1.0f;
        const int tpos = tag.x * kTileRows + m;
        const uint32_t acc = tbase + a * 128;
        // 64-column loads of 64 / H rows; a remainder of fewer rows in 32-column loads
        constexpr int kRpl = 64 / H;
        int r = 0;
        for (; r + kRpl <= nrows; r += kRpl) {
            uint32_t v[64];
            tc_ld_32x32b_x64(acc + r * H, v);
            tc_wait_ld_regs<64>(v);
#pragma unroll
            for (int i = 0; i < kRpl; ++i)
                emit_row(p, row0 + r + i, tpos, head_sum<H>(v + i * H, wsm + (r + i) * H, ksm),
                         __shfl_sync(0xFFFFFFFFu, end_l, r + i), (hist_m >> (r + i)) & 1,
                         gh + (r + i) * (kHistBins / 2));
        }
        if constexpr (H < 64) {
            for (; r < nrows; r += 32 / H) {
                uint32_t v[32];
                tc_ld_32x32b_x32(acc + r * H, v);   // within the accumulator's 128 columns
                tc_wait_ld_regs<32>(v);
#pragma unroll
                for (int i = 0; i < 32 / H; ++i)
                    if (r + i < nrows)
                        emit_row(p, row0 + r + i, tpos, head_sum<H>(v + i * H, wsm + (r + i) * H, ksm),
                                 __shfl_sync(0xFFFFFFFFu, end_l, r + i), (hist_m >> (r + i)) & 1,
                                 gh + (r + i) * (kHistBins / 2));
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) smem_add_release(released + a, 1u);
    }
    if (cur >= 0 && !aborted && hist_m) flush_group_hist(p, gh, group, row0, nrows, hist_m, e);
}

template <int F, int H>
__global__ void __launch_bounds__(kScoreThreads, 1)
    score_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap smap,
                 const __grid_constant__ CUtensorMap qmap, const ScoreArgs args) {
    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* full = bars;
    uint64_t* empty = bars + kMaxStages;
    uint64_t* qfull = bars + 2 * kMaxStages;
    uint64_t* tfull = qfull + 2;
    uint64_t* done_bar = tfull + kAcc * kEpiGroups;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    volatile int* abort = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
    uint32_t* released = reinterpret_cast<uint32_t*>(smem + OFF_MISC + 16);   // per accumulator
    uint32_t* published = reinterpret_cast<uint32_t*>(smem + OFF_MISC + 32);
    uint32_t* consumed = reinterpret_cast<uint32_t*>(smem + OFF_MISC + 48);   // per copy warp
    uint32_t* armed = consumed + kCopyWarps;                                   // per copy warp
    const int warp = threadIdx.x >> 5;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kMaxStages; ++s) {
            mbar_init(full + s, 1);   // the tile's copy warp (its tag and bytes)
            mbar_init(empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) mbar_init(qfull + b, 1);
        for (int b = 0; b < kAcc * kEpiGroups; ++b) mbar_init(tfull + b, 2);
        for (int b = 0; b < kAcc; ++b) released[b] = 0u;
        *published = 0u;
        for (int c = 0; c < kCopyWarps; ++c) consumed[c] = armed[c] = 0u;
        mbar_init(done_bar, kMmaWarps);
        *abort = 0;
        mbar_fence_init();
        tma_prefetch(&kmap);
        tma_prefetch(&smap);
        tma_prefetch(&qmap);
    }
    if (warp == 1) tc_alloc(tmem_slot, TM_COLS);
    for (int i = threadIdx.x; i < kEpiGroups * kGroupHistWords; i += blockDim.x)
        reinterpret_cast<uint32_t*>(smem + OFF_HIST)[i] = 0u;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    pdl_launch_dependents();
    pdl_wait();   // the plan kernel's segments and tile prefix

    if (warp == 0) {
        const int4 range = args.cta[blockIdx.x];   // {first tile, end tile, first segment, segments}
        const int t0 = range.x, t1 = range.y, S = range.w;
        const int seg = (t0 < t1 && range.z < 0) ? find_segment(args.seg_prefix, S, t0) : range.z;
        Producer<F, H> pr{&kmap,
                    &smap,
                    &qmap,
                    smem,
                    full,
                    empty,
                    qfull,
                    abort,
                    reinterpret_cast<int4*>(smem + OFF_PRING),
                    published,
                    consumed,
                    armed};
        producer_role(pr, args, t0, t1, seg, S);
    } else if (warp < kFirstEpiWarp) {
        mma_role<F, H>(args, smem, tmem, full, empty, qfull, tfull, released, done_bar, abort);
    } else if (warp < kFirstCopyWarp) {
        epilogue_role<F, H>(args, smem, tmem, tfull, released, abort);
    } else {
        copy_role<F>(args, &kmap, &smap, smem, full, empty, published, consumed, armed, abort, warp - kFirstCopyWarp);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tc_dealloc(tmem, TM_COLS);
    }
}

// ----------------------------------------------------------------- host
static void* g_time_before = nullptr;
static void* g_time_after = nullptr;

static bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace dsa

using namespace dsa;

extern "C" void dsa_set_score_timing(void* before, void* after) {
    g_time_before = before;
    g_time_after = after;
}

extern "C" int dsa_timing_event_create(void** event) {
    if (!event) return DSA_ERR_INVALID;
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return DSA_ERR_CUDA;
    *event = static_cast<void*>(e);
    return DSA_OK;
}

extern "C" int dsa_timing_event_destroy(void* event) {
    return cudaEventDestroy(static_cast<cudaEvent_t>(event)) == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

extern "C" int dsa_timing_elapsed_ms(void* start, void* end, float* ms) {
    if (!start || !end || !ms) return DSA_ERR_INVALID;
    if (cudaEventSynchronize(static_cast<cudaEvent_t>(end)) != cudaSuccess) return DSA_ERR_CUDA;
    return cudaEventElapsedTime(ms, static_cast<cudaEvent_t>(start), static_cast<cudaEvent_t>(end)) == cudaSuccess
               ? DSA_OK
               : DSA_ERR_CUDA;
}

extern "C" size_t dsa_workspace_size(int fmt, int64_t rows, int64_t num_requests, int64_t max_pages, int64_t k) {
    (void)fmt;
    (void)num_requests;
    (void)k;
    if (rows < 0 || max_pages < 0) return 0;
    return workspace_layout(rows, max_pages * kPage, true, true).total;
}

namespace dsa {

// Query operands of one scoring call: `heads` heads per row, payload row r at
// q + r * q_stride (FP8: 32 x 128 codes; MXFP4: heads x 64 packed bytes), MXFP4
// scales of row r at q_scales + r * qs_stride (group-major or head-major),
// BF16 weights of row r at w + r * w_stride.
struct QueryOperands {
    int heads;
    const void* q;
    int64_t q_stride;
    const void* q_scales;
    int64_t qs_stride;
    bool qs_group_major;
    const void* w;
    int64_t w_stride;
};

// The step's preparation (dsa_decode_step): its inputs, the rest being the
// scoring call's own (cache, queries and weights out, row bounds out, status).
struct PrepareCall {
    const void* q;
    int64_t q_row_stride;
    const void* wv;
    int64_t wv_row_stride;
    const void* k;
    int64_t k_row_stride;
    const float* gamma;
    const float* beta;
    float eps;
    const int64_t* slots;
    int64_t n;
    const int32_t* seq_lens;
    int64_t num_seq;
    const int32_t* query_lens;
};

// prep: when non-null, the preparation runs first, in one launch that also
// lays out the plan (in place of plan_kernel); its outputs are q_rows, w,
// starts and row_ends.
static int score_paged_impl(int fmt, const QueryOperands& qo, const void* cache, int64_t page_stride,
                            int64_t num_pages, const int32_t* block_table, int64_t bt_stride, int64_t max_pages,
                            const int32_t* starts, const int32_t* row_ends, int64_t num_requests, int64_t rows,
                            int64_t max_query_len, float* logits, int64_t logits_ld, int64_t k, int32_t* topk,
                            void* workspace, size_t workspace_bytes, int32_t* status, cudaStream_t stream,
                            const PrepareCall* prep = nullptr) {
    if (fmt < DSA_FMT_FP8 || fmt > DSA_FMT_MXFP4_RG) return DSA_ERR_UNSUPPORTED;
    if (rows < 0 || num_requests < 0 || max_pages < 0 || num_pages < 0 || k < 0 || max_query_len < 0)
        return DSA_ERR_INVALID;
    if (rows == 0) return DSA_OK;
    const bool fp4 = fmt_fp4(fmt);
    const bool rg = (fmt == DSA_FMT_MXFP4_RG);
    const int64_t width = max_pages * kPage;
    if (rows > (1 << 30) || num_requests > (1 << 30) || width > (int64_t(1) << 30) || num_pages > 0x7FFFFFFF)
        return DSA_ERR_UNSUPPORTED;
    const void* q_rows = qo.q;
    const void* w = qo.w;
    if (!q_rows || !w || !starts || !row_ends || !workspace || (fp4 && !qo.q_scales)) return DSA_ERR_INVALID;
    if (num_pages > 0 && !cache) return DSA_ERR_INVALID;
    if (max_pages > 0 && num_requests > 0 && (!block_table || bt_stride < max_pages)) return DSA_ERR_INVALID;
    const int64_t min_stride = fp4 ? DSA_FP4_PAGE_BYTES : DSA_FP8_PAGE_BYTES;
    if (page_stride < min_stride || page_stride % 16) return DSA_ERR_INVALID;
    if (!aligned(cache, 16) || !aligned(q_rows, 16) || !aligned(workspace, 256) || !aligned(w, 2) ||
        (fp4 && !aligned(qo.q_scales, 16)) || qo.q_stride % 16 || qo.qs_stride % 16)
        return DSA_ERR_INVALID;
    if (logits && (logits_ld < width || !aligned(logits, 4))) return DSA_ERR_INVALID;
    const bool want_topk = (k > 0 && topk != nullptr);
    if (k > (int64_t(1) << 30)) return DSA_ERR_UNSUPPORTED;
    const WsLayout L = workspace_layout(rows, width, true, logits == nullptr);
    if (workspace_bytes < L.total) return DSA_ERR_INVALID;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    float* out_logits = logits ? logits : reinterpret_cast<float*>(ws + L.logits);
    const int64_t ld = logits ? logits_ld : width;
    const int heads = qo.heads;
    const int seg_rows = heads > 32 ? 128 / heads : kSegRows;

    // Tensor maps: key pages, key scales, query rows.
    CUtensorMap kmap, smap, qmap;
    const cuuint64_t np = static_cast<cuuint64_t>(num_pages > 0 ? num_pages : 1);
    uint8_t* cache_b = static_cast<uint8_t*>(const_cast<void*>(cache));
    void* cache_addr = cache_b ? static_cast<void*>(cache_b) : workspace;   // unused when there are no pages
    if (rg) {
        // {16 code bytes, 64 keys, 4 column groups, pages}: one box = one group of one page
        const cuuint64_t dims[4] = {16, 64, 4, np};
        const cuuint64_t strides[3] = {16, kRgGroupBytes, static_cast<cuuint64_t>(page_stride)};
        const cuuint32_t box[4] = {16, 64, 1, 1};
        if (encode_tiled(&kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, cache_addr, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
            return DSA_ERR_CUDA;
    } else {
        // {row bytes, 64 keys, pages}: FP8 rows of 128 bytes (128-byte swizzle), MXFP4 rows of
        // 64 packed bytes (64-byte swizzle)
        const cuuint64_t row = fp4 ? 64 : 128;
        const cuuint64_t dims[3] = {row, 64, np};
        const cuuint64_t strides[2] = {row, static_cast<cuuint64_t>(page_stride)};
        const cuuint32_t box[3] = {static_cast<cuuint32_t>(row), 64, 1};
        if (encode_tiled(&kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, cache_addr, dims, strides, box,
                         fp4 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
            return DSA_ERR_CUDA;
    }
    {
        const cuuint64_t dims[2] = {64, np};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(page_stride)};
        const cuuint32_t box[2] = {64, 1};
        uint8_t* sbase = cache_b ? cache_b + (fp4 ? kFp4KeyBytes : kFp8KeyBytes) : static_cast<uint8_t*>(workspace);
        if (encode_tiled(&smap, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, sbase, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
            return DSA_ERR_CUDA;
    }
    if (rg) {
        // {64 code bytes, heads, rows}: one box = one 16-byte column chunk of a row's heads
        const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(rows)};
        const cuuint64_t strides[2] = {64, static_cast<cuuint64_t>(qo.q_stride)};
        const cuuint32_t box[3] = {16, static_cast<cuuint32_t>(heads), 1};
        if (encode_tiled(&qmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(q_rows), dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
            return DSA_ERR_CUDA;
    } else {
        const cuuint64_t row = fp4 ? 64 : 128;
        const cuuint64_t dims[3] = {row, static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(rows)};
        const cuuint64_t strides[2] = {row, static_cast<cuuint64_t>(qo.q_stride)};
        const cuuint32_t box[3] = {static_cast<cuuint32_t>(row), static_cast<cuuint32_t>(heads), 1};
        if (encode_tiled(&qmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(q_rows), dims, strides, box,
                         fp4 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
            return DSA_ERR_CUDA;
    }

    int* info = reinterpret_cast<int*>(ws + L.info);
    int4* segs = reinterpret_cast<int4*>(ws + L.segs);
    int* seg_prefix = reinterpret_cast<int*>(ws + L.seg_prefix);
    int* eff_end = reinterpret_cast<int*>(ws + L.eff_end);
    int4* cta = reinterpret_cast<int4*>(ws + L.cta);
    const int grid = device_sm_count() < kMaxScoreCtas ? device_sm_count() : kMaxScoreCtas;
    if (prep) {
        const int rc = launch_prepare(fmt, prep->q, prep->q_row_stride, prep->wv, prep->wv_row_stride, rows,
                                      const_cast<void*>(q_rows), const_cast<void*>(w), prep->k, prep->k_row_stride,
                                      prep->gamma, prep->beta, prep->eps, prep->slots, prep->n,
                                      const_cast<void*>(cache), page_stride, num_pages, prep->seq_lens, prep->num_seq,
                                      prep->query_lens, num_requests, rows, const_cast<int32_t*>(starts),
                                      const_cast<int32_t*>(row_ends), status, stream);
        if (rc != DSA_OK) return rc;
    }
    if (launch_pdl(plan_kernel, dim3(1), dim3(kPlanThreads), 0, stream, starts, row_ends, static_cast<int>(num_requests),
                   static_cast<int>(rows), static_cast<int>(width), info, segs, seg_prefix, eff_end, cta, grid, seg_rows,
                   status) != cudaSuccess)
        return DSA_ERR_CUDA;

    // One kernel per (format, heads); its shared-memory limit is an attribute of
    // each device's copy of it.
    using ScoreFn = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const ScoreArgs);
    ScoreFn fn = nullptr;
    int variant = 0;
    switch (fmt) {
        case DSA_FMT_FP8: fn = score_kernel<DSA_FMT_FP8, 32>; variant = 0; break;
        case DSA_FMT_FP8_MX: fn = score_kernel<DSA_FMT_FP8_MX, 32>; variant = 1; break;
        case DSA_FMT_MXFP4:
            fn = heads == 16 ? score_kernel<DSA_FMT_MXFP4, 16>
                             : heads == 64 ? score_kernel<DSA_FMT_MXFP4, 64> : score_kernel<DSA_FMT_MXFP4, 32>;
            variant = 2 + (heads == 16 ? 0 : heads == 64 ? 2 : 1);
            break;
        default:
            fn = heads == 16 ? score_kernel<DSA_FMT_MXFP4_RG, 16>
                             : heads == 64 ? score_kernel<DSA_FMT_MXFP4_RG, 64> : score_kernel<DSA_FMT_MXFP4_RG, 32>;
            variant = 5 + (heads == 16 ? 0 : heads == 64 ? 2 : 1);
            break;
    }
    if (!fp4 && heads != 32) return DSA_ERR_UNSUPPORTED;
    static bool attr_set[64][8] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DSA_ERR_CUDA;
    if (!attr_set[dev][variant]) {
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kScoreSmem) != cudaSuccess)
            return DSA_ERR_CUDA;
        attr_set[dev][variant] = true;
    }
    ScoreArgs a;
    a.fmt = fmt;
    a.num_pages = static_cast<int>(num_pages);
    a.block_table = block_table;
    a.bt_stride = bt_stride;
    a.q_rows = static_cast<const uint8_t*>(q_rows);
    a.w = static_cast<const __nv_bfloat16*>(w);
    a.segs = segs;
    a.seg_prefix = seg_prefix;
    a.eff_end = eff_end;
    a.cta = cta;
    a.logits = out_logits;
    a.ld = ld;
    a.hist_k = want_topk ? static_cast<int>(k) : -1;
    a.hist = reinterpret_cast<unsigned*>(ws + L.hist);
    a.status = status;
    a.heads = heads;
    a.q_scales = static_cast<const uint8_t*>(qo.q_scales);
    a.qs_stride = qo.qs_stride;
    a.qs_group_major = qo.qs_group_major ? 1 : 0;
    a.w_stride = qo.w_stride;
    a.rows = static_cast<int>(rows);
    if (g_time_before && g_time_after)   // external: kept as a record node under stream capture
        cudaEventRecordWithFlags(static_cast<cudaEvent_t>(g_time_before), stream, cudaEventRecordExternal);
    if (launch_pdl(fn, dim3(grid), dim3(kScoreThreads), kScoreSmem, stream, kmap, smap, qmap, a) != cudaSuccess)
        return DSA_ERR_CUDA;
    if (g_time_before && g_time_after)
        cudaEventRecordWithFlags(static_cast<cudaEvent_t>(g_time_after), stream, cudaEventRecordExternal);
    if (!want_topk && !logits) return DSA_OK;
    return launch_select(out_logits, logits, ld, width, eff_end, rows, want_topk ? k : 0, want_topk ? topk : nullptr,
                         ws, L, stream, true);
}

}  // namespace dsa

using namespace dsa;

extern "C" int dsa_score_paged(int fmt, const void* q_rows, const void* w, const void* cache, int64_t page_stride,
                               int64_t num_pages, const int32_t* block_table, int64_t bt_stride, int64_t max_pages,
                               const int32_t* starts, const int32_t* row_ends, int64_t num_requests, int64_t rows,
                               int64_t max_query_len, float* logits, int64_t logits_ld, int64_t k, int32_t* topk,
                               void* workspace, size_t workspace_bytes, int32_t* status, void* stream) {
    // 4096-byte query rows of 32 heads; MXFP4 rows carry their scales at byte 2048
    // (head-major, or group-major in the row-group format)
    QueryOperands qo{kHeads, q_rows, kQRowBytes,
                     q_rows ? static_cast<const uint8_t*>(q_rows) + kFp4Scales : nullptr, kQRowBytes,
                     fmt == DSA_FMT_MXFP4_RG, w, kHeads};
    return score_paged_impl(fmt, qo, cache, page_stride, num_pages, block_table, bt_stride, max_pages, starts,
                            row_ends, num_requests, rows, max_query_len, logits, logits_ld, k, topk, workspace,
                            workspace_bytes, status, static_cast<cudaStream_t>(stream));
}

extern "C" int dsa_score_paged_heads(int fmt, int64_t heads, const void* payload, const void* q_scales, const void* w,
                                     const void* cache, int64_t page_stride, int64_t num_pages,
                                     const int32_t* block_table, int64_t bt_stride, int64_t max_pages,
                                     const int32_t* starts, const int32_t* row_ends, int64_t num_requests,
                                     int64_t rows, int64_t max_query_len, float* logits, int64_t logits_ld, int64_t k,
                                     int32_t* topk, void* workspace, size_t workspace_bytes, int32_t* status,
                                     void* stream) {
    if (!fmt_fp4(fmt) || (heads != 16 && heads != 32 && heads != 64)) return DSA_ERR_UNSUPPORTED;
    QueryOperands qo{static_cast<int>(heads), payload, heads * 64, q_scales, 4 * kRgQuerySlots, true, w, heads};
    return score_paged_impl(fmt, qo, cache, page_stride, num_pages, block_table, bt_stride, max_pages, starts,
                            row_ends, num_requests, rows, max_query_len, logits, logits_ld, k, topk, workspace,
                            workspace_bytes, status, static_cast<cudaStream_t>(stream));
}

extern "C" int dsa_decode_step(int fmt, const void* q, int64_t q_row_stride, const void* wv, int64_t wv_row_stride,
                               const void* k, int64_t k_row_stride, const float* gamma, const float* beta, float eps,
                               const int64_t* slots, int64_t n, void* cache, int64_t page_stride, int64_t num_pages,
                               const int32_t* seq_lens, int64_t num_seq, const int32_t* query_lens,
                               int64_t num_requests, int64_t num_rows, const int32_t* block_table, int64_t bt_stride,
                               int64_t max_pages, int64_t max_query_len, void* q_out, void* w_out, int32_t* starts,
                               int32_t* row_ends, float* logits, int64_t logits_ld, int64_t top_k, int32_t* topk,
                               void* workspace, size_t workspace_bytes, int32_t* status, void* stream) {
    // The preparation's 32-head query rows and weights, read by the scoring as dsa_score_paged reads them.
    QueryOperands qo{kHeads, q_out, kQRowBytes,
                     q_out ? static_cast<const uint8_t*>(q_out) + kFp4Scales : nullptr, kQRowBytes,
                     fmt == DSA_FMT_MXFP4_RG, w_out, kHeads};
    const PrepareCall prep{q, q_row_stride, wv, wv_row_stride, k, k_row_stride, gamma, beta, eps, slots, n,
                           seq_lens, num_seq, query_lens};
    // the preparation's argument errors first, before any work of the scoring's
    const int rc = check_prepare(fmt, q, q_row_stride, wv, wv_row_stride, num_rows, q_out, w_out, k, k_row_stride,
                                 gamma, beta, slots, n, cache, page_stride, num_pages, seq_lens, num_seq, query_lens,
                                 num_requests, num_rows, starts, row_ends);
    if (rc != DSA_OK) return rc;
    if (num_rows == 0)   // nothing to score; the step's keys are still inserted
        return launch_prepare(fmt, q, q_row_stride, wv, wv_row_stride, 0, q_out, w_out, k, k_row_stride, gamma, beta,
                              eps, slots, n, cache, page_stride, num_pages, seq_lens, num_seq, query_lens,
                              num_requests, 0, starts, row_ends, status, static_cast<cudaStream_t>(stream));
    return score_paged_impl(fmt, qo, cache, page_stride, num_pages, block_table, bt_stride, max_pages, starts,
                            row_ends, num_requests, num_rows, max_query_len, logits, logits_ld, top_k, topk,
                            workspace, workspace_bytes, status, static_cast<cudaStream_t>(stream), &prep);
}
