// Top-k selection over per-row scores (radix select on order-preserving bits).
//
// Page "cutedsl.dsa.overlap": the indexer path is "wq_b -> DsaIndex -> scoring
// and top-k"; page "amd.ops.fp4_indexer", decode_tile_size, budgets per-row
// selection scratch next to the logits.
//
// Pass 1 (fused into the scoring epilogue, or hist_kernel here): a 2048-bin
// histogram of the top 11 bits of each row's order-preserving score keys.
// Pass 2 (select_kernel): the boundary bin B is where the count from the top
// reaches k; positions in bins above B are winners, bin B holds the
// candidates, resolved by two more radix levels (bits 20..10, then 9..0).
// Rows of at most 8192 positions take one CTA that holds the row in
// registers and its candidates in shared memory.  Longer rows take one CTA
// per 4096 positions; each appends its candidates to a per-row buffer, and
// the last CTA of the row (a done counter, no waiting) resolves them.  Every
// placement uses block scans, not contended atomics.  The row's histogram and
// counters are cleared at the end, so the workspace is zero for the next call.
#include <mutex>

#include "host.h"
#include "scan.cuh"

namespace dsa {

constexpr int kSelThreads = 1024;
constexpr int kChunk = 4096;   // positions per select CTA
constexpr int kPerThread = kChunk / kSelThreads;
constexpr int kRefineCap = 4096;   // boundary candidates the last CTA keeps in shared memory

struct SelectArgs {
    const float* logits;
    float* fill;         // when non-null: write -inf at [end, width) of each row
    int64_t ld;
    int64_t width;
    const int32_t* ends;
    int k;               // 0: fill only
    int32_t* out;
    unsigned* hist;
    int* counters;
    uint2* cand;
};

__device__ __forceinline__ int clamp_end(const int32_t* ends, int row, int64_t width) {
    const int64_t e = ends[row];
    return static_cast<int>(e < 0 ? 0 : (e > width ? width : e));
}

// Copies a row's 2048-bin histogram to shared memory, all loads in flight.
__device__ __forceinline__ void load_hist(unsigned* h, const unsigned* ghist) {
    unsigned r[kHistBins / kSelThreads];
#pragma unroll
    for (int i = 0; i < kHistBins / kSelThreads; ++i) r[i] = ghist[i * kSelThreads + threadIdx.x];
#pragma unroll
    for (int i = 0; i < kHistBins / kSelThreads; ++i) h[i * kSelThreads + threadIdx.x] = r[i];
}

// Finds, over `bins` counts in shared memory, the bin B where the count from
// the top first reaches `need`; stores B and the count strictly above it.
__device__ void find_boundary(const unsigned* h, int bins, int need, int* out_bin, int* out_above, int* tmp) {
    const int per = bins / kSelThreads;   // bins per thread (8 or 4)
    const int first = bins - (threadIdx.x + 1) * per;   // thread 0 owns the top bins
    int local = 0;
    for (int i = 0; i < per; ++i) local += static_cast<int>(h[first + i]);
    int total;
    const int inc = block_inclusive_scan(local, tmp, &total);
    int cum = inc - local;   // count in bins above this thread's range
    for (int b = first + per - 1; b >= first; --b) {
        const int c = static_cast<int>(h[b]);
        if (cum < need && cum + c >= need) {
            *out_bin = b;
            *out_above = cum;
        }
        cum += c;
    }
}

__global__ void __launch_bounds__(kSelThreads) hist_kernel(const float* __restrict__ logits, int64_t ld,
                                                           int64_t width, const int32_t* __restrict__ ends, int k,
                                                           unsigned* __restrict__ hist) {
    __shared__ unsigned h[kHistBins];
    pdl_launch_dependents();
    pdl_wait();
    const int row = blockIdx.x;
    const int n = clamp_end(ends, row, width);
    if (n <= k) return;
    const int64_t lo = static_cast<int64_t>(blockIdx.y) * kChunk;
    if (lo >= n) return;
    const int64_t hi = min(static_cast<int64_t>(n), lo + kChunk);
    for (int i = threadIdx.x; i < kHistBins; i += kSelThreads) h[i] = 0;
    __syncthreads();
    const float* src = logits + static_cast<int64_t>(row) * ld;
    float v[kPerThread];
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
        const int64_t t = lo + i * kSelThreads + threadIdx.x;
        v[i] = t < hi ? src[t] : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < kPerThread; ++i)
        if (lo + i * kSelThreads + threadIdx.x < hi) atomicAdd(&h[hist_bin(v[i])], 1u);
    __syncthreads();
    for (int i = threadIdx.x; i < kHistBins; i += kSelThreads)
        if (h[i]) atomicAdd(hist + static_cast<int64_t>(row) * kHistBins + i, h[i]);
}

// Streams the boundary-bin candidates of a row: from shared memory when they
// fit, else from the candidate buffer when it did not overflow, else by
// re-reading the row and keeping bin == B.
struct CandSource {
    const uint2* buf;
    int count;
    int mode;   // 0: shared-memory copy, 1: global buffer, 2: re-read the row
    const float* row;
    int n;
    uint32_t bin;
    template <typename F>
    __device__ __forceinline__ void for_each(F&& f) const {
        if (mode != 2) {
            for (int i = threadIdx.x; i < count; i += kSelThreads) {
                const uint2 c = buf[i];
                f(c.x, static_cast<int>(c.y));
            }
        } else {
            for (int t = threadIdx.x; t < n; t += kSelThreads) {
                const uint32_t key = order_key(row[t]);
                if ((key >> (32 - kHistBits)) == bin) f(key, t);
            }
        }
    }
};

// Writes the positions of the candidates matching `pred` to out[base ..),
// at most `limit` of them, placed by a block scan (no shared atomics).
// Returns how many candidates matched (every thread gets the same value).
template <typename Pred>
__device__ int emit_matching(const CandSource& src, Pred pred, int32_t* out, int base, int limit, int* tmp,
                             int* s_tot) {
    int mine = 0;
    src.for_each([&](uint32_t key, int) { mine += pred(key) ? 1 : 0; });
    int pos = block_inclusive_scan(mine, tmp, s_tot) - mine;
    const int total = *s_tot;
    if (mine) {
        src.for_each([&](uint32_t key, int t) {
            if (pred(key)) {
                if (pos < limit) out[base + pos] = t;
                ++pos;
            }
        });
    }
    __syncthreads();
    return total;
}

// Top `need` of at most kRankMax candidates held in shared memory, by rank
// counting: rank(c) = candidates with a larger key, plus equal keys earlier in
// the list.  Ranks are distinct, so exactly min(need, ncand) positions are
// written.  Four threads share a candidate, each scanning every fourth group
// of four keys of `keys` (a copy padded with zeros, which never outrank a real
// key); two shuffles add their counts.
constexpr int kRankMax = kSelThreads / 4;
__device__ void rank_select(const uint2* c, uint32_t* keys, int ncand, int32_t* out, int above, int need) {
    const int i = threadIdx.x;
    const int padded = (ncand + 15) & ~15;
    if (i < ncand) keys[i] = c[i].x;
    else if (i < padded) keys[i] = 0u;
    __syncthreads();
    const int cand = i >> 2, part = i & 3;
    uint2 me = make_uint2(0u, 0u);
    int rank = 0;
    if (cand < ncand) {
        me = c[cand];
        for (int j = part * 4; j < ncand; j += 16) {
            const uint4 k4 = *reinterpret_cast<const uint4*>(keys + j);
            rank += (k4.x > me.x || (k4.x == me.x && j + 0 < cand)) ? 1 : 0;
            rank += (k4.y > me.x || (k4.y == me.x && j + 1 < cand)) ? 1 : 0;
            rank += (k4.z > me.x || (k4.z == me.x && j + 2 < cand)) ? 1 : 0;
            rank += (k4.w > me.x || (k4.w == me.x && j + 3 < cand)) ? 1 : 0;
        }
    }
    rank += __shfl_xor_sync(0xFFFFFFFFu, rank, 1);
    rank += __shfl_xor_sync(0xFFFFFFFFu, rank, 2);
    if (cand < ncand && part == 0 && rank < need) out[above + rank] = static_cast<int>(me.y);
}

// Resolves the boundary bin of a row: `need` more positions come from the
// candidates (keys whose top 11 bits equal the bin B), chosen by two more
// radix levels (bits 20..10, then 9..0); positions go to out[above ..).
__device__ void refine_boundary(const CandSource& src, uint32_t B, int32_t* out, int above, int need,
                                unsigned* h, int* tmp, int* s_bin, int* s_above, int* s_tot) {
    // level 2: bits [20:10]
    for (int i = threadIdx.x; i < kHistBins; i += kSelThreads) h[i] = 0;
    if (threadIdx.x == 0) {
        *s_bin = 0;
        *s_above = 0;
    }
    __syncthreads();
    src.for_each([&](uint32_t key, int) { atomicAdd(&h[(key >> 10) & 0x7FF], 1u); });
    __syncthreads();
    find_boundary(h, kHistBins, need, s_bin, s_above, tmp);
    __syncthreads();
    const uint32_t B2 = static_cast<uint32_t>(*s_bin);
    const int n2 = emit_matching(src, [&](uint32_t key) { return ((key >> 10) & 0x7FF) > B2; }, out, above, need,
                                 tmp, s_tot);
    // level 3: bits [9:0] within level-2 bin B2
    for (int i = threadIdx.x; i < 1024; i += kSelThreads) h[i] = 0;
    if (threadIdx.x == 0) {
        *s_bin = 0;
        *s_above = 0;
    }
    __syncthreads();
    src.for_each([&](uint32_t key, int) {
        if (((key >> 10) & 0x7FF) == B2) atomicAdd(&h[key & 0x3FF], 1u);
    });
    __syncthreads();
    const int need2 = need - n2;
    find_boundary(h, 1024, need2, s_bin, s_above, tmp);
    __syncthreads();
    const uint32_t B3 = static_cast<uint32_t>(*s_bin);
    const int n3 = emit_matching(
        src, [&](uint32_t key) { return ((key >> 10) & 0x7FF) == B2 && (key & 0x3FF) > B3; }, out, above + n2,
        need2, tmp, s_tot);
    // equal keys at the boundary: the first ones in candidate order
    const uint32_t kB = (B << (32 - kHistBits)) | (B2 << 10) | B3;
    const int left = need2 - n3;
    const int n4 = emit_matching(src, [&](uint32_t key) { return key == kB; }, out, above + n2 + n3, left, tmp,
                                 s_tot);
    // Short only when the histogram disagreed with the scores (an aborted scoring pass).
    for (int e = n2 + n3 + min(n4, left) + threadIdx.x; e < need; e += kSelThreads) out[above + e] = -1;
}

// Rows of at most kSingleRow positions are selected by one CTA holding the
// whole row in registers; longer rows are split into kChunk-position CTAs.
constexpr int kSingleRow = 8192;
constexpr int kSelDynSmem = kSingleRow * sizeof(float);   // the staged row

__global__ void __launch_bounds__(kSelThreads) select_kernel(const SelectArgs a, int pdl) {
    __shared__ __align__(16) unsigned h[kHistBins];   // histogram, then rank_select's key copy
    __shared__ int tmp[32];
    __shared__ int s_bin, s_above, s_last, s_wbase, s_cbase, s_tot;
    __shared__ uint64_t s_bar;
    __shared__ int s_ww[kSelThreads / 32], s_wb[kSelThreads / 32];
    __shared__ uint2 cbuf[kRefineCap];
    if (pdl) pdl_wait();
    const int row = blockIdx.x;
    const int64_t lo = static_cast<int64_t>(blockIdx.y) * kChunk;
    const int n = clamp_end(a.ends, row, a.width);
    if (a.fill) {
        float* dst = a.fill + static_cast<int64_t>(row) * a.ld;
        const int64_t hi = min(a.width, lo + kChunk);
        for (int64_t t = max(lo, static_cast<int64_t>(n)) + threadIdx.x; t < hi; t += kSelThreads)
            dst[t] = -__int_as_float(0x7F800000);
    }
    const int k = a.k;
    if (k <= 0) return;
    int32_t* out = a.out + static_cast<int64_t>(row) * k;
    if (n <= k) {
        const int64_t hi = min(static_cast<int64_t>(k), lo + kChunk);
        for (int64_t pos = lo + threadIdx.x; pos < hi; pos += kSelThreads) out[pos] = pos < n ? static_cast<int>(pos) : -1;
        return;
    }
    unsigned* ghist = a.hist + static_cast<int64_t>(row) * kHistBins;
    const float* src = a.logits + static_cast<int64_t>(row) * a.ld;

    if (n <= kSingleRow) {
        // ---- one CTA per row: the row staged in shared memory by one bulk
        // copy (while the histogram is read), then compact loops over it.
        if (blockIdx.y != 0) return;
        extern __shared__ __align__(16) float srow[];
        const int n4 = (n + 3) & ~3;
        const bool bulk = (reinterpret_cast<uintptr_t>(src) % 16) == 0 && n4 <= a.ld;
        if (threadIdx.x == 0) {
            s_bin = 0;
            s_above = 0;
            if (bulk) {
                mbar_init(&s_bar, 1);
                mbar_fence_init();
                mbar_arrive_expect_tx(&s_bar, static_cast<uint32_t>(n4) * 4u);
                bulk_load(srow, src, static_cast<uint32_t>(n4) * 4u, &s_bar);
            }
        }
        if (!bulk)
            for (int t = threadIdx.x; t < n; t += kSelThreads) srow[t] = src[t];
        load_hist(h, ghist);
        __syncthreads();
        find_boundary(h, kHistBins, k, &s_bin, &s_above, tmp);
        if (bulk) mbar_drain(&s_bar, 0);   // bounded wait for the row
        __syncthreads();
        const uint32_t B = static_cast<uint32_t>(s_bin);
        const int above = s_above;
        // Place winners (bin > B) and candidates (bin == B) with warp ballots:
        // each warp writes one contiguous run per iteration, so stores coalesce.
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        const unsigned lt = (1u << lane) - 1u;
        int wwin = 0, wbnd = 0;
        for (int t0 = 0; t0 < n; t0 += kSelThreads) {
            const int t = t0 + threadIdx.x;
            const uint32_t b = t < n ? order_key(srow[t]) >> (32 - kHistBits) : 0u;
            wwin += __popc(__ballot_sync(0xFFFFFFFFu, t < n && b > B));
            wbnd += __popc(__ballot_sync(0xFFFFFFFFu, t < n && b == B));
        }
        if (lane == 0) {
            s_ww[warp] = wwin;
            s_wb[warp] = wbnd;
        }
        __syncthreads();
        int pw = 0, pc = 0, ncand = 0;
        for (int i = 0; i < kSelThreads / 32; ++i) {
            if (i < warp) {
                pw += s_ww[i];
                pc += s_wb[i];
            }
            ncand += s_wb[i];
        }
        for (int t0 = 0; t0 < n; t0 += kSelThreads) {
            const int t = t0 + threadIdx.x;
            const uint32_t key = t < n ? order_key(srow[t]) : 0u;
            const uint32_t b = key >> (32 - kHistBits);
            const unsigned mw = __ballot_sync(0xFFFFFFFFu, t < n && b > B);
            const unsigned mb = __ballot_sync(0xFFFFFFFFu, t < n && b == B);
            if (t < n && b > B) {
                const int pos = pw + __popc(mw & lt);
                if (pos < k) out[pos] = t;
            } else if (t < n && b == B) {
                const int pos = pc + __popc(mb & lt);
                if (pos < kRefineCap) cbuf[pos] = make_uint2(key, static_cast<uint32_t>(t));
            }
            pw += __popc(mw);
            pc += __popc(mb);
        }
        __syncthreads();
        if (ncand <= kRankMax) {
            rank_select(cbuf, h, ncand, out, above, k - above);
        } else {
            const CandSource srcs{cbuf, min(ncand, kRefineCap), ncand <= kRefineCap ? 0 : 2, src, n, B};
            refine_boundary(srcs, B, out, above, k - above, h, tmp, &s_bin, &s_above, &s_tot);
        }
        __syncthreads();
        for (int i = threadIdx.x; i < kHistBins; i += kSelThreads) ghist[i] = 0;
        return;
    }

    // ---- several CTAs per row
    const int nch = (n + kChunk - 1) / kChunk;
    if (blockIdx.y >= nch) return;
    int* ctr = a.counters + static_cast<int64_t>(row) * 4;
    uint2* cand = a.cand + static_cast<int64_t>(row) * kCandCap;
    const int64_t hi = min(static_cast<int64_t>(n), lo + kChunk);
    float v[kPerThread];   // this CTA's scores, loaded while the histogram is read
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
        const int64_t t = lo + i * kSelThreads + threadIdx.x;
        v[i] = t < hi ? src[t] : 0.0f;
    }
    load_hist(h, ghist);
    if (threadIdx.x == 0) {
        s_bin = 0;
        s_above = 0;
    }
    __syncthreads();
    find_boundary(h, kHistBins, k, &s_bin, &s_above, tmp);
    __syncthreads();
    const uint32_t B = static_cast<uint32_t>(s_bin);
    // Place winners and candidates with warp ballots (coalesced runs per warp
    // and iteration); the CTA's bases come from one global add per counter.
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned lt = (1u << lane) - 1u;
    int wwin = 0, wbnd = 0;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
        const int64_t t = lo + i * kSelThreads + threadIdx.x;
        const uint32_t b = order_key(v[i]) >> (32 - kHistBits);
        wwin += __popc(__ballot_sync(0xFFFFFFFFu, t < hi && b > B));
        wbnd += __popc(__ballot_sync(0xFFFFFFFFu, t < hi && b == B));
    }
    if (lane == 0) {
        s_ww[warp] = wwin;
        s_wb[warp] = wbnd;
    }
    __syncthreads();
    int pw = 0, pc = 0, tot_w = 0, tot_b = 0;
    for (int i = 0; i < kSelThreads / 32; ++i) {
        if (i < warp) {
            pw += s_ww[i];
            pc += s_wb[i];
        }
        tot_w += s_ww[i];
        tot_b += s_wb[i];
    }
    if (threadIdx.x == 0) {
        s_wbase = tot_w ? atomicAdd(ctr + 0, tot_w) : 0;
        s_cbase = tot_b ? atomicAdd(ctr + 1, tot_b) : 0;
    }
    __syncthreads();
    pw += s_wbase;
    pc += s_cbase;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
        const int64_t t = lo + i * kSelThreads + threadIdx.x;
        const uint32_t key = order_key(v[i]);
        const uint32_t b = key >> (32 - kHistBits);
        const unsigned mw = __ballot_sync(0xFFFFFFFFu, t < hi && b > B);
        const unsigned mb = __ballot_sync(0xFFFFFFFFu, t < hi && b == B);
        if (t < hi && b > B) {
            const int pos = pw + __popc(mw & lt);
            if (pos < k) out[pos] = static_cast<int>(t);
        } else if (t < hi && b == B) {
            const int pos = pc + __popc(mb & lt);
            if (pos < kCandCap) cand[pos] = make_uint2(key, static_cast<uint32_t>(t));
        }
        pw += __popc(mw);
        pc += __popc(mb);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = (atomicAdd(ctr + 2, 1) == nch - 1) ? 1 : 0;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // Last CTA of the row: resolve the boundary bin.
    const int above = s_above;
    const int ncand = *reinterpret_cast<volatile int*>(ctr + 1);
    CandSource srcs{cand, min(ncand, kCandCap), ncand > kCandCap ? 2 : 1, src, n, B};
    if (ncand <= kRefineCap) {
        for (int i = threadIdx.x; i < ncand; i += kSelThreads) cbuf[i] = cand[i];
        srcs.buf = cbuf;
        srcs.mode = 0;
    }
    __syncthreads();
    if (srcs.mode == 0 && ncand <= kRankMax)
        rank_select(cbuf, h, ncand, out, above, k - above);
    else
        refine_boundary(srcs, B, out, above, k - above, h, tmp, &s_bin, &s_above, &s_tot);
    __syncthreads();
    for (int i = threadIdx.x; i < kHistBins; i += kSelThreads) ghist[i] = 0;
    if (threadIdx.x < 4) ctr[threadIdx.x] = 0;
}

// ----------------------------------------------------------------- host utilities
static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

WsLayout workspace_layout(int64_t rows, int64_t width, bool with_plan, bool with_logits) {
    WsLayout L{};
    size_t off = 0;
    const size_t r = static_cast<size_t>(rows);
    L.info = off;
    off = align256(off + (with_plan ? 8 * sizeof(int) : 0));
    L.segs = off;
    off = align256(off + (with_plan ? (r + 1) * sizeof(int4) : 0));
    L.seg_prefix = off;
    off = align256(off + (with_plan ? (r + 2) * sizeof(int) : 0));
    L.eff_end = off;
    off = align256(off + (with_plan ? r * sizeof(int) : 0));
    L.cta = off;
    off = align256(off + (with_plan ? kMaxScoreCtas * sizeof(int4) : 0));
    L.hist = off;
    off = align256(off + r * kHistBins * sizeof(unsigned));
    L.counters = off;
    off = align256(off + r * 4 * sizeof(int));
    L.cand = off;
    off = align256(off + r * kCandCap * sizeof(uint2));
    L.logits = off;
    off = align256(off + (with_logits ? r * static_cast<size_t>(width) * sizeof(float) : 0));
    L.total = off;
    return L;
}

int device_sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (!cache[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = n > 0 ? n : 1;
    }
    return cache[dev];
}

CUresult encode_tiled(CUtensorMap* map, CUtensorMapDataType type, cuuint32_t rank, void* addr,
                      const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                      CUtensorMapSwizzle swizzle) {
    using Fn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                            const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                            CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    static Fn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<Fn>(p);
    });
    if (!fn) return CUDA_ERROR_NOT_FOUND;
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return fn(map, type, rank, addr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

int launch_select(const float* logits, float* logits_fill, int64_t ld, int64_t width, const int32_t* ends,
                  int64_t rows, int64_t k, int32_t* out, uint8_t* ws, const WsLayout& L, cudaStream_t stream,
                  bool pdl) {
    SelectArgs a;
    a.logits = logits;
    a.fill = logits_fill;
    a.ld = ld;
    a.width = width;
    a.ends = ends;
    a.k = static_cast<int>(k);
    a.out = out;
    a.hist = reinterpret_cast<unsigned*>(ws + L.hist);
    a.counters = reinterpret_cast<int*>(ws + L.counters);
    a.cand = reinterpret_cast<uint2*>(ws + L.cand);
    const int64_t span = (k > width) ? k : width;
    const int64_t chunks = (span + kChunk - 1) / kChunk;
    if (chunks == 0 || rows == 0) return DSA_OK;
    if (chunks > 65535 || rows > 0x7FFFFFFF) return DSA_ERR_UNSUPPORTED;
    const dim3 grid(static_cast<unsigned>(rows), static_cast<unsigned>(chunks));
    cudaError_t err;
    static bool attr_set[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DSA_ERR_CUDA;
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSelDynSmem) !=
            cudaSuccess)
            return DSA_ERR_CUDA;
        attr_set[dev] = true;
    }
    if (pdl) err = launch_pdl(select_kernel, grid, dim3(kSelThreads), kSelDynSmem, stream, a, 1);
    else {
        select_kernel<<<grid, kSelThreads, kSelDynSmem, stream>>>(a, 0);
        err = cudaGetLastError();
    }
    return err == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace dsa

using namespace dsa;

extern "C" size_t dsa_topk_workspace_size(int64_t rows, int64_t k) {
    (void)k;
    if (rows < 0) return 0;
    return workspace_layout(rows, 0, false, false).total;
}

extern "C" int dsa_topk(const float* logits, int64_t ld, const int32_t* row_ends, int64_t rows, int64_t width,
                        int64_t k, int32_t* out, void* workspace, size_t workspace_bytes, void* stream_) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (rows < 0 || width < 0 || k < 0 || ld < width) return DSA_ERR_INVALID;
    if (rows == 0 || k == 0) return DSA_OK;
    if (!row_ends || !out || !workspace || (width > 0 && !logits)) return DSA_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(workspace) % 256) return DSA_ERR_INVALID;
    if (k > (int64_t(1) << 30) || width > (int64_t(1) << 30)) return DSA_ERR_UNSUPPORTED;
    const WsLayout L = workspace_layout(rows, 0, false, false);
    if (workspace_bytes < L.total) return DSA_ERR_INVALID;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const int64_t chunks = (width + kChunk - 1) / kChunk;
    if (chunks > 65535 || rows > 0x7FFFFFFF) return DSA_ERR_UNSUPPORTED;
    if (chunks > 0) {
        if (launch_pdl(hist_kernel, dim3(static_cast<unsigned>(rows), static_cast<unsigned>(chunks)),
                       dim3(kSelThreads), 0, stream, logits, ld, width, row_ends, static_cast<int>(k),
                       reinterpret_cast<unsigned*>(ws + L.hist)) != cudaSuccess)
            return DSA_ERR_CUDA;
    }
    return launch_select(logits, nullptr, ld, width, row_ends, rows, k, out, ws, L, stream, true);
}

extern "C" const char* dsa_version(void) { return "dsa-gb300 0.1.0"; }

// ----------------------------------------------------------------- top-k without allocation
// Some callers cannot allocate device memory when they call the library: a
// serving engine that reserved nearly all HBM for its KV cache up front and
// forbids further cudaMalloc, or a plugin host that hands a kernel its inputs
// and outputs but no allocator.  dsa_topk_noalloc serves them with scratch that
// lives in this file-scope array instead of a caller workspace.  Every GPU that
// loads the library holds the array until the process exits.
namespace dsa {

constexpr size_t noalloc_align(size_t x) { return (x + 255) & ~size_t(255); }
constexpr size_t kNoAllocBytes = noalloc_align(size_t(DSA_TOPK_NOALLOC_MAX_ROWS) * kHistBins * sizeof(unsigned)) +
                                 noalloc_align(size_t(DSA_TOPK_NOALLOC_MAX_ROWS) * 4 * sizeof(int)) +
                                 noalloc_align(size_t(DSA_TOPK_NOALLOC_MAX_ROWS) * kCandCap * sizeof(uint2));

static __device__ __align__(256) uint8_t g_topk_scratch[kNoAllocBytes];

// Device address of g_topk_scratch on the current device, looked up once per
// device (in host code the array's name is only a stand-in, not an address).
static int noalloc_scratch(uint8_t** ptr) {
    static std::mutex mu;
    static uint8_t* addr[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DSA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_topk_scratch) != cudaSuccess || !p) return DSA_ERR_CUDA;
        addr[dev] = static_cast<uint8_t*>(p);
    }
    *ptr = addr[dev];
    return DSA_OK;
}

}  // namespace dsa

extern "C" int dsa_topk_noalloc(const float* logits, int64_t ld, const int32_t* row_ends, int64_t rows,
                                int64_t width, int64_t k, int32_t* out, void* stream_) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (rows < 0 || width < 0 || k < 0 || ld < width) return DSA_ERR_INVALID;
    if (rows > DSA_TOPK_NOALLOC_MAX_ROWS) return DSA_ERR_UNSUPPORTED;   // past the static scratch
    if (rows == 0 || k == 0) return DSA_OK;
    if (!row_ends || !out || (width > 0 && !logits)) return DSA_ERR_INVALID;
    if (k > (int64_t(1) << 30) || width > (int64_t(1) << 30)) return DSA_ERR_UNSUPPORTED;
    const int64_t chunks = (width + kChunk - 1) / kChunk;
    if (chunks > 65535) return DSA_ERR_UNSUPPORTED;
    uint8_t* ws = nullptr;
    const int rc = noalloc_scratch(&ws);
    if (rc != DSA_OK) return rc;
    const WsLayout L = workspace_layout(rows, 0, false, false);
    if (L.total > kNoAllocBytes) return DSA_ERR_UNSUPPORTED;
    // The array keeps the last call's contents: clear the histograms and counters.
    if (cudaMemsetAsync(ws + L.hist, 0, L.cand - L.hist, stream) != cudaSuccess) return DSA_ERR_CUDA;
    if (chunks > 0) {
        if (launch_pdl(hist_kernel, dim3(static_cast<unsigned>(rows), static_cast<unsigned>(chunks)),
                       dim3(kSelThreads), 0, stream, logits, ld, width, row_ends, static_cast<int>(k),
                       reinterpret_cast<unsigned*>(ws + L.hist)) != cudaSuccess)
            return DSA_ERR_CUDA;
    }
    return launch_select(logits, nullptr, ld, width, row_ends, rows, k, out, ws, L, stream, true);
}
