// Top-k selection over per-row scores (radix select on order-preserving bits).
//
// Page "cutedsl.dsa.overlap": the indexer path is "wq_b -> DsaIndex -> scoring
// and top-k"; page "amd.ops.fp4_indexer", decode_tile_size, budgets per-row
// selection scratch next to the logits.
//
// Level 1 (fused into the scoring epilogue, or hist_kernel here): a 2048-bin
// histogram of the top 11 bits of each row's order-preserving score keys.
// select_kernel gives each span of a row (the whole row unless the batch has
// too few rows to fill the GPU) one 512-thread CTA, two per SM.  A CTA finds
// the level-1 boundary bin B1 (where the count from the top reaches k) and
// streams its span in tiles of 4096 positions, two tiles of loads in flight:
// positions above B1 are winners, positions in B1 are candidates, kept in
// shared memory and counted in a level-2 histogram (key bits 20..10).  A row
// of one span places its winners at once; the spans of a longer row publish
// winners, candidates and level-2 counts to the row's global buffers, and the
// last span to finish (a done counter, no waiting) settles the row.  One pass
// over the candidates places the level-2 winners and keeps the candidates of
// the level-2 boundary bin, which settle the rest (a rank count in one warp
// when they are few, else a level-3 histogram of bits 9..0, equal keys last).
// Positions within the top k come out in no particular order.  Histograms and
// counters are cleared at the end, so the workspace is zero for the next call.
#include <mutex>

#include "host.h"
#include "scan.cuh"

namespace dsa {

constexpr int kSelThreads = 512;
constexpr int kPerThread = 8;                       // values per thread in one tile
constexpr int kChunk = kSelThreads * kPerThread;    // positions per tile (and per hist_kernel CTA)
constexpr int kRefineCap = 3584;   // level-1 candidates kept in shared memory
constexpr int kLevel3Cap = 512;    // level-3 candidates kept in shared memory
constexpr int kWinCap = 4096;      // level-1 winners a CTA buffers in shared memory (k up to this)
constexpr int kRing = 3;           // score tiles in flight per CTA (shared-memory ring)
constexpr int kSpanMin = 2 * kChunk;   // shortest span worth a CTA of its own (rows this long stay whole)
constexpr int kSelDynSmem = kRing * kChunk * sizeof(float) + kRefineCap * sizeof(uint2) +
                            kLevel3Cap * sizeof(uint2) + kWinCap * sizeof(int);

struct SelectArgs {
    const float* logits;
    float* fill;         // when non-null: write -inf at [end, width) of each row
    int64_t ld;
    int64_t width;
    const int32_t* ends;  // row bounds; null: every row holds `width` scores
    int k;               // 0: fill only
    int32_t* out;
    unsigned* hist;      // level-1 histograms, [rows][2048]
    int* counters;       // [rows][4]: winners published, candidates published, spans done, spare
    uint2* cand;         // [rows][kCandCap]: level-1 candidates of split rows (key, position)
    int span;            // positions per CTA, a multiple of kChunk
};

__device__ __forceinline__ int clamp_end(const int32_t* ends, int row, int64_t width) {
    if (!ends) return static_cast<int>(width);   // every row holds width scores
    const int64_t e = ends[row];
    return static_cast<int>(e < 0 ? 0 : (e > width ? width : e));
}

// Finds, over `bins` counts in shared memory, the bin B where the count from
// the top first reaches `need`; stores B and the count strictly above it.
// Leaves both untouched when the counts never reach `need`.
__device__ void find_boundary(const unsigned* h, int bins, int need, int* out_bin, int* out_above, int* tmp) {
    const int per = bins / kSelThreads;   // bins per thread
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

// This thread's four adjacent bins of a 2048-bin histogram, for
// find_boundary4: bins 2048 - 4 (tid + 1) .. 2048 - 4 tid - 1, so that
// thread 0 holds the top four.
static_assert(kHistBins == 4 * kSelThreads, "four histogram bins per thread");
__device__ __forceinline__ uint4 hist_quad(const unsigned* h) {
    return reinterpret_cast<const uint4*>(h)[kHistBins / 4 - 1 - threadIdx.x];
}

// find_boundary over a 2048-bin histogram held as hist_quad in registers.
__device__ void find_boundary4(uint4 q, int need, int* out_bin, int* out_above, int* tmp) {
    const int first = kHistBins - 4 * (threadIdx.x + 1);
    const int c[4] = {static_cast<int>(q.x), static_cast<int>(q.y), static_cast<int>(q.z), static_cast<int>(q.w)};
    const int local = c[0] + c[1] + c[2] + c[3];
    int total;
    const int inc = block_inclusive_scan(local, tmp, &total);
    int cum = inc - local;   // count in bins above this thread's four
#pragma unroll
    for (int j = 3; j >= 0; --j) {
        if (cum < need && cum + c[j] >= need) {
            *out_bin = first + j;
            *out_above = cum;
        }
        cum += c[j];
    }
}

// Position for this lane among the lanes of its warp where `pred` holds, the
// warp's run taken from `counter` with one atomic; -1 where `pred` is false.
// Every lane of the warp must call it.
__device__ __forceinline__ int warp_slot(bool pred, int* counter) {
    const unsigned m = __ballot_sync(0xFFFFFFFFu, pred);
    if (m == 0) return -1;
    const int lane = threadIdx.x & 31;
    const int leader = __ffs(m) - 1;
    int base = 0;
    if (lane == leader) base = atomicAdd(counter, __popc(m));
    base = __shfl_sync(0xFFFFFFFFu, base, leader);
    return pred ? base + __popc(m & ((1u << lane) - 1u)) : -1;
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

// The level-1 candidates of a row (keys in bin B1): a buffer of `count`
// (key, position) pairs in shared or global memory, or, when the buffer
// overflowed, the row itself filtered by bin.  for_each calls f(valid, key,
// position) with the same trip count on every lane of a warp.
struct CandSource {
    const uint2* buf;   // nullptr: re-read the row
    int count;
    const float* row;
    int n;
    uint32_t b1;
    template <typename F>
    __device__ __forceinline__ void for_each(F&& f) const {
        const int lane = threadIdx.x & 31;
        const int w0 = threadIdx.x - lane;
        if (buf) {
            constexpr int U = 4;
            for (int base = w0; base < count; base += kSelThreads * U) {
                uint2 c[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int i = base + u * kSelThreads + lane;
                    c[u] = i < count ? buf[i] : make_uint2(0u, 0u);
                }
#pragma unroll
                for (int u = 0; u < U; ++u)
                    f(base + u * kSelThreads + lane < count, c[u].x, static_cast<int>(c[u].y));
            }
        } else {
            constexpr int U = 8;
            for (int base = w0; base < n; base += kSelThreads * U) {
                float x[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int t = base + u * kSelThreads + lane;
                    x[u] = t < n ? row[t] : 0.0f;
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int t = base + u * kSelThreads + lane;
                    const uint32_t key = order_key(x[u]);
                    f(t < n && (key >> (32 - kHistBits)) == b1, key, t);
                }
            }
        }
    }
};

// Top `need` of n3 <= 32 level-3 candidates by one warp: rank(c) = the
// candidates with a larger key, plus equal keys earlier in the list.
__device__ __forceinline__ void warp_rank_select(const uint2* c3, int n3, int32_t* out, int base, int need, int k) {
    const int lane = threadIdx.x & 31;
    const uint2 me = lane < n3 ? c3[lane] : make_uint2(0u, 0u);
    int rank = 0;
    for (int j = 0; j < n3; ++j) {
        const uint32_t kj = __shfl_sync(0xFFFFFFFFu, me.x, j);
        rank += (kj > me.x || (kj == me.x && j < lane)) ? 1 : 0;
    }
    if (lane < n3 && rank < need && base + rank < k) out[base + rank] = static_cast<int>(me.y);
}

__global__ void __launch_bounds__(kSelThreads, 2) select_kernel(const SelectArgs a, int pdl) {
    __shared__ unsigned h1[kHistBins];   // level-1 histogram, then level 3
    __shared__ __align__(16) unsigned h2[kHistBins];   // level-2 histogram (read as uint4)
    __shared__ int tmp[32];
    __shared__ int s_b1, s_a1, s_b2, s_a2, s_b3, s_a3;
    __shared__ int s_wc[2];   // level-1 winners and candidates placed
    __shared__ int s_w2, s_c3, s_w3, s_tie, s_last, s_wbase, s_cbase;
    extern __shared__ float4 sel_dyn[];
    float4* ring = sel_dyn;                                                    // kRing tiles of scores
    uint2* cbuf = reinterpret_cast<uint2*>(sel_dyn + kRing * kChunk / 4);     // level-1 candidates
    uint2* c3buf = cbuf + kRefineCap;                                          // level-3 candidates
    int* wbuf = reinterpret_cast<int*>(c3buf + kLevel3Cap);                    // level-1 winners
    if (pdl) pdl_wait();
    const int row = blockIdx.x;
    const int64_t lo = static_cast<int64_t>(blockIdx.y) * a.span;
    const int k = a.k;
    unsigned* ghist = a.hist + static_cast<int64_t>(row) * kHistBins;
    int* ctr = a.counters + static_cast<int64_t>(row) * 4;
    uint2* gcand = a.cand + static_cast<int64_t>(row) * kCandCap;
    const float* src = a.logits + static_cast<int64_t>(row) * a.ld;
    const int lane = threadIdx.x & 31;
    const int lo32 = static_cast<int>(lo);

    // ---- level 1: the row's histogram, then the span in tiles through a
    // ring of kRing tiles in shared memory.  Each thread copies, and later
    // reads, the same 8 scores of a tile: positions base + 4 * tid + j and
    // base + kChunk / 2 + 4 * tid + j (j < 4), so no barrier guards the ring.
    const bool vec = (reinterpret_cast<uintptr_t>(src) & 15) == 0;
    auto issue_tile = [&](int i, int bound) {   // tile i of the span into ring slot i % kRing, up to `bound`
        const int base = lo32 + i * kChunk;
        float4* slot = ring + (i % kRing) * (kChunk / 4);
#pragma unroll
        for (int h = 0; h < 2 && base < bound; ++h) {
            const int p = base + h * (kChunk / 2) + 4 * threadIdx.x;
            const int avail = max(0, min(4, bound - p));
            float4* d = slot + h * (kChunk / 8) + threadIdx.x;
            if (vec) {
                cp_async16(d, avail ? src + p : src, 4u * avail);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    cp_async4(reinterpret_cast<float*>(d) + j, j < avail ? src + p + j : src, j < avail ? 4u : 0u);
            }
        }
        cp_async_commit();
    };
    // The row's histogram does not depend on the row's bound: it goes out
    // together with the bound's load, and so do the first tiles of the row's
    // first span (the one span that is needed whenever the row is longer than
    // k), read up to the end of the span within the row's width; positions
    // past the bound are never classified.  Later spans may lie past the
    // bound and wait for it.
    uint4 hq1 = make_uint4(0u, 0u, 0u, 0u);
    const bool early = k > 0 && blockIdx.y == 0;
    if (k > 0) hq1 = hist_quad(ghist);
    if (early) {
        const int wend = static_cast<int>(min(a.width, lo + a.span));
#pragma unroll
        for (int i = 0; i < kRing; ++i) issue_tile(i, wend);
    }
    const int n = clamp_end(a.ends, row, a.width);
    if (a.fill) {
        float* dst = a.fill + static_cast<int64_t>(row) * a.ld;
        const int64_t hi = min(a.width, lo + a.span);
        for (int64_t t = max(lo, static_cast<int64_t>(n)) + threadIdx.x; t < hi; t += kSelThreads)
            dst[t] = -__int_as_float(0x7F800000);
    }
    if (k <= 0) return;
    int32_t* out = a.out + static_cast<int64_t>(row) * k;
    if (n <= k) {
        cp_async_wait<0>();   // no copy into this CTA's ring may outlive it
        const int64_t hi = min(static_cast<int64_t>(k), lo + a.span);
        for (int64_t pos = lo + threadIdx.x; pos < hi; pos += kSelThreads) out[pos] = pos < n ? static_cast<int>(pos) : -1;
        return;
    }
    const int nsp = static_cast<int>((n + a.span - 1) / a.span);
    if (static_cast<int>(blockIdx.y) >= nsp) {
        cp_async_wait<0>();
        return;
    }
    const bool split = nsp > 1;
    const int hi = static_cast<int>(min(static_cast<int64_t>(n), lo + a.span));
    if (!early) {
#pragma unroll
        for (int i = 0; i < kRing; ++i) issue_tile(i, hi);
    }
    // Winners wait in shared memory (written out coalesced after the pass)
    // when k allows; else they go straight to the output.
    const bool wbuffered = k <= kWinCap;
    if (!split)   // a split row's last span builds its level-2 histogram from scratch
        for (int i = threadIdx.x; i < kHistBins; i += kSelThreads) h2[i] = 0;
    if (threadIdx.x == 0) {
        s_b1 = 0; s_a1 = 0; s_b2 = 0; s_a2 = 0; s_b3 = 0; s_a3 = 0;
        s_wc[0] = 0; s_wc[1] = 0; s_w2 = 0; s_c3 = 0; s_w3 = 0; s_tie = 0;
    }
    __syncthreads();
    find_boundary4(hq1, k, &s_b1, &s_a1, tmp);
    __syncthreads();
    const uint32_t B1 = static_cast<uint32_t>(s_b1);
    const int above1 = s_a1;
    const uint32_t kwin = (B1 + 1u) << (32 - kHistBits);   // keys >= kwin: winners (0 when B1 is the top bin)
    const uint32_t kcand = B1 << (32 - kHistBits);         // keys in [kcand, kwin): candidates
    const bool top_bin = B1 == kHistBins - 1;
    // Classifies tile i (waiting for this thread's copies of it), then reuses
    // its slot for tile i + kRing.  Bit u of wm / cm marks value u as a winner
    // (key > kw) / candidate (kcand <= key <= kw); the warp's runs come from
    // one scan of both counts and one shared 64-bit add of both, and only
    // marked values are placed.
    const uint32_t kw = top_bin ? 0xFFFFFFFFu : kwin - 1u;
    const uint32_t crange = kw - kcand;
    const bool pos_bounds = kcand >= 0x80000000u;   // the level-1 bin lies at or above +0
    const int tw = static_cast<int>(kw & 0x7FFFFFFFu);   // winners: bits above, as a signed integer
    const uint32_t tc = kcand & 0x7FFFFFFFu;            // candidates: bits in [tc, tc + crange]
    const int ntiles = (hi - lo32 + kChunk - 1) / kChunk;
    const float* ringf = reinterpret_cast<const float*>(ring);
    for (int i = 0; i < ntiles; ++i) {
        cp_async_wait<kRing - 1>();
        const int base = lo32 + i * kChunk;
        const int slot = (i % kRing) * kChunk;   // float offset of the slot
        const float4 va = ring[slot / 4 + threadIdx.x], vb = ring[slot / 4 + kChunk / 8 + threadIdx.x];
        const float x[kPerThread] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
        uint32_t wm = 0, cm = 0;
        if (pos_bounds) {
            // Both bounds among non-negative scores: the raw bits order those
            // as the key does, and every score with the sign bit set lies
            // below them (as a signed integer, or past kw unsigned).
#pragma unroll
            for (int u = 0; u < kPerThread; ++u) {
                const uint32_t b = __float_as_uint(x[u]);
                if (static_cast<int>(b) > tw) wm |= 1u << u;
                if (b - tc <= crange) cm |= 1u << u;
            }
        } else {
#pragma unroll
            for (int u = 0; u < kPerThread; ++u) {
                const uint32_t key = order_key(x[u]);
                if (key > kw) wm |= 1u << u;
                if (key - kcand <= crange) cm |= 1u << u;
            }
        }
        if (base + kChunk > hi) {   // last, partial tile: drop positions past the end
            uint32_t inm = 0;
#pragma unroll
            for (int u = 0; u < kPerThread; ++u)
                if (base + (u >> 2) * (kChunk / 2) + 4 * threadIdx.x + (u & 3) < hi) inm |= 1u << u;
            wm &= inm;
            cm &= inm;
        }
        const int cw = __popc(wm), cc = __popc(cm);
        int inc = (cw << 16) | cc;   // both counts stay below 2^16
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, inc, d);
            if (lane >= d) inc += y;
        }
        // Lanes 30 and 31 reserve the warp's runs of winners and candidates with
        // one shared add each (one instruction, two counters).
        const int tot = __shfl_sync(0xFFFFFFFFu, inc, 31);
        const int want = lane == 30 ? tot >> 16 : (tot & 0xFFFF);
        int o = 0;
        if (lane >= 30 && want) o = atomicAdd(&s_wc[lane - 30], want);
        int pw = __shfl_sync(0xFFFFFFFFu, o, 30) + (inc >> 16) - cw;
        int pc = __shfl_sync(0xFFFFFFFFu, o, 31) + (inc & 0xFFFF) - cc;
        const int tb = base + 4 * threadIdx.x;   // position of value 0 of this thread
        if (wbuffered) {
            // predicated over the 8 values: no loop as long as the warp's busiest lane.
            // A row has fewer than k <= kWinCap winners, so the bound is tested once
            // (it only fails when the histogram disagreed with the scores).
            if (pw + cw <= kWinCap) {
#pragma unroll
                for (int u = 0; u < kPerThread; ++u)
                    if ((wm >> u) & 1u) wbuf[pw++] = tb + (u >> 2) * (kChunk / 2) + (u & 3);
            } else {
#pragma unroll
                for (int u = 0; u < kPerThread; ++u) {
                    if ((wm >> u) & 1u) {
                        if (pw < kWinCap) wbuf[pw] = tb + (u >> 2) * (kChunk / 2) + (u & 3);
                        ++pw;
                    }
                }
            }
            wm = 0;
        }
        while (wm) {
            const int u = __ffs(wm) - 1;
            wm &= wm - 1u;
            const int t = tb + (u >> 2) * (kChunk / 2) + (u & 3);
            if (!split) {
                if (pw < k) out[pw] = t;
            } else {
                const int g = atomicAdd(ctr + 0, 1);
                if (g < k) out[g] = t;
            }
            ++pw;
        }
        while (cm) {
            const int u = __ffs(cm) - 1;
            cm &= cm - 1u;
            const int off = (u >> 2) * (kChunk / 2) + (u & 3);
            const uint32_t key = order_key(ringf[slot + 4 * threadIdx.x + off]);
            if (!split) atomicAdd(&h2[(key >> 10) & 0x7FF], 1u);   // a split row's last span counts them all
            if (pc < kRefineCap) cbuf[pc] = make_uint2(key, static_cast<uint32_t>(tb + off));
            ++pc;
        }
        issue_tile(i + kRing, hi);   // this thread is done with the slot
    }
    cp_async_wait<0>();
    __syncthreads();
    const int nwin = s_wc[0], mycand = s_wc[1];
    int ncand = mycand;
    const uint2* cand_src = ncand <= kRefineCap ? cbuf : nullptr;
    if (!split && wbuffered)
        for (int i = threadIdx.x; i < nwin; i += kSelThreads)
            if (i < k) out[i] = wbuf[i];
    if (split) {
        // Publish this span's winners, candidates and level-2 counts; the last
        // span of the row to finish reads the row's totals back and settles it.
        if (threadIdx.x == 0) {
            s_wbase = (wbuffered && nwin) ? atomicAdd(ctr + 0, nwin) : 0;
            s_cbase = mycand ? atomicAdd(ctr + 1, mycand) : 0;
        }
        __syncthreads();
        if (wbuffered)
            for (int i = threadIdx.x; i < nwin; i += kSelThreads)
                if (s_wbase + i < k) out[s_wbase + i] = wbuf[i];
        if (ncand <= kRefineCap)
            for (int i = threadIdx.x; i < ncand; i += kSelThreads)
                if (s_cbase + i < kCandCap) gcand[s_cbase + i] = cbuf[i];
        if (threadIdx.x == 0 && ncand > kRefineCap) atomicAdd(ctr + 3, 1);   // candidates dropped
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            s_last = (atomicAdd(ctr + 2, 1) == nsp - 1) ? 1 : 0;
        }
        __syncthreads();
        if (!s_last) return;
        __threadfence();
        ncand = *reinterpret_cast<volatile int*>(ctr + 1);
        const bool dropped = *reinterpret_cast<volatile int*>(ctr + 3) != 0;
        cand_src = (!dropped && ncand <= kCandCap) ? gcand : nullptr;
        // The row's level-2 counts, from every span's candidates (or from the
        // row itself when a candidate buffer overflowed).
        for (int i = threadIdx.x; i < kHistBins; i += kSelThreads) h2[i] = 0;
        __syncthreads();
        const CandSource all{cand_src, ncand, src, n, B1};
        all.for_each([&](bool valid, uint32_t kk, int) {
            if (valid) atomicAdd(&h2[(kk >> 10) & 0x7FF], 1u);
        });
    }
    for (int i = threadIdx.x; i < kHistBins; i += kSelThreads) h1[i] = 0;   // level 3 from here on
    __syncthreads();

    // ---- level 2: one pass over the candidates
    const int need = k - above1;
    find_boundary4(hist_quad(h2), need, &s_b2, &s_a2, tmp);
    __syncthreads();
    const uint32_t B2 = static_cast<uint32_t>(s_b2);
    const int above2 = s_a2;
    const CandSource cs{cand_src, ncand, src, n, B1};
    const int base2 = above1, base3 = above1 + above2;
    cs.for_each([&](bool valid, uint32_t kk, int t) {
        if (!__any_sync(0xFFFFFFFFu, valid)) return;   // uniform over the warp
        const uint32_t b2 = (kk >> 10) & 0x7FF;
        const int pw = warp_slot(valid && b2 > B2, &s_w2);
        if (pw >= 0 && base2 + pw < k) out[base2 + pw] = t;
        const bool c3 = valid && b2 == B2;
        const int pc = warp_slot(c3, &s_c3);
        if (c3) {
            atomicAdd(&h1[kk & 0x3FF], 1u);
            if (pc < kLevel3Cap) c3buf[pc] = make_uint2(kk, static_cast<uint32_t>(t));
        }
    });
    __syncthreads();

    // ---- level 3 and equal keys
    const int need2 = need - above2;
    const int n3 = s_c3;
    int placed;
    if (n3 <= 32) {
        // few enough to rank in one warp (their keys agree on bits 31..10)
        if (threadIdx.x < 32) warp_rank_select(c3buf, n3, out, base3, need2, k);
        placed = base3 + min(n3, need2);
    } else {
        find_boundary(h1, 1024, need2, &s_b3, &s_a3, tmp);
        __syncthreads();
        const uint32_t B3 = static_cast<uint32_t>(s_b3);
        const int above3 = s_a3;
        const int left = need2 - above3;   // equal keys to take
        auto level3 = [&](bool valid, uint32_t kk, int t) {
            const uint32_t b3 = kk & 0x3FF;
            const int pw = warp_slot(valid && b3 > B3, &s_w3);
            if (pw >= 0 && base3 + pw < k) out[base3 + pw] = t;
            const int pt = warp_slot(valid && b3 == B3, &s_tie);
            if (pt >= 0 && pt < left && base3 + above3 + pt < k) out[base3 + above3 + pt] = t;
        };
        if (n3 <= kLevel3Cap) {
            const CandSource c3s{c3buf, n3, src, n, B1};
            c3s.for_each(level3);
        } else {
            cs.for_each([&](bool valid, uint32_t kk, int t) { level3(valid && ((kk >> 10) & 0x7FF) == B2, kk, t); });
        }
        __syncthreads();
        placed = base3 + above3 + min(s_tie, left);
    }
    // Short only when the histogram disagreed with the scores (an aborted scoring pass).
    for (int e = placed + threadIdx.x; e < k; e += kSelThreads) out[e] = -1;
    for (int i = threadIdx.x; i < kHistBins; i += kSelThreads) ghist[i] = 0;
    if (split && threadIdx.x < 4) ctr[threadIdx.x] = 0;
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
    if (rows == 0 || (k == 0 && (!logits_fill || width == 0))) return DSA_OK;
    if (rows > 0x7FFFFFFF) return DSA_ERR_UNSUPPORTED;
    // Span per CTA: about four CTAs per SM over rows x width, a multiple of
    // kChunk, at least kSpanMin positions (rows that short stay whole: a split
    // row pays for its merge) -- unless spans of kSpanMin would leave fewer
    // CTAs than SMs (a few long rows), when spans go down to kChunk.
    const int64_t sms = device_sm_count();
    const int64_t target = 4 * sms;
    int64_t span = (rows * width + target - 1) / target;
    const bool few = width > kSpanMin && rows * ((width + kSpanMin - 1) / kSpanMin) < sms;
    const int64_t span_min = few ? kChunk : kSpanMin;
    span = span < span_min ? span_min : span;
    span = (span + kChunk - 1) / kChunk * kChunk;
    if (span > (int64_t(1) << 30)) span = int64_t(1) << 30;
    a.span = static_cast<int>(span);
    const int64_t reach = (k > width) ? k : width;
    const int64_t spans = (reach + span - 1) / span;
    if (spans > 65535) return DSA_ERR_UNSUPPORTED;
    const dim3 grid(static_cast<unsigned>(rows), static_cast<unsigned>(spans > 0 ? spans : 1));
    cudaError_t err;
    static bool attr_set[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DSA_ERR_CUDA;
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSelDynSmem) !=
                cudaSuccess ||
            cudaFuncSetAttribute(select_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared) != cudaSuccess)
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
// A 2048-bin histogram per row (8 KB), 16 bytes of counters per row and 8192
// candidates of 8 bytes per split row (64 KB): with 64 rows 512 KB + 1 KB + 4 MB.
constexpr size_t kNoAllocBytes = noalloc_align(size_t(DSA_TOPK_NOALLOC_MAX_ROWS) * kHistBins * sizeof(unsigned)) +
                                 noalloc_align(size_t(DSA_TOPK_NOALLOC_MAX_ROWS) * 4 * sizeof(int)) +
                                 noalloc_align(size_t(DSA_TOPK_NOALLOC_MAX_ROWS) * kCandCap * sizeof(uint2));
static_assert(kNoAllocBytes == DSA_TOPK_NOALLOC_SCRATCH_BYTES, "the header states the array's size");

static __device__ __align__(256) uint8_t g_topk_scratch[kNoAllocBytes];

// Device address of g_topk_scratch on the current device.  In host code the
// array's name is only a stand-in, not an address.  The lookup is made on
// every call: it is a host-side query that allocates nothing, and a cached
// address would go stale if the device's context were reset (the module is
// then loaded again, possibly elsewhere).  The first lookup on a device loads
// the library's device code there.
static int noalloc_scratch(uint8_t** ptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_topk_scratch) != cudaSuccess || !p) return DSA_ERR_CUDA;
    *ptr = static_cast<uint8_t*>(p);
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

// ----------------------------------------------------------------- DCP top-k merge
// Page "cutedsl.dsa.overlap": under DCP the indexer path ends with the top-k
// merge and the local slots.  Each row holds every rank's local top-k
// candidates (rank w's at columns w*k .. w*k + k - 1: scores, rank-local
// positions); the select above picks the k_out best columns, and this kernel
// turns a column into the candidate's global key position (and, for one
// rank, its rank-local slot when that rank owns it).
namespace dsa {

__global__ void __launch_bounds__(256) merge_positions_kernel(int32_t* __restrict__ out, int64_t rows, int64_t k_out,
                                                              const int32_t* __restrict__ idx, int64_t idx_ld,
                                                              int64_t k, int64_t world, int64_t inter, int64_t rank,
                                                              int32_t* __restrict__ out_local) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= rows * k_out) return;
    const int64_t r = i / k_out;
    const int c = out[i];
    int64_t g = -1;
    if (c >= 0) {
        const int64_t l = idx[r * idx_ld + c];
        if (l >= 0) g = (l / inter) * (world * inter) + (c / k) * inter + l % inter;
    }
    out[i] = static_cast<int32_t>(g);
    if (out_local) {
        const bool mine = g >= 0 && (g / inter) % world == rank;
        out_local[i] = mine ? static_cast<int32_t>((g / (world * inter)) * inter + g % inter) : -1;
    }
}

}  // namespace dsa

extern "C" int dsa_topk_merge(const float* scores, int64_t scores_ld, const int32_t* idx, int64_t idx_ld,
                              int64_t rows, int64_t world, int64_t k, int64_t interleave, int64_t k_out,
                              int32_t* out, int64_t rank, int32_t* out_local, void* workspace,
                              size_t workspace_bytes, void* stream_) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (rows < 0 || world < 1 || k < 0 || interleave < 1 || k_out < 0) return DSA_ERR_INVALID;
    if (rows == 0 || k_out == 0) return DSA_OK;
    const int64_t width = world * k;
    if (scores_ld < width || idx_ld < width) return DSA_ERR_INVALID;
    if (!out || !workspace || (width > 0 && (!scores || !idx))) return DSA_ERR_INVALID;
    if (out_local && (rank < 0 || rank >= world)) return DSA_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(workspace) % 256) return DSA_ERR_INVALID;
    if (k_out > (int64_t(1) << 30) || width > (int64_t(1) << 30) || interleave > (int64_t(1) << 30) ||
        world > (int64_t(1) << 20))
        return DSA_ERR_UNSUPPORTED;
    const WsLayout L = workspace_layout(rows, 0, false, false);
    if (workspace_bytes < L.total) return DSA_ERR_INVALID;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const int64_t chunks = (width + kChunk - 1) / kChunk;
    if (chunks > 65535 || rows > 0x7FFFFFFF) return DSA_ERR_UNSUPPORTED;
    if (chunks > 0) {
        if (launch_pdl(hist_kernel, dim3(static_cast<unsigned>(rows), static_cast<unsigned>(chunks)),
                       dim3(kSelThreads), 0, stream, scores, scores_ld, width, static_cast<const int32_t*>(nullptr),
                       static_cast<int>(k_out), reinterpret_cast<unsigned*>(ws + L.hist)) != cudaSuccess)
            return DSA_ERR_CUDA;
    }
    int rc = launch_select(scores, nullptr, scores_ld, width, nullptr, rows, k_out, out, ws, L, stream, true);
    if (rc != DSA_OK) return rc;
    const int64_t n = rows * k_out;
    const int64_t blocks = (n + 255) / 256;
    if (blocks > 0x7FFFFFFF) return DSA_ERR_UNSUPPORTED;
    return launch_pdl(merge_positions_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, out, rows,
                      k_out, idx, idx_ld, k, world, interleave, out_local ? rank : int64_t(0), out_local) ==
                   cudaSuccess
               ? DSA_OK
               : DSA_ERR_CUDA;
}
