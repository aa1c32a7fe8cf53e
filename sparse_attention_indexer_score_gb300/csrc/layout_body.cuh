// Request grouping and causal key bounds of the decode step's query rows, as
// a block-wide device function (one CTA, any multiple of 32 threads), shared
// by decode_layout_kernel and the fused step-preparation kernel.
//
// Page "amd.ops.fp4_indexer", decode_layout: starts = [0, cumsum(query_lens)];
// row r belongs to the request searchsorted(starts[1:], r, right=True) capped at
// R - 1, and scores keys t < max(0, seq_len - query_len + (r - start) + 1);
// rows at or past starts[R] are padding with bound 0.  Under DCP (world > 1)
// key runs of `interleave` positions go to the ranks round-robin and the bound
// becomes the number of the rank's own keys below it: with
// full = E / (world * interleave) * interleave,
// E_local = full + clamp(E - full * world - rank * interleave, 0, interleave).
#pragma once

#include "scan.cuh"

namespace dsa {

// Requests up to which the row-to-request search and the per-request offsets
// stay in shared memory (12 KB, which keeps a 256-thread step-preparation
// block at eight per SM); more requests read them from global memory.
constexpr int kLayoutSmemReq = 1024;

__device__ __forceinline__ void decode_layout_block(const int32_t* __restrict__ seq_lens,
                                                    const int32_t* __restrict__ query_lens, int num_req,
                                                    int64_t num_rows, int32_t* __restrict__ starts,
                                                    int32_t* __restrict__ row_ends, int64_t dcp_rank = 0,
                                                    int64_t dcp_world = 1, int64_t interleave = 1) {
    __shared__ int warp_tmp[32];
    __shared__ int chunk_total;
    __shared__ int s_starts[kLayoutSmemReq + 1];     // starts[1 .. R] when the requests fit
    __shared__ long long s_off[kLayoutSmemReq];      // seq_len - query_len - start + 1 of each request
    const bool fit = num_req <= kLayoutSmemReq;
    int carry = 0;
    if (threadIdx.x == 0) starts[0] = 0;
    for (int base = 0; base < num_req; base += blockDim.x) {
        const int i = base + threadIdx.x;
        const int v = (i < num_req) ? query_lens[i] : 0;
        const int sl = (fit && i < num_req) ? seq_lens[i] : 0;
        const int inc = block_inclusive_scan(v, warp_tmp, &chunk_total);
        if (i < num_req) {
            starts[i + 1] = carry + inc;
            if (fit) {
                s_starts[i + 1] = carry + inc;
                s_off[i] = static_cast<long long>(sl) - v - (carry + inc - v) + 1;
            }
        }
        carry += chunk_total;
        __syncthreads();
    }
    __syncthreads();
    const int last = carry;   // starts[R]
    for (int64_t r = threadIdx.x; r < num_rows; r += blockDim.x) {
        int end = 0;
        if (num_req > 0 && r < last) {
            // first q with starts[q + 1] > r  (searchsorted right on starts[1:])
            int lo = 0, hi = num_req;
            int64_t e;
            if (fit) {
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (static_cast<int64_t>(s_starts[mid + 1]) > r) hi = mid; else lo = mid + 1;
                }
                e = s_off[min(lo, num_req - 1)] + r;
            } else {
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (static_cast<int64_t>(starts[mid + 1]) > r) hi = mid; else lo = mid + 1;
                }
                const int q = min(lo, num_req - 1);
                e = static_cast<int64_t>(seq_lens[q]) - query_lens[q] + (r - starts[q]) + 1;
            }
            e = e > 0 ? e : 0;
            if (dcp_world > 1) {
                const int64_t full = e / (dcp_world * interleave) * interleave;
                const int64_t part = e - full * dcp_world - dcp_rank * interleave;
                e = full + (part < 0 ? 0 : (part > interleave ? interleave : part));
            }
            end = static_cast<int>(e);
        }
        row_ends[r] = end;
    }
}

}  // namespace dsa
