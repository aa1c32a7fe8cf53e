// Block-wide prefix sums for the single-CTA bookkeeping kernels.
#pragma once

#include "common.cuh"

namespace dsa {

// Inclusive scan of one int per thread over a block of up to 1024 threads.
// `warp_tmp` is shared scratch of 32 ints.  Returns the inclusive prefix; the
// block total is written to *total, which must be shared memory (all threads
// read it after the call; one thread writes it).
__device__ __forceinline__ int block_inclusive_scan(int v, int* warp_tmp, int* total) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int o = __shfl_up_sync(0xFFFFFFFFu, v, d);
        if (lane >= d) v += o;
    }
    if (lane == 31) warp_tmp[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int s = (lane < nwarps) ? warp_tmp[lane] : 0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int o = __shfl_up_sync(0xFFFFFFFFu, s, d);
            if (lane >= d) s += o;
        }
        warp_tmp[lane] = s;   // inclusive prefix over warps
        if (lane == 31) *total = s;
    }
    __syncthreads();
    const int before = (warp > 0) ? warp_tmp[warp - 1] : 0;
    const int result = v + before;
    __syncthreads();   // warp_tmp may be reused by the caller's next scan
    return result;
}

// Two inclusive scans (of a and of b) over the block with one set of
// barriers; `warp_tmp` holds 64 ints, totals go to total_a / total_b (shared).
__device__ __forceinline__ void block_inclusive_scan2(int& a, int& b, int* warp_tmp, int* total_a, int* total_b) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int oa = __shfl_up_sync(0xFFFFFFFFu, a, d);
        const int ob = __shfl_up_sync(0xFFFFFFFFu, b, d);
        if (lane >= d) {
            a += oa;
            b += ob;
        }
    }
    if (lane == 31) {
        warp_tmp[warp] = a;
        warp_tmp[32 + warp] = b;
    }
    __syncthreads();
    if (warp == 0) {
        int sa = (lane < nwarps) ? warp_tmp[lane] : 0;
        int sb = (lane < nwarps) ? warp_tmp[32 + lane] : 0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int oa = __shfl_up_sync(0xFFFFFFFFu, sa, d);
            const int ob = __shfl_up_sync(0xFFFFFFFFu, sb, d);
            if (lane >= d) {
                sa += oa;
                sb += ob;
            }
        }
        warp_tmp[lane] = sa;
        warp_tmp[32 + lane] = sb;
        if (lane == 31) {
            *total_a = sa;
            *total_b = sb;
        }
    }
    __syncthreads();
    if (warp > 0) {
        a += warp_tmp[warp - 1];
        b += warp_tmp[32 + warp - 1];
    }
    __syncthreads();   // warp_tmp may be reused by the caller's next scan
}

}  // namespace dsa
