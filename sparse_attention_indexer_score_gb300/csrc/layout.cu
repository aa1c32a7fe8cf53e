// Request grouping and causal key bounds of the decode step's query rows.
//
// Page "amd.ops.fp4_indexer", decode_layout: starts = [0, cumsum(query_lens)];
// row r belongs to the request searchsorted(starts[1:], r, right=True) capped at
// R - 1, and scores keys t < max(0, seq_len - query_len + (r - start) + 1);
// rows at or past starts[R] are padding with bound 0.  No device-to-host
// reads: one CTA scans the query lengths, then bounds every row.
#include "host.h"
#include "scan.cuh"

namespace dsa {

__global__ void __launch_bounds__(1024) decode_layout_kernel(const int32_t* __restrict__ seq_lens,
                                                             const int32_t* __restrict__ query_lens, int num_req,
                                                             int64_t num_rows, int32_t* __restrict__ starts,
                                                             int32_t* __restrict__ row_ends) {
    __shared__ int warp_tmp[32];
    __shared__ int chunk_total;
    pdl_launch_dependents();
    pdl_wait();
    int carry = 0;
    if (threadIdx.x == 0) starts[0] = 0;
    for (int base = 0; base < num_req; base += blockDim.x) {
        const int i = base + threadIdx.x;
        const int v = (i < num_req) ? query_lens[i] : 0;
        const int inc = block_inclusive_scan(v, warp_tmp, &chunk_total);
        if (i < num_req) starts[i + 1] = carry + inc;
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
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (static_cast<int64_t>(starts[mid + 1]) > r) hi = mid; else lo = mid + 1;
            }
            const int q = min(lo, num_req - 1);
            const int64_t e = static_cast<int64_t>(seq_lens[q]) - query_lens[q] + (r - starts[q]) + 1;
            end = static_cast<int>(e > 0 ? e : 0);
        }
        row_ends[r] = end;
    }
}

}  // namespace dsa

using namespace dsa;

extern "C" int dsa_decode_layout(const int32_t* seq_lens, int64_t num_seq, const int32_t* query_lens,
                                 int64_t num_requests, int64_t num_rows, int32_t* starts, int32_t* row_ends,
                                 void* stream) {
    if (num_rows < 0 || num_requests < 0 || num_seq < num_requests) return DSA_ERR_INVALID;
    if (num_requests > 0x7FFFFFFF - 1 || num_rows > 0x7FFFFFFF) return DSA_ERR_UNSUPPORTED;
    if (!starts || (num_rows > 0 && !row_ends) || (num_requests > 0 && (!seq_lens || !query_lens)))
        return DSA_ERR_INVALID;
    const cudaError_t err = launch_pdl(decode_layout_kernel, dim3(1), dim3(1024), 0, static_cast<cudaStream_t>(stream),
                                       seq_lens, query_lens, static_cast<int>(num_requests), num_rows, starts,
                                       row_ends);
    return err == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
