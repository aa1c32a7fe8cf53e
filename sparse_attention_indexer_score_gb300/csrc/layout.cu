// Request grouping and causal key bounds of the decode step's query rows.
//
// Page "amd.ops.fp4_indexer", decode_layout (the definition is restated in
// layout_body.cuh).  No device-to-host reads: one CTA scans the query lengths,
// then bounds every row.
#include "host.h"
#include "layout_body.cuh"

namespace dsa {

__global__ void __launch_bounds__(1024) decode_layout_kernel(const int32_t* __restrict__ seq_lens,
                                                             const int32_t* __restrict__ query_lens, int num_req,
                                                             int64_t num_rows, int32_t* __restrict__ starts,
                                                             int32_t* __restrict__ row_ends, int64_t dcp_rank,
                                                             int64_t dcp_world, int64_t interleave) {
    pdl_launch_dependents();
    pdl_wait();
    decode_layout_block(seq_lens, query_lens, num_req, num_rows, starts, row_ends, dcp_rank, dcp_world, interleave);
}

}  // namespace dsa

using namespace dsa;

extern "C" int dsa_decode_layout(const int32_t* seq_lens, int64_t num_seq, const int32_t* query_lens,
                                 int64_t num_requests, int64_t num_rows, int32_t* starts, int32_t* row_ends,
                                 void* stream) {
    if (num_rows < 0 || num_requests < 0 || num_seq < num_requests) return DSA_ERR_INVALID;
    if (num_requests > 0x7FFFFFFF - 1 || num_rows > 0x7FFFFFFF) return DSA_ERR_UNSUPPORTED;
    if (!starts || (num_rows > 0 && !row_ends) || (num_requests > 0 && (!seq_lens || !query_lens)))
        return DSA_ERR_INVALID;   // (the same checks as dsa_prepare_step's layout part)
    const cudaError_t err = launch_pdl(decode_layout_kernel, dim3(1), dim3(1024), 0, static_cast<cudaStream_t>(stream),
                                       seq_lens, query_lens, static_cast<int>(num_requests), num_rows, starts,
                                       row_ends, int64_t(0), int64_t(1), int64_t(1));
    return err == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

extern "C" int dsa_decode_layout_dcp(const int32_t* seq_lens, int64_t num_seq, const int32_t* query_lens,
                                     int64_t num_requests, int64_t num_rows, int64_t dcp_rank,
                                     int64_t dcp_world_size, int64_t interleave, int32_t* starts,
                                     int32_t* row_ends, void* stream) {
    if (dcp_world_size < 1 || dcp_rank < 0 || dcp_rank >= dcp_world_size || interleave < 1) return DSA_ERR_INVALID;
    if (dcp_world_size > (int64_t(1) << 20) || interleave > (int64_t(1) << 30)) return DSA_ERR_UNSUPPORTED;
    if (num_rows < 0 || num_requests < 0 || num_seq < num_requests) return DSA_ERR_INVALID;
    if (num_requests > 0x7FFFFFFF - 1 || num_rows > 0x7FFFFFFF) return DSA_ERR_UNSUPPORTED;
    if (!starts || (num_rows > 0 && !row_ends) || (num_requests > 0 && (!seq_lens || !query_lens)))
        return DSA_ERR_INVALID;
    const cudaError_t err = launch_pdl(decode_layout_kernel, dim3(1), dim3(1024), 0, static_cast<cudaStream_t>(stream),
                                       seq_lens, query_lens, static_cast<int>(num_requests), num_rows, starts,
                                       row_ends, dcp_rank, dcp_world_size, interleave);
    return err == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

// ----------------------------------------------------------------- failure detection self-check
// One thread waits, with the kernels' own bounded wait, on an mbarrier that
// nothing arrives on: the wait gives up after its time limit and flags
// DSA_STATUS_TIMEOUT, and the kernel returns normally.
namespace dsa {
__global__ void wait_selftest_kernel(int32_t* status) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, status);
}
}  // namespace dsa

extern "C" int dsa_selftest_wait_timeout(int32_t* status, void* stream) {
    if (!status) return DSA_ERR_INVALID;
    wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status);
    return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
