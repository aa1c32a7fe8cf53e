// Tensor-core rate probe: the dense MMA throughput of the two operand kinds
// the scoring kernel uses, measured on this GPU rather than taken from a
// nominal figure.
//
// One persistent CTA per SM issues `iters` tcgen05.mma instructions back to
// back on operands resident in shared memory (no memory traffic), all into
// one TMEM accumulator, at the scoring kernel's shape: M = 128, N = 128 and
// K = 32 (kind::f8f6f4, E4M3 x E4M3) or K = 64 (kind::mxf4, packed E2M1 with
// UE8M0 block scales).  The caller times the launch with CUDA events:
// FLOPs = 2 * M * N * K * iters * CTAs.
#include "common.cuh"
#include "host.h"

namespace dsa {

constexpr int kProbeThreads = 128;
constexpr int kProbeA = 128 * 128;   // A: 128 rows of 128 bytes (FP8) or 64 bytes (packed E2M1)
constexpr int kProbeB = 128 * 128;
constexpr int kProbeSmem = kProbeA + kProbeB + 2 * 512 + 64 + 1024;

__global__ void __launch_bounds__(kProbeThreads, 1) mma_probe_kernel(int kind, int64_t iters, int32_t* status) {
    extern __shared__ uint8_t dyn[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn) + 1023) & ~uintptr_t(1023));
    uint8_t* a = smem;
    uint8_t* b = smem + kProbeA;
    uint8_t* sfa = b + kProbeB;
    uint8_t* sfb = sfa + 512;
    uint64_t* bar = reinterpret_cast<uint64_t*>(sfb + 512);
    uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Operand bytes: a fixed non-zero pattern (E4M3 / E2M1 codes of small
    // values, no NaN); scale bytes 127 (2^0).
    for (int i = threadIdx.x; i < (kProbeA + kProbeB) / 4; i += kProbeThreads)
        reinterpret_cast<uint32_t*>(a)[i] = 0x3A2C1B34u ^ (static_cast<uint32_t>(i) * 0x01010101u & 0x07070707u);
    for (int i = threadIdx.x; i < 2 * 512 / 4; i += kProbeThreads) reinterpret_cast<uint32_t*>(sfa)[i] = 0x7F7F7F7Fu;
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        mbar_fence_init();
    }
    fence_proxy_async_smem();
    if (warp == 0) tc_alloc(slot, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    if (warp == 0 && lane == 0) {
        const uint32_t d = tmem;                       // accumulator: columns 0..127
        const uint32_t ts_a = tmem + 128, ts_b = tmem + 132;
        const bool fp4 = (kind == 1);
        if (fp4) {
            tc_cp_32x128b_warpx4(ts_a, desc_rows16(smem_u32(sfa)));
            tc_cp_32x128b_warpx4(ts_b, desc_rows16(smem_u32(sfb)));
        }
        const uint64_t ad = fp4 ? desc_sw64(smem_u32(a)) : desc_sw128(smem_u32(a));
        const uint64_t bd = fp4 ? desc_sw64(smem_u32(b)) : desc_sw128(smem_u32(b));
        const uint32_t id8 = idesc_f8f6f4(kMmaE4M3, kMmaE4M3, 128, 128);
        const uint32_t id4 = idesc_mx(kMmaMxf4E2M1, kMmaMxf4E2M1, 128, 128, 0, 0);
        for (int64_t i = 0; i < iters; ++i) {
            const uint32_t kk = static_cast<uint32_t>(i & 3);
            if (fp4)
                tc_mma_mxf4(d, ad + 2 * (kk & 1), bd + 2 * (kk & 1), id4, ts_a, ts_b, i > 0);
            else
                tc_mma_f8f6f4(d, ad + 2 * kk, bd + 2 * kk, id8, i > 0);
        }
        tc_commit(bar);
        mbar_drain(bar, 0, globaltimer() + kWaitLimitNs, status);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tc_dealloc(tmem, 256);
    }
}

}  // namespace dsa

using namespace dsa;

extern "C" int dsa_probe_mma(int kind, int64_t iters, int32_t* status, void* stream_) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    // at most 2^22 MMAs per CTA (a fraction of a second), well inside the final wait's limit
    if ((kind != 0 && kind != 1) || iters < 1 || iters > (int64_t(1) << 22)) return DSA_ERR_INVALID;
    static bool attr_set[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DSA_ERR_CUDA;
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(mma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmem) !=
            cudaSuccess)
            return DSA_ERR_CUDA;
        attr_set[dev] = true;
    }
    mma_probe_kernel<<<device_sm_count(), kProbeThreads, kProbeSmem, stream>>>(kind, iters, status);
    return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
