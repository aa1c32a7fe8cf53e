// QueryNorm: the q_a RMSNorm of the packed projection -> q_c, BF16.
//
// Page "cutedsl.dsa.overlap", class QueryNorm: every row of 1536 BF16
// columns is scaled by rr = 1 / sqrt(mean square + eps) and by the BF16
// weights; the page's two kernels fix the FP32 order of the sum of squares,
// and both are provided:
//   per-row form  one row per 256-thread CTA; thread t < 192 holds columns
//                 8t..8t+7, sums their squares with sequential FMAs, the
//                 warps reduce by xor butterfly and the 8 warp sums are added
//                 in warp order;
//   tiled form    one row per warp; lane l holds columns 256i + 8l + j
//                 (i < 6, j < 8) as values e = 8i + j, whose squares go to
//                 four FMA chains by e mod 4, added as (c0 + c1) + (c2 + c3)
//                 before the butterfly.
// rr = 1 / sqrt(total / 1536 + eps) and y = BF16((x * rr) * w), each FP32
// operation rounded on its own (no contraction).
#include "host.h"
#include "common.cuh"

namespace dsa {

constexpr int kNormCols = 1536;
constexpr int kTiledFrom = 64;   // default: batches of at least this many rows take the tiled form

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(a));
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(b));
    return lo | (hi << 16);
}
__device__ __forceinline__ float warp_butterfly_sum(float v) {
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, d));
    return v;
}
__device__ __forceinline__ float norm_rsqrt(float total, float eps) {
    return __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(total, static_cast<float>(kNormCols)), eps)));
}
__device__ __forceinline__ void unpack8(uint4 r, float (&v)[8]) {
    v[0] = bf16_lo(r.x); v[1] = bf16_hi(r.x); v[2] = bf16_lo(r.y); v[3] = bf16_hi(r.y);
    v[4] = bf16_lo(r.z); v[5] = bf16_hi(r.z); v[6] = bf16_lo(r.w); v[7] = bf16_hi(r.w);
}

__global__ void __launch_bounds__(256) query_norm_row_kernel(const uint16_t* __restrict__ x, int64_t xs,
                                                             const uint16_t* __restrict__ w, float eps,
                                                             uint16_t* __restrict__ out, int64_t os) {
    __shared__ float ss[8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t row = blockIdx.x;
    float g[8];
    unpack8(*reinterpret_cast<const uint4*>(w + (tid % 192) * 8), g);
    pdl_launch_dependents();
    pdl_wait();
    float v[8];
    float acc = 0.0f;
    if (tid < 192) {
        unpack8(*reinterpret_cast<const uint4*>(x + row * xs + tid * 8), v);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc = fmaf(v[i], v[i], acc);
    }
    acc = warp_butterfly_sum(acc);
    if (lane == 0) ss[warp] = acc;
    __syncthreads();
    if (tid < 192) {
        float total = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) total = __fadd_rn(total, ss[k]);
        const float rr = norm_rsqrt(total, eps);
        uint4 o;
        uint32_t* ow = &o.x;
#pragma unroll
        for (int i = 0; i < 8; i += 2)
            ow[i / 2] = pack_bf16x2(__fmul_rn(__fmul_rn(v[i], rr), g[i]), __fmul_rn(__fmul_rn(v[i + 1], rr), g[i + 1]));
        *reinterpret_cast<uint4*>(out + row * os + tid * 8) = o;
    }
}

__global__ void __launch_bounds__(256) query_norm_tiled_kernel(const uint16_t* __restrict__ x, int64_t xs,
                                                               const uint16_t* __restrict__ w, float eps,
                                                               int64_t batch, uint16_t* __restrict__ out,
                                                               int64_t os) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + warp;
    float g[48];
#pragma unroll
    for (int i = 0; i < 6; ++i) {
        float t[8];
        unpack8(*reinterpret_cast<const uint4*>(w + 256 * i + 8 * lane), t);
#pragma unroll
        for (int j = 0; j < 8; ++j) g[8 * i + j] = t[j];
    }
    pdl_launch_dependents();
    pdl_wait();
    if (row >= batch) return;
    float v[48];
#pragma unroll
    for (int i = 0; i < 6; ++i) {
        float t[8];
        unpack8(*reinterpret_cast<const uint4*>(x + row * xs + 256 * i + 8 * lane), t);
#pragma unroll
        for (int j = 0; j < 8; ++j) v[8 * i + j] = t[j];
    }
    float c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int e = 0; e < 48; ++e) c[e % 4] = fmaf(v[e], v[e], c[e % 4]);
    const float total = warp_butterfly_sum(__fadd_rn(__fadd_rn(c[0], c[1]), __fadd_rn(c[2], c[3])));
    const float rr = norm_rsqrt(total, eps);
#pragma unroll
    for (int i = 0; i < 6; ++i) {
        uint4 o;
        uint32_t* ow = &o.x;
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
            const int e = 8 * i + j;
            ow[j / 2] = pack_bf16x2(__fmul_rn(__fmul_rn(v[e], rr), g[e]), __fmul_rn(__fmul_rn(v[e + 1], rr), g[e + 1]));
        }
        *reinterpret_cast<uint4*>(out + row * os + 256 * i + 8 * lane) = o;
    }
}

}  // namespace dsa

using namespace dsa;

extern "C" int dsa_query_norm(const void* x, int64_t x_row_stride, const void* w, float eps, int64_t batch,
                              void* out, int64_t out_row_stride, int variant, void* stream_) {
    if (batch < 0 || variant < -1 || variant > 1) return DSA_ERR_INVALID;
    if (batch == 0) return DSA_OK;
    if (!x || !w || !out) return DSA_ERR_INVALID;
    if (x_row_stride < kNormCols || out_row_stride < kNormCols || x_row_stride % 8 || out_row_stride % 8)
        return DSA_ERR_INVALID;
    const auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
    if (!a16(x) || !a16(w) || !a16(out)) return DSA_ERR_INVALID;
    const bool tiled = variant == 1 || (variant == -1 && batch >= kTiledFrom);
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    const uint16_t* xp = static_cast<const uint16_t*>(x);
    const uint16_t* wp = static_cast<const uint16_t*>(w);
    uint16_t* op = static_cast<uint16_t*>(out);
    cudaError_t err;
    if (tiled) {
        const int64_t blocks = (batch + 7) / 8;
        if (blocks > 0x7FFFFFFF) return DSA_ERR_UNSUPPORTED;
        err = launch_pdl(query_norm_tiled_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, xp,
                         x_row_stride, wp, eps, batch, op, out_row_stride);
    } else {
        if (batch > 0x7FFFFFFF) return DSA_ERR_UNSUPPORTED;
        err = launch_pdl(query_norm_row_kernel, dim3(static_cast<unsigned>(batch)), dim3(256), 0, stream, xp,
                         x_row_stride, wp, eps, op, out_row_stride);
    }
    return err == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
