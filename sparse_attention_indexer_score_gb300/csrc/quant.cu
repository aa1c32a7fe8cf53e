// Query quantisation (FP8 with a per-head power-of-two scale folded into the
// head weights, or MXFP4) and key LayerNorm + quantise + paged insert.
//
// Page "cutedsl.dsa.index": DsaIndex.fp8_query, quantize_fp4_query,
// insert_key, insert_fp4_key, mxfp4_scale (definition only), e2m1x2.
#include "host.h"
#include "common.cuh"
#include "layout_body.cuh"

namespace dsa {

// ----------------------------------------------------------------- codecs
// Four FP32 -> four E4M3 bytes (round to nearest even, satfinite), a in byte 0.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
    unsigned short lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}
// Two FP32 -> one byte of two E2M1 (round to nearest even, satfinite), lo in the low nibble.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %2, %1;\n\tcvt.u32.u8 %0, t;\n\t}"
        : "=r"(r)
        : "f"(lo), "f"(hi));
    return r;
}
// 2^e as an FP32, e in [-126, 127].
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float(static_cast<uint32_t>(e + 127) << 23); }

// Smallest e with 448 * 2^e >= a, for a positive normal FP32 a: with
// a = m * 2^E (1 <= m < 2) and 448 = 1.75 * 2^8, e = E - 8, plus one when m > 1.75.
__device__ __forceinline__ int fp8_exponent(float a) {
    const uint32_t u = __float_as_uint(a);
    const int E = static_cast<int>((u >> 23) & 0xFFu) - 127;
    return E - 8 + ((u & 0x7FFFFFu) > 0x600000u ? 1 : 0);
}
// MXFP4 block exponent: the smallest e with 6 * 2^e >= max(amax, 6 * 2^-126),
// clamped to [-127, 127]; with 6 = 1.5 * 2^2, e = E - 2, plus one when m > 1.5.
__device__ __forceinline__ int mx_exponent(float amax) {
    const float a = fmaxf(amax, 6.0f * 0x1p-126f);
    const uint32_t u = __float_as_uint(a);
    const int E = static_cast<int>((u >> 23) & 0xFFu) - 127;
    const int e = E - 2 + ((u & 0x7FFFFFu) > 0x400000u ? 1 : 0);
    return min(max(e, -127), 127);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// MXFP4 of a 128-column head held by a warp (lane l: columns 4l..4l+3; amax:
// the lane's max |x|): returns the lane's two bytes of E2M1 pairs (column 4l
// in the low nibble) and sets *scale_byte to the UE8M0 byte of its 32-column
// block (8 lanes per block).
__device__ __forceinline__ uint32_t mxfp4_lane(float x0, float x1, float x2, float x3, float amax,
                                               uint32_t* scale_byte) {
#pragma unroll
    for (int d = 4; d >= 1; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, d));
    const int e = mx_exponent(amax);
    const float inv = exp2i(-e);
    const uint32_t b01 = e2m1x2(__fmul_rn(x0, inv), __fmul_rn(x1, inv));
    const uint32_t b23 = e2m1x2(__fmul_rn(x2, inv), __fmul_rn(x3, inv));
    *scale_byte = static_cast<uint32_t>(e + 127);
    return b01 | (b23 << 8);
}

// ----------------------------------------------------------------- query rows
// One warp per (row, head); lane l holds columns 4l..4l+3.  `block` is the
// block index within this part of the grid (256 threads per block).
__device__ __forceinline__ void quantize_query_block(int fmt, const uint16_t* __restrict__ q, int64_t q_stride,
                                                     const uint16_t* __restrict__ wv, int64_t wv_stride,
                                                     int64_t rows, uint8_t* __restrict__ q_out,
                                                     __nv_bfloat16* __restrict__ w_out, int64_t block) {
    const int64_t gw = (block * 256 + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (gw >= rows * kHeads) return;
    const int64_t row = gw >> 5;
    const int head = static_cast<int>(gw & 31);
    const uint2 raw = *reinterpret_cast<const uint2*>(q + row * q_stride + head * kDim + lane * 4);
    const float x0 = bf16_bits_to_f32(raw.x & 0xFFFFu), x1 = bf16_bits_to_f32(raw.x >> 16);
    const float x2 = bf16_bits_to_f32(raw.y & 0xFFFFu), x3 = bf16_bits_to_f32(raw.y >> 16);
    float amax = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
    uint8_t* out_row = q_out + row * kQRowBytes;
    const float wvf = bf16_bits_to_f32(wv[row * wv_stride + head]);
    if (!fmt_fp4(fmt)) {
        amax = fmaxf(amax, 1e-10f);
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, d));
        const int e = fp8_exponent(amax);
        const float inv = exp2i(-e);
        const uint32_t word = e4m3x4(__fmul_rn(x0, inv), __fmul_rn(x1, inv), __fmul_rn(x2, inv), __fmul_rn(x3, inv));
        *reinterpret_cast<uint32_t*>(out_row + head * kDim + lane * 4) = word;
        if (lane == 0) {
            const float fold = __fmul_rn(__fmul_rn(wvf, exp2i(e)), 0.015625f);   // (wv * scale) / 64
            w_out[row * kHeads + head] = __float2bfloat16_rn(fold);
        }
    } else {
        uint32_t byte;
        *reinterpret_cast<uint16_t*>(out_row + head * (kDim / 2) + lane * 2) =
            static_cast<uint16_t>(mxfp4_lane(x0, x1, x2, x3, amax, &byte));
        if (fmt == DSA_FMT_MXFP4_RG) {
            // row-group scales: block g of head h at g * 64 + h
            if ((lane & 7) == 0) out_row[kFp4Scales + (lane >> 3) * kRgQuerySlots + head] = static_cast<uint8_t>(byte);
        } else {
            const uint32_t b1 = __shfl_sync(0xFFFFFFFFu, byte, 8);
            const uint32_t b2 = __shfl_sync(0xFFFFFFFFu, byte, 16);
            const uint32_t b3 = __shfl_sync(0xFFFFFFFFu, byte, 24);
            if (lane == 0)
                *reinterpret_cast<uint32_t*>(out_row + kFp4Scales + head * 4) =
                    byte | (b1 << 8) | (b2 << 16) | (b3 << 24);
        }
        if (lane == 0) w_out[row * kHeads + head] = __float2bfloat16_rn(__fmul_rn(wvf, 0.015625f));
    }
}

__global__ void __launch_bounds__(256) quantize_query_kernel(int fmt, const uint16_t* __restrict__ q,
                                                             int64_t q_stride, const uint16_t* __restrict__ wv,
                                                             int64_t wv_stride, int64_t rows,
                                                             uint8_t* __restrict__ q_out,
                                                             __nv_bfloat16* __restrict__ w_out) {
    pdl_launch_dependents();
    pdl_wait();
    quantize_query_block(fmt, q, q_stride, wv, wv_stride, rows, q_out, w_out, blockIdx.x);
}

// ----------------------------------------------------------------- keys
// One half-warp per key; lane j of the half holds columns 8j..8j+7.  `block`
// is the block index within this part of the grid (256 threads per block).
__device__ __forceinline__ void insert_key_block(int fmt, const uint16_t* __restrict__ k, int64_t k_stride,
                                                 const float* __restrict__ gamma, const float* __restrict__ beta,
                                                 float eps, const int64_t* __restrict__ slots, int64_t n,
                                                 uint8_t* __restrict__ cache, int64_t page_stride,
                                                 int64_t num_pages, int32_t* status, int64_t block) {
    const int64_t key = (block * 256 + threadIdx.x) >> 4;
    const int j = threadIdx.x & 15;
    const unsigned hmask = (threadIdx.x & 16) ? 0xFFFF0000u : 0x0000FFFFu;
    if (key >= n) return;
    const int64_t slot = slots[key];
    if (slot < 0) return;                                  // padding: nothing written
    if (slot >= num_pages * kPage) {
        if (j == 0 && status) atomicOr(status, DSA_STATUS_BAD_SLOT);
        return;
    }
    const uint4 raw = *reinterpret_cast<const uint4*>(k + key * k_stride + j * 8);
    float x[8];
    const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = bf16_bits_to_f32(w4[i] & 0xFFFFu);
        x[2 * i + 1] = bf16_bits_to_f32(w4[i] >> 16);
    }
    // LayerNorm in FP32, fixed order: 8-term sums, xor butterfly over 16 lanes.
    float total = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) total = __fadd_rn(total, x[i]);
#pragma unroll
    for (int d = 8; d >= 1; d >>= 1) total = __fadd_rn(total, __shfl_xor_sync(hmask, total, d, 16));
    const float mean = __fdiv_rn(total, 128.0f);
    float dx[8];
    float square = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        dx[i] = __fsub_rn(x[i], mean);
        square = __fadd_rn(square, __fmul_rn(dx[i], dx[i]));
    }
#pragma unroll
    for (int d = 8; d >= 1; d >>= 1) square = __fadd_rn(square, __shfl_xor_sync(hmask, square, d, 16));
    const float variance = __fdiv_rn(square, 128.0f);
    const float rstd = __frcp_rn(__fsqrt_rn(__fadd_rn(variance, eps)));
    float normed[8];
    float amax = 0.0f;
    const float4 g0 = *reinterpret_cast<const float4*>(gamma + j * 8);
    const float4 g1 = *reinterpret_cast<const float4*>(gamma + j * 8 + 4);
    const float4 c0 = *reinterpret_cast<const float4*>(beta + j * 8);
    const float4 c1 = *reinterpret_cast<const float4*>(beta + j * 8 + 4);
    const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    const float b[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float y = __fadd_rn(__fmul_rn(__fmul_rn(dx[i], rstd), g[i]), b[i]);
        normed[i] = __bfloat162float(__float2bfloat16_rn(y));
        amax = fmaxf(amax, fabsf(normed[i]));
    }
    const int64_t page = slot / kPage;
    const int off = static_cast<int>(slot % kPage);
    uint8_t* base = cache + page * page_stride;
    if (!fmt_fp4(fmt)) {
#pragma unroll
        for (int d = 8; d >= 1; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(hmask, amax, d, 16));
        const int e = fp8_exponent(fmaxf(amax, 1e-10f));
        const float inv = exp2i(-e);
        uint2 words;
        words.x = e4m3x4(__fmul_rn(normed[0], inv), __fmul_rn(normed[1], inv), __fmul_rn(normed[2], inv),
                         __fmul_rn(normed[3], inv));
        words.y = e4m3x4(__fmul_rn(normed[4], inv), __fmul_rn(normed[5], inv), __fmul_rn(normed[6], inv),
                         __fmul_rn(normed[7], inv));
        *reinterpret_cast<uint2*>(base + off * kDim + j * 8) = words;
        if (j == 0) {
            const uint32_t sc = (fmt == DSA_FMT_FP8) ? __float_as_uint(exp2i(e))
                                                     : static_cast<uint32_t>(e + 127) * 0x01010101u;
            *reinterpret_cast<uint32_t*>(base + kFp8KeyBytes + off * 4) = sc;
        }
    } else {
        // 4 lanes hold one 32-column block
#pragma unroll
        for (int d = 2; d >= 1; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(hmask, amax, d, 16));
        const int e = mx_exponent(amax);
        const float inv = exp2i(-e);
        uint32_t word = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            word |= e2m1x2(__fmul_rn(normed[2 * i], inv), __fmul_rn(normed[2 * i + 1], inv)) << (8 * i);
        const uint32_t byte = static_cast<uint32_t>(e + 127);
        if (fmt == DSA_FMT_MXFP4_RG) {
            // lane j: bytes 4(j mod 4) .. +3 of group j / 4's 16 bytes; its first lane writes the scale
            const int g = j >> 2;
            *reinterpret_cast<uint32_t*>(base + g * kRgGroupBytes + off * 16 + (j & 3) * 4) = word;
            if ((j & 3) == 0) base[kFp4KeyBytes + g * kRgScaleGroup + off] = static_cast<uint8_t>(byte);
        } else {
            *reinterpret_cast<uint32_t*>(base + off * (kDim / 2) + j * 4) = word;
            const uint32_t b1 = __shfl_sync(hmask, byte, 4, 16);
            const uint32_t b2 = __shfl_sync(hmask, byte, 8, 16);
            const uint32_t b3 = __shfl_sync(hmask, byte, 12, 16);
            if (j == 0)
                *reinterpret_cast<uint32_t*>(base + kFp4KeyBytes + off * 4) =
                    byte | (b1 << 8) | (b2 << 16) | (b3 << 24);
        }
    }
}

__global__ void __launch_bounds__(256) insert_key_kernel(int fmt, const uint16_t* __restrict__ k, int64_t k_stride,
                                                         const float* __restrict__ gamma,
                                                         const float* __restrict__ beta, float eps,
                                                         const int64_t* __restrict__ slots, int64_t n,
                                                         uint8_t* __restrict__ cache, int64_t page_stride,
                                                         int64_t num_pages, int32_t* status) {
    pdl_launch_dependents();
    pdl_wait();
    insert_key_block(fmt, k, k_stride, gamma, beta, eps, slots, n, cache, page_stride, num_pages, status, blockIdx.x);
}

// ----------------------------------------------------------------- row-group queries
// Page "amd.ops.fp4_indexer", quantize_queries: one warp per (row, head slot
// of 64); slots past `heads` only clear their four scale bytes.
__global__ void __launch_bounds__(256) quantize_queries_rg_kernel(const uint16_t* __restrict__ q, int64_t row_stride,
                                                                  int64_t head_stride, int heads, int64_t rows,
                                                                  uint8_t* __restrict__ payload,
                                                                  uint8_t* __restrict__ scales) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t gw = (static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (gw >= rows * kRgQuerySlots) return;
    const int64_t row = gw / kRgQuerySlots;
    const int h = static_cast<int>(gw % kRgQuerySlots);
    uint8_t* srow = scales + row * (4 * kRgQuerySlots);
    if (h >= heads) {
        if (lane < 4) srow[lane * kRgQuerySlots + h] = 0;
        return;
    }
    const uint2 raw = *reinterpret_cast<const uint2*>(q + row * row_stride + h * head_stride + lane * 4);
    const float x0 = bf16_bits_to_f32(raw.x & 0xFFFFu), x1 = bf16_bits_to_f32(raw.x >> 16);
    const float x2 = bf16_bits_to_f32(raw.y & 0xFFFFu), x3 = bf16_bits_to_f32(raw.y >> 16);
    const float amax = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
    uint32_t byte;
    *reinterpret_cast<uint16_t*>(payload + (row * heads + h) * (kDim / 2) + lane * 2) =
        static_cast<uint16_t>(mxfp4_lane(x0, x1, x2, x3, amax, &byte));
    if ((lane & 7) == 0) srow[(lane >> 3) * kRgQuerySlots + h] = static_cast<uint8_t>(byte);
}

// ----------------------------------------------------------------- fused step preparation
// One launch for the three independent parts of a decode step's preparation:
// block 0 computes the request starts and row bounds, the next blocks insert
// the step's keys, the rest quantise the query rows.  The parts write
// disjoint buffers, so the result is that of the three calls in any order.
struct PrepareArgs {
    int fmt;
    // query rows
    const uint16_t* q;
    int64_t q_stride;
    const uint16_t* wv;
    int64_t wv_stride;
    int64_t rows;
    uint8_t* q_out;
    __nv_bfloat16* w_out;
    int64_t q_blocks;
    // keys
    const uint16_t* k;
    int64_t k_stride;
    const float* gamma;
    const float* beta;
    float eps;
    const int64_t* slots;
    int64_t n;
    uint8_t* cache;
    int64_t page_stride;
    int64_t num_pages;
    int32_t* status;
    int64_t k_blocks;
    // layout
    const int32_t* seq_lens;
    const int32_t* query_lens;
    int num_req;
    int64_t num_rows;
    int32_t* starts;
    int32_t* row_ends;
};

__global__ void __launch_bounds__(256) prepare_step_kernel(const PrepareArgs a) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t b = blockIdx.x;
    if (b == 0) {
        decode_layout_block(a.seq_lens, a.query_lens, a.num_req, a.num_rows, a.starts, a.row_ends);
    } else if (b <= a.k_blocks) {
        insert_key_block(a.fmt, a.k, a.k_stride, a.gamma, a.beta, a.eps, a.slots, a.n, a.cache, a.page_stride,
                         a.num_pages, a.status, b - 1);
    } else {
        quantize_query_block(a.fmt, a.q, a.q_stride, a.wv, a.wv_stride, a.rows, a.q_out, a.w_out,
                             b - 1 - a.k_blocks);
    }
}

}  // namespace dsa

using namespace dsa;

static bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Argument checks shared by the single calls and dsa_prepare_step; each
// returns DSA_OK and the number of 256-thread blocks its part needs (0 when
// there is nothing to do).
static int check_quantize(int fmt, const void* q, int64_t q_row_stride, const void* wv, int64_t wv_row_stride,
                          int64_t rows, const void* q_out, const void* w_out, int64_t* blocks) {
    *blocks = 0;
    if (fmt < DSA_FMT_FP8 || fmt > DSA_FMT_MXFP4_RG) return DSA_ERR_UNSUPPORTED;
    if (rows < 0) return DSA_ERR_INVALID;
    if (rows == 0) return DSA_OK;
    if (!q || !wv || !q_out || !w_out) return DSA_ERR_INVALID;
    if (q_row_stride < kHeads * kDim || q_row_stride % 8 || wv_row_stride < kHeads) return DSA_ERR_INVALID;
    if (!aligned(q, 16) || !aligned(q_out, 16) || !aligned(w_out, 2) || !aligned(wv, 2)) return DSA_ERR_INVALID;
    *blocks = (rows * kHeads * 32 + 255) / 256;
    return *blocks > 0x7FFFFFFF ? DSA_ERR_UNSUPPORTED : DSA_OK;
}

static int check_insert(int fmt, const void* k, int64_t k_row_stride, const float* gamma, const float* beta,
                        const int64_t* slots, int64_t n, const void* cache, int64_t page_stride, int64_t num_pages,
                        int64_t* blocks) {
    *blocks = 0;
    if (fmt < DSA_FMT_FP8 || fmt > DSA_FMT_MXFP4_RG) return DSA_ERR_UNSUPPORTED;
    if (n < 0 || num_pages < 0) return DSA_ERR_INVALID;
    if (n == 0) return DSA_OK;
    if (!k || !gamma || !beta || !slots || !cache) return DSA_ERR_INVALID;
    const int64_t min_stride = fmt_fp4(fmt) ? DSA_FP4_PAGE_BYTES : DSA_FP8_PAGE_BYTES;
    if (page_stride < min_stride || page_stride % 16) return DSA_ERR_INVALID;
    if (k_row_stride < kDim || k_row_stride % 8) return DSA_ERR_INVALID;
    if (!aligned(k, 16) || !aligned(gamma, 16) || !aligned(beta, 16) || !aligned(cache, 16) || !aligned(slots, 8))
        return DSA_ERR_INVALID;
    *blocks = (n * 16 + 255) / 256;
    return *blocks > 0x7FFFFFFF ? DSA_ERR_UNSUPPORTED : DSA_OK;
}

static int check_layout(const int32_t* seq_lens, int64_t num_seq, const int32_t* query_lens, int64_t num_requests,
                        int64_t num_rows, const int32_t* starts, const int32_t* row_ends) {
    if (num_rows < 0 || num_requests < 0 || num_seq < num_requests) return DSA_ERR_INVALID;
    if (num_requests > 0x7FFFFFFF - 1 || num_rows > 0x7FFFFFFF) return DSA_ERR_UNSUPPORTED;
    if (!starts || (num_rows > 0 && !row_ends) || (num_requests > 0 && (!seq_lens || !query_lens)))
        return DSA_ERR_INVALID;
    return DSA_OK;
}

extern "C" int dsa_quantize_query(int fmt, const void* q, int64_t q_row_stride, const void* wv,
                                  int64_t wv_row_stride, int64_t rows, void* q_out, void* w_out, void* stream) {
    int64_t blocks = 0;
    const int rc = check_quantize(fmt, q, q_row_stride, wv, wv_row_stride, rows, q_out, w_out, &blocks);
    if (rc != DSA_OK || blocks == 0) return rc;
    const cudaError_t err = launch_pdl(quantize_query_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                                       static_cast<cudaStream_t>(stream), fmt, static_cast<const uint16_t*>(q),
                                       q_row_stride, static_cast<const uint16_t*>(wv), wv_row_stride, rows,
                                       static_cast<uint8_t*>(q_out), static_cast<__nv_bfloat16*>(w_out));
    return err == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

extern "C" int dsa_quantize_queries_rg(const void* q, int64_t q_row_stride, int64_t q_head_stride, int64_t heads,
                                       int64_t rows, void* payload, void* scales, void* stream) {
    if (heads != 16 && heads != 32 && heads != 64) return DSA_ERR_UNSUPPORTED;
    if (rows < 0) return DSA_ERR_INVALID;
    if (rows == 0) return DSA_OK;
    if (!q || !payload || !scales) return DSA_ERR_INVALID;
    if (q_head_stride < kDim || q_head_stride % 4 || q_row_stride < 0 || q_row_stride % 4) return DSA_ERR_INVALID;
    if (!aligned(q, 8) || !aligned(payload, 2)) return DSA_ERR_INVALID;
    if (rows > (int64_t(1) << 40) / (kRgQuerySlots * 32)) return DSA_ERR_UNSUPPORTED;
    const int64_t blocks = (rows * kRgQuerySlots * 32 + 255) / 256;
    if (blocks > 0x7FFFFFFF) return DSA_ERR_UNSUPPORTED;
    const cudaError_t err =
        launch_pdl(quantize_queries_rg_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                   static_cast<cudaStream_t>(stream), static_cast<const uint16_t*>(q), q_row_stride, q_head_stride,
                   static_cast<int>(heads), rows, static_cast<uint8_t*>(payload), static_cast<uint8_t*>(scales));
    return err == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

extern "C" int dsa_insert_key(int fmt, const void* k, int64_t k_row_stride, const float* gamma, const float* beta,
                              float eps, const int64_t* slots, int64_t n, void* cache, int64_t page_stride,
                              int64_t num_pages, int32_t* status, void* stream) {
    int64_t blocks = 0;
    const int rc = check_insert(fmt, k, k_row_stride, gamma, beta, slots, n, cache, page_stride, num_pages, &blocks);
    if (rc != DSA_OK || blocks == 0) return rc;
    const cudaError_t err = launch_pdl(insert_key_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                                       static_cast<cudaStream_t>(stream), fmt, static_cast<const uint16_t*>(k),
                                       k_row_stride, gamma, beta, eps, slots, n, static_cast<uint8_t*>(cache),
                                       page_stride, num_pages, status);
    return err == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

namespace dsa {

// The three parts' checks; *qb and *kb get the blocks of the quantise and
// insert parts.
static int check_prepare_blocks(int fmt, const void* q, int64_t q_row_stride, const void* wv, int64_t wv_row_stride,
                                int64_t rows, const void* q_out, const void* w_out, const void* k,
                                int64_t k_row_stride, const float* gamma, const float* beta, const int64_t* slots,
                                int64_t n, const void* cache, int64_t page_stride, int64_t num_pages,
                                const int32_t* seq_lens, int64_t num_seq, const int32_t* query_lens,
                                int64_t num_requests, int64_t num_rows, const int32_t* starts,
                                const int32_t* row_ends, int64_t* qb_out, int64_t* kb_out) {
    int64_t qb = 0, kb = 0;
    int rc = check_quantize(fmt, q, q_row_stride, wv, wv_row_stride, rows, const_cast<void*>(q_out),
                            const_cast<void*>(w_out), &qb);
    if (rc != DSA_OK) return rc;
    rc = check_insert(fmt, k, k_row_stride, gamma, beta, slots, n, const_cast<void*>(cache), page_stride, num_pages,
                      &kb);
    if (rc != DSA_OK) return rc;
    rc = check_layout(seq_lens, num_seq, query_lens, num_requests, num_rows, const_cast<int32_t*>(starts),
                      const_cast<int32_t*>(row_ends));
    if (rc != DSA_OK) return rc;
    *qb_out = qb;
    *kb_out = kb;
    return (1 + kb + qb > 0x7FFFFFFF) ? DSA_ERR_UNSUPPORTED : DSA_OK;
}

int check_prepare(int fmt, const void* q, int64_t q_row_stride, const void* wv, int64_t wv_row_stride, int64_t rows,
                  const void* q_out, const void* w_out, const void* k, int64_t k_row_stride, const float* gamma,
                  const float* beta, const int64_t* slots, int64_t n, const void* cache, int64_t page_stride,
                  int64_t num_pages, const int32_t* seq_lens, int64_t num_seq, const int32_t* query_lens,
                  int64_t num_requests, int64_t num_rows, const int32_t* starts, const int32_t* row_ends) {
    int64_t qb = 0, kb = 0;
    return check_prepare_blocks(fmt, q, q_row_stride, wv, wv_row_stride, rows, q_out, w_out, k, k_row_stride, gamma,
                                beta, slots, n, cache, page_stride, num_pages, seq_lens, num_seq, query_lens,
                                num_requests, num_rows, starts, row_ends, &qb, &kb);
}

int launch_prepare(int fmt, const void* q, int64_t q_row_stride, const void* wv, int64_t wv_row_stride, int64_t rows,
                   void* q_out, void* w_out, const void* k, int64_t k_row_stride, const float* gamma,
                   const float* beta, float eps, const int64_t* slots, int64_t n, void* cache, int64_t page_stride,
                   int64_t num_pages, const int32_t* seq_lens, int64_t num_seq, const int32_t* query_lens,
                   int64_t num_requests, int64_t num_rows, int32_t* starts, int32_t* row_ends, int32_t* status,
                   cudaStream_t stream) {
    int64_t qb = 0, kb = 0;
    const int rc = check_prepare_blocks(fmt, q, q_row_stride, wv, wv_row_stride, rows, q_out, w_out, k, k_row_stride,
                                        gamma, beta, slots, n, cache, page_stride, num_pages, seq_lens, num_seq,
                                        query_lens, num_requests, num_rows, starts, row_ends, &qb, &kb);
    if (rc != DSA_OK) return rc;
    PrepareArgs a;
    a.fmt = fmt;
    a.q = static_cast<const uint16_t*>(q);
    a.q_stride = q_row_stride;
    a.wv = static_cast<const uint16_t*>(wv);
    a.wv_stride = wv_row_stride;
    a.rows = rows;
    a.q_out = static_cast<uint8_t*>(q_out);
    a.w_out = static_cast<__nv_bfloat16*>(w_out);
    a.q_blocks = qb;
    a.k = static_cast<const uint16_t*>(k);
    a.k_stride = k_row_stride;
    a.gamma = gamma;
    a.beta = beta;
    a.eps = eps;
    a.slots = slots;
    a.n = n;
    a.cache = static_cast<uint8_t*>(cache);
    a.page_stride = page_stride;
    a.num_pages = num_pages;
    a.status = status;
    a.k_blocks = kb;
    a.seq_lens = seq_lens;
    a.query_lens = query_lens;
    a.num_req = static_cast<int>(num_requests);
    a.num_rows = num_rows;
    a.starts = starts;
    a.row_ends = row_ends;
    const dim3 grid(static_cast<unsigned>(1 + kb + qb));
    const cudaError_t err = launch_pdl(prepare_step_kernel, grid, dim3(256), 0, stream, a);
    return err == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace dsa

extern "C" int dsa_prepare_step(int fmt, const void* q, int64_t q_row_stride, const void* wv, int64_t wv_row_stride,
                                int64_t rows, void* q_out, void* w_out, const void* k, int64_t k_row_stride,
                                const float* gamma, const float* beta, float eps, const int64_t* slots, int64_t n,
                                void* cache, int64_t page_stride, int64_t num_pages, const int32_t* seq_lens,
                                int64_t num_seq, const int32_t* query_lens, int64_t num_requests, int64_t num_rows,
                                int32_t* starts, int32_t* row_ends, int32_t* status, void* stream) {
    return launch_prepare(fmt, q, q_row_stride, wv, wv_row_stride, rows, q_out, w_out, k, k_row_stride, gamma, beta,
                          eps, slots, n, cache, page_stride, num_pages, seq_lens, num_seq, query_lens, num_requests,
                          num_rows, starts, row_ends, status, static_cast<cudaStream_t>(stream));
}
