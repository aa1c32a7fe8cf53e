// Host-side helpers shared by the launchers: workspace layout, device
// properties, tensor-map encoding and PDL launches.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace dsa {

// Byte offsets of the regions of a dsa_score_paged / dsa_topk workspace.
// Every region starts on a 256-byte boundary.  `hist` and `counters`
// must be zero on entry and are zero again when a call completes.
constexpr int kMaxScoreCtas = 1024;   // largest scoring grid the plan table holds

struct WsLayout {
    size_t info;        // int[8]: segment count, tile count
    size_t segs;        // int4[rows + 1]: request, first row, rows, largest bound
    size_t seg_prefix;  // int[rows + 2]: exclusive prefix of tiles per segment
    size_t eff_end;     // int[rows]: row bounds after validation (0 outside every request)
    size_t cta;         // int4[kMaxScoreCtas]: per scoring CTA {first tile, end tile, first segment, segments}
    size_t hist;        // uint32[rows][2048]: histogram of the top 11 order-preserving score bits
    size_t counters;    // int[rows][4]: winners published, candidates published, spans done, candidates dropped
    size_t cand;        // uint2[rows][kCandCap]: level-1 candidates of split rows (key, position)
    size_t logits;      // float[rows][width] when the caller keeps no logits
    size_t total;
};

WsLayout workspace_layout(int64_t rows, int64_t width, bool with_plan, bool with_logits);

int device_sm_count();

// cuTensorMapEncodeTiled through the runtime's driver entry point.
CUresult encode_tiled(CUtensorMap* map, CUtensorMapDataType type, cuuint32_t rank, void* addr,
                      const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                      CUtensorMapSwizzle swizzle);

// Launch with programmatic stream serialization (the kernel may start while
// the previous kernel on the stream finishes; it must call griddepcontrol.wait
// before reading that kernel's results).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// dsa_prepare_step's argument checks alone (no launch).
int check_prepare(int fmt, const void* q, int64_t q_row_stride, const void* wv, int64_t wv_row_stride, int64_t rows,
                  const void* q_out, const void* w_out, const void* k, int64_t k_row_stride, const float* gamma,
                  const float* beta, const int64_t* slots, int64_t n, const void* cache, int64_t page_stride,
                  int64_t num_pages, const int32_t* seq_lens, int64_t num_seq, const int32_t* query_lens,
                  int64_t num_requests, int64_t num_rows, const int32_t* starts, const int32_t* row_ends);

// dsa_prepare_step's checks and launch.
int launch_prepare(int fmt, const void* q, int64_t q_row_stride, const void* wv, int64_t wv_row_stride, int64_t rows,
                   void* q_out, void* w_out, const void* k, int64_t k_row_stride, const float* gamma,
                   const float* beta, float eps, const int64_t* slots, int64_t n, void* cache, int64_t page_stride,
                   int64_t num_pages, const int32_t* seq_lens, int64_t num_seq, const int32_t* query_lens,
                   int64_t num_requests, int64_t num_rows, int32_t* starts, int32_t* row_ends, int32_t* status,
                   cudaStream_t stream);

// Top-k selection launcher shared by dsa_score_paged and dsa_topk.
int launch_select(const float* logits, float* logits_fill, int64_t ld, int64_t width, const int32_t* ends,
                  int64_t rows, int64_t k, int32_t* out, uint8_t* ws, const WsLayout& L, cudaStream_t stream,
                  bool pdl);

}  // namespace dsa
