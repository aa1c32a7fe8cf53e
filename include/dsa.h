/*
 * dsa.h - C ABI of the GB300 DSA lightning-indexer decode step.
 *
 * One decode step of the DeepSeek-style sparse-attention indexer, as the
 * indexer pages state it:
 *   1. dsa_quantize_query  per-head FP8 (power-of-two scale folded into the
 *                          head weights) or MXFP4 query rows;
 *   2. dsa_insert_key      LayerNorm (FP32) + quantise + paged insert of the
 *                          shared 128-column indexer key;
 *   3. dsa_decode_layout   request grouping and causal key bounds of the
 *                          (speculative-verify) query rows;
 *   4. dsa_score_paged     paged MQA logits score[t] = sum_h w_h * ReLU(q_h . k_t),
 *                          with the top-k selection fused behind it;
 *   5. dsa_topk            top-k of an existing logits matrix.
 *
 * Conventions for every call:
 *   - Every pointer argument except `stream` is a DEVICE pointer owned by the
 *     caller.  The library allocates no device memory; scratch comes from a
 *     caller workspace sized by dsa_workspace_size / dsa_topk_workspace_size.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call
 *     only enqueues work and returns; nothing waits for the GPU.
 *   - Return value: DSA_OK, or a negative DSA_ERR_* code.  Argument checks
 *     happen on the host before anything is enqueued, so an error return
 *     means no work was queued (except DSA_ERR_CUDA, which reports a failed
 *     launch).
 *   - Invalid *device data* (a page id outside the pool, a slot past the
 *     cache, row bounds past the block table, inconsistent request starts) is
 *     never trapped on: the offending access is skipped (or clamped) and a bit
 *     is OR-ed into the optional caller-provided int32 `status` word.
 *   - Empty inputs (zero rows, zero keys) return DSA_OK and launch nothing.
 *
 * Constants: 32 heads x 128 columns per query row, 128-column keys, 64-token
 * cache pages (page "cutedsl.dsa.index", module docstring and DsaIndex).
 */
#ifndef DSA_H
#define DSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSA_HEADS 32
#define DSA_DIM 128
#define DSA_PAGE_TOKENS 64
#define DSA_Q_ROW_BYTES 4096          /* one quantised query row: 32 x 128 B */
#define DSA_FP4_SCALES 2048           /* byte offset of the MXFP4 query scales in a row */
#define DSA_FP8_PAGE_BYTES 8448       /* 64 x (128 B E4M3 + 4 B scale) */
#define DSA_FP4_PAGE_BYTES 4352       /* 64 x (64 B E2M1 + 4 B UE8M0) */

/* Key / query formats.  Page "cutedsl.dsa.index", module docstring:
 *  DSA_FMT_FP8     E4M3 keys, one power-of-two FP32 scale per token (132 B/token);
 *                  E4M3 queries with the per-head scale folded into the weights.
 *  DSA_FMT_FP8_MX  as DSA_FMT_FP8, but the key scale is stored as its exponent
 *                  in four UE8M0 bytes (the "mx" scales).  The scorer applies
 *                  byte b to columns 32b..32b+31 (MX block scales, inside a
 *                  block-scaled MMA), so caches with unequal bytes score as
 *                  such; the writer stores the token's one exponent four times.
 *  DSA_FMT_MXFP4   E2M1 keys and queries, one UE8M0 scale per 32 columns
 *                  (68 B/token); the head weights carry only the 1/64 factor.
 *  DSA_FMT_MXFP4_RG  the codes and scales of DSA_FMT_MXFP4, placed group-major
 *                  ("row-group") in the 4352-byte page section (page
 *                  "amd.ops.fp4_indexer", cache_views): the 16 code bytes of
 *                  column group g (columns 32g..32g+31) of token t at
 *                  g * 1024 + t * 16, its UE8M0 byte at 4096 + g * 64 + t.
 *                  Queries and weights as DSA_FMT_MXFP4. */
typedef enum {
    DSA_FMT_FP8 = 0,
    DSA_FMT_FP8_MX = 1,
    DSA_FMT_MXFP4 = 2,
    DSA_FMT_MXFP4_RG = 3
} dsa_format;

/* Return codes. */
#define DSA_OK 0
#define DSA_ERR_INVALID (-1)      /* bad shape, stride, alignment, null pointer, count */
#define DSA_ERR_UNSUPPORTED (-2)  /* unknown format or a size the kernels do not handle */
#define DSA_ERR_CUDA (-3)         /* a kernel launch or a driver call failed */

/* Bits of the device status word (OR-ed in by the kernels). */
#define DSA_STATUS_BAD_SLOT 1       /* a slot >= num_pages * 64 was skipped */
#define DSA_STATUS_BAD_PAGE 2       /* a block-table entry outside [0, num_pages) was not loaded; scores of its keys are unspecified */
#define DSA_STATUS_BAD_GEOMETRY 4   /* starts / row bounds out of range were clamped */
#define DSA_STATUS_TIMEOUT 8        /* an internal pipeline wait gave up (about 1 s); results invalid */

/*
 * dsa_quantize_query - quantise indexer query rows and fold the head weights.
 *
 * Page "cutedsl.dsa.index": DsaIndex.kernel, DsaIndex.fp8_query,
 * quantize_fp4_query, fp4_query_views.
 *
 *   q       BF16, row r head h column c at q[r * q_row_stride + h * 128 + c];
 *           q_row_stride >= 4096 elements, a multiple of 8; q 16-byte aligned.
 *   wv      BF16 head-weight logits, wv[r * wv_row_stride + h].
 *   rows    number of query rows (>= 0).
 *   q_out   uint8 [rows][4096], 16-byte aligned.
 *           FP8 formats: head h's 128 E4M3 codes at h * 128, codes of v / 2^e where
 *             2^e is the smallest power of two with 448 * 2^e >= max(1e-10, amax_h).
 *           DSA_FMT_MXFP4: head h's 64 bytes of E2M1 pairs at h * 64 (column 2j in the
 *             low nibble of byte j), its four UE8M0 bytes (column block b at byte b)
 *             at 2048 + h * 4; bytes 2176..4095 are not written.
 *           DSA_FMT_MXFP4_RG: the same pairs; the UE8M0 byte of block b of head h
 *             at 2048 + b * 64 + h (the row-group order of dsa_quantize_queries_rg);
 *             the slots of heads 32..63 and bytes 2304..4095 are not written.
 *   w_out   BF16 [rows][32]: FP8: BF16(wv * 2^e / 64); MXFP4: BF16(wv / 64).
 */
int dsa_quantize_query(int fmt, const void* q, int64_t q_row_stride,
                       const void* wv, int64_t wv_row_stride, int64_t rows,
                       void* q_out, void* w_out, void* stream);

/*
 * dsa_quantize_queries_rg - MXFP4 of [rows, heads, 128] queries in the
 * row-group layout, no scale folded into head weights.
 *
 * Page "amd.ops.fp4_indexer": quantize_queries (payload [rows, heads, 64],
 * scales [rows, 1, 4, 16, 4]; heads 16, 32 or 64).  The page fixes the scale
 * tensor's shape but not its order; the order taken is group-major, like the
 * cache's scale view [pages, 1, 4, 64]: the byte of column block g of head h at
 * flat position g * 64 + h of the row's 256 bytes.
 *
 *   q        BF16, row r head h column c at q[r * q_row_stride + h * q_head_stride + c];
 *            q_head_stride >= 128 and both strides multiples of 4 elements; q 8-byte aligned.
 *   heads    16, 32 or 64 (else DSA_ERR_UNSUPPORTED).
 *   payload  uint8 [rows][heads][64], 2-byte aligned: head h's E2M1 pairs (column 2j
 *            in the low nibble of byte j), codes of v / 2^e for its block scale 2^e.
 *   scales   uint8 [rows][256]; the slots of heads >= `heads` are written 0.
 * The codec is dsa_quantize_query's MXFP4 one, bit for bit.
 */
int dsa_quantize_queries_rg(const void* q, int64_t q_row_stride, int64_t q_head_stride,
                            int64_t heads, int64_t rows, void* payload, void* scales,
                            void* stream);

/*
 * dsa_insert_key - LayerNorm (FP32) + BF16 + quantise + insert of indexer keys.
 *
 * Page "cutedsl.dsa.index": insert_key, insert_fp4_key, module docstring;
 * page "amd.ops.fp4_indexer": store_keys (negative slots are padding).
 *
 *   k            BF16 wk projections, key i column c at k[i * k_row_stride + c];
 *                k_row_stride >= 128 and a multiple of 8; k 16-byte aligned.
 *   gamma, beta  FP32 [128] LayerNorm weight and bias; eps the LayerNorm epsilon.
 *   slots        int64 [n]: slot = page * 64 + offset; < 0 = padding (no write);
 *                >= num_pages * 64 is skipped and flagged DSA_STATUS_BAD_SLOT.
 *   cache        uint8, page p at cache + p * page_stride (16-byte aligned,
 *                page_stride a multiple of 16 and >= 8448 (FP8) or 4352 (MXFP4)).
 *                FP8 page: 64 x 128 B E4M3 codes at offset * 128, then 64 x 4 B
 *                scales at 8192 + offset * 4 (FP32 2^e, or the byte e + 127 four
 *                times for DSA_FMT_FP8_MX).  MXFP4 page: 64 x 64 B E2M1 at
 *                offset * 64, then 64 x 4 UE8M0 at 4096 + offset * 4.
 *                DSA_FMT_MXFP4_RG page: the same bytes group-major (see the
 *                format list); page_stride >= 4352 and a multiple of 16.
 *   status       optional int32 device word (may be NULL).
 *
 * The LayerNorm is computed in a fixed order: per 8-column group a sequential
 * FP32 sum, the 16 group sums combined by an xor butterfly (8, 4, 2, 1),
 * correctly rounded division, square root and reciprocal, no fused
 * multiply-add.  Keys with the same slot in one call race (last writer wins).
 */
int dsa_insert_key(int fmt, const void* k, int64_t k_row_stride,
                   const float* gamma, const float* beta, float eps,
                   const int64_t* slots, int64_t n,
                   void* cache, int64_t page_stride, int64_t num_pages,
                   int32_t* status, void* stream);

/*
 * dsa_decode_layout - group verify rows by request and bound their keys.
 *
 * Page "amd.ops.fp4_indexer": decode_layout (without its DCP branch).
 *
 *   seq_lens     int32 [num_seq] global sequence lengths (num_seq >= num_requests;
 *                entries past num_requests are ignored).
 *   query_lens   int32 [num_requests] rows per request (>= 0).
 *   num_rows     rows to bound (>= 0); rows past the last request are padding.
 *   starts       int32 [num_requests + 1] out: [0, cumsum(query_lens)].
 *   row_ends     int32 [num_rows] out: for row r of request q,
 *                max(0, seq_len[q] - query_len[q] + (r - starts[q]) + 1); 0 for padding.
 * Errors (DSA_ERR_INVALID): num_rows < 0, num_requests < 0, num_seq < num_requests.
 */
int dsa_decode_layout(const int32_t* seq_lens, int64_t num_seq,
                      const int32_t* query_lens, int64_t num_requests,
                      int64_t num_rows, int32_t* starts, int32_t* row_ends,
                      void* stream);

/*
 * dsa_decode_layout_dcp - dsa_decode_layout with decode context parallelism.
 *
 * Page "amd.ops.fp4_indexer", decode_layout(..., dcp_rank, dcp_world_size,
 * interleave): a request's key positions are dealt to dcp_world_size ranks
 * in runs of `interleave` consecutive positions (run n to rank n mod world);
 * each rank scores only its own keys, numbered consecutively.  starts are as
 * without DCP; row_ends are rank-local: for a global bound E,
 *   full = E / (world * interleave) * interleave,
 *   row_ends = full + clamp(E - full * world - dcp_rank * interleave, 0, interleave).
 * dcp_world_size == 1 gives dsa_decode_layout's result.
 * Errors (DSA_ERR_INVALID): dcp_rank outside [0, dcp_world_size),
 * dcp_world_size < 1, interleave < 1, and dsa_decode_layout's cases.
 */
int dsa_decode_layout_dcp(const int32_t* seq_lens, int64_t num_seq,
                          const int32_t* query_lens, int64_t num_requests,
                          int64_t num_rows, int64_t dcp_rank,
                          int64_t dcp_world_size, int64_t interleave,
                          int32_t* starts, int32_t* row_ends, void* stream);

/*
 * dsa_prepare_step - dsa_quantize_query, dsa_insert_key and dsa_decode_layout
 * of one decode step in a single launch.
 *
 * Page "cutedsl.dsa.index" (DsaIndex) handles the query and the new key of a
 * token together; page "cutedsl.dsa.overlap" runs this preparation ahead of
 * scoring.  The three parts read and write disjoint buffers, so the results
 * are exactly those of the three calls (in any order); the arguments keep
 * their meaning, layout and checks:
 *   fmt, q, q_row_stride, wv, wv_row_stride, rows, q_out, w_out   as dsa_quantize_query;
 *   k, k_row_stride, gamma, beta, eps, slots, n, cache, page_stride,
 *   num_pages, status                                            as dsa_insert_key;
 *   seq_lens, num_seq, query_lens, num_requests, num_rows,
 *   starts, row_ends                                             as dsa_decode_layout.
 * Any argument error of a part returns that error and launches nothing.
 * Ownership: every buffer belongs to the caller; nothing is allocated.
 */
int dsa_prepare_step(int fmt, const void* q, int64_t q_row_stride,
                     const void* wv, int64_t wv_row_stride, int64_t rows,
                     void* q_out, void* w_out,
                     const void* k, int64_t k_row_stride,
                     const float* gamma, const float* beta, float eps,
                     const int64_t* slots, int64_t n,
                     void* cache, int64_t page_stride, int64_t num_pages,
                     const int32_t* seq_lens, int64_t num_seq,
                     const int32_t* query_lens, int64_t num_requests,
                     int64_t num_rows, int32_t* starts, int32_t* row_ends,
                     int32_t* status, void* stream);

/*
 * dsa_query_norm - the q_a RMSNorm of the packed projection -> q_c (QueryNorm).
 *
 * Page "cutedsl.dsa.overlap", class QueryNorm: row r of q_c is
 * BF16((x[r] * rr) * w) with rr = 1 / sqrt(sum_c x[r][c]^2 / 1536 + eps), in
 * FP32, in one of the page's two summation orders:
 *   variant 0  per-row form: one row per CTA, 8 columns per thread, sequential
 *              FMAs, warp butterfly sums added in warp order;
 *   variant 1  tiled form: one row per warp, 48 columns per lane in four FMA
 *              chains by value index mod 4;
 *   variant -1 the tiled form from 64 rows on, else the per-row form (the
 *              pages do not print their threshold).
 *   x        BF16 [batch][x_row_stride >= 1536, multiple of 8]: columns 0..1535
 *            of each row are q_a; 16-byte aligned.
 *   w        BF16 [1536] weights, 16-byte aligned.
 *   eps      added to the mean square.
 *   out      BF16 [batch][out_row_stride >= 1536, multiple of 8], 16-byte aligned.
 * batch == 0 launches nothing.  Errors: DSA_ERR_INVALID for a negative batch,
 * a bad variant, null pointers, strides or alignment as above.
 */
int dsa_query_norm(const void* x, int64_t x_row_stride, const void* w, float eps,
                   int64_t batch, void* out, int64_t out_row_stride, int variant,
                   void* stream);

/*
 * dsa_workspace_size - bytes of scratch dsa_score_paged needs for these sizes
 * (rows query rows, num_requests requests, max_pages block-table columns, top-k k).
 * The workspace must be zero-filled before its first use; every call that
 * completes leaves it zero-filled again, so it can be reused without clearing.
 */
size_t dsa_workspace_size(int fmt, int64_t rows, int64_t num_requests,
                          int64_t max_pages, int64_t k);

/*
 * dsa_score_paged - paged MQA logits of grouped query rows, fused with top-k.
 *
 * Page "cutedsl.dsa.index" (module docstring: the MQA logits take the FP8 /
 * MXFP4 query and the paged indexer cache); page "amd.ops.fp4_indexer":
 * score_paged (block table, query_starts, row_ends, logits width
 * max_pages * 64); page "cutedsl.dsa.overlap" (scoring and top-k).
 *
 *   q_rows        uint8 [rows][4096] from dsa_quantize_query, 16-byte aligned.
 *   w             BF16 [rows][32] head weights from dsa_quantize_query.
 *   cache         paged cache written by dsa_insert_key (same layout rules:
 *                 base 16-byte aligned, page_stride a multiple of 16).
 *   block_table   int32, request q's page j at block_table[q * bt_stride + j],
 *                 max_pages columns.
 *   starts        int32 [num_requests + 1]: rows starts[q] .. starts[q+1]-1 form
 *                 request q and share its keys.
 *   row_ends      int32 [rows]: row r scores positions t < row_ends[r]
 *                 (bounded by max_pages * 64).  Rows outside every request score
 *                 nothing.
 *   max_query_len the largest starts[q+1] - starts[q] (>= 0; informational).
 *   logits        optional FP32 [rows][logits_ld] out (logits_ld >= max_pages * 64):
 *                 score[r][t] for t < row_ends[r], -inf for the rest of the
 *                 max_pages * 64 columns.  NULL keeps the logits in the workspace.
 *   k, topk       optional top-k (k > 0 and topk != NULL): int32 [rows][k] of
 *                 positions t (logical key indices of the request) of the k
 *                 largest scores of each row, in no particular order; rows with
 *                 at most k keys list 0..row_end-1 in order, then -1.
 *   workspace     scratch of at least dsa_workspace_size(...) bytes, 256-byte
 *                 aligned, zero-filled before first use.
 *   status        optional int32 device word.
 *
 * score[r][t] = sum_h w[r][h] * ReLU(q_h . k_t), q and k dequantised (FP8 keys
 * times their scale; MXFP4 values times their block scales), accumulated in
 * FP32 on the tensor cores.  Keys come from page block_table[q][t / 64], token
 * t % 64.
 */
int dsa_score_paged(int fmt, const void* q_rows, const void* w,
                    const void* cache, int64_t page_stride, int64_t num_pages,
                    const int32_t* block_table, int64_t bt_stride, int64_t max_pages,
                    const int32_t* starts, const int32_t* row_ends,
                    int64_t num_requests, int64_t rows, int64_t max_query_len,
                    float* logits, int64_t logits_ld,
                    int64_t k, int32_t* topk,
                    void* workspace, size_t workspace_bytes,
                    int32_t* status, void* stream);

/*
 * dsa_decode_step - one decode step in one call: dsa_prepare_step, then
 * dsa_score_paged on what it produced.
 *
 * Page "cutedsl.dsa.overlap": the indexer path runs the preparation ahead of
 * "scoring and top-k"; page "cutedsl.dsa.index" (DsaIndex) quantises the query
 * and inserts the new key of a token together.  The call checks every
 * argument of both parts before its first launch and then issues the same
 * launches as the two calls (preparation, plan, scoring, selection), chained
 * by programmatic dependent launch.  Results are those of
 *   dsa_prepare_step(fmt, q, q_row_stride, wv, wv_row_stride, num_rows, q_out,
 *                    w_out, k, k_row_stride, gamma, beta, eps, slots, n, cache,
 *                    page_stride, num_pages, seq_lens, num_seq, query_lens,
 *                    num_requests, num_rows, starts, row_ends, status)
 * followed by
 *   dsa_score_paged(fmt, q_out, w_out, cache, page_stride, num_pages,
 *                   block_table, bt_stride, max_pages, starts, row_ends,
 *                   num_requests, num_rows, max_query_len, logits, logits_ld,
 *                   top_k, topk, workspace, workspace_bytes, status),
 * every argument with the meaning, layout and checks it has there (q_out is
 * uint8 [num_rows][4096], w_out BF16 [num_rows][32]).  Any argument error of
 * either returns that error and launches nothing.  With num_rows = 0 only the
 * keys are inserted.  Ownership: every buffer belongs to the caller; nothing is
 * allocated; the workspace is dsa_score_paged's (dsa_workspace_size).
 */
int dsa_decode_step(int fmt, const void* q, int64_t q_row_stride,
                    const void* wv, int64_t wv_row_stride,
                    const void* k, int64_t k_row_stride,
                    const float* gamma, const float* beta, float eps,
                    const int64_t* slots, int64_t n,
                    void* cache, int64_t page_stride, int64_t num_pages,
                    const int32_t* seq_lens, int64_t num_seq,
                    const int32_t* query_lens, int64_t num_requests, int64_t num_rows,
                    const int32_t* block_table, int64_t bt_stride, int64_t max_pages,
                    int64_t max_query_len, void* q_out, void* w_out,
                    int32_t* starts, int32_t* row_ends,
                    float* logits, int64_t logits_ld, int64_t top_k, int32_t* topk,
                    void* workspace, size_t workspace_bytes,
                    int32_t* status, void* stream);

/*
 * dsa_score_paged_heads - dsa_score_paged for MXFP4 queries of 16, 32 or 64
 * heads in the quantize_queries form.
 *
 * Page "amd.ops.fp4_indexer": score_paged quantises [rows, heads, 128] queries
 * with quantize_queries (heads 16, 32 or 64) and scores them against the
 * MXFP4 cache; its weights carry the head factors but no group scales.
 *
 *   fmt           DSA_FMT_MXFP4 or DSA_FMT_MXFP4_RG (the cache's placement);
 *                 other formats return DSA_ERR_UNSUPPORTED.
 *   heads         16, 32 or 64 (else DSA_ERR_UNSUPPORTED).
 *   payload       uint8 [rows][heads][64] from dsa_quantize_queries_rg, 16-byte
 *                 aligned: head h's E2M1 pairs.
 *   q_scales      uint8 [rows][256] from dsa_quantize_queries_rg (block g of
 *                 head h at g * 64 + h), 16-byte aligned.
 *   w             BF16 [rows][heads] head weights.
 *   every other argument as dsa_score_paged, whose workspace size it uses.
 *
 * score[r][t] = sum_h w[r][h] * ReLU(q_h . k_t) over the query's heads.  A
 * request's rows are scored in groups of min(4, 128 / heads) rows per key
 * read.
 */
int dsa_score_paged_heads(int fmt, int64_t heads, const void* payload, const void* q_scales, const void* w,
                          const void* cache, int64_t page_stride, int64_t num_pages,
                          const int32_t* block_table, int64_t bt_stride, int64_t max_pages,
                          const int32_t* starts, const int32_t* row_ends,
                          int64_t num_requests, int64_t rows, int64_t max_query_len,
                          float* logits, int64_t logits_ld,
                          int64_t k, int32_t* topk,
                          void* workspace, size_t workspace_bytes,
                          int32_t* status, void* stream);

/*
 * dsa_topk_workspace_size - bytes of scratch dsa_topk needs (zero-filled before
 * first use, left zero-filled by every completed call).
 */
size_t dsa_topk_workspace_size(int64_t rows, int64_t k);

/*
 * dsa_topk - top-k positions of each row of an FP32 logits matrix.
 *
 * Page "cutedsl.dsa.overlap" (the indexer path ends in "scoring and top-k");
 * page "amd.ops.fp4_indexer": decode_tile_size (per-row selection scratch).
 *
 *   logits    FP32 [rows][ld], row r valid for t < min(row_ends[r], width).
 *   row_ends  int32 [rows].
 *   out       int32 [rows][k]: positions of the k largest values (any order);
 *             rows with at most k valid entries list them in order, then -1.
 * Equal values at the k-th place are broken arbitrarily.
 */
int dsa_topk(const float* logits, int64_t ld, const int32_t* row_ends,
             int64_t rows, int64_t width, int64_t k, int32_t* out,
             void* workspace, size_t workspace_bytes, void* stream);

/*
 * dsa_topk_merge - the DCP top-k merge and the local slots.
 *
 * Page "cutedsl.dsa.overlap" names this step of the indexer path under DCP
 * (it prints no code).  Every rank has selected its local top-k of a row;
 * the caller gathers all ranks' candidates (for instance with an all-gather)
 * and this call keeps the k_out best of them:
 *   scores     FP32 [rows][scores_ld >= world * k]: rank w's candidates at
 *              columns w*k .. w*k + k - 1; empty candidates -inf.
 *   idx        int32 [rows][idx_ld >= world * k]: their rank-local key
 *              positions (as dsa_decode_layout_dcp numbers them), -1 empty.
 *   interleave the DCP run length.
 *   out        int32 [rows][k_out] out: global key positions of the k_out best
 *              candidates, in no particular order; -1 where a row has fewer
 *              valid candidates (those -1 entries may sit anywhere in the row).
 *   rank, out_local  optional (out_local may be NULL): rank-local positions of
 *              the selected keys that `rank` owns, -1 elsewhere.
 *   workspace  at least dsa_topk_workspace_size(rows, k_out) bytes, 256-byte
 *              aligned, zero-filled before first use (left zero-filled).
 * Errors (DSA_ERR_INVALID): negative sizes, world < 1, interleave < 1, short
 * leading dimensions, null pointers, rank outside [0, world) with out_local.
 */
int dsa_topk_merge(const float* scores, int64_t scores_ld, const int32_t* idx,
                   int64_t idx_ld, int64_t rows, int64_t world, int64_t k,
                   int64_t interleave, int64_t k_out, int32_t* out,
                   int64_t rank, int32_t* out_local, void* workspace,
                   size_t workspace_bytes, void* stream);

/*
 * dsa_topk_noalloc - dsa_topk for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this call; it exists for callers that
 * cannot obtain scratch memory when they call the library: a serving engine
 * that reserved nearly all HBM for its KV cache up front and forbids further
 * cudaMalloc, or a plugin host that passes a kernel its inputs and outputs but
 * no allocator.  It computes what dsa_topk computes, with the same arguments
 * minus the workspace.  Its scratch is a file-scope device array of
 * DSA_TOPK_NOALLOC_SCRATCH_BYTES (about 4.5 MB: for each of the
 * DSA_TOPK_NOALLOC_MAX_ROWS rows an 8 KB histogram, 16 bytes of counters and
 * 64 KB of candidates), held by every GPU that loads the library until the
 * process exits.
 *
 *   - rows > DSA_TOPK_NOALLOC_MAX_ROWS returns DSA_ERR_UNSUPPORTED (split the rows
 *     over several calls).
 *   - Every call looks up the array's device address on the current device
 *     (cudaGetSymbolAddress, a host-side query).  The first call on a device
 *     also loads the library's device code there: make that first call before
 *     any stream capture.
 *   - Every call shares the one array: it clears the parts that must start at
 *     zero on its stream, but calls that overlap on the GPU (other streams or
 *     other threads) race and must be serialised by the caller.
 *   - It calls no cudaMalloc, cudaFree or other allocating routine.
 */
#define DSA_TOPK_NOALLOC_MAX_ROWS 64
#define DSA_TOPK_NOALLOC_SCRATCH_BYTES 4719616
int dsa_topk_noalloc(const float* logits, int64_t ld, const int32_t* row_ends,
                     int64_t rows, int64_t width, int64_t k, int32_t* out, void* stream);

/*
 * dsa_set_score_timing - profiling hook: when both events are non-NULL,
 * dsa_score_paged records `before` just ahead of its scoring kernel and
 * `after` just behind it on the call's stream, so the scoring kernel alone can
 * be timed.  Pass NULLs to switch it off.  Not thread-safe.  The records are
 * "external", so a call captured into a CUDA graph records them on every
 * replay.
 */
void dsa_set_score_timing(void* before, void* after);

/* dsa_timing_event_create / _destroy / _elapsed_ms - CUDA events of the
 * library's runtime for dsa_set_score_timing.  _elapsed_ms waits for `end`
 * and writes the milliseconds between the two records.  Return DSA_OK or
 * DSA_ERR_CUDA. */
int dsa_timing_event_create(void** event);
int dsa_timing_event_destroy(void* event);
int dsa_timing_elapsed_ms(void* start, void* end, float* ms);

/*
 * dsa_probe_mma - measurement helper: the dense tensor-core rate of the MMA
 * kinds the scorer uses, on this GPU.  The pages have no counterpart; it
 * exists so that the scorer's tensor-side roofline has a measured peak.
 *
 * Launches one CTA per SM; each issues `iters` tcgen05.mma instructions of
 * M = 128, N = 128 back to back on operands held in shared memory, into one
 * accumulator in tensor memory: kind 0 = kind::f8f6f4 E4M3 x E4M3 (K = 32),
 * kind 1 = kind::mxf4 packed E2M1 with UE8M0 block scales (K = 64).  Time the
 * launch on `stream` with CUDA events: FLOPs = 2 * 128 * 128 * K * iters * SMs.
 *   status  optional int32 device word: DSA_STATUS_TIMEOUT if the final wait
 *           for the MMAs gave up (then the timing is invalid).
 * Returns DSA_ERR_INVALID for another kind or iters outside [1, 2^22].
 */
int dsa_probe_mma(int kind, int64_t iters, int32_t* status, void* stream);

/* dsa_version - library version string. */
const char* dsa_version(void);

/*
 * dsa_selftest_wait_timeout - exercise the failure detection of the kernels.
 *
 * Launches one thread that waits, with the bounded wait every kernel of this
 * library uses, on a barrier that nothing completes.  The wait gives up after
 * its time limit (about one second), sets DSA_STATUS_TIMEOUT in *status and
 * the kernel returns: the context stays usable.  status: int32 device word.
 * Returns DSA_ERR_INVALID for a null status.
 */
int dsa_selftest_wait_timeout(int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H */
