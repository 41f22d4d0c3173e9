/*
 * irs.h — C ABI of the indexer-routed sparse attention library (libirs.so, sm_103a).
 *
 * The library computes, on one GPU, the hot path of indexer-routed sparse GQA
 * attention as described by the NVIDIA NeMo AutoModel API reference pages
 *   "nemo_automodel.components.models.qwen3_8_flash_next.qsa"       (QSA page),
 *   "nemo_automodel.components.models.step5.sparse"                 (Step-5 sparse page),
 *   "nemo_automodel.components.models.step5.layers" / "...step5.fa4" (windowed GQA),
 *   "nemo_automodel.components.models.common.cudnn_sparse_attention" (latent attention page):
 *
 *   1. a compressed-block indexer: FP32 mean of every c consecutive index keys of a
 *      document, a weighted-ReLU score per (query, visible block) on tensor cores,
 *      and a per-query top-k over blocks;
 *   2. expansion of the chosen blocks into an int32 route row of global token IDs;
 *   3. attention forward over exactly the routed keys and values;
 *   4. its backward (query, key and value gradients over the same routes).
 *
 * Conventions for every call
 *   - All tensor pointers are DEVICE pointers unless stated otherwise, owned by the
 *     caller. The library allocates no memory: scratch space is passed in.
 *   - "bf16" pointers point to IEEE bfloat16 data; they are typed `const void*`.
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default stream)
 *     and is asynchronous: a return value of IRS_OK means the arguments were valid
 *     and the kernels were launched, not that they have finished.
 *   - Host-side validation raises by category, like the pages' error taxonomy
 *     (TypeError / ValueError / RuntimeError): see irs_status. Nothing falls back to
 *     another implementation.
 *   - Conditions only the device can see (route IDs out of range, malformed
 *     cu_seqlens, a bounded wait that gave up) are OR-ed into *err_flag
 *     (IRS_DEVERR_* bits) when err_flag is not NULL. The caller reads it after the
 *     stream has synchronised. No kernel traps.
 *   - irs_last_error() returns a thread-local message for the last non-OK status.
 */
#ifndef IRS_H_
#define IRS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* irs_stream_t;

typedef enum {
  IRS_OK = 0,
  IRS_ERR_TYPE = 1,    /* unsupported element type or layout class (pages: TypeError)   */
  IRS_ERR_VALUE = 2,   /* bad size, shape, stride, alignment, width, scale, NULL, buffer
                          too small (pages: ValueError)                                   */
  IRS_ERR_RUNTIME = 3  /* no usable sm_103 device, or a CUDA launch error (RuntimeError)  */
} irs_status;

/* Bits OR-ed into *err_flag by the kernels. */
#define IRS_DEVERR_ROUTE_ID 0x1   /* a route entry outside [-1, Tk); it was treated as padding */
#define IRS_DEVERR_CU_SEQLENS 0x2 /* cu_seqlens not strictly increasing from 0 to T, or a
                                     document longer than max_doc_len; no route was written  */
#define IRS_DEVERR_TIMEOUT 0x4    /* a bounded on-device wait gave up; outputs are undefined */

/* Version of this ABI (incremented on incompatible change). */
int irs_abi_version(void);

/* Message describing the last non-OK status returned on this host thread. */
const char* irs_last_error(void);

/*
 * Scratch bytes irs_sparse_index_score_topk needs for these sizes (0 on invalid sizes).
 * QSA page, `Qwen3_8_FlashNextQSAIndexer` (the pooled keys [B, floor(S/c), 1, D_index]) and
 * `select_qsa_token_ids` (the FP32 score tensor, which the page bounds by chunking rows).
 * The scratch holds the per-document layout, the pooled bf16 block keys
 * [floor(T/c), Di] and, when the caller passes no score buffer, the FP32 score rows
 * [T, max_doc_len / c].
 */
size_t irs_index_workspace_bytes(int T, int Hi, int Di, int c, int budget, int ndocs, int max_doc_len,
                                 int with_score_buffer);

/*
 * sparse_index_score_topk(qI, kI, w, cu_seqlens, c, budget) -> route_ids
 *
 * QSA page, `select_qsa_token_ids` and `Qwen3_8_FlashNextQSAIndexer`; Step-5 sparse
 * page, `indexer_score_tile` (per-head FP32 weights) and `pack_region_bitmap`.
 *
 * For a query at document-local position tau (document d = [s_d, e_d) of cu_seqlens):
 *   nvis = floor((tau+1)/c) complete blocks are visible; block b is the FP32 mean of
 *   index keys s_d + b*c .. s_d + b*c + c-1 (sequential FP32 sum, one division by c),
 *   rounded once to bf16;
 *   score[b] = sum_h w[t,h] * ReLU(sum_d qI[t,h,d] * kbar[b,d])   (FP32 accumulation);
 *   if nvis > budget/c the budget/c highest scores are kept (ties: lower block index),
 *   otherwise every visible block is kept.
 * Route row t (width W = budget + c - 1, int32, global token IDs):
 *   slots [0, budget): the kept blocks in ascending block order, c tokens each, then -1;
 *   slots [budget, W): the (tau+1) % c tokens s_d + nvis*c .. t of the incomplete block,
 *   then -1. Routes never leave the query's document.
 *
 * qI          bf16 [T, Hi, Di] contiguous (row t*Hi + h has Di elements), 16-byte aligned
 * kI          bf16 [T, Di] contiguous, 16-byte aligned
 * w           fp32 [T, Hi] contiguous
 * cu_seqlens  int32 [ndocs + 1] DEVICE, strictly increasing, 0 .. T
 * ndocs, max_doc_len  host values: number of documents and the longest document
 * T, Hi, Di, c, budget  sizes; Hi a power of two in [1, 256] (IRS_ERR_VALUE otherwise),
 *             Di in {64, 128}, c >= 1, budget % c == 0
 * route_ids   int32 [T, budget + c - 1] output
 * scores_dbg  NULL, or fp32 [T, ld_scores] output: for rows with nvis > budget/c the
 *             entries [0, nvis) receive the block scores; other entries are untouched.
 *             ld_scores >= max_doc_len / c. When not NULL it also serves as the score
 *             scratch, so the workspace may be sized with with_score_buffer = 0.
 * workspace   scratch of at least irs_index_workspace_bytes(...) bytes, 256-byte aligned
 * err_flag    NULL or one device int32 (IRS_DEVERR_* bits are OR-ed in)
 */
irs_status irs_sparse_index_score_topk(const void* qI, const void* kI, const float* w, const int32_t* cu_seqlens,
                                       int ndocs, int max_doc_len, int T, int Hi, int Di, int c, int budget,
                                       int32_t* route_ids, float* scores_dbg, int64_t ld_scores, void* workspace,
                                       size_t workspace_bytes, int32_t* err_flag, irs_stream_t stream);

/*
 * The indexer with its front half: sparse_index_score_topk over normalised and rotated
 * index queries and keys.
 *
 * QSA page, `Qwen3_8_FlashNextQSAIndexer` (the FP32 group means get K RMSNorm and
 * group-start RoPE; the index queries RMSNorm and RoPE) and `apply_qsa_rope` (per-token
 * rotary values cat(cos, sin) over the first rope_dims dims, the rest unchanged). Before
 * scoring:
 *   pooled key b (FP32 group mean, first token s_b):  k~_b = bf16(rope(rmsnorm(kbar_b, k_weight), rope[s_b]))
 *   query row (t, h):                                 q~   = bf16(rope(rmsnorm(qI[t,h], q_weight), rope[t]))
 * with rmsnorm(x, g)_d = (x_d / sqrt(sum_e x_e^2 / Di + eps)) * g_d and rope pairing dims d
 * and d + rope_dims/2 (rotate-half): (y_d cos_d - y_{d+h} sin_d, y_{d+h} cos_d + y_d sin_d).
 * Everything is FP32 with each operation rounded on its own (sum of squares in ascending
 * dim order, IEEE division and square root), then one rounding to bf16, so the transformed
 * operands are reproducible bit for bit. Scoring, top-k and routes are then those of
 * irs_sparse_index_score_topk.
 *
 * q_weight, k_weight  fp32 [Di] DEVICE, 16-byte aligned
 * eps                 >= 0
 * rope                fp32 [T, rope_dims] DEVICE, 16-byte aligned: row t = cat(cos, sin) for
 *                     token t (the caller composes it for document-local positions); NULL if
 *                     rope_dims = 0
 * rope_dims           a multiple of 16 in [0, Di]
 * workspace           at least irs_index_front_workspace_bytes(...) bytes (the plain
 *                     indexer's scratch plus the transformed queries [T, Hi, Di] bf16 and the
 *                     FP32 group means [floor(T/c), Di])
 * Other arguments as for irs_sparse_index_score_topk.
 */
size_t irs_index_front_workspace_bytes(int T, int Hi, int Di, int c, int budget, int ndocs, int max_doc_len,
                                       int with_score_buffer);
irs_status irs_sparse_index_score_topk_front(const void* qI, const void* kI, const float* w,
                                             const int32_t* cu_seqlens, int ndocs, int max_doc_len, int T, int Hi,
                                             int Di, int c, int budget, const float* q_weight, const float* k_weight,
                                             float eps, const float* rope, int rope_dims, int32_t* route_ids,
                                             float* scores_dbg, int64_t ld_scores, void* workspace,
                                             size_t workspace_bytes, int32_t* err_flag, irs_stream_t stream);

/*
 * The front half alone, for checking the transformed operands bit for bit: q_out bf16
 * [T, Hi, Di] receives the transformed queries, k_out bf16 [floor(T/c), Di] the transformed
 * pooled keys in pooled order (document by document; rows past the last complete block are
 * zero). Same definitions and arguments as irs_sparse_index_score_topk_front; the
 * workspace is sized by irs_index_front_workspace_bytes(..., with_score_buffer = 0).
 */
irs_status irs_index_front_operands(const void* qI, const void* kI, const int32_t* cu_seqlens, int ndocs,
                                    int max_doc_len, int T, int Hi, int Di, int c, int budget, const float* q_weight,
                                    const float* k_weight, float eps, const float* rope, int rope_dims, void* q_out,
                                    void* k_out, void* workspace, size_t workspace_bytes, int32_t* err_flag,
                                    irs_stream_t stream);

/*
 * The indexer with a separate selection per KV group.
 *
 * Step-5 sparse page, `Step5SparseIndexer.forward` (region IDs per KV group) and
 * `indexer_score_tile` (one weighted-ReLU score per group, with that group's FP32 head
 * weights; signed weights allowed). Group g of token t scores the shared pooled keys with
 * its own Hi query heads and weights and selects its own blocks, each group exactly as
 * irs_sparse_index_score_topk does for one (same kernels, run once per group).
 *
 * qI          bf16 [T, G, Hi, Di] contiguous;  w  fp32 [T, G, Hi] contiguous
 * route_ids   int32 [T, G, budget + c - 1]
 * scores_dbg  NULL or fp32 [T, G, ld_scores] (row (t, g) at (t*G + g) * ld_scores)
 * workspace   irs_index_workspace_bytes(T, Hi, Di, c, budget, ndocs, max_doc_len, ...) bytes:
 *             the score scratch is reused group after group
 * Other arguments as for irs_sparse_index_score_topk; G >= 1.
 */
irs_status irs_sparse_index_score_topk_grouped(const void* qI, const void* kI, const float* w,
                                               const int32_t* cu_seqlens, int ndocs, int max_doc_len, int T, int G,
                                               int Hi, int Di, int c, int budget, int32_t* route_ids,
                                               float* scores_dbg, int64_t ld_scores, void* workspace,
                                               size_t workspace_bytes, int32_t* err_flag, irs_stream_t stream);

/*
 * The indexer with FP8 E4M3 scoring operands.
 *
 * Step-5 sparse page, `indexer_score_tile` (queries and summaries rounded to FP8 E4M3) and
 * `_summarize_region_payload` (summaries keep both roundings, BF16 then FP8). Queries are
 * rounded bf16 -> E4M3, pooled keys FP32 mean -> bf16 -> E4M3 (to nearest, ties to even,
 * saturating at +-448), and the block scores run on the kind::f8f6f4 tensor-core path
 * (products of E4M3 values accumulated in FP32); top-k and routes as in
 * irs_sparse_index_score_topk. Di must be 128. The workspace is
 * irs_index_e4m3_workspace_bytes(...) bytes (the plain scratch plus the byte copies of the
 * queries [T, Hi, Di] and pooled keys [floor(T/c), Di]). Other arguments as for
 * irs_sparse_index_score_topk.
 */
size_t irs_index_e4m3_workspace_bytes(int T, int Hi, int Di, int c, int budget, int ndocs, int max_doc_len,
                                      int with_score_buffer);
irs_status irs_sparse_index_score_topk_e4m3(const void* qI, const void* kI, const float* w, const int32_t* cu_seqlens,
                                            int ndocs, int max_doc_len, int T, int Hi, int Di, int c, int budget,
                                            int32_t* route_ids, float* scores_dbg, int64_t ld_scores, void* workspace,
                                            size_t workspace_bytes, int32_t* err_flag, irs_stream_t stream);

/*
 * The indexer's projections: queries, raw keys and signed head weights from hidden states.
 *
 * QSA page, the indexer class (`Qwen3_8_FlashNextQSAIndexer`): one fused projection gives
 * the raw query/key layout [B, S, (H_index + 1) * D_index], split into queries
 * [B, S, H_index, D_index] and raw keys [B, S, 1, D_index]. Step-5 sparse page,
 * `Step5IndexerWeightProjection`: FP32 source weights matched by a BF16 projection give
 * signed FP32 head weights. Here one weight matrix holds all three (N = (Hi+1)*Di + Hi):
 *   out[t, n] = sum_k hidden[t, k] * weight[n, k]   (products of bf16 values, FP32 sums)
 *   qI[t, h, d] = bf16(out[t, h*Di + d])             (round to nearest even)
 *   kI[t, d]    = bf16(out[t, Hi*Di + d])
 *   w[t, h]     = out[t, (Hi+1)*Di + h]              (FP32)
 * It runs as one tcgen05 GEMM (128 tokens x 256 columns per tile, K in 64-wide steps).
 *
 * hidden  bf16 [T, H] contiguous, 16-byte aligned; H a positive multiple of 8
 * weight  bf16 [N, H] contiguous, 16-byte aligned (row n gives output column n)
 * qI      bf16 [T, Hi, Di] out, 16-byte aligned; Di a positive multiple of 8
 * kI      bf16 [T, Di] out, 16-byte aligned
 * w       fp32 [T, Hi] out
 * Errors: IRS_ERR_VALUE for NULL or unaligned pointers and unsupported sizes, before any
 * work is queued; IRS_ERR_RUNTIME when a launch fails. err_flag as elsewhere (a bounded
 * wait that gave up).
 */
irs_status irs_indexer_projection(const void* hidden, const void* weight, int T, int H, int Hi, int Di, void* qI,
                                  void* kI, float* w, int32_t* err_flag, irs_stream_t stream);

/*
 * The projection with the query side of the indexer front half fused into its epilogue
 * (QSA page, the indexer class: RMSNorm and RoPE of the queries; `apply_qsa_rope`). qI
 * receives the transformed queries, equal bit for bit to
 * irs_index_front_operands' queries computed from irs_indexer_projection's qI: each head
 * row is rounded to bf16, normalised with q_weight and rotated with the token's rotary
 * row, in the FP32 order documented for irs_sparse_index_score_topk_front, then rounded to
 * bf16. kI stays raw (the keys get their front half after pooling) and w is unchanged.
 * Di must be 64 or 128; q_weight fp32 [Di] and rope fp32 [T, rope_dims] as for
 * irs_sparse_index_score_topk_front (16-byte aligned).
 */
irs_status irs_indexer_projection_front(const void* hidden, const void* weight, int T, int H, int Hi, int Di,
                                        const float* q_weight, float eps, const float* rope, int rope_dims, void* qI,
                                        void* kI, float* w, int32_t* err_flag, irs_stream_t stream);

/*
 * irs_sparse_index_score_topk_front for queries that arrive already transformed (from
 * irs_indexer_projection_front): the pooled keys get K RMSNorm and group-start RoPE with
 * k_weight, the queries are scored as given. Workspace, arguments and errors as for
 * irs_sparse_index_score_topk_front (without q_weight).
 */
irs_status irs_sparse_index_score_topk_front_keys(const void* qI, const void* kI, const float* w,
                                                  const int32_t* cu_seqlens, int ndocs, int max_doc_len, int T, int Hi,
                                                  int Di, int c, int budget, const float* k_weight, float eps,
                                                  const float* rope, int rope_dims, int32_t* route_ids,
                                                  float* scores_dbg, int64_t ld_scores, void* workspace,
                                                  size_t workspace_bytes, int32_t* err_flag, irs_stream_t stream);

/*
 * Step-5 learned-logit region summaries.
 *
 * Step-5 sparse page: `Step5SparseIndexer.project_keys` returns the index keys and
 * per-dimension compression logits shaped like them; `_summarize_region_payload` turns
 * them into region summaries in FP32 and keeps both roundings (bf16, then FP8 E4M3);
 * `indexer_score_tile` scores E4M3-rounded bf16 region summaries; `region_metadata` resets
 * the regions at every document boundary. A region is a run of c consecutive tokens of
 * one document (as the pooled blocks of irs_sparse_index_score_topk). Per region and dim d:
 *   m_d = max_j z[j, d]
 *   e_j = exp(z[j, d] - m_d)
 *   summary_d = e4m3(bf16((sum_j e_j k[j, d]) / (sum_j e_j)))
 * The sums run over the region's tokens in order, in FP32, without fused multiply-add.
 * exp is evaluated in FP32 as follows, each operation rounded to nearest:
 *   t = x * log2(e),  n = rint(t),  f = t - n;
 *   2^f by its degree-7 Taylor polynomial in Horner form;
 *   the result times 2^n, and 0 where t < -125.
 * E4M3 rounding is to nearest, ties to even, saturating at +-448.
 *
 * irs_region_summaries writes the summaries alone:
 *   kI, z      bf16 [T, Di] contiguous (keys and compression logits), 16-byte aligned
 *   out        bf16 [floor(T/c), Di]: row blk_off[d] + b is region b of document d (blk_off
 *              the running count of floor(len/c) over documents); rows past the last region
 *              are zeroed
 *   workspace  irs_region_summaries_workspace_bytes(T, Di, c, ndocs, max_doc_len) bytes,
 *              256-byte aligned
 *   Di 64 or 128; other arguments as for irs_sparse_index_score_topk.
 *
 * irs_sparse_index_score_topk_summaries is the per-group indexer of
 * irs_sparse_index_score_topk_grouped with these summaries as the block keys instead of
 * the means:
 *   - e4m3_queries = 0: bf16 queries, Di 64 or 128;
 *   - e4m3_queries = 1: queries rounded bf16 -> E4M3 and the scores on the kind::f8f6f4
 *     path, as in irs_sparse_index_score_topk_e4m3; Di must be 128.
 * qI [T, G, Hi, Di], w [T, G, Hi], route_ids [T, G, budget + c - 1] and scores_dbg as in
 * irs_sparse_index_score_topk_grouped (G = 1 is the ungrouped indexer). The workspace is
 * irs_index_summaries_workspace_bytes(...) bytes.
 * Errors: IRS_ERR_VALUE for NULL or unaligned pointers and unsupported sizes, before any
 * work is queued; IRS_ERR_RUNTIME when a launch fails.
 */
size_t irs_region_summaries_workspace_bytes(int T, int Di, int c, int ndocs, int max_doc_len);
irs_status irs_region_summaries(const void* kI, const void* z, const int32_t* cu_seqlens, int ndocs, int max_doc_len,
                                int T, int Di, int c, void* out, void* workspace, size_t workspace_bytes,
                                int32_t* err_flag, irs_stream_t stream);
size_t irs_index_summaries_workspace_bytes(int T, int G, int Hi, int Di, int c, int budget, int ndocs,
                                           int max_doc_len, int e4m3_queries, int with_score_buffer);
irs_status irs_sparse_index_score_topk_summaries(const void* qI, const void* kI, const void* z, const float* w,
                                                 const int32_t* cu_seqlens, int ndocs, int max_doc_len, int T, int G,
                                                 int Hi, int Di, int c, int budget, int e4m3_queries,
                                                 int32_t* route_ids, float* scores_dbg, int64_t ld_scores,
                                                 void* workspace, size_t workspace_bytes, int32_t* err_flag,
                                                 irs_stream_t stream);

/*
 * irs_sparse_index_score_topk without a workspace: the same computation and arguments,
 * minus `workspace` / `workspace_bytes`. The reference pages have no counterpart; this
 * entry point exists for callers that cannot allocate device memory for the library,
 * such as plugins of inference runtimes that are given no allocator, or loops that must
 * not risk the device-wide synchronisation a cudaMalloc can cause. It allocates nothing:
 * its scratch is one fixed 16 MiB device array inside libirs.so (every GPU that loads
 * the library holds it until the process exits).
 *
 * - Sizes whose scratch (irs_index_workspace_bytes(..., with_score_buffer)) exceeds
 *   16 MiB are rejected with IRS_ERR_VALUE. Passing a score buffer (scores_dbg) keeps
 *   the FP32 score rows out of the scratch; the rest is small (the pooled keys
 *   [floor(T/c), Di] bf16 plus per-document offsets).
 * - The first call on a device looks up the array's device address for that device;
 *   make that first call before any stream capture.
 * - All calls share the one array, which keeps whatever the last call left there. Each
 *   call writes every scratch word it later reads (pooled-key rows past the last complete
 *   block are zeroed, not left over), so nothing of an earlier call leaks into a result.
 *   Calls whose work overlaps on the GPU (different streams, or different host threads)
 *   race on it: serialise them.
 */
irs_status irs_sparse_index_score_topk_noalloc(const void* qI, const void* kI, const float* w,
                                               const int32_t* cu_seqlens, int ndocs, int max_doc_len, int T, int Hi,
                                               int Di, int c, int budget, int32_t* route_ids, float* scores_dbg,
                                               int64_t ld_scores, int32_t* err_flag, irs_stream_t stream);

/*
 * Top-k, bitmap packing and expansion from given FP32 scores (the second half of
 * irs_sparse_index_score_topk), so that routes can be compared bit for bit with an
 * independent implementation that selects from the same scores. QSA page,
 * `select_qsa_token_ids` (top budget/c blocks, expanded to token IDs, tail appended);
 * Step-5 sparse page, `pack_region_bitmap` (the selection as 32-bit words). It runs the
 * same top-k kernels as irs_sparse_index_score_topk.
 *
 * scores      fp32 [T, ld_scores]; for row t with nvis > budget/c, entries [0, nvis)
 *             are read (NaN is outside the contract); other rows are not read.
 * Other arguments as in irs_sparse_index_score_topk.
 */
irs_status irs_topk_from_scores(const float* scores, int64_t ld_scores, const int32_t* cu_seqlens, int ndocs,
                                int max_doc_len, int T, int c, int budget, int32_t* route_ids, int32_t* err_flag,
                                irs_stream_t stream);

/*
 * Sliding window in front of an indexer route (Step-5 layers page: the attention keys
 * come from a sliding window or from the CSA selection; the windowed workload uses both).
 *   out[t, j]          = t - window + 1 + j if that token is in t's document, else -1
 *   out[t, window + j] = route_ids[t, j] if it is < t - window + 1, else -1
 * so the composed row never repeats an ID.
 * route_ids int32 [T, W]; out int32 [T, window + W]; window >= 1.
 */
irs_status irs_compose_window_routes(const int32_t* route_ids, int W, const int32_t* cu_seqlens, int ndocs,
                                     int T, int window, int32_t* out, int32_t* err_flag, irs_stream_t stream);

/*
 * sparse_gqa_attn_fwd(q, k, v, route_ids, scale) -> out, lse
 *
 * QSA page, `gathered_qsa_gqa_attention`; latent attention page,
 * `cudnn_sparse_attention` (keys = full latent rows, values = their first Dv dims,
 * passed as v = k with Dv < Dqk).
 *
 * For query t and query head h, with KV head g = h / (Hq/Hkv) (consecutive query
 * heads share a KV head) and R_t = { r = route_ids[t, i] : 0 <= r < Tk }:
 *   s_r   = scale * q[t,h,:] . k[r,g,:]
 *   out   = sum_r exp(s_r - m) v[r,g,:] / sum_r exp(s_r - m),   m = max_r s_r
 *   lse   = m + ln sum_r exp(s_r - m)                (natural log)
 * A row with no valid entry gives out = 0 and lse = -inf. Entries equal to -1 are
 * padding; other entries outside [0, Tk) are also padding and set IRS_DEVERR_ROUTE_ID.
 * IDs within a row must be distinct (a repeated ID is counted twice).
 *
 * q     bf16, element (t,h,d) at q + t*q_stride_t + h*q_stride_h + d
 * k     bf16, element (r,g,d) at k + r*k_stride_t + g*k_stride_h + d
 * v     bf16, element (r,g,d) at v + r*v_stride_t + g*v_stride_h + d (may alias k)
 *       strides are in elements; rows must be 16-byte aligned (strides multiple of 8)
 * route_ids  int32, entry (t,i) at route_ids + t*route_stride + i, 0 <= i < W
 * sizes: Hq % Hkv == 0, Dqk % 64 == 0 and Dqk <= 576, Dv % 128 == 0 and Dv <= 512,
 *        one chunk of 128 gathered key rows (plus value rows unless v aliases k) and
 *        the query tile must fit in 227 KB of shared memory (IRS_ERR_VALUE otherwise;
 *        about Dqk + Dv <= 704 without aliasing),
 *        1 <= W <= 4096
 * scale > 0 (finite)
 * out   bf16 [T, Hq, Dv] contiguous;  lse  fp32 [T, Hq] contiguous (may be NULL)
 *
 * Kernels (results are the same definition either way): latent shapes (Hkv == 1, v the
 * first Dv dims of k, Hq % 64 == 0, Dqk >= Dv + 64, W <= 2048) run a kernel that keeps
 * 64 query heads' output in tensor memory; all other shapes run the GQA kernel, which
 * loads runs of 64 consecutive routed rows as TMA tiles when the K/V rows exceed half the
 * L2. Every on-device wait is bounded; one that gives up sets IRS_DEVERR_TIMEOUT.
 */
irs_status irs_sparse_gqa_attn_fwd(const void* q, int64_t q_stride_t, int64_t q_stride_h, const void* k,
                                   int64_t k_stride_t, int64_t k_stride_h, const void* v, int64_t v_stride_t,
                                   int64_t v_stride_h, const int32_t* route_ids, int64_t route_stride, int T,
                                   int Tk, int Hq, int Hkv, int Dqk, int Dv, int W, float scale, void* out,
                                   float* lse, int32_t* err_flag, irs_stream_t stream);

/*
 * sparse_gqa_attn_fwd with a route per KV group.
 *
 * Step-5 sparse page, `Step5SparseIndexer.forward` (region IDs per KV group); the query
 * heads of KV head g (h / (Hq/Hkv) == g) attend the entries of route row (t, g) at
 * route_ids + t*route_stride + g*route_group_stride (W entries, -1 padding), with the
 * definitions of irs_sparse_gqa_attn_fwd. route_group_stride >= W. Runs the GQA kernel once
 * per KV head.
 */
irs_status irs_sparse_gqa_attn_fwd_grouped(const void* q, int64_t q_stride_t, int64_t q_stride_h, const void* k,
                                           int64_t k_stride_t, int64_t k_stride_h, const void* v, int64_t v_stride_t,
                                           int64_t v_stride_h, const int32_t* route_ids, int64_t route_stride,
                                           int64_t route_group_stride, int T, int Tk, int Hq, int Hkv, int Dqk,
                                           int Dv, int W, float scale, void* out, float* lse, int32_t* err_flag,
                                           irs_stream_t stream);

/*
 * sparse_gqa_attn_fwd with a sliding window in front of every route row.
 *
 * Step-5 layers page, `Step5Attention` (a query's keys come from a sliding window and from
 * the indexer's selection). The result equals irs_compose_window_routes followed by
 * irs_sparse_gqa_attn_fwd, without the composed route tensor: query t (document d =
 * [s_d, e_d) of cu_seqlens) attends the tokens max(s_d, t - window + 1) .. t, then the
 * entries of route row t that lie before t - window + 1 (entries inside the window are
 * skipped, so no key counts twice). Keys are taken in that order, the order of the composed
 * route, so the outputs are bit-identical to the composed call. The window's keys are not
 * read from memory: 64 consecutive window tokens load as one TMA row tile when the K/V
 * rows exceed half the L2.
 *
 * cu_seqlens  int32 [ndocs + 1] DEVICE, strictly increasing from 0 to T (as for the
 *             indexer); ndocs >= 1. Queries and keys share token positions (Tk >= T).
 * window      >= 1; W + window <= 4096.
 * Other arguments and limits as for irs_sparse_gqa_attn_fwd; every shape runs the GQA
 * kernel (latent shapes included).
 */
irs_status irs_sparse_gqa_attn_fwd_windowed(const void* q, int64_t q_stride_t, int64_t q_stride_h, const void* k,
                                            int64_t k_stride_t, int64_t k_stride_h, const void* v,
                                            int64_t v_stride_t, int64_t v_stride_h, const int32_t* route_ids,
                                            int64_t route_stride, const int32_t* cu_seqlens, int ndocs, int window,
                                            int T, int Tk, int Hq, int Hkv, int Dqk, int Dv, int W, float scale,
                                            void* out, float* lse, int32_t* err_flag, irs_stream_t stream);

/*
 * sparse_gqa_attn_bwd(q, k, v, route_ids, out, lse, dout, scale) -> dq, dk, dv
 *
 * Latent attention page, `_CudnnSparseAttention.backward` (the BF16 output gradient is
 * mapped to gradients of the query and of the gathered K/V rows); the same gradients
 * for the GQA routes of the QSA page. The backward of irs_sparse_gqa_attn_fwd for the
 * loss sum(out * dout). With the notation above and the forward's out and lse:
 *   p_r   = exp(s_r - lse),   D = dout[t,h,:] . out[t,h,:]
 *   ds_r  = p_r (dout[t,h,:] . v[r,g,:] - D)
 *   dq[t,h,:]  = scale * sum_r ds_r k[r,g,:]          (written)
 *   dk[r,g,:] += scale * ds_r q[t,h,:]                  (added, over every t and h in g)
 *   dv[r,g,:] += p_r dout[t,h,:]                        (added)
 * D is taken from the BF16 forward output, as the forward saves it; route semantics
 * (padding, IRS_DEVERR_ROUTE_ID, distinct IDs) are those of the forward.
 *
 * q, k, v, route_ids, T, Tk, Hq, Hkv, Dqk, Dv, W, scale: as for the forward (same limits)
 * out   bf16 [T, Hq, Dv] contiguous: the forward's output
 * lse   fp32 [T, Hq] contiguous: the forward's lse (natural log; required)
 * dout  bf16 [T, Hq, Dv] contiguous
 * dq    fp32 [T, Hq, Dqk] contiguous, overwritten
 * dk    fp32 [Tk, Hkv, Dqk] contiguous, 16-byte aligned, ACCUMULATED (zero it first)
 * dv    fp32 [Tk, Hkv, Dv] contiguous, 16-byte aligned, accumulated; dv may equal dk
 *       only when v is a view of k's first Dv dims (same pointer and strides, Dv <= Dqk;
 *       IRS_ERR_VALUE otherwise): the value gradient is then added into the first Dv dims
 *       of each dk row, which is the gradient of latent rows used as keys and values
 * The accumulation uses FP32 atomics, so dk and dv are not bit-reproducible across runs.
 * One CTA per (query, KV head, block of up to 16 query heads), waiting on nothing outside
 * itself. Blocks of 8 or more heads with separate K and V (dims multiples of 64 up to 256)
 * run on the tensor cores, where P and ds are rounded once to bf16 as product operands (as
 * the forward rounds P); smaller blocks and latent rows run in FP32 on the CUDA cores.
 */
irs_status irs_sparse_gqa_attn_bwd(const void* q, int64_t q_stride_t, int64_t q_stride_h, const void* k,
                                   int64_t k_stride_t, int64_t k_stride_h, const void* v, int64_t v_stride_t,
                                   int64_t v_stride_h, const int32_t* route_ids, int64_t route_stride,
                                   const void* out, const float* lse, const void* dout, int T, int Tk, int Hq,
                                   int Hkv, int Dqk, int Dv, int W, float scale, float* dq, float* dk, float* dv,
                                   int32_t* err_flag, irs_stream_t stream);

/*
 * Failure-detection self-test (no counterpart on the reference pages). Launches one
 * bounded on-device wait on a barrier phase that nothing completes: after limit_ns
 * (1e6 .. 2e9) the wait gives up, ORs IRS_DEVERR_TIMEOUT into *err_flag and the kernel
 * returns, leaving the context usable. It is the same bounded wait every kernel of this
 * library uses, so a caller can check on its own device that a stalled pipeline reports
 * an error instead of hanging. err_flag: one device int32 (required).
 */
irs_status irs_check_bounded_wait(uint64_t limit_ns, int32_t* err_flag, irs_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* IRS_H_ */
