// Internal declarations shared by the translation units of libirs.so.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/irs.h"

namespace irs {

// Sizes and scratch offsets of one indexer call.
constexpr int kMaxIndexCtas = 160;   // persistent CTAs of the score kernel (>= one per SM)

// Indexer front half: RMSNorm weights of queries and keys, eps, and the per-token rotary
// table [T, rope_dims] = cat(cos, sin) (device pointers).
struct FrontHalf {
  const float* q_weight;   // nullptr: the queries are already transformed (keys only)
  const float* k_weight;
  float eps;
  const float* rope;
  int rope_dims;
};

struct IndexPlan {
  int kb;              // blocks kept per query (budget / c)
  int QT;              // queries per score tile (256 / Hi)
  int tau_sparse;      // first document-local position with more than kb visible blocks
  int nblk_cap;        // rows of the pooled-key buffer (T / c)
  int64_t ldS;         // row stride of the score buffer (max_doc_len / c)
  int stages;          // 64-dim key atoms in the score kernel's TMA ring
  size_t off_meta, off_blk, off_tile, off_kbar, off_scores, ws_bytes;
  size_t off_qfront, off_kbar32;   // front half only: transformed queries, FP32 group means
  size_t off_q8, off_k8;           // E4M3 operands only: queries and pooled keys, one byte each
  size_t score_smem, topk_smem;
};

IndexPlan plan_index(int T, int Hi, int Di, int c, int budget, int ndocs, int max_doc_len, bool with_scores,
                     bool front = false, bool e4m3 = false, int G = 1);
size_t topk_smem_bytes(int nvis_cap, int kb);

cudaError_t configure_score_kernels(size_t smem);
cudaError_t configure_topk_kernel(size_t smem);
// front == nullptr: the plain indexer. Otherwise the scores use the transformed queries
// (tm_q must map ws + p.off_qfront) and the transformed pooled keys. G > 1: per-group
// selection; tm_q maps [T][G*Hi][Di], w is [T, G, Hi], route [T, G, W], and group g's score
// rows start at scores + g * scores_group_stride (row stride ldS). e4m3: queries and pooled
// keys are rounded to FP8 E4M3 and scored with kind::f8f6f4 (tm_q / tm_k map the byte copies
// at ws + p.off_q8 / p.off_k8; Di = 128). z != nullptr: the block keys are the Step-5
// learned-logit summaries of kI under the compression logits z [T, Di] (E4M3 values; as bytes
// for e4m3, else as bf16) instead of the means.
cudaError_t launch_index(const IndexPlan& p, const __nv_bfloat16* qI, const __nv_bfloat16* kI, const float* w,
                         const int32_t* cu, int ndocs, int max_doc_len, int T, int Hi, int Di, int c, int budget,
                         int32_t* route, float* scores, int64_t ldS, uint8_t* ws, int32_t* err,
                         const CUtensorMap& tm_q, const CUtensorMap& tm_k, int num_sms, cudaStream_t stream,
                         const FrontHalf* front = nullptr, int G = 1, int64_t scores_group_stride = 0,
                         bool e4m3 = false, const __nv_bfloat16* z = nullptr);
// The learned-logit summaries alone, as E4M3-valued bf16 [nblk_cap, Di] into out (rows past
// the region count zeroed); uses the plan's layout scratch.
cudaError_t launch_summaries(const IndexPlan& p, const __nv_bfloat16* kI, const __nv_bfloat16* z, const int32_t* cu,
                             int ndocs, int max_doc_len, int T, int Di, int c, uint8_t* ws, int32_t* err,
                             __nv_bfloat16* out, cudaStream_t stream);
// The front half alone: transformed queries [T*Hi, Di] into q_out, pooled keys [T/c, Di]
// into k_out (rows past the last complete block zeroed).
cudaError_t launch_front_operands(const IndexPlan& p, const __nv_bfloat16* qI, const __nv_bfloat16* kI,
                                  const int32_t* cu, int ndocs, int max_doc_len, int T, int Hi, int Di, int c,
                                  uint8_t* ws, int32_t* err, const FrontHalf& front, __nv_bfloat16* q_out,
                                  __nv_bfloat16* k_out, cudaStream_t stream);
cudaError_t launch_topk_from_scores(const float* scores, int64_t ldS, const int32_t* cu, int ndocs, int max_doc_len,
                                    int T, int c, int budget, int32_t* route, int32_t* err, cudaStream_t stream);
cudaError_t launch_compose_window(const int32_t* route, int W, const int32_t* cu, int ndocs, int T, int window,
                                  int32_t* out, int32_t* err, cudaStream_t stream);

// The indexer's projections (one GEMM): out[T, N] = X[T, H] . W[N, H]^T with N =
// (Hi+1)*Di + Hi; columns [0, Hi*Di) -> qI (bf16), the next Di -> kI (bf16), the last Hi
// -> w (fp32).
struct ProjArgs {
  int T, H, N, Hi, Di;
  __nv_bfloat16* qI;
  __nv_bfloat16* kI;
  float* w;
  int32_t* err;
  int tiles_m, tiles_n;
  // query front half fused into the epilogue (q_weight == nullptr: off; Di 64 or 128)
  const float* q_weight;
  float eps;
  const float* rope;   // [T, rope_dims] = cat(cos, sin)
  int rope_dims;
};
size_t proj_smem_bytes();
cudaError_t configure_proj_kernel();
cudaError_t launch_proj(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const ProjArgs& a, int num_sms,
                        cudaStream_t stream);

// Gathered sparse attention.
constexpr int kMaxKvMaps = 8;   // KV heads handled by one launch (one row-tile map per head)

struct AttnMaps {
  CUtensorMap k[kMaxKvMaps];    // [Tk rows x Dqk] of KV head g0+i, box {64, 64}, SW128
  CUtensorMap v[kMaxKvMaps];    // [Tk rows x Dv]  (unused when v aliases k)
};

struct AttnArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  int64_t q_st, q_sh, k_st, k_sh, v_st, v_sh;
  const int32_t* route;
  int64_t route_stride;
  __nv_bfloat16* out;
  float* lse;
  int32_t* err;
  int T, Tk, Hq, Hkv, Dqk, Dv, W;
  int G;          // query heads per KV head
  int HB;         // query heads handled by one sub-item (<= 16)
  int nhb;        // head blocks per KV head
  int g0, ng;     // KV heads [g0, g0+ng) handled by this launch
  int v_alias;    // 1: values are the first Dv dims of the gathered key rows
  int tile_runs;  // 1: the maps are valid; 64 consecutive routed rows load as one TMA tile
  int stages;
  float scale_log2;  // scale * log2(e)
  // sliding window in front of the route (0 = none): query t also attends the tokens
  // max(s_d, t - window + 1) .. t of its document (cu: cu_seqlens, ndocs entries + 1), and
  // route IDs inside that window are skipped
  const int32_t* cu;
  int ndocs;
  int window;
  int flag_routes;   // 1: this launch reports route IDs out of range (each route row once)
};

struct AttnPlan {
  int stages;
  size_t smem;
  int grid;
  long long items;
  int nh_class;   // 4, 8 or 16: head loop length of the softmax warps
};

AttnPlan plan_attn(const AttnArgs& a, int num_sms);

// Latent attention (one KV head whose rows are keys and, by their first Dv dims, values):
// 64 query heads per work item with the output accumulated in TMEM.
bool mla_supported(const AttnArgs& a);
size_t mla_smem_bytes(const AttnArgs& a);
cudaError_t configure_mla_kernel(size_t smem);
cudaError_t launch_mla(const AttnArgs& a, int num_sms, cudaStream_t stream);
cudaError_t configure_attn_kernel(size_t smem);
cudaError_t launch_attn(const AttnMaps& maps, const AttnArgs& a, const AttnPlan& p, cudaStream_t stream);

// Attention backward (CUDA cores): one CTA per (query, KV head, block of <= 16 heads).
struct BwdArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  int64_t q_st, q_sh, k_st, k_sh, v_st, v_sh;
  const int32_t* route;
  int64_t route_stride;
  const __nv_bfloat16* out;   // [T, Hq, Dv] contiguous
  const float* lse;           // [T, Hq]
  const __nv_bfloat16* dout;  // [T, Hq, Dv] contiguous
  float* dq;                  // [T, Hq, Dqk], written
  float* dk;                  // [Tk, Hkv, Dqk], added to
  float* dv;                  // [Tk, Hkv, Dv], added to (unused when dv_alias)
  int32_t* err;
  int T, Tk, Hq, Hkv, Dqk, Dv, W;
  int G, HB, nhb;
  int v_alias;    // 1: value rows are the first Dv dims of the key rows
  int dv_alias;   // 1: the value gradient is added into the first Dv dims of dk's rows
  int nkc;        // routed rows staged per step
  float scale, scale_log2;
};

size_t bwd_smem_bytes(const BwdArgs& a);
int bwd_pick_rows(const BwdArgs& a, size_t max_smem);
int bwd_max_heads();
cudaError_t configure_bwd_kernel(size_t smem);
cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream);
// The tensor-core backward (separate K and V, Dqk and Dv multiples of 64 up to 256).
bool bwd_tc_supported(const BwdArgs& a);
cudaError_t launch_bwd_tc(const BwdArgs& a, unsigned items, cudaStream_t stream);

}  // namespace irs
