// C ABI of libirs.so: argument validation (by the pages' error categories), device
// checks, TMA descriptor encoding and kernel launches. See include/irs.h for the
// contract of every entry point.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "irs_internal.h"
#include "irs_ptx.cuh"

namespace {

thread_local char g_msg[512] = "";

irs_status fail(irs_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return s;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

struct DeviceInfo {
  bool checked = false;
  bool ok = false;
  int num_sms = 0;
  size_t l2_bytes = 0;
  size_t score_smem = 0, topk_smem = 0, attn_smem = 0, mla_smem = 0, bwd_smem = 0;   // largest configured so far
  bool proj_configured = false;
};
constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// The current device must be an sm_103 GPU; returns its slot.
irs_status current_device(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(IRS_ERR_RUNTIME, "no CUDA device: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(IRS_ERR_RUNTIME, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.checked) {
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int l2 = 0;
    cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
    d.l2_bytes = (size_t)(l2 > 0 ? l2 : 0);
    d.checked = true;
    d.ok = (major == 10 && minor == 3);
    d.num_sms = sms;
  }
  if (!d.ok) return fail(IRS_ERR_RUNTIME, "libirs needs an sm_103 (GB300) device; device %d is not one", dev);
  *out = &d;
  return IRS_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 tensor map [rows][inner] (inner contiguous), SW128 boxes of {64, box_rows}.
irs_status make_tmap(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return fail(IRS_ERR_RUNTIME, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(IRS_ERR_RUNTIME, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return IRS_OK;
}

// 2-D bf16 row-tile map: rows of `inner` elements `row_stride` elements apart, box {64, 64}
// (one SW128 atom of 64 consecutive rows).
irs_status make_row_tile_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t row_stride) {
  auto fn = encode_fn();
  if (fn == nullptr) return fail(IRS_ERR_RUNTIME, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_stride * 2};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(IRS_ERR_RUNTIME, "cuTensorMapEncodeTiled (row tiles) failed (%d)", (int)r);
  return IRS_OK;
}

// 3-D bf16 map of index queries [T][rows_per_token][Di] (contiguous), box {64, Hi, 256/Hi}:
// the (query, head) rows of one score tile, for any head group of the token.
irs_status make_query_tiles_map(CUtensorMap* m, const void* base, uint64_t Di, uint64_t rows_per_token, uint64_t T,
                                uint32_t Hi) {
  auto fn = encode_fn();
  if (fn == nullptr) return fail(IRS_ERR_RUNTIME, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[3] = {Di, rows_per_token, T};
  cuuint64_t strides[2] = {Di * 2, rows_per_token * Di * 2};
  cuuint32_t box[3] = {64, Hi, 256 / Hi};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(IRS_ERR_RUNTIME, "cuTensorMapEncodeTiled (query tiles) failed (%d)", (int)r);
  return IRS_OK;
}

// Byte maps for E4M3 operands (128-byte SW128 rows of 128 elements): the queries as
// [T][rows_per_token][Di] with box {128, Hi, 256/Hi} (rows_per_token = G*Hi), the pooled keys
// as [krows][Di] with box {128, 128}.
irs_status make_e4m3_maps(CUtensorMap* tq, CUtensorMap* tk, const void* q8, const void* k8, uint64_t Di, uint64_t Hi,
                          uint64_t rows_per_token, uint64_t T, uint64_t krows) {
  auto fn = encode_fn();
  if (fn == nullptr) return fail(IRS_ERR_RUNTIME, "cuTensorMapEncodeTiled is unavailable");
  {
    cuuint64_t dims[3] = {Di, rows_per_token, T};
    cuuint64_t strides[2] = {Di, rows_per_token * Di};
    cuuint32_t box[3] = {128, (cuuint32_t)Hi, (cuuint32_t)(256 / Hi)};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(q8), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(IRS_ERR_RUNTIME, "cuTensorMapEncodeTiled (E4M3 queries) failed (%d)", (int)r);
  }
  cuuint64_t dims[2] = {Di, krows};
  cuuint64_t strides[1] = {Di};
  cuuint32_t box[2] = {128, 128};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(k8), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(IRS_ERR_RUNTIME, "cuTensorMapEncodeTiled (E4M3 keys) failed (%d)", (int)r);
  return IRS_OK;
}

irs_status launch_status(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return fail(IRS_ERR_RUNTIME, "%s: %s", what, cudaGetErrorString(e));
  return IRS_OK;
}

constexpr size_t kMaxSmem = 227 * 1024;

irs_status check_index_sizes(int T, int Hi, int Di, int c, int budget, int ndocs, int max_doc_len) {
  if (T < 1) return fail(IRS_ERR_VALUE, "T must be >= 1 (got %d)", T);
  if (ndocs < 1 || ndocs > T) return fail(IRS_ERR_VALUE, "ndocs must be in [1, T] (got %d)", ndocs);
  if (max_doc_len < 1 || max_doc_len > T) return fail(IRS_ERR_VALUE, "max_doc_len must be in [1, T]");
  if (!pow2(Hi) || Hi > 256) return fail(IRS_ERR_VALUE, "Hi must be a power of two in [1, 256] (got %d)", Hi);
  if (Di != 64 && Di != 128) return fail(IRS_ERR_VALUE, "Di must be 64 or 128 (got %d)", Di);
  if (c < 1) return fail(IRS_ERR_VALUE, "c must be >= 1 (got %d)", c);
  if (budget < c || budget % c != 0) return fail(IRS_ERR_VALUE, "budget must be a positive multiple of c");
  if ((long long)T * Hi >= (1LL << 31)) return fail(IRS_ERR_VALUE, "T*Hi too large");
  if ((long long)budget + c - 1 >= (1LL << 24)) return fail(IRS_ERR_VALUE, "route width too large");
  if (irs::topk_smem_bytes(max_doc_len / c > 0 ? max_doc_len / c : 1, budget / c) > kMaxSmem)
    return fail(IRS_ERR_VALUE, "max_doc_len / c too large for the on-chip top-k (max about 48k blocks)");
  return IRS_OK;
}

// Raise the dynamic shared-memory limits of the indexer kernels to what this call needs.
irs_status configure_index(DeviceInfo* dev, const irs::IndexPlan& p) {
  if (p.score_smem > kMaxSmem) return fail(IRS_ERR_VALUE, "score tile does not fit in shared memory");
  std::lock_guard<std::mutex> lk(g_dev_mu);
  irs_status s = IRS_OK;
  if (dev->score_smem < p.score_smem) {
    if ((s = launch_status(irs::configure_score_kernels(p.score_smem), "configuring scoring")) != IRS_OK) return s;
    dev->score_smem = p.score_smem;
  }
  if (dev->topk_smem < p.topk_smem) {
    if ((s = launch_status(irs::configure_topk_kernel(p.topk_smem), "configuring top-k")) != IRS_OK) return s;
    dev->topk_smem = p.topk_smem;
  }
  return IRS_OK;
}

}  // namespace

extern "C" {

int irs_abi_version(void) { return 1; }

const char* irs_last_error(void) { return g_msg; }

size_t irs_index_workspace_bytes(int T, int Hi, int Di, int c, int budget, int ndocs, int max_doc_len,
                                 int with_score_buffer) {
  if (check_index_sizes(T, Hi, Di, c, budget, ndocs, max_doc_len) != IRS_OK) return 0;
  return irs::plan_index(T, Hi, Di, c, budget, ndocs, max_doc_len, with_score_buffer != 0).ws_bytes;
}

}  // extern "C"

namespace {

irs_status check_front(const float* q_weight, const float* k_weight, float eps, const float* rope, int rope_dims,
                       int Di) {
  if (!q_weight || !k_weight) return fail(IRS_ERR_VALUE, "NULL RMSNorm weights");
  if (!aligned16(q_weight) || !aligned16(k_weight) || (rope != nullptr && !aligned16(rope)))
    return fail(IRS_ERR_VALUE, "RMSNorm weights and the rotary table must be 16-byte aligned");
  if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(IRS_ERR_VALUE, "eps must be finite and >= 0");
  if (rope_dims < 0 || rope_dims > Di || rope_dims % 16 != 0)
    return fail(IRS_ERR_VALUE, "rope_dims must be a multiple of 16 in [0, Di] (got %d)", rope_dims);
  if (rope_dims > 0 && rope == nullptr) return fail(IRS_ERR_VALUE, "NULL rotary table");
  return IRS_OK;
}

// The indexer with or without its front half (front == nullptr).
irs_status index_impl(const void* qI, const void* kI, const float* w, const int32_t* cu_seqlens, int ndocs,
                      int max_doc_len, int T, int Hi, int Di, int c, int budget, const irs::FrontHalf* front,
                      int32_t* route_ids, float* scores_dbg, int64_t ld_scores, void* workspace,
                      size_t workspace_bytes, int32_t* err_flag, irs_stream_t stream, int G = 1,
                      bool e4m3 = false, const void* z = nullptr) {
  irs_status s = check_index_sizes(T, Hi, Di, c, budget, ndocs, max_doc_len);
  if (s != IRS_OK) return s;
  if (e4m3 && (Di != 128 || front != nullptr))
    return fail(IRS_ERR_VALUE, "E4M3 scoring needs Di = 128 (no front half)");
  if (z != nullptr && !aligned16(z)) return fail(IRS_ERR_VALUE, "the compression logits must be 16-byte aligned");
  if (G < 1 || (long long)T * G * Hi >= (1LL << 31)) return fail(IRS_ERR_VALUE, "bad group count %d", G);
  if (!qI || !kI || !w || !cu_seqlens || !route_ids || !workspace)
    return fail(IRS_ERR_VALUE, "NULL tensor pointer");
  if (!aligned16(qI) || !aligned16(kI)) return fail(IRS_ERR_VALUE, "qI and kI must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(IRS_ERR_VALUE, "workspace must be 256-byte aligned");
  const irs::IndexPlan p =
      irs::plan_index(T, Hi, Di, c, budget, ndocs, max_doc_len, scores_dbg == nullptr, front != nullptr, e4m3, G);
  if (scores_dbg != nullptr && ld_scores < p.ldS)
    return fail(IRS_ERR_VALUE, "ld_scores must be >= max_doc_len / c (%lld)", (long long)p.ldS);
  if (workspace_bytes < p.ws_bytes)
    return fail(IRS_ERR_VALUE, "workspace too small: %zu < %zu bytes", workspace_bytes, p.ws_bytes);
  DeviceInfo* dev = nullptr;
  if ((s = current_device(&dev)) != IRS_OK) return s;
  if ((s = configure_index(dev, p)) != IRS_OK) return s;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // score rows: the caller's [T, G, ld_scores] (group g of token t at (t*G + g) * ld_scores),
  // or the workspace's [T, ldS], reused group after group
  float* scores = scores_dbg != nullptr ? scores_dbg : reinterpret_cast<float*>(ws + p.off_scores);
  const int64_t ldS = scores_dbg != nullptr ? ld_scores * G : p.ldS;
  const int64_t group_stride = scores_dbg != nullptr ? ld_scores : 0;
  CUtensorMap tm_q, tm_k;
  // with the front half the scores read the transformed queries from the workspace (unless
  // the caller's queries are already transformed)
  const void* qsrc =
      (front != nullptr && front->q_weight != nullptr) ? static_cast<const void*>(ws + p.off_qfront) : qI;
  if (e4m3) {
    if ((s = make_e4m3_maps(&tm_q, &tm_k, ws + p.off_q8, ws + p.off_k8, (uint64_t)Di, (uint64_t)Hi,
                            (uint64_t)G * Hi, (uint64_t)T, (uint64_t)p.nblk_cap)) != IRS_OK)
      return s;
  } else {
    if ((s = make_query_tiles_map(&tm_q, qsrc, (uint64_t)Di, (uint64_t)G * Hi, (uint64_t)T, (uint32_t)Hi)) != IRS_OK)
      return s;
    if ((s = make_tmap(&tm_k, ws + p.off_kbar, (uint64_t)Di, (uint64_t)p.nblk_cap, 128)) != IRS_OK) return s;
  }
  return launch_status(irs::launch_index(p, static_cast<const __nv_bfloat16*>(qI),
                                         static_cast<const __nv_bfloat16*>(kI), w, cu_seqlens, ndocs, max_doc_len, T,
                                         Hi, Di, c, budget, route_ids, scores, ldS, ws, err_flag, tm_q, tm_k,
                                         dev->num_sms, reinterpret_cast<cudaStream_t>(stream), front, G,
                                         group_stride, e4m3, static_cast<const __nv_bfloat16*>(z)),
                       "launching the indexer");
}

}  // namespace

extern "C" {

irs_status irs_sparse_index_score_topk(const void* qI, const void* kI, const float* w, const int32_t* cu_seqlens,
                                       int ndocs, int max_doc_len, int T, int Hi, int Di, int c, int budget,
                                       int32_t* route_ids, float* scores_dbg, int64_t ld_scores, void* workspace,
                                       size_t workspace_bytes, int32_t* err_flag, irs_stream_t stream) {
  return index_impl(qI, kI, w, cu_seqlens, ndocs, max_doc_len, T, Hi, Di, c, budget, nullptr, route_ids, scores_dbg,
                    ld_scores, workspace, workspace_bytes, err_flag, stream);
}

size_t irs_index_front_workspace_bytes(int T, int Hi, int Di, int c, int budget, int ndocs, int max_doc_len,
                                       int with_score_buffer) {
  if (check_index_sizes(T, Hi, Di, c, budget, ndocs, max_doc_len) != IRS_OK) return 0;
  return irs::plan_index(T, Hi, Di, c, budget, ndocs, max_doc_len, with_score_buffer != 0, true).ws_bytes;
}

irs_status irs_sparse_index_score_topk_front(const void* qI, const void* kI, const float* w,
                                             const int32_t* cu_seqlens, int ndocs, int max_doc_len, int T, int Hi,
                                             int Di, int c, int budget, const float* q_weight, const float* k_weight,
                                             float eps, const float* rope, int rope_dims, int32_t* route_ids,
                                             float* scores_dbg, int64_t ld_scores, void* workspace,
                                             size_t workspace_bytes, int32_t* err_flag, irs_stream_t stream) {
  irs_status s = check_front(q_weight, k_weight, eps, rope, rope_dims, Di);
  if (s != IRS_OK) return s;
  const irs::FrontHalf f{q_weight, k_weight, eps, rope, rope_dims};
  return index_impl(qI, kI, w, cu_seqlens, ndocs, max_doc_len, T, Hi, Di, c, budget, &f, route_ids, scores_dbg,
                    ld_scores, workspace, workspace_bytes, err_flag, stream);
}

irs_status irs_sparse_index_score_topk_grouped(const void* qI, const void* kI, const float* w,
                                               const int32_t* cu_seqlens, int ndocs, int max_doc_len, int T, int G,
                                               int Hi, int Di, int c, int budget, int32_t* route_ids,
                                               float* scores_dbg, int64_t ld_scores, void* workspace,
                                               size_t workspace_bytes, int32_t* err_flag, irs_stream_t stream) {
  return index_impl(qI, kI, w, cu_seqlens, ndocs, max_doc_len, T, Hi, Di, c, budget, nullptr, route_ids, scores_dbg,
                    ld_scores, workspace, workspace_bytes, err_flag, stream, G);
}

size_t irs_index_e4m3_workspace_bytes(int T, int Hi, int Di, int c, int budget, int ndocs, int max_doc_len,
                                      int with_score_buffer) {
  if (check_index_sizes(T, Hi, Di, c, budget, ndocs, max_doc_len) != IRS_OK || Di != 128) return 0;
  return irs::plan_index(T, Hi, Di, c, budget, ndocs, max_doc_len, with_score_buffer != 0, false, true).ws_bytes;
}

irs_status irs_sparse_index_score_topk_e4m3(const void* qI, const void* kI, const float* w, const int32_t* cu_seqlens,
                                            int ndocs, int max_doc_len, int T, int Hi, int Di, int c, int budget,
                                            int32_t* route_ids, float* scores_dbg, int64_t ld_scores, void* workspace,
                                            size_t workspace_bytes, int32_t* err_flag, irs_stream_t stream) {
  return index_impl(qI, kI, w, cu_seqlens, ndocs, max_doc_len, T, Hi, Di, c, budget, nullptr, route_ids, scores_dbg,
                    ld_scores, workspace, workspace_bytes, err_flag, stream, 1, true);
}

size_t irs_index_summaries_workspace_bytes(int T, int G, int Hi, int Di, int c, int budget, int ndocs,
                                           int max_doc_len, int e4m3_queries, int with_score_buffer) {
  if (check_index_sizes(T, Hi, Di, c, budget, ndocs, max_doc_len) != IRS_OK || G < 1) return 0;
  if (e4m3_queries != 0 && Di != 128) return 0;
  return irs::plan_index(T, Hi, Di, c, budget, ndocs, max_doc_len, with_score_buffer != 0, false, e4m3_queries != 0,
                         G)
      .ws_bytes;
}

irs_status irs_sparse_index_score_topk_summaries(const void* qI, const void* kI, const void* z, const float* w,
                                                 const int32_t* cu_seqlens, int ndocs, int max_doc_len, int T, int G,
                                                 int Hi, int Di, int c, int budget, int e4m3_queries,
                                                 int32_t* route_ids, float* scores_dbg, int64_t ld_scores,
                                                 void* workspace, size_t workspace_bytes, int32_t* err_flag,
                                                 irs_stream_t stream) {
  if (z == nullptr) return fail(IRS_ERR_VALUE, "NULL compression logits");
  return index_impl(qI, kI, w, cu_seqlens, ndocs, max_doc_len, T, Hi, Di, c, budget, nullptr, route_ids, scores_dbg,
                    ld_scores, workspace, workspace_bytes, err_flag, stream, G, e4m3_queries != 0, z);
}

size_t irs_region_summaries_workspace_bytes(int T, int Di, int c, int ndocs, int max_doc_len) {
  if (check_index_sizes(T, 1, Di, c, c, ndocs, max_doc_len) != IRS_OK) return 0;
  return irs::plan_index(T, 1, Di, c, c, ndocs, max_doc_len, false).ws_bytes;
}

irs_status irs_region_summaries(const void* kI, const void* z, const int32_t* cu_seqlens, int ndocs, int max_doc_len,
                                int T, int Di, int c, void* out, void* workspace, size_t workspace_bytes,
                                int32_t* err_flag, irs_stream_t stream) {
  irs_status s = check_index_sizes(T, 1, Di, c, c, ndocs, max_doc_len);
  if (s != IRS_OK) return s;
  if (!kI || !z || !cu_seqlens || !out || !workspace) return fail(IRS_ERR_VALUE, "NULL tensor pointer");
  if (!aligned16(kI) || !aligned16(z) || !aligned16(out))
    return fail(IRS_ERR_VALUE, "kI, z and out must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(IRS_ERR_VALUE, "workspace must be 256-byte aligned");
  const irs::IndexPlan p = irs::plan_index(T, 1, Di, c, c, ndocs, max_doc_len, false);
  if (workspace_bytes < p.ws_bytes)
    return fail(IRS_ERR_VALUE, "workspace too small: %zu < %zu bytes", workspace_bytes, p.ws_bytes);
  DeviceInfo* dev = nullptr;
  if ((s = current_device(&dev)) != IRS_OK) return s;
  return launch_status(irs::launch_summaries(p, static_cast<const __nv_bfloat16*>(kI),
                                             static_cast<const __nv_bfloat16*>(z), cu_seqlens, ndocs, max_doc_len, T,
                                             Di, c, static_cast<uint8_t*>(workspace), err_flag,
                                             static_cast<__nv_bfloat16*>(out), reinterpret_cast<cudaStream_t>(stream)),
                       "launching the region summaries");
}

}  // extern "C"

namespace {

irs_status projection_impl(const void* hidden, const void* weight, int T, int H, int Hi, int Di, void* qI, void* kI,
                           float* w, int32_t* err_flag, irs_stream_t stream, const float* q_weight, float eps,
                           const float* rope, int rope_dims) {
  if (T < 1 || H < 8 || H % 8 != 0) return fail(IRS_ERR_VALUE, "need T >= 1 and H a positive multiple of 8");
  if (Hi < 1 || Di < 8 || Di % 8 != 0) return fail(IRS_ERR_VALUE, "need Hi >= 1 and Di a positive multiple of 8");
  const long long N = (long long)(Hi + 1) * Di + Hi;
  if (N >= (1LL << 24) || (long long)T * N >= (1LL << 40)) return fail(IRS_ERR_VALUE, "projection too large");
  if (!hidden || !weight || !qI || !kI || !w) return fail(IRS_ERR_VALUE, "NULL tensor pointer");
  if (!aligned16(hidden) || !aligned16(weight) || !aligned16(qI) || !aligned16(kI))
    return fail(IRS_ERR_VALUE, "hidden, weight, qI and kI must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(w) & 3u) != 0) return fail(IRS_ERR_VALUE, "w must be 4-byte aligned");
  DeviceInfo* dev = nullptr;
  irs_status s = current_device(&dev);
  if (s != IRS_OK) return s;
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!dev->proj_configured) {
      if ((s = launch_status(irs::configure_proj_kernel(), "configuring the projection")) != IRS_OK) return s;
      dev->proj_configured = true;
    }
  }
  CUtensorMap tm_x, tm_w;
  if ((s = make_tmap(&tm_x, hidden, (uint64_t)H, (uint64_t)T, 128)) != IRS_OK) return s;
  if ((s = make_tmap(&tm_w, weight, (uint64_t)H, (uint64_t)N, 256)) != IRS_OK) return s;
  irs::ProjArgs a{T, H, (int)N, Hi, Di, static_cast<__nv_bfloat16*>(qI), static_cast<__nv_bfloat16*>(kI), w,
                  err_flag, (T + 127) / 128, (int)((N + 255) / 256), q_weight, eps, rope, rope_dims};
  return launch_status(irs::launch_proj(tm_x, tm_w, a, dev->num_sms, reinterpret_cast<cudaStream_t>(stream)),
                       "launching the projection");
}

}  // namespace

extern "C" {

irs_status irs_indexer_projection(const void* hidden, const void* weight, int T, int H, int Hi, int Di, void* qI,
                                  void* kI, float* w, int32_t* err_flag, irs_stream_t stream) {
  return projection_impl(hidden, weight, T, H, Hi, Di, qI, kI, w, err_flag, stream, nullptr, 0.f, nullptr, 0);
}

irs_status irs_sparse_index_score_topk_front_keys(const void* qI, const void* kI, const float* w,
                                                  const int32_t* cu_seqlens, int ndocs, int max_doc_len, int T, int Hi,
                                                  int Di, int c, int budget, const float* k_weight, float eps,
                                                  const float* rope, int rope_dims, int32_t* route_ids,
                                                  float* scores_dbg, int64_t ld_scores, void* workspace,
                                                  size_t workspace_bytes, int32_t* err_flag, irs_stream_t stream) {
  irs_status s = check_front(k_weight, k_weight, eps, rope, rope_dims, Di);
  if (s != IRS_OK) return s;
  const irs::FrontHalf f{nullptr, k_weight, eps, rope, rope_dims};
  return index_impl(qI, kI, w, cu_seqlens, ndocs, max_doc_len, T, Hi, Di, c, budget, &f, route_ids, scores_dbg,
                    ld_scores, workspace, workspace_bytes, err_flag, stream);
}

irs_status irs_indexer_projection_front(const void* hidden, const void* weight, int T, int H, int Hi, int Di,
                                        const float* q_weight, float eps, const float* rope, int rope_dims, void* qI,
                                        void* kI, float* w, int32_t* err_flag, irs_stream_t stream) {
  if (Di != 64 && Di != 128) return fail(IRS_ERR_VALUE, "the fused front half needs Di = 64 or 128 (got %d)", Di);
  irs_status s = check_front(q_weight, q_weight, eps, rope, rope_dims, Di);
  if (s != IRS_OK) return s;
  return projection_impl(hidden, weight, T, H, Hi, Di, qI, kI, w, err_flag, stream, q_weight, eps, rope, rope_dims);
}

irs_status irs_index_front_operands(const void* qI, const void* kI, const int32_t* cu_seqlens, int ndocs,
                                    int max_doc_len, int T, int Hi, int Di, int c, int budget, const float* q_weight,
                                    const float* k_weight, float eps, const float* rope, int rope_dims, void* q_out,
                                    void* k_out, void* workspace, size_t workspace_bytes, int32_t* err_flag,
                                    irs_stream_t stream) {
  irs_status s = check_index_sizes(T, Hi, Di, c, budget, ndocs, max_doc_len);
  if (s != IRS_OK) return s;
  if ((s = check_front(q_weight, k_weight, eps, rope, rope_dims, Di)) != IRS_OK) return s;
  if (!qI || !kI || !cu_seqlens || !q_out || !k_out || !workspace) return fail(IRS_ERR_VALUE, "NULL tensor pointer");
  if (!aligned16(qI) || !aligned16(kI) || !aligned16(q_out) || !aligned16(k_out))
    return fail(IRS_ERR_VALUE, "qI, kI, q_out and k_out must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(IRS_ERR_VALUE, "workspace must be 256-byte aligned");
  const irs::IndexPlan p = irs::plan_index(T, Hi, Di, c, budget, ndocs, max_doc_len, false, true);
  if (workspace_bytes < p.ws_bytes)
    return fail(IRS_ERR_VALUE, "workspace too small: %zu < %zu bytes", workspace_bytes, p.ws_bytes);
  DeviceInfo* dev = nullptr;
  if ((s = current_device(&dev)) != IRS_OK) return s;
  const irs::FrontHalf f{q_weight, k_weight, eps, rope, rope_dims};
  return launch_status(irs::launch_front_operands(p, static_cast<const __nv_bfloat16*>(qI),
                                                  static_cast<const __nv_bfloat16*>(kI), cu_seqlens, ndocs,
                                                  max_doc_len, T, Hi, Di, c, static_cast<uint8_t*>(workspace),
                                                  err_flag, f, static_cast<__nv_bfloat16*>(q_out),
                                                  static_cast<__nv_bfloat16*>(k_out),
                                                  reinterpret_cast<cudaStream_t>(stream)),
                       "launching the indexer front half");
}

irs_status irs_topk_from_scores(const float* scores, int64_t ld_scores, const int32_t* cu_seqlens, int ndocs,
                                int max_doc_len, int T, int c, int budget, int32_t* route_ids, int32_t* err_flag,
                                irs_stream_t stream) {
  irs_status s = check_index_sizes(T, 1, 64, c, budget, ndocs, max_doc_len);
  if (s != IRS_OK) return s;
  if (!scores || !cu_seqlens || !route_ids) return fail(IRS_ERR_VALUE, "NULL tensor pointer");
  if (ld_scores < max_doc_len / c) return fail(IRS_ERR_VALUE, "ld_scores must be >= max_doc_len / c");
  DeviceInfo* dev = nullptr;
  if ((s = current_device(&dev)) != IRS_OK) return s;
  const size_t smem = irs::topk_smem_bytes(max_doc_len / c > 0 ? max_doc_len / c : 1, budget / c);
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (dev->topk_smem < smem) {
      if ((s = launch_status(irs::configure_topk_kernel(smem), "configuring top-k")) != IRS_OK) return s;
      dev->topk_smem = smem;
    }
  }
  return launch_status(irs::launch_topk_from_scores(scores, ld_scores, cu_seqlens, ndocs, max_doc_len, T, c, budget,
                                                    route_ids, err_flag, reinterpret_cast<cudaStream_t>(stream)),
                       "launching top-k");
}

irs_status irs_compose_window_routes(const int32_t* route_ids, int W, const int32_t* cu_seqlens, int ndocs,
                                     int T, int window, int32_t* out, int32_t* err_flag, irs_stream_t stream) {
  if (T < 1 || W < 1 || window < 1 || ndocs < 1 || ndocs > T)
    return fail(IRS_ERR_VALUE, "bad sizes (T=%d W=%d window=%d ndocs=%d)", T, W, window, ndocs);
  if ((long long)W + window >= (1LL << 24)) return fail(IRS_ERR_VALUE, "composed width too large");
  if (!route_ids || !cu_seqlens || !out) return fail(IRS_ERR_VALUE, "NULL tensor pointer");
  DeviceInfo* dev = nullptr;
  irs_status s = current_device(&dev);
  if (s != IRS_OK) return s;
  return launch_status(irs::launch_compose_window(route_ids, W, cu_seqlens, ndocs, T, window, out, err_flag,
                                                  reinterpret_cast<cudaStream_t>(stream)),
                       "launching window composition");
}

}  // extern "C"

namespace {

// Forward attention over routes, optionally with a sliding window in front of each route
// (window > 0: cu_seqlens / ndocs give the documents the window stays inside).
irs_status attn_fwd_impl(const void* q, int64_t q_stride_t, int64_t q_stride_h, const void* k, int64_t k_stride_t,
                         int64_t k_stride_h, const void* v, int64_t v_stride_t, int64_t v_stride_h,
                         const int32_t* route_ids, int64_t route_stride, int T, int Tk, int Hq, int Hkv, int Dqk,
                         int Dv, int W, float scale, const int32_t* cu_seqlens, int ndocs, int window, void* out,
                         float* lse, int32_t* err_flag, irs_stream_t stream, int64_t route_group_stride = 0) {
  if (T < 0 || Tk < 1 || Hq < 1 || Hkv < 1) return fail(IRS_ERR_VALUE, "bad sizes (T=%d Tk=%d Hq=%d Hkv=%d)", T, Tk, Hq, Hkv);
  if (Hq % Hkv != 0) return fail(IRS_ERR_VALUE, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
  if (Dqk < 64 || Dqk > 576 || Dqk % 64 != 0) return fail(IRS_ERR_VALUE, "Dqk must be a multiple of 64 in [64, 576]");
  if (Dv < 128 || Dv > 512 || Dv % 128 != 0) return fail(IRS_ERR_VALUE, "Dv must be a multiple of 128 in [128, 512]");
  if (W < 1 || W > 4096) return fail(IRS_ERR_VALUE, "route width W must be in [1, 4096] (got %d)", W);
  if (route_stride < W) return fail(IRS_ERR_VALUE, "route_stride must be >= W");
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(IRS_ERR_VALUE, "scale must be positive and finite");
  if (T == 0) return IRS_OK;
  if (!q || !k || !v || !route_ids || !out) return fail(IRS_ERR_VALUE, "NULL tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(IRS_ERR_VALUE, "q, k, v and out must be 16-byte aligned");
  if (q_stride_t % 8 || q_stride_h % 8 || k_stride_t % 8 || k_stride_h % 8 || v_stride_t % 8 || v_stride_h % 8)
    return fail(IRS_ERR_VALUE, "q/k/v strides must be multiples of 8 elements (16 bytes)");
  if (q_stride_t < 0 || q_stride_h < 0 || k_stride_t < 0 || k_stride_h < 0 || v_stride_t < 0 || v_stride_h < 0)
    return fail(IRS_ERR_VALUE, "negative strides are not supported");
  DeviceInfo* dev = nullptr;
  irs_status s = current_device(&dev);
  if (s != IRS_OK) return s;

  irs::AttnArgs a{};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.q_st = q_stride_t; a.q_sh = q_stride_h;
  a.k_st = k_stride_t; a.k_sh = k_stride_h;
  a.v_st = v_stride_t; a.v_sh = v_stride_h;
  a.route = route_ids;
  a.route_stride = route_stride;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.lse = lse;
  a.err = err_flag;
  a.T = T; a.Tk = Tk; a.Hq = Hq; a.Hkv = Hkv; a.Dqk = Dqk; a.Dv = Dv; a.W = W;
  a.G = Hq / Hkv;
  a.HB = a.G < 16 ? a.G : 16;
  a.nhb = (a.G + a.HB - 1) / a.HB;
  a.v_alias = (v == k && v_stride_t == k_stride_t && v_stride_h == k_stride_h && Dv <= Dqk) ? 1 : 0;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.cu = cu_seqlens;
  a.ndocs = ndocs;
  a.window = window;
  a.flag_routes = 1;
  if (window == 0 && route_group_stride == 0 && irs::mla_supported(a)) {
    const size_t smem = irs::mla_smem_bytes(a);
    {
      std::lock_guard<std::mutex> lk(g_dev_mu);
      if (dev->mla_smem < smem) {
        if ((s = launch_status(irs::configure_mla_kernel(smem), "configuring latent attention")) != IRS_OK) return s;
        dev->mla_smem = smem;
      }
    }
    return launch_status(irs::launch_mla(a, dev->num_sms, reinterpret_cast<cudaStream_t>(stream)),
                         "launching latent attention");
  }
  const irs::AttnPlan p = irs::plan_attn(a, dev->num_sms);
  if (p.smem > kMaxSmem) return fail(IRS_ERR_VALUE, "attention tile does not fit in shared memory");
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (dev->attn_smem < p.smem) {
      if ((s = launch_status(irs::configure_attn_kernel(p.smem), "configuring attention")) != IRS_OK) return s;
      dev->attn_smem = p.smem;
    }
  }
  // one launch per group of up to kMaxKvMaps KV heads (one row-tile map per head and operand)
  // per-group routes: one launch per KV head, on that head's route rows
  const int gstep = route_group_stride != 0 ? 1 : irs::kMaxKvMaps;
  for (int g0 = 0; g0 < Hkv; g0 += gstep) {
    const int ng = Hkv - g0 < gstep ? Hkv - g0 : gstep;
    a.route = route_ids + (int64_t)g0 * route_group_stride;
    a.flag_routes = (route_group_stride != 0 || g0 == 0) ? 1 : 0;
    irs::AttnMaps maps;
    memset(&maps, 0, sizeof(maps));
    // Runs of 64 consecutive routed rows load as TMA row tiles when the key/value rows cannot
    // stay L2-resident (more than half the L2): the tiles keep many more bytes in flight for
    // DRAM latency than 16-byte copies. Rows that do stay in L2 are served faster by the copies.
    const double kv_bytes = (double)Tk * Hkv * (Dqk + (a.v_alias ? 0 : Dv)) * 2.0;
    a.tile_runs = (Tk >= 64 && kv_bytes > 0.5 * (double)dev->l2_bytes) ? 1 : 0;
    for (int i = 0; i < ng && a.tile_runs; ++i) {
      const __nv_bfloat16* kb = a.k + (int64_t)(g0 + i) * k_stride_h;
      if ((s = make_row_tile_map(&maps.k[i], kb, (uint64_t)Dqk, (uint64_t)Tk, (uint64_t)k_stride_t)) != IRS_OK)
        return s;
      if (!a.v_alias) {
        const __nv_bfloat16* vb = a.v + (int64_t)(g0 + i) * v_stride_h;
        if ((s = make_row_tile_map(&maps.v[i], vb, (uint64_t)Dv, (uint64_t)Tk, (uint64_t)v_stride_t)) != IRS_OK)
          return s;
      }
    }
    a.g0 = g0;
    a.ng = ng;
    if ((s = launch_status(irs::launch_attn(maps, a, p, reinterpret_cast<cudaStream_t>(stream)),
                           "launching attention")) != IRS_OK)
      return s;
  }
  return IRS_OK;
}

}  // namespace

extern "C" {

irs_status irs_sparse_gqa_attn_fwd(const void* q, int64_t q_stride_t, int64_t q_stride_h, const void* k,
                                   int64_t k_stride_t, int64_t k_stride_h, const void* v, int64_t v_stride_t,
                                   int64_t v_stride_h, const int32_t* route_ids, int64_t route_stride, int T,
                                   int Tk, int Hq, int Hkv, int Dqk, int Dv, int W, float scale, void* out,
                                   float* lse, int32_t* err_flag, irs_stream_t stream) {
  return attn_fwd_impl(q, q_stride_t, q_stride_h, k, k_stride_t, k_stride_h, v, v_stride_t, v_stride_h, route_ids,
                       route_stride, T, Tk, Hq, Hkv, Dqk, Dv, W, scale, nullptr, 0, 0, out, lse, err_flag, stream);
}

irs_status irs_sparse_gqa_attn_fwd_grouped(const void* q, int64_t q_stride_t, int64_t q_stride_h, const void* k,
                                           int64_t k_stride_t, int64_t k_stride_h, const void* v, int64_t v_stride_t,
                                           int64_t v_stride_h, const int32_t* route_ids, int64_t route_stride,
                                           int64_t route_group_stride, int T, int Tk, int Hq, int Hkv, int Dqk,
                                           int Dv, int W, float scale, void* out, float* lse, int32_t* err_flag,
                                           irs_stream_t stream) {
  if (route_group_stride < W) return fail(IRS_ERR_VALUE, "route_group_stride must be >= W");
  return attn_fwd_impl(q, q_stride_t, q_stride_h, k, k_stride_t, k_stride_h, v, v_stride_t, v_stride_h, route_ids,
                       route_stride, T, Tk, Hq, Hkv, Dqk, Dv, W, scale, nullptr, 0, 0, out, lse, err_flag, stream,
                       route_group_stride);
}

irs_status irs_sparse_gqa_attn_fwd_windowed(const void* q, int64_t q_stride_t, int64_t q_stride_h, const void* k,
                                            int64_t k_stride_t, int64_t k_stride_h, const void* v,
                                            int64_t v_stride_t, int64_t v_stride_h, const int32_t* route_ids,
                                            int64_t route_stride, const int32_t* cu_seqlens, int ndocs, int window,
                                            int T, int Tk, int Hq, int Hkv, int Dqk, int Dv, int W, float scale,
                                            void* out, float* lse, int32_t* err_flag, irs_stream_t stream) {
  if (window < 1) return fail(IRS_ERR_VALUE, "window must be >= 1 (got %d)", window);
  if (W < 1 || (long long)W + window > 4096)
    return fail(IRS_ERR_VALUE, "route width plus window must be in [2, 4096] (W=%d, window=%d)", W, window);
  if (ndocs < 1 || ndocs > T) return fail(IRS_ERR_VALUE, "ndocs must be in [1, T] (got %d)", ndocs);
  if (Tk < T) return fail(IRS_ERR_VALUE, "the window needs key positions for every query (Tk >= T)");
  if (cu_seqlens == nullptr) return fail(IRS_ERR_VALUE, "NULL cu_seqlens");
  return attn_fwd_impl(q, q_stride_t, q_stride_h, k, k_stride_t, k_stride_h, v, v_stride_t, v_stride_h, route_ids,
                       route_stride, T, Tk, Hq, Hkv, Dqk, Dv, W, scale, cu_seqlens, ndocs, window, out, lse, err_flag,
                       stream);
}


irs_status irs_sparse_gqa_attn_bwd(const void* q, int64_t q_stride_t, int64_t q_stride_h, const void* k,
                                   int64_t k_stride_t, int64_t k_stride_h, const void* v, int64_t v_stride_t,
                                   int64_t v_stride_h, const int32_t* route_ids, int64_t route_stride,
                                   const void* out, const float* lse, const void* dout, int T, int Tk, int Hq,
                                   int Hkv, int Dqk, int Dv, int W, float scale, float* dq, float* dk, float* dv,
                                   int32_t* err_flag, irs_stream_t stream) {
  if (T < 0 || Tk < 1 || Hq < 1 || Hkv < 1) return fail(IRS_ERR_VALUE, "bad sizes (T=%d Tk=%d Hq=%d Hkv=%d)", T, Tk, Hq, Hkv);
  if (Hq % Hkv != 0) return fail(IRS_ERR_VALUE, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
  if (Dqk < 64 || Dqk > 576 || Dqk % 64 != 0) return fail(IRS_ERR_VALUE, "Dqk must be a multiple of 64 in [64, 576]");
  if (Dv < 128 || Dv > 512 || Dv % 128 != 0) return fail(IRS_ERR_VALUE, "Dv must be a multiple of 128 in [128, 512]");
  if (W < 1 || W > 4096) return fail(IRS_ERR_VALUE, "route width W must be in [1, 4096] (got %d)", W);
  if (route_stride < W) return fail(IRS_ERR_VALUE, "route_stride must be >= W");
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(IRS_ERR_VALUE, "scale must be positive and finite");
  if (T == 0) return IRS_OK;
  if (!q || !k || !v || !route_ids || !out || !lse || !dout || !dq || !dk || !dv)
    return fail(IRS_ERR_VALUE, "NULL tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dk) || !aligned16(dv))
    return fail(IRS_ERR_VALUE, "q, k, v, dk and dv must be 16-byte aligned");
  if (q_stride_t % 8 || q_stride_h % 8 || k_stride_t % 8 || k_stride_h % 8 || v_stride_t % 8 || v_stride_h % 8)
    return fail(IRS_ERR_VALUE, "q/k/v strides must be multiples of 8 elements (16 bytes)");
  if (q_stride_t < 0 || q_stride_h < 0 || k_stride_t < 0 || k_stride_h < 0 || v_stride_t < 0 || v_stride_h < 0)
    return fail(IRS_ERR_VALUE, "negative strides are not supported");
  if (dv == dk) {
    // one gradient buffer for keys and values is the gradient of latent rows used as both;
    // for separate value rows it would silently add the value gradient into the key gradient
    if (Dv > Dqk) return fail(IRS_ERR_VALUE, "dv may share dk's buffer only when Dv <= Dqk");
    if (!(v == k && v_stride_t == k_stride_t && v_stride_h == k_stride_h))
      return fail(IRS_ERR_VALUE, "dv may share dk's buffer only when v is a view of k's first Dv dims");
  }
  if ((long long)T * Hkv * ((Hq / Hkv + irs::bwd_max_heads() - 1) / irs::bwd_max_heads()) > 0x7fffffffLL)
    return fail(IRS_ERR_VALUE, "too many work items");
  DeviceInfo* dev = nullptr;
  irs_status s = current_device(&dev);
  if (s != IRS_OK) return s;

  irs::BwdArgs a{};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.q_st = q_stride_t; a.q_sh = q_stride_h;
  a.k_st = k_stride_t; a.k_sh = k_stride_h;
  a.v_st = v_stride_t; a.v_sh = v_stride_h;
  a.route = route_ids;
  a.route_stride = route_stride;
  a.out = static_cast<const __nv_bfloat16*>(out);
  a.lse = lse;
  a.dout = static_cast<const __nv_bfloat16*>(dout);
  a.dq = dq; a.dk = dk; a.dv = dv;
  a.err = err_flag;
  a.T = T; a.Tk = Tk; a.Hq = Hq; a.Hkv = Hkv; a.Dqk = Dqk; a.Dv = Dv; a.W = W;
  a.G = Hq / Hkv;
  a.HB = a.G < irs::bwd_max_heads() ? a.G : irs::bwd_max_heads();
  a.nhb = (a.G + a.HB - 1) / a.HB;
  a.v_alias = (v == k && v_stride_t == k_stride_t && v_stride_h == k_stride_h && Dv <= Dqk) ? 1 : 0;
  a.dv_alias = dv == dk ? 1 : 0;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.nkc = irs::bwd_pick_rows(a, kMaxSmem);
  if (a.nkc == 0) return fail(IRS_ERR_VALUE, "backward tile does not fit in shared memory");
  const size_t smem = irs::bwd_smem_bytes(a);
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (dev->bwd_smem < smem) {
      if ((s = launch_status(irs::configure_bwd_kernel(smem), "configuring the backward")) != IRS_OK) return s;
      dev->bwd_smem = smem;
    }
  }
  return launch_status(irs::launch_bwd(a, reinterpret_cast<cudaStream_t>(stream)), "launching the backward");
}

}  // extern "C"

// =====================================================================================
// Indexer without allocation: the scratch lives in one fixed device array.
//
// For callers that cannot hand the library a workspace: code that runs where cudaMalloc
// is not allowed or not wanted, e.g. plugin interfaces of inference runtimes that give a
// plugin no allocator, or latency-critical loops that must not risk the device-wide
// synchronisation an allocation can cause. The array is a file-scope __device__ object,
// so every GPU that loads this library holds it until the process exits.
// =====================================================================================
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;   // 16 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];
void* g_noalloc_addr[kMaxDevices] = {};
std::mutex g_noalloc_mu;

}  // namespace

extern "C" irs_status irs_sparse_index_score_topk_noalloc(const void* qI, const void* kI, const float* w,
                                                          const int32_t* cu_seqlens, int ndocs, int max_doc_len, int T,
                                                          int Hi, int Di, int c, int budget, int32_t* route_ids,
                                                          float* scores_dbg, int64_t ld_scores, int32_t* err_flag,
                                                          irs_stream_t stream) {
  irs_status s = check_index_sizes(T, Hi, Di, c, budget, ndocs, max_doc_len);
  if (s != IRS_OK) return s;
  if (!qI || !kI || !w || !cu_seqlens || !route_ids) return fail(IRS_ERR_VALUE, "NULL tensor pointer");
  if (!aligned16(qI) || !aligned16(kI)) return fail(IRS_ERR_VALUE, "qI and kI must be 16-byte aligned");
  const irs::IndexPlan p = irs::plan_index(T, Hi, Di, c, budget, ndocs, max_doc_len, scores_dbg == nullptr);
  if (scores_dbg != nullptr && ld_scores < p.ldS)
    return fail(IRS_ERR_VALUE, "ld_scores must be >= max_doc_len / c (%lld)", (long long)p.ldS);
  if (p.ws_bytes > kNoAllocScratchBytes)
    return fail(IRS_ERR_VALUE,
                "these sizes need %zu bytes of scratch but the fixed array holds %zu: pass a score buffer "
                "(scores_dbg) to drop the score rows from the scratch, or use irs_sparse_index_score_topk",
                p.ws_bytes, kNoAllocScratchBytes);
  DeviceInfo* dev = nullptr;
  if ((s = current_device(&dev)) != IRS_OK) return s;
  int ordinal = 0;
  if (cudaGetDevice(&ordinal) != cudaSuccess) return fail(IRS_ERR_RUNTIME, "cudaGetDevice failed");
  uint8_t* ws = nullptr;
  {
    // once per device, with that device current: the array's device address
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_addr[ordinal] == nullptr) {
      void* addr = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
      if (e != cudaSuccess)
        return fail(IRS_ERR_RUNTIME, "cudaGetSymbolAddress of the fixed scratch failed: %s", cudaGetErrorString(e));
      g_noalloc_addr[ordinal] = addr;
    }
    ws = static_cast<uint8_t*>(g_noalloc_addr[ordinal]);
  }
  if ((s = configure_index(dev, p)) != IRS_OK) return s;
  float* scores = scores_dbg != nullptr ? scores_dbg : reinterpret_cast<float*>(ws + p.off_scores);
  const int64_t ldS = scores_dbg != nullptr ? ld_scores : p.ldS;
  CUtensorMap tm_q, tm_k;
  if ((s = make_query_tiles_map(&tm_q, qI, (uint64_t)Di, (uint64_t)Hi, (uint64_t)T, (uint32_t)Hi)) != IRS_OK) return s;
  if ((s = make_tmap(&tm_k, ws + p.off_kbar, (uint64_t)Di, (uint64_t)p.nblk_cap, 128)) != IRS_OK) return s;
  return launch_status(irs::launch_index(p, static_cast<const __nv_bfloat16*>(qI),
                                         static_cast<const __nv_bfloat16*>(kI), w, cu_seqlens, ndocs, max_doc_len, T,
                                         Hi, Di, c, budget, route_ids, scores, ldS, ws, err_flag, tm_q, tm_k,
                                         dev->num_sms, reinterpret_cast<cudaStream_t>(stream)),
                       "launching the indexer (fixed scratch)");
}

// =====================================================================================
// Failure-detection self-test: one bounded wait on an mbarrier phase that nothing
// completes. The wait gives up after limit_ns, records IRS_DEVERR_TIMEOUT and the kernel
// returns, so the context stays usable (no trap, no fault, no endless loop).
// =====================================================================================
namespace {

__global__ void bounded_wait_probe_kernel(int32_t* err, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_word;
  if (threadIdx.x != 0) return;
  irs::mbar_init(&bar, 1);
  abort_word = 0;
  irs::fence_mbar_init();
  volatile int* abort_flag = &abort_word;
  (void)irs::mbar_wait(&bar, 0, abort_flag, err, limit_ns);   // nobody arrives: gives up
}

}  // namespace

extern "C" irs_status irs_check_bounded_wait(uint64_t limit_ns, int32_t* err_flag, irs_stream_t stream) {
  if (err_flag == nullptr) return fail(IRS_ERR_VALUE, "err_flag must be a device int32");
  if (limit_ns < 1000000ull || limit_ns > 2000000000ull)
    return fail(IRS_ERR_VALUE, "limit_ns must be in [1e6, 2e9] (got %llu)", (unsigned long long)limit_ns);
  DeviceInfo* dev = nullptr;
  irs_status s = current_device(&dev);
  if (s != IRS_OK) return s;
  bounded_wait_probe_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(err_flag, limit_ns);
  return launch_status(cudaGetLastError(), "launching the bounded-wait check");
}
