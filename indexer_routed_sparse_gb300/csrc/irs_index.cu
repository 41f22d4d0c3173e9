// Compressed-block indexer on sm_103a: document layout, FP32 block mean-pool,
// tensor-core weighted-ReLU scoring, per-query top-k, bitmap packing and route
// expansion, plus the sliding-window route composition.
//
// Definitions follow the QSA page (nemo_automodel.components.models.qwen3_8_flash_next.qsa:
// `select_qsa_token_ids`, `Qwen3_8_FlashNextQSAIndexer`, `_forward_packed`) and the Step-5
// sparse page (nemo_automodel.components.models.step5.sparse: `indexer_score_tile`,
// `pack_region_bitmap`).
#include <cuda_fp8.h>

#include "irs_index_score.cuh"

namespace irs {

// =====================================================================================
// a1: document layout. One CTA validates cu_seqlens and writes, per document, the first
// pooled-block row and the first score tile; it also resets the tile counter of the
// persistent score kernel. meta[0] = 1 when the layout is valid.
// =====================================================================================
__global__ void __launch_bounds__(1024) layout_kernel(const int32_t* __restrict__ cu, int ndocs, int T, int c,
                                                      int tau_sparse, int QT, int max_doc_len,
                                                      int32_t* __restrict__ meta, int32_t* __restrict__ blk_off,
                                                      int32_t* __restrict__ tile_off, int32_t* err) {
  __shared__ int s_warp[2][32];
  __shared__ int s_carry[2];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int ok = 1;
  if (tid == 0) {
    s_carry[0] = 0;
    s_carry[1] = 0;
    blk_off[0] = 0;
    tile_off[0] = 0;
    if (cu[0] != 0 || cu[ndocs] != T) ok = 0;
  }
  __syncthreads();
  for (int base = 0; base < ndocs; base += 1024) {
    const int d = base + tid;
    int nb = 0, nt = 0;
    if (d < ndocs) {
      const int L = cu[d + 1] - cu[d];
      if (L <= 0 || L > max_doc_len) ok = 0;
      if (L > 0) {
        nb = L / c;
        nt = L > tau_sparse ? (L - tau_sparse + QT - 1) / QT : 0;
      }
    }
    // inclusive block scan of (nb, nt)
    int a = nb, b = nt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int ya = __shfl_up_sync(0xffffffffu, a, o), yb = __shfl_up_sync(0xffffffffu, b, o);
      if (lane >= o) { a += ya; b += yb; }
    }
    if (lane == 31) { s_warp[0][warp] = a; s_warp[1][warp] = b; }
    __syncthreads();
    if (warp == 0) {
      int wa = s_warp[0][lane], wb = s_warp[1][lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int ya = __shfl_up_sync(0xffffffffu, wa, o), yb = __shfl_up_sync(0xffffffffu, wb, o);
        if (lane >= o) { wa += ya; wb += yb; }
      }
      s_warp[0][lane] = wa;
      s_warp[1][lane] = wb;
    }
    __syncthreads();
    const int pa = (warp > 0 ? s_warp[0][warp - 1] : 0) + s_carry[0];
    const int pb = (warp > 0 ? s_warp[1][warp - 1] : 0) + s_carry[1];
    if (d < ndocs) {
      blk_off[d + 1] = pa + a;
      tile_off[d + 1] = pb + b;
    }
    __syncthreads();
    if (tid == 1023) { s_carry[0] = pa + a; s_carry[1] = pb + b; }
    __syncthreads();
  }
  ok = __syncthreads_and(ok);
  if (tid == 0) {
    meta[0] = ok;
    meta[1] = s_carry[0];
    meta[2] = s_carry[1];
    meta[3] = 0;   // tile counter of the score kernel
    if (!ok) record_error(err, IRS_DEVERR_CU_SEQLENS);
  }
}

// =====================================================================================
// a2: block mean-pool. Thread = (pooled block, 8 consecutive dims). FP32 sequential sum
// over the c rows in token order, one IEEE division by c, then round-to-nearest-even
// to bf16 (the scoring operand). Rows past the last complete block (up to the buffer's
// T/c rows) are zeroed: key tiles that reach into them only feed masked scores, but the
// scratch then never holds values of an earlier call.
// =====================================================================================
__global__ void __launch_bounds__(256) pool_kernel(const __nv_bfloat16* __restrict__ kI,
                                                   const int32_t* __restrict__ cu, int ndocs, int Di, int c,
                                                   int nblk_cap, const int32_t* __restrict__ meta,
                                                   const int32_t* __restrict__ blk_off,
                                                   __nv_bfloat16* __restrict__ kbar, float* __restrict__ kbar32,
                                                   uint8_t* __restrict__ kbar8) {
  if (meta[0] != 1) return;
  const int nblk = meta[1];
  const int chunks = Di >> 3;
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int gb = (int)(gid / chunks);
  const int ch = (int)(gid % chunks);
  if (gb >= nblk_cap) return;
  if (gb >= nblk) {
    if (kbar8 != nullptr) reinterpret_cast<uint2*>(kbar8 + (long long)gb * Di)[ch] = make_uint2(0, 0);
    else if (kbar32 == nullptr) reinterpret_cast<uint4*>(kbar + (long long)gb * Di)[ch] = make_uint4(0, 0, 0, 0);
    return;
  }
  const int d = find_le(blk_off, ndocs, gb);
  const int b = gb - blk_off[d];
  const long long row0 = (long long)cu[d] + (long long)b * c;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  const uint4* src = reinterpret_cast<const uint4*>(kI + row0 * Di) + ch;
  for (int j = 0; j < c; ++j) {
    const uint4 u = __ldg(src + (long long)j * chunks);
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(p[i]);
      acc[2 * i] = __fadd_rn(acc[2 * i], f.x);
      acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], f.y);
    }
  }
  const float fc = (float)c;
  if (kbar32 != nullptr) {
    // the FP32 means themselves, for the front half (normalised and rotated before rounding)
    float4* o4 = reinterpret_cast<float4*>(kbar32 + (long long)gb * Di + ch * 8);
    o4[0] = make_float4(__fdiv_rn(acc[0], fc), __fdiv_rn(acc[1], fc), __fdiv_rn(acc[2], fc), __fdiv_rn(acc[3], fc));
    o4[1] = make_float4(__fdiv_rn(acc[4], fc), __fdiv_rn(acc[5], fc), __fdiv_rn(acc[6], fc), __fdiv_rn(acc[7], fc));
    return;
  }
  if (kbar8 != nullptr) {
    // Step-5 E4M3 summaries: the FP32 mean rounded to bf16, then to E4M3 (nearest even,
    // saturating at 448)
    uint8_t b[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float m = __bfloat162float(__float2bfloat16_rn(__fdiv_rn(acc[i], fc)));
      b[i] = (uint8_t)__nv_cvt_float_to_fp8(m, __NV_SATFINITE, __NV_E4M3);
    }
    reinterpret_cast<uint2*>(kbar8 + (long long)gb * Di)[ch] = *reinterpret_cast<const uint2*>(b);
    return;
  }
  uint4 o;
  __nv_bfloat162* q = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    q[i] = __floats2bfloat162_rn(__fdiv_rn(acc[2 * i], fc), __fdiv_rn(acc[2 * i + 1], fc));
  reinterpret_cast<uint4*>(kbar + (long long)gb * Di)[ch] = o;
}

// Step-5 E4M3 queries: every bf16 index query value rounded to E4M3 (nearest even,
// saturating at 448). Thread = 16 consecutive values.
__global__ void __launch_bounds__(256) quantize_e4m3_kernel(const __nv_bfloat16* __restrict__ x, long long n16,
                                                            uint8_t* __restrict__ y) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n16) return;
  const uint4* src = reinterpret_cast<const uint4*>(x) + 2 * i;
  uint8_t b[16];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float f[8];
    const uint4 u = __ldg(src + h);
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 v = __bfloat1622float2(p[k]);
      f[2 * k] = v.x;
      f[2 * k + 1] = v.y;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) b[8 * h + k] = (uint8_t)__nv_cvt_float_to_fp8(f[k], __NV_SATFINITE, __NV_E4M3);
  }
  reinterpret_cast<uint4*>(y)[i] = *reinterpret_cast<const uint4*>(b);
}

// =====================================================================================
// Step-5 learned-logit region summaries (Step-5 sparse page: `project_keys` gives per-dim
// compression logits shaped like the keys; `_summarize_region_payload` makes the region
// summaries in FP32 and keeps the bf16 and E4M3 roundings; regions reset at document
// boundaries). Per region and dim, the softmax of the logits over the region's c tokens
// weights the keys: m = max_j z_j, e_j = exp(z_j - m), summary = (sum_j e_j k_j) / (sum_j e_j)
// with both sums sequential in token order, then bf16, then E4M3.
// =====================================================================================

// e^x for x <= 0, evaluated in FP32 with every operation rounded to nearest and no fused
// multiply-add, so that its value is a fixed function of x: Cody and Waite's reduction to
// base 2 (t = x log2(e), n = rint(t), f = t - n, exact), 2^f from its degree-7 Taylor
// polynomial (coefficients (ln 2)^k / k! rounded to FP32) in Horner form, times 2^n (exact,
// the result stays normal). Where t < -125 the value is 0.
__device__ __forceinline__ float exp_stated(float x) {
  const float t = __fmul_rn(x, 0x1.715476p+0f);
  if (t < -125.f) return 0.f;
  const float n = rintf(t);
  const float f = __fsub_rn(t, n);
  float p = 0x1.ffcbfcp-17f;
  p = __fadd_rn(__fmul_rn(p, f), 0x1.430912p-13f);
  p = __fadd_rn(__fmul_rn(p, f), 0x1.5d87fep-10f);
  p = __fadd_rn(__fmul_rn(p, f), 0x1.3b2ab6p-7f);
  p = __fadd_rn(__fmul_rn(p, f), 0x1.c6b08ep-5f);
  p = __fadd_rn(__fmul_rn(p, f), 0x1.ebfbe0p-3f);
  p = __fadd_rn(__fmul_rn(p, f), 0x1.62e430p-1f);
  p = __fadd_rn(__fmul_rn(p, f), 1.0f);
  return __fmul_rn(p, __int_as_float(((int)n + 127) << 23));
}

// Thread = (region, pair of dims): pass 1 takes the logits' max, pass 2 the two sums.
// Output: E4M3 bytes into kbar8, or (kbar8 == nullptr) the E4M3 values as bf16 into kbar.
// Rows from the region count up to nblk_cap are zeroed.
__global__ void __launch_bounds__(256) summary_kernel(const __nv_bfloat16* __restrict__ kI,
                                                      const __nv_bfloat16* __restrict__ z,
                                                      const int32_t* __restrict__ cu, int ndocs, int Di, int c,
                                                      int nblk_cap, const int32_t* __restrict__ meta,
                                                      const int32_t* __restrict__ blk_off,
                                                      __nv_bfloat16* __restrict__ kbar, uint8_t* __restrict__ kbar8) {
  if (meta[0] != 1) return;
  const int nblk = meta[1];
  const int pairs = Di >> 1;
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int gb = (int)(gid / pairs);
  const int pr = (int)(gid % pairs);
  if (gb >= nblk_cap) return;
  if (gb >= nblk) {
    if (kbar8 != nullptr) reinterpret_cast<uint16_t*>(kbar8 + (long long)gb * Di)[pr] = 0;
    else reinterpret_cast<uint32_t*>(kbar + (long long)gb * Di)[pr] = 0u;
    return;
  }
  const int d = find_le(blk_off, ndocs, gb);
  const long long row0 = (long long)cu[d] + (long long)(gb - blk_off[d]) * c;
  const __nv_bfloat162* zs = reinterpret_cast<const __nv_bfloat162*>(z + row0 * Di) + pr;
  const __nv_bfloat162* ks = reinterpret_cast<const __nv_bfloat162*>(kI + row0 * Di) + pr;
  float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll 8
  for (int j = 0; j < c; ++j) {
    const float2 v = __bfloat1622float2(zs[(long long)j * pairs]);
    m0 = fmaxf(m0, v.x);
    m1 = fmaxf(m1, v.y);
  }
  float s0 = 0.f, s1 = 0.f, n0 = 0.f, n1 = 0.f;
#pragma unroll 8
  for (int j = 0; j < c; ++j) {
    const float2 v = __bfloat1622float2(zs[(long long)j * pairs]);
    const float2 k = __bfloat1622float2(ks[(long long)j * pairs]);
    const float e0 = exp_stated(__fsub_rn(v.x, m0));
    const float e1 = exp_stated(__fsub_rn(v.y, m1));
    s0 = __fadd_rn(s0, e0);
    s1 = __fadd_rn(s1, e1);
    n0 = __fadd_rn(n0, __fmul_rn(e0, k.x));
    n1 = __fadd_rn(n1, __fmul_rn(e1, k.y));
  }
  const __nv_fp8_storage_t b0 = __nv_cvt_float_to_fp8(
      __bfloat162float(__float2bfloat16_rn(__fdiv_rn(n0, s0))), __NV_SATFINITE, __NV_E4M3);
  const __nv_fp8_storage_t b1 = __nv_cvt_float_to_fp8(
      __bfloat162float(__float2bfloat16_rn(__fdiv_rn(n1, s1))), __NV_SATFINITE, __NV_E4M3);
  if (kbar8 != nullptr) {
    reinterpret_cast<uint16_t*>(kbar8 + (long long)gb * Di)[pr] = (uint16_t)(b0 | ((uint16_t)b1 << 8));
    return;
  }
  const float f0 = __half2float(__half(__nv_cvt_fp8_to_halfraw(b0, __NV_E4M3)));
  const float f1 = __half2float(__half(__nv_cvt_fp8_to_halfraw(b1, __NV_E4M3)));
  reinterpret_cast<__nv_bfloat162*>(kbar + (long long)gb * Di)[pr] = __floats2bfloat162_rn(f0, f1);
}

// =====================================================================================
// Indexer front half (QSA page, `Qwen3_8_FlashNextQSAIndexer`: the FP32 group means get K
// RMSNorm and group-start RoPE, the queries RMSNorm and RoPE; `apply_qsa_rope`: per-token
// rotary values cat(cos, sin) over the first rope_dims dims, the rest unchanged). One
// thread per row of Di values, all in FP32 with every operation rounded on its own (no
// fused multiply-add), in the order the oracle uses:
//   ss = sum_d x_d * x_d (ascending d), r = sqrt(ss / Di + eps), y_d = (x_d / r) * wt_d,
//   then for d < h = rope_dims / 2: (y_d cos_d - y_{d+h} sin_d, y_{d+h} cos_d + y_d sin_d),
// and one rounding to bf16 at the end.
// =====================================================================================
template <typename In>
__device__ __forceinline__ void load8(const In* p, float (&f)[8]);
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&f)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 x = __bfloat1622float2(b[i]);
    f[2 * i] = x.x;
    f[2 * i + 1] = x.y;
  }
}
template <>
__device__ __forceinline__ void load8<float>(const float* p, float (&f)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint4 o;
  __nv_bfloat162* q = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
  for (int i = 0; i < 4; ++i) q[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return o;
}

// One row: x (Di values) -> out (bf16), normalised with wt and rotated with rope (cos | sin).
// out may be x itself (bf16 rows staged in shared memory): every 8-value chunk is read
// before it is written, and later chunks are read before their own writes.
template <typename In>
__device__ __forceinline__ void front_row(const In* x, int Di, const float* __restrict__ wt, float eps,
                                          const float* __restrict__ rope, int rope_dims, __nv_bfloat16* out) {
  float ss = 0.f;
  for (int d0 = 0; d0 < Di; d0 += 8) {
    float f[8];
    load8<In>(x + d0, f);
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = __fadd_rn(ss, __fmul_rn(f[i], f[i]));
  }
  const float r = __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)Di), eps));
  const int h = rope_dims >> 1;
  // weights and rotary values by 16-byte loads (the C ABI requires 16-byte alignment of
  // both tables; every offset below is a multiple of 8 floats)
  for (int d0 = 0; d0 < h; d0 += 8) {
    float a[8], b[8], ya[8], yb[8], wa[8], wb[8], cs[8], sn[8];
    load8<In>(x + d0, a);
    load8<In>(x + d0 + h, b);
    load8<float>(wt + d0, wa);
    load8<float>(wt + d0 + h, wb);
    load8<float>(rope + d0, cs);
    load8<float>(rope + h + d0, sn);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float y1 = __fmul_rn(__fdiv_rn(a[i], r), wa[i]);
      const float y2 = __fmul_rn(__fdiv_rn(b[i], r), wb[i]);
      ya[i] = __fsub_rn(__fmul_rn(y1, cs[i]), __fmul_rn(y2, sn[i]));
      yb[i] = __fadd_rn(__fmul_rn(y2, cs[i]), __fmul_rn(y1, sn[i]));
    }
    *reinterpret_cast<uint4*>(out + d0) = pack8(ya);
    *reinterpret_cast<uint4*>(out + d0 + h) = pack8(yb);
  }
  for (int d0 = rope_dims; d0 < Di; d0 += 8) {
    float a[8], wa[8];
    load8<In>(x + d0, a);
    load8<float>(wt + d0, wa);
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = __fmul_rn(__fdiv_rn(a[i], r), wa[i]);
    *reinterpret_cast<uint4*>(out + d0) = pack8(a);
  }
}

// Pooled keys: block gb takes the rotary values of its first token; rows past the last
// complete block are zeroed (as pool_kernel does without the front half).
__global__ void __launch_bounds__(128) front_keys_kernel(const float* __restrict__ kbar32, int nblk_cap, int Di,
                                                         const int32_t* __restrict__ meta,
                                                         const int32_t* __restrict__ blk_off,
                                                         const int32_t* __restrict__ cu, int ndocs, int c,
                                                         const float* __restrict__ k_weight, float eps,
                                                         const float* __restrict__ rope, int rope_dims,
                                                         __nv_bfloat16* __restrict__ kbar) {
  if (meta[0] != 1) return;
  const int gb = blockIdx.x * blockDim.x + threadIdx.x;
  if (gb >= nblk_cap) return;
  __nv_bfloat16* out = kbar + (long long)gb * Di;
  if (gb >= meta[1]) {
    for (int d0 = 0; d0 < Di; d0 += 8) *reinterpret_cast<uint4*>(out + d0) = make_uint4(0, 0, 0, 0);
    return;
  }
  const int d = find_le(blk_off, ndocs, gb);
  const long long tok = (long long)cu[d] + (long long)(gb - blk_off[d]) * c;
  front_row<float>(kbar32 + (long long)gb * Di, Di, k_weight, eps, rope + tok * rope_dims, rope_dims, out);
}

// Queries: row t*Hi + h takes the rotary values of token t. A CTA stages 128 rows in
// shared memory with coalesced 16-byte loads (rows padded by one 16-byte chunk, so the
// per-thread row reads of 8 consecutive threads fall in distinct banks), each thread
// transforms its row in place, and the CTA stores the rows back coalesced.
constexpr int kFrontRows = 128;

__global__ void __launch_bounds__(kFrontRows) front_queries_kernel(const __nv_bfloat16* __restrict__ qI,
                                                                   long long rows, int Hi, int Di,
                                                                   const float* __restrict__ q_weight, float eps,
                                                                   const float* __restrict__ rope, int rope_dims,
                                                                   __nv_bfloat16* __restrict__ qout) {
  extern __shared__ uint4 stage[];
  const int cpr = Di >> 3;        // 16-byte chunks per row
  const int pitch = cpr + 1;
  const long long row0 = (long long)blockIdx.x * kFrontRows;
  const int nrows = rows - row0 < kFrontRows ? (int)(rows - row0) : kFrontRows;
  const uint4* src = reinterpret_cast<const uint4*>(qI + row0 * Di);
  for (int i = threadIdx.x; i < nrows * cpr; i += kFrontRows) stage[(i / cpr) * pitch + i % cpr] = __ldg(src + i);
  __syncthreads();
  if (threadIdx.x < nrows) {
    __nv_bfloat16* r = reinterpret_cast<__nv_bfloat16*>(stage + threadIdx.x * pitch);
    const long long t = (row0 + threadIdx.x) / Hi;
    front_row<__nv_bfloat16>(r, Di, q_weight, eps, rope + t * rope_dims, rope_dims, r);
  }
  __syncthreads();
  uint4* dst = reinterpret_cast<uint4*>(qout + row0 * Di);
  for (int i = threadIdx.x; i < nrows * cpr; i += kFrontRows) dst[i] = stage[(i / cpr) * pitch + i % cpr];
}

// =====================================================================================
// a4 + a5: per-query top-k (radix select on order-preserving keys, ties to the lower
// block index), bitmap packing and route expansion. One CTA of 128 threads per query row.
// =====================================================================================
constexpr int kTopkThreads = 128;

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;                       // -0 == +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // larger score -> larger key
}

struct TopkArgs {
  const float* scores;
  int64_t ldS;
  const int32_t* cu;
  const int32_t* meta;   // nullable: layout validated by layout_kernel
  int32_t* route;
  int32_t* err;
  int ndocs, T, c, budget, max_doc_len;
  int nvis_cap;          // shared-memory capacity in blocks
  int64_t route_ts;      // elements between the route rows of consecutive tokens
};

__global__ void __launch_bounds__(kTopkThreads) topk_expand_kernel(TopkArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const int nw_cap = (a.nvis_cap + 31) / 32;
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem_raw);
  uint32_t* gtw = keys + a.nvis_cap;
  uint32_t* eqw = gtw + nw_cap;
  int32_t* pfx = reinterpret_cast<int32_t*>(eqw + nw_cap);
  const int kb = a.budget / a.c;
  int32_t* sel = pfx + nw_cap;
  __shared__ int hist[2 * 4 * 256];   // two buffers x one histogram per warp
  __shared__ int s_digit, s_above, s_bin;
  __shared__ uint32_t s_diff[4];

  if (a.meta != nullptr && a.meta[0] != 1) return;
  const int t = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int W = a.budget + a.c - 1;
  int32_t* out = a.route + (long long)t * a.route_ts;

  const int d = find_doc(a.cu, a.ndocs, t);
  const int s = a.cu[d], e = a.cu[d + 1];
  if (!(s <= t && t < e && e <= a.T && e - s <= a.max_doc_len)) {
    if (tid == 0) record_error(a.err, IRS_DEVERR_CU_SEQLENS);
    return;
  }
  const int tau = t - s;
  const int nvis = (tau + 1) / a.c;
  const int ntail = (tau + 1) % a.c;
  const bool sparse = nvis > kb;
  const int nsel = sparse ? kb : nvis;

  if (sparse) {
    const float* row = a.scores + (long long)t * a.ldS;
    uint32_t diff = 0;
    const uint32_t key0 = order_key(__ldg(row));
    for (int i = tid; i < nvis; i += kTopkThreads) {
      const uint32_t k = order_key(__ldg(row + i));
      keys[i] = k;
      diff |= k ^ key0;
    }
    // bits above the highest differing bit are common to every key of the row: the radix
    // passes start below them (scores of one row share sign and most exponent bits)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) diff |= __shfl_xor_sync(0xffffffffu, diff, o);
    if (lane == 0) s_diff[warp] = diff;
    for (int i = tid; i < 1024; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    diff = s_diff[0] | s_diff[1] | s_diff[2] | s_diff[3];
    // ---- radix select: the kb-th largest key, MSB first, 8-bit digits ----
    const int hb = diff ? 31 - __clz(diff) : -1;
    // all keys equal (hb < 0): the threshold is that key and the lowest indices win
    uint32_t mask = hb < 0 ? 0xFFFFFFFFu : (hb >= 31 ? 0u : ~((2u << hb) - 1u));
    uint32_t prefix = key0 & mask;
    int rem = kb;
    int buf = 0;
    for (int top = hb; top >= 0; top -= 8) {
      const int shift = top - 7 > 0 ? top - 7 : 0;
      const int width = top - shift + 1;
      const uint32_t dmask = (1u << width) - 1u;
      int* hw = hist + buf * 1024 + warp * 256;
      for (int i = tid; i < nvis; i += kTopkThreads) {
        const uint32_t k = keys[i];
        if ((k & mask) == prefix) atomicAdd(&hw[(k >> shift) & dmask], 1);
      }
      // clear the other histogram for the next pass while this one is counted
      for (int i = tid; i < 1024; i += kTopkThreads) hist[(buf ^ 1) * 1024 + i] = 0;
      __syncthreads();
      if (warp == 0) {
        const int* h = hist + buf * 1024;
        int loc[8], lsum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int bin = 255 - 8 * lane - i;
          loc[i] = h[bin] + h[256 + bin] + h[512 + bin] + h[768 + bin];
          lsum += loc[i];
        }
        int incl = lsum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const int excl = incl - lsum;
        if (excl < rem && rem <= incl) {
          int run = excl;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (run + loc[i] >= rem) { s_digit = 255 - 8 * lane - i; s_above = run; s_bin = loc[i]; break; }
            run += loc[i];
          }
        }
      }
      __syncthreads();
      prefix |= (uint32_t)s_digit << shift;
      mask |= dmask << shift;
      rem -= s_above;
      buf ^= 1;
      // the threshold bin is taken whole: no lower digit can change the selection
      if (s_bin == rem) break;
    }
    // selected: (key & mask) > prefix, plus the `rem` lowest-index keys with (key & mask) == prefix
    const uint32_t thr = prefix;
    // ---- bitmap words of "greater" and "equal" elements ----
    const int nw = (nvis + 31) / 32;
    for (int base = 0; base < nw * 32; base += kTopkThreads) {
      const int i = base + tid;
      const uint32_t k = i < nvis ? keys[i] : 0u;
      const uint32_t km = k & mask;
      const uint32_t g = __ballot_sync(0xffffffffu, i < nvis && km > thr);
      const uint32_t q = __ballot_sync(0xffffffffu, i < nvis && km == thr);
      const int wi = (base >> 5) + warp;
      if (lane == 0 && wi < nw) { gtw[wi] = g; eqw[wi] = q; }
    }
    __syncthreads();
    // ---- take the `rem` lowest-index equal elements; prefix popcounts of the bitmap ----
    if (warp == 0) {
      int eq_run = 0, sel_run = 0;
      for (int wb = 0; wb < nw; wb += 32) {
        const int wi = wb + lane;
        uint32_t g = 0, q = 0;
        if (wi < nw) { g = gtw[wi]; q = eqw[wi]; }
        // equal elements before this word (inclusive scan over lanes)
        const int qc = __popc(q);
        int qi = qc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, qi, o);
          if (lane >= o) qi += y;
        }
        const int q_before = eq_run + qi - qc;
        uint32_t take = 0;
        if (q_before < rem) {
          const int want = rem - q_before;   // >= 1
          if (want >= qc) take = q;
          else {
            uint32_t x = q;
            for (int r = 0; r < want; ++r) { take |= x & (~x + 1u); x &= x - 1u; }
          }
        }
        const uint32_t bits = g | take;
        const int bc = __popc(bits);
        int bi = bc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, bi, o);
          if (lane >= o) bi += y;
        }
        if (wi < nw) { gtw[wi] = bits; pfx[wi] = sel_run + bi - bc; }
        eq_run += __shfl_sync(0xffffffffu, qi, 31);
        sel_run += __shfl_sync(0xffffffffu, bi, 31);
      }
    }
    __syncthreads();
    // ---- ascending list of selected blocks ----
    for (int wi = tid; wi < nw; wi += kTopkThreads) {
      uint32_t x = gtw[wi];
      int r = pfx[wi];
      while (x) {
        const int b = __ffs(x) - 1;
        if (r < kb) sel[r] = wi * 32 + b;
        ++r;
        x &= x - 1u;
      }
    }
    __syncthreads();
  }
  // ---- route row: [selected blocks x c tokens | -1 ...][tail tokens | -1 ...] ----
  const int c = a.c;
  const int nblk_slots = nsel * c;
  if ((c & (c - 1)) == 0) {
    const int cs = __ffs(c) - 1;
    for (int slot = tid; slot < nblk_slots; slot += kTopkThreads) {
      const int r = slot >> cs;
      const int b = sparse ? sel[r] : r;
      out[slot] = s + (b << cs) + (slot & (c - 1));
    }
  } else {
    for (int r = tid; r < nsel; r += kTopkThreads) {
      const int b = sparse ? sel[r] : r;
      for (int j = 0; j < c; ++j) out[r * c + j] = s + b * c + j;
    }
  }
  for (int slot = nblk_slots + tid; slot < W; slot += kTopkThreads) {
    const int j = slot - a.budget;
    out[slot] = (j >= 0 && j < ntail) ? s + nvis * c + j : -1;
  }
}

// Register variant of the per-row CTA kernel for rows of at most 128*KPT visible blocks:
// the row's keys stay in registers (element i = tid + 128k) and every scan is done by all
// 128 threads (block scans), so no warp waits on a serial section. Same selection rule and
// route layout as topk_expand_kernel.
struct BlockScan2 {
  int a, b;
};

// Exclusive block-wide scan of two ints over 128 threads (ascending thread order); also
// returns the totals. `red` is 8 ints of shared scratch. Contains two __syncthreads.
__device__ __forceinline__ BlockScan2 block_exscan2(int x, int y, int* red, int& tx, int& ty) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int ix = x, iy = y;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int ux = __shfl_up_sync(0xffffffffu, ix, o), uy = __shfl_up_sync(0xffffffffu, iy, o);
    if (lane >= o) { ix += ux; iy += uy; }
  }
  if (lane == 31) { red[warp] = ix; red[4 + warp] = iy; }
  __syncthreads();
  int bx = 0, by = 0;
  tx = 0;
  ty = 0;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const int rx = red[w], ry = red[4 + w];
    if (w < warp) { bx += rx; by += ry; }
    tx += rx;
    ty += ry;
  }
  __syncthreads();
  return BlockScan2{bx + ix - x, by + iy - y};
}

template <int KPT>
__global__ void __launch_bounds__(kTopkThreads) topk_reg_kernel(TopkArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const int kb = a.budget / a.c;
  int32_t* sel = reinterpret_cast<int32_t*>(smem_raw);   // [kb]
  __shared__ int hist[256];
  __shared__ int red[8];
  __shared__ int s_res[4];
  __shared__ uint32_t s_diff[4];
  __shared__ uint32_t s_bits[KPT * 4];
  if (a.meta != nullptr && a.meta[0] != 1) return;
  const int t = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int W = a.budget + a.c - 1;
  int32_t* out = a.route + (long long)t * a.route_ts;
  const int d = find_doc(a.cu, a.ndocs, t);
  const int s = a.cu[d], e = a.cu[d + 1];
  if (!(s <= t && t < e && e <= a.T && e - s <= a.max_doc_len)) {
    if (tid == 0) record_error(a.err, IRS_DEVERR_CU_SEQLENS);
    return;
  }
  const int tau = t - s;
  const int nvis = (tau + 1) / a.c;
  const int ntail = (tau + 1) % a.c;
  const bool sparse = nvis > kb;
  const int nsel = sparse ? kb : nvis;
  if (sparse) {
    const float* row = a.scores + (long long)t * a.ldS;
    const uint32_t key0 = order_key(__ldg(row));
    uint32_t key[KPT];
    uint32_t diff = 0;
#pragma unroll
    for (int k = 0; k < KPT; ++k) {
      const int i = tid + kTopkThreads * k;
      key[k] = i < nvis ? order_key(__ldg(row + i)) : 0u;
      if (i < nvis) diff |= key[k] ^ key0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) diff |= __shfl_xor_sync(0xffffffffu, diff, o);
    if (lane == 0) s_diff[warp] = diff;
    hist[tid] = 0;
    hist[tid + 128] = 0;
    __syncthreads();
    diff = s_diff[0] | s_diff[1] | s_diff[2] | s_diff[3];
    const int hb = diff ? 31 - __clz(diff) : -1;
    uint32_t mask = hb < 0 ? 0xFFFFFFFFu : (hb >= 31 ? 0u : ~((2u << hb) - 1u));
    uint32_t prefix = key0 & mask;
    int rem = kb;
    for (int top = hb; top >= 0; top -= 8) {
      const int shift = top - 7 > 0 ? top - 7 : 0;
      const uint32_t dmask = (1u << (top - shift + 1)) - 1u;
#pragma unroll
      for (int k = 0; k < KPT; ++k) {
        const int i = tid + kTopkThreads * k;
        if (i < nvis && (key[k] & mask) == prefix) atomicAdd(&hist[(key[k] >> shift) & dmask], 1);
      }
      __syncthreads();
      // thread i owns bins 255-2i and 254-2i (descending digit order)
      const int h0 = hist[255 - 2 * tid], h1 = hist[254 - 2 * tid];
      int tot_unused, tot2;
      const BlockScan2 ex = block_exscan2(h0 + h1, 0, red, tot_unused, tot2);
      // digits above this thread's pair hold ex.a keys
      if (ex.a < rem && rem <= ex.a + h0 + h1) {
        if (rem <= ex.a + h0) { s_res[0] = 255 - 2 * tid; s_res[1] = ex.a; s_res[2] = h0; }
        else { s_res[0] = 254 - 2 * tid; s_res[1] = ex.a + h0; s_res[2] = h1; }
      }
      hist[tid] = 0;              // every read of hist is behind the scan's barriers
      hist[tid + 128] = 0;
      __syncthreads();
      prefix |= (uint32_t)s_res[0] << shift;
      mask |= dmask << shift;
      rem -= s_res[1];
      const int bin = s_res[2];
      __syncthreads();            // s_res is rewritten by the next pass
      if (bin == rem) break;      // the threshold bin is taken whole
    }
    const uint32_t thr = prefix;
    // ---- bitmap words: word 4k + warp = blocks 128k + 32 warp .. +31 ----
#pragma unroll
    for (int k = 0; k < KPT; ++k) {
      const int i = tid + kTopkThreads * k;
      const uint32_t km = key[k] & mask;
      const uint32_t g = __ballot_sync(0xffffffffu, i < nvis && km > thr);
      const uint32_t q = __ballot_sync(0xffffffffu, i < nvis && km == thr);
      if (lane == 0) { s_bits[4 * k + warp] = g; hist[4 * k + warp] = (int)q; }
    }
    __syncthreads();
    // thread i owns word i (KPT*4 <= 128 words)
    const int nw = (nvis + 31) / 32;
    const uint32_t g = tid < nw ? s_bits[tid] : 0u;
    const uint32_t q = tid < nw ? (uint32_t)hist[tid] : 0u;
    int te, ts;
    const BlockScan2 eqx = block_exscan2(__popc(q), 0, red, te, ts);
    uint32_t take = 0;
    if (eqx.a < rem) {
      const int want = rem - eqx.a;
      if (want >= __popc(q)) take = q;
      else {
        uint32_t x = q;
        for (int r = 0; r < want; ++r) { take |= x & (~x + 1u); x &= x - 1u; }
      }
    }
    const uint32_t bits = g | take;
    const BlockScan2 selx = block_exscan2(__popc(bits), 0, red, te, ts);
    uint32_t x = bits;
    int r = selx.a;
    while (x) {
      const int b = __ffs(x) - 1;
      if (r < kb) sel[r] = tid * 32 + b;
      ++r;
      x &= x - 1u;
    }
    __syncthreads();
  }
  const int c = a.c;
  const int nblk_slots = nsel * c;
  if ((c & (c - 1)) == 0) {
    const int cs = __ffs(c) - 1;
    for (int slot = tid; slot < nblk_slots; slot += kTopkThreads) {
      const int rr = slot >> cs;
      const int b = sparse ? sel[rr] : rr;
      out[slot] = s + (b << cs) + (slot & (c - 1));
    }
  } else {
    for (int rr = tid; rr < nsel; rr += kTopkThreads) {
      const int b = sparse ? sel[rr] : rr;
      for (int j = 0; j < c; ++j) out[rr * c + j] = s + b * c + j;
    }
  }
  for (int slot = nblk_slots + tid; slot < W; slot += kTopkThreads) {
    const int j = slot - a.budget;
    out[slot] = (j >= 0 && j < ntail) ? s + nvis * c + j : -1;
  }
}

// Warp-per-row variant for small selections (kb <= 32) of rows of at most 32*KPL visible
// blocks; eight rows per CTA, no block barriers. Lane l holds blocks l, l+32, ... of its row.
// The threshold (the kb-th largest key) is found in two steps. The kb-th largest of the 32
// lane maxima, L, is a lower bound for it: the kb lanes whose maxima are >= L hold kb keys
// >= L. So every key >= the threshold is >= L, and only those candidates (about 32 ln 2 + kb
// of them on continuous scores) need ranking. With at most 32 candidates, one per lane,
// three 32-lane bitonic sorts in registers give L, the threshold and the ascending list of
// selected blocks. More candidates (many keys tied near the top) take a general path: an
// exact rank count over up to kTopkCand candidates in shared memory, else a bit-serial
// radix select over all keys, and the selection from bitmap words (ballots of the lanes'
// j-th keys). Both paths select the keys above the threshold plus the lowest-index keys
// equal to it, as the other variants do.
constexpr int kTopkWarpRows = 8;
constexpr int kTopkCand = 128;

// 32-lane bitonic sort of one value per lane: descending (lane 0 the largest) or ascending.
template <bool kDescending>
__device__ __forceinline__ uint32_t warp_bitonic_sort(uint32_t v, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const uint32_t o = __shfl_xor_sync(0xffffffffu, v, j);
      // within a run of k lanes sorted in direction `dir`, the lower lane of each pair keeps
      // the value that comes first in that direction
      const bool dir = ((lane & k) == 0) == kDescending;
      const bool lower = (lane & j) == 0;
      const uint32_t hi = v > o ? v : o, lo = v > o ? o : v;
      v = (lower == dir) ? hi : lo;
    }
  }
  return v;
}

template <int KPL>
__global__ void __launch_bounds__(kTopkWarpRows * 32) topk_warp_kernel(TopkArgs a) {
  static_assert(KPL % 8 == 0, "keys are handled in chunks of 8 words");
  extern __shared__ uint8_t smem_raw[];
  const int kb = a.budget / a.c;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t lt = (1u << lane) - 1u;   // lanes below this one
  uint32_t* cand = reinterpret_cast<uint32_t*>(smem_raw) + warp * 2 * kTopkCand;   // keys
  uint32_t* cidx = cand + kTopkCand;                                              // their blocks
  if (a.meta != nullptr && a.meta[0] != 1) return;
  const int t = blockIdx.x * kTopkWarpRows + warp;
  if (t >= a.T) return;
  const int W = a.budget + a.c - 1;
  int32_t* out = a.route + (long long)t * a.route_ts;
  const int d = find_doc(a.cu, a.ndocs, t);
  const int s = a.cu[d], e = a.cu[d + 1];
  if (!(s <= t && t < e && e <= a.T && e - s <= a.max_doc_len)) {
    if (lane == 0) record_error(a.err, IRS_DEVERR_CU_SEQLENS);
    return;
  }
  const int tau = t - s;
  const int nvis = (tau + 1) / a.c;
  const int ntail = (tau + 1) % a.c;
  const bool sparse = nvis > kb;
  const int nsel = sparse ? kb : nvis;
  // lane r < nsel ends up holding the r-th selected block (ascending)
  uint32_t selv = (uint32_t)lane;
  if (sparse) {
    const float* row = a.scores + (long long)t * a.ldS;
    const int nw = (nvis + 31) >> 5;   // words with at least one visible block (uniform)
    uint32_t key[KPL];
    // per-key work runs on chunks of 8 words, skipped past the row's last visible block;
    // every load is issued before any key is used
#pragma unroll
    for (int j = 0; j < KPL; ++j) {
      key[j] = 0u;
      if (8 * (j >> 3) < nw) {
        const int i = lane + 32 * j;
        if (i < nvis) key[j] = __float_as_uint(__ldg(row + i));
      }
    }
    uint32_t mx = 0;   // 0 is below every key of a real score (order_key(-inf) > 0)
#pragma unroll
    for (int j = 0; j < KPL; ++j) {
      if (8 * (j >> 3) < nw) {
        const int i = lane + 32 * j;
        key[j] = i < nvis ? order_key(__uint_as_float(key[j])) : 0u;
        mx = key[j] > mx ? key[j] : mx;
      }
    }
    const uint32_t L = __shfl_sync(0xffffffffu, warp_bitonic_sort<true>(mx, lane), kb - 1);
    // candidates (keys >= L) compacted by ballots in ascending block order
    int C = 0;
#pragma unroll
    for (int j = 0; j < KPL; ++j) {
      if (8 * (j >> 3) < nw) {
        const bool p = key[j] >= L;
        const uint32_t bal = __ballot_sync(0xffffffffu, p);
        const int o = C + __popc(bal & lt);
        if (p && o < kTopkCand) { cand[o] = key[j]; cidx[o] = (uint32_t)(lane + 32 * j); }
        C += __popc(bal);
      }
    }
    __syncwarp();
    if (C <= 32) {
      // ---- common path: one candidate per lane, lanes in ascending block order ----
      const uint32_t ck = lane < C ? cand[lane] : 0u;
      const uint32_t ci = lane < C ? cidx[lane] : 0u;
      const uint32_t thr = __shfl_sync(0xffffffffu, warp_bitonic_sort<true>(ck, lane), kb - 1);
      const uint32_t gt = __ballot_sync(0xffffffffu, ck > thr);
      const uint32_t eq = __ballot_sync(0xffffffffu, ck == thr);
      const int rem = kb - __popc(gt);
      // keys above the threshold, and the rem lowest blocks (= lowest lanes) equal to it
      const bool take = ck > thr || (ck == thr && __popc(eq & lt) < rem);
      const uint32_t tk = __ballot_sync(0xffffffffu, take);
      __syncwarp();
      if (take) cidx[__popc(tk & lt)] = ci;
      __syncwarp();
      selv = lane < kb ? cidx[lane] : 0u;
    } else {
      // ---- general path ----
      uint32_t thr;
      int rem;
      if (C <= kTopkCand) {
        bool found = false;
        uint32_t my_thr = 0;
        int my_rem = 0;
        for (int i = lane; i < C; i += 32) {
          const uint32_t v = cand[i];
          int gt = 0, ge = 0;
          for (int q = 0; q < C; ++q) {
            const uint32_t u = cand[q];
            gt += u > v ? 1 : 0;
            ge += u >= v ? 1 : 0;
          }
          if (gt < kb && kb <= ge) { found = true; my_thr = v; my_rem = kb - gt; }
        }
        const int src = __ffs(__ballot_sync(0xffffffffu, found)) - 1;
        thr = __shfl_sync(0xffffffffu, my_thr, src);
        rem = __shfl_sync(0xffffffffu, my_rem, src);
      } else {
        // bit-serial radix select: the rem-th largest among the keys that match the prefix
        uint32_t prefix = 0, mask = 0;
        rem = kb;
        for (int bit = 31; bit >= 0; --bit) {
          const uint32_t m2 = mask | (1u << bit), want = prefix | (1u << bit);
          int c1 = 0;
#pragma unroll
          for (int j = 0; j < KPL; ++j) c1 += (key[j] & m2) == want ? 1 : 0;
          const int tot = __reduce_add_sync(0xffffffffu, c1);
          if (tot >= rem) prefix = want;
          else rem -= tot;
          mask = m2;
        }
        thr = prefix;
      }
      // bitmap word j = ballot of the lanes' j-th keys; selected blocks in ascending order
      int eq_before = 0, sel_before = 0;
#pragma unroll
      for (int j = 0; j < KPL; ++j) {
        if (j >= nw) break;
        const uint32_t g = __ballot_sync(0xffffffffu, key[j] > thr);
        const uint32_t q = __ballot_sync(0xffffffffu, key[j] == thr);
        uint32_t tk = 0;
        if (eq_before < rem) {
          const int want = rem - eq_before;
          if (want >= __popc(q)) tk = q;
          else {
            uint32_t x = q;
            for (int r = 0; r < want; ++r) { tk |= x & (~x + 1u); x &= x - 1u; }
          }
        }
        eq_before += __popc(q);
        const uint32_t bits = g | tk;
        // the n-th set bit of this word goes to lane sel_before + n
        const int n_here = __popc(bits);
        const int r = lane - sel_before;
        if (r >= 0 && r < n_here) {
          uint32_t x = bits;
          for (int q2 = 0; q2 < r; ++q2) x &= x - 1u;
          selv = 32u * j + (uint32_t)(__ffs(x) - 1);
        }
        sel_before += n_here;
      }
    }
  }
  // ---- route row: [selected blocks x c tokens | -1 ...][tail tokens | -1 ...] ----
  const int c = a.c;
  const int nblk_slots = nsel * c;
  if ((c & 31) == 0) {
    for (int r = 0; r < nsel; ++r) {
      const int base = s + (int)__shfl_sync(0xffffffffu, selv, r) * c;
      for (int j = lane; j < c; j += 32) out[r * c + j] = base + j;
    }
  } else {
    const bool pow2 = (c & (c - 1)) == 0;
    const int cs = __ffs(c) - 1;
    for (int slot0 = 0; slot0 < nblk_slots; slot0 += 32) {
      const int slot = slot0 + lane;
      const int rr = slot < nblk_slots ? (pow2 ? slot >> cs : slot / c) : 0;
      const int b = (int)__shfl_sync(0xffffffffu, selv, rr);
      if (slot < nblk_slots) out[slot] = s + b * c + (slot - rr * c);
    }
  }
  for (int slot = nblk_slots + lane; slot < W; slot += 32) {
    const int j = slot - a.budget;
    out[slot] = (j >= 0 && j < ntail) ? s + nvis * c + j : -1;
  }
}

// Launch the top-k + expansion for every row: the warp-per-row variant for kb <= 32 and
// rows of at most 2048 visible blocks, the register variant for larger kb on such rows,
// else the shared-memory variant.
static cudaError_t launch_topk(const TopkArgs& ta, int kb, cudaStream_t stream, size_t cta_smem) {
  const int nv = ta.nvis_cap;
  if (kb <= 32 && nv <= 2048) {
    const size_t wsmem = (size_t)kTopkWarpRows * 2 * kTopkCand * 4;
    const unsigned grid = (unsigned)((ta.T + kTopkWarpRows - 1) / kTopkWarpRows);
    if (nv <= 256) topk_warp_kernel<8><<<grid, kTopkWarpRows * 32, wsmem, stream>>>(ta);
    else if (nv <= 512) topk_warp_kernel<16><<<grid, kTopkWarpRows * 32, wsmem, stream>>>(ta);
    else if (nv <= 1024) topk_warp_kernel<32><<<grid, kTopkWarpRows * 32, wsmem, stream>>>(ta);
    else topk_warp_kernel<64><<<grid, kTopkWarpRows * 32, wsmem, stream>>>(ta);
    return cudaGetLastError();
  }
  const size_t smem = (size_t)kb * 4;
  if (nv <= 2048 && smem <= 48 * 1024) {
    if (nv <= 256) topk_reg_kernel<2><<<ta.T, kTopkThreads, smem, stream>>>(ta);
    else if (nv <= 512) topk_reg_kernel<4><<<ta.T, kTopkThreads, smem, stream>>>(ta);
    else if (nv <= 1024) topk_reg_kernel<8><<<ta.T, kTopkThreads, smem, stream>>>(ta);
    else topk_reg_kernel<16><<<ta.T, kTopkThreads, smem, stream>>>(ta);
    return cudaGetLastError();
  }
  topk_expand_kernel<<<ta.T, kTopkThreads, cta_smem, stream>>>(ta);
  return cudaGetLastError();
}

// =====================================================================================
// a5': sliding window composed in front of an indexer route.
// =====================================================================================
__global__ void __launch_bounds__(128) compose_window_kernel(const int32_t* __restrict__ route, int W,
                                                             const int32_t* __restrict__ cu, int ndocs, int T,
                                                             int window, int32_t* __restrict__ out, int32_t* err) {
  const int t = blockIdx.x;
  const int d = find_doc(cu, ndocs, t);
  const int s = cu[d], e = cu[d + 1];
  const int Wo = window + W;
  int32_t* o = out + (long long)t * Wo;
  if (!(s <= t && t < e && e <= T)) {
    if (threadIdx.x == 0) record_error(err, IRS_DEVERR_CU_SEQLENS);
    return;
  }
  const int lo = t - window + 1;
  const int32_t* r = route + (long long)t * W;
  for (int j = threadIdx.x; j < Wo; j += blockDim.x) {
    int v;
    if (j < window) {
      const int tok = lo + j;
      v = tok >= s ? tok : -1;
    } else {
      const int x = r[j - window];
      v = x < lo ? x : -1;
    }
    o[j] = v;
  }
}

// =====================================================================================
// host launchers
// =====================================================================================
IndexPlan plan_index(int T, int Hi, int Di, int c, int budget, int ndocs, int max_doc_len, bool with_scores,
                     bool front, bool e4m3, int G) {
  IndexPlan p{};
  p.kb = budget / c;
  p.QT = kIdxN / Hi;
  p.tau_sparse = (p.kb + 1) * c - 1;
  p.nblk_cap = T / c > 0 ? T / c : 1;
  p.ldS = max_doc_len / c > 0 ? max_doc_len / c : 1;
  size_t off = 0;
  auto take = [&](size_t bytes, size_t align) {
    off = (off + align - 1) / align * align;
    const size_t o = off;
    off += bytes;
    return o;
  };
  p.off_meta = take(64, 256);
  p.off_blk = take(sizeof(int32_t) * (size_t)(ndocs + 1), 256);
  p.off_tile = take(sizeof(int32_t) * (size_t)(ndocs + 1), 256);
  p.off_kbar = take((size_t)p.nblk_cap * Di * 2, 1024);
  p.off_scores = with_scores ? take((size_t)T * p.ldS * sizeof(float), 1024) : 0;
  p.off_qfront = front ? take((size_t)T * Hi * Di * 2, 1024) : 0;
  p.off_kbar32 = front ? take((size_t)p.nblk_cap * Di * sizeof(float), 1024) : 0;
  p.off_q8 = e4m3 ? take((size_t)T * G * Hi * Di, 1024) : 0;
  p.off_k8 = e4m3 ? take((size_t)p.nblk_cap * Di, 1024) : 0;
  p.ws_bytes = (off + 255) / 256 * 256;
  if (e4m3) {   // one 128-byte atom per key tile
    p.stages = 8;
    p.score_smem = IdxSmem<128, true>::total(p.stages);
  } else {
    p.stages = Di == 64 ? 8 : 5;
    p.score_smem = Di == 64 ? IdxSmem<64>::total(p.stages) : IdxSmem<128>::total(p.stages);
  }
  p.topk_smem = topk_smem_bytes(p.ldS, p.kb);
  return p;
}

size_t topk_smem_bytes(int nvis_cap, int kb) {
  const size_t nw = (size_t)(nvis_cap + 31) / 32;
  return (size_t)nvis_cap * 4 + nw * 4 * 3 + (size_t)kb * 4 + 16;
}

// Layout, pooling and (with `front`) the front half's transforms: pooled bf16 keys into
// kbar, transformed queries into qfront.
static void launch_pool(const IndexPlan& p, const __nv_bfloat16* qI, const __nv_bfloat16* kI, const int32_t* cu,
                        int ndocs, int max_doc_len, int T, int Hi, int Di, int c, uint8_t* ws, int32_t* err,
                        const FrontHalf* front, __nv_bfloat16* kbar, __nv_bfloat16* qfront, cudaStream_t stream,
                        bool e4m3 = false, const __nv_bfloat16* z = nullptr, int G = 1) {
  int32_t* meta = reinterpret_cast<int32_t*>(ws + p.off_meta);
  int32_t* blk_off = reinterpret_cast<int32_t*>(ws + p.off_blk);
  int32_t* tile_off = reinterpret_cast<int32_t*>(ws + p.off_tile);
  float* kbar32 = reinterpret_cast<float*>(ws + p.off_kbar32);

  layout_kernel<<<1, 1024, 0, stream>>>(cu, ndocs, T, c, p.tau_sparse, p.QT, max_doc_len, meta, blk_off, tile_off,
                                        err);
  if (z != nullptr) {
    const long long threads = (long long)p.nblk_cap * (Di / 2);
    summary_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, stream>>>(kI, z, cu, ndocs, Di, c, p.nblk_cap, meta,
                                                                          blk_off, kbar,
                                                                          e4m3 ? ws + p.off_k8 : nullptr);
  } else {
    const long long threads = (long long)p.nblk_cap * (Di / 8);
    const int grid = (int)((threads + 255) / 256);
    pool_kernel<<<grid, 256, 0, stream>>>(kI, cu, ndocs, Di, c, p.nblk_cap, meta, blk_off, kbar,
                                          front ? kbar32 : nullptr, e4m3 ? ws + p.off_k8 : nullptr);
  }
  if (e4m3) {
    const long long n16 = (long long)T * G * Hi * Di / 16;
    quantize_e4m3_kernel<<<(unsigned)((n16 + 255) / 256), 256, 0, stream>>>(qI, n16, ws + p.off_q8);
  }
  if (front) {
    front_keys_kernel<<<(p.nblk_cap + 127) / 128, 128, 0, stream>>>(kbar32, p.nblk_cap, Di, meta, blk_off, cu, ndocs, c,
                                                                    front->k_weight, front->eps, front->rope,
                                                                    front->rope_dims, kbar);
  }
  if (front && front->q_weight != nullptr) {   // (no q_weight: the queries arrive transformed)
    const long long rows = (long long)T * Hi;
    const size_t stage_bytes = (size_t)kFrontRows * (Di / 8 + 1) * 16;
    front_queries_kernel<<<(unsigned)((rows + kFrontRows - 1) / kFrontRows), kFrontRows, stage_bytes, stream>>>(
        qI, rows, Hi, Di, front->q_weight, front->eps, front->rope, front->rope_dims, qfront);
  }
}

cudaError_t launch_index(const IndexPlan& p, const __nv_bfloat16* qI, const __nv_bfloat16* kI, const float* w,
                         const int32_t* cu, int ndocs, int max_doc_len, int T, int Hi, int Di, int c, int budget,
                         int32_t* route, float* scores, int64_t ldS, uint8_t* ws, int32_t* err,
                         const CUtensorMap& tm_q, const CUtensorMap& tm_k, int num_sms, cudaStream_t stream,
                         const FrontHalf* front, int G, int64_t scores_group_stride, bool e4m3,
                         const __nv_bfloat16* z) {
  int32_t* meta = reinterpret_cast<int32_t*>(ws + p.off_meta);
  int32_t* blk_off = reinterpret_cast<int32_t*>(ws + p.off_blk);
  int32_t* tile_off = reinterpret_cast<int32_t*>(ws + p.off_tile);
  __nv_bfloat16* kbar = reinterpret_cast<__nv_bfloat16*>(ws + p.off_kbar);
  launch_pool(p, qI, kI, cu, ndocs, max_doc_len, T, Hi, Di, c, ws, err, front, kbar,
              reinterpret_cast<__nv_bfloat16*>(ws + p.off_qfront), stream, e4m3, z, G);
  const int grid = num_sms < kMaxIndexCtas ? num_sms : kMaxIndexCtas;
  const int W = budget + c - 1;
  // one score + top-k pass per KV group (Step-5 selects per group), sharing the pooled keys;
  // passes run in stream order, so they can share the score scratch
  for (int g = 0; g < G; ++g) {
    // the score kernel's tile counter (meta[3]) starts at 0 for every pass (the layout
    // kernel has reset it for the first)
    if (g > 0) {
      const cudaError_t me = cudaMemsetAsync(meta + 3, 0, sizeof(int32_t), stream);
      if (me != cudaSuccess) return me;
    }
    float* sg = scores + (int64_t)g * scores_group_stride;
    IndexArgs ia{w + (int64_t)g * Hi, cu, blk_off, tile_off, meta, sg, ldS, err, ndocs, T, c, p.QT, p.tau_sparse,
                 p.stages, (int64_t)G * Hi, g * Hi};
    const cudaError_t le = e4m3 ? launch_score_e4m3(Hi, grid, p.score_smem, stream, tm_q, tm_k, ia)
                           : (Di == 64 ? launch_score_64(Hi, grid, p.score_smem, stream, tm_q, tm_k, ia)
                                       : launch_score_128(Hi, grid, p.score_smem, stream, tm_q, tm_k, ia));
    if (le != cudaSuccess) return le;
    TopkArgs ta{sg, ldS, cu, meta, route + (int64_t)g * W, err, ndocs, T, c, budget, max_doc_len, (int)p.ldS,
                (int64_t)G * W};
    const cudaError_t te = launch_topk(ta, p.kb, stream, p.topk_smem);
    if (te != cudaSuccess) return te;
  }
  return cudaSuccess;
}

cudaError_t launch_front_operands(const IndexPlan& p, const __nv_bfloat16* qI, const __nv_bfloat16* kI,
                                  const int32_t* cu, int ndocs, int max_doc_len, int T, int Hi, int Di, int c,
                                  uint8_t* ws, int32_t* err, const FrontHalf& front, __nv_bfloat16* q_out,
                                  __nv_bfloat16* k_out, cudaStream_t stream) {
  launch_pool(p, qI, kI, cu, ndocs, max_doc_len, T, Hi, Di, c, ws, err, &front, k_out, q_out, stream);
  return cudaGetLastError();
}

cudaError_t launch_summaries(const IndexPlan& p, const __nv_bfloat16* kI, const __nv_bfloat16* z, const int32_t* cu,
                             int ndocs, int max_doc_len, int T, int Di, int c, uint8_t* ws, int32_t* err,
                             __nv_bfloat16* out, cudaStream_t stream) {
  int32_t* meta = reinterpret_cast<int32_t*>(ws + p.off_meta);
  int32_t* blk_off = reinterpret_cast<int32_t*>(ws + p.off_blk);
  int32_t* tile_off = reinterpret_cast<int32_t*>(ws + p.off_tile);
  layout_kernel<<<1, 1024, 0, stream>>>(cu, ndocs, T, c, p.tau_sparse, p.QT, max_doc_len, meta, blk_off, tile_off,
                                        err);
  const long long threads = (long long)p.nblk_cap * (Di / 2);
  summary_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, stream>>>(kI, z, cu, ndocs, Di, c, p.nblk_cap, meta,
                                                                        blk_off, out, nullptr);
  return cudaGetLastError();
}

cudaError_t launch_topk_from_scores(const float* scores, int64_t ldS, const int32_t* cu, int ndocs, int max_doc_len,
                                    int T, int c, int budget, int32_t* route, int32_t* err, cudaStream_t stream) {
  const int nvis_cap = max_doc_len / c > 0 ? max_doc_len / c : 1;
  TopkArgs ta{scores, ldS, cu, nullptr, route, err, ndocs, T, c, budget, max_doc_len, nvis_cap, budget + c - 1};
  return launch_topk(ta, budget / c, stream, topk_smem_bytes(nvis_cap, budget / c));
}

cudaError_t launch_compose_window(const int32_t* route, int W, const int32_t* cu, int ndocs, int T, int window,
                                  int32_t* out, int32_t* err, cudaStream_t stream) {
  compose_window_kernel<<<T, 128, 0, stream>>>(route, W, cu, ndocs, T, window, out, err);
  return cudaGetLastError();
}

cudaError_t configure_score_kernels(size_t smem) {
  cudaError_t e = configure_score_64(smem);
  if (e != cudaSuccess) return e;
  if ((e = configure_score_128(smem)) != cudaSuccess) return e;
  return configure_score_e4m3(smem);
}

cudaError_t configure_topk_kernel(size_t smem) {
  return cudaFuncSetAttribute(topk_expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

}  // namespace irs
