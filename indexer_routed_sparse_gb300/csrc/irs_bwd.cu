// Sparse attention backward over routed keys on sm_103a (CUDA cores, FP32).
//
// Semantics: latent attention page (`_CudnnSparseAttention.backward`): the BF16 output
// gradient is mapped to gradients of the query and of the gathered K/V rows; the GQA
// routes of the QSA page get the same gradients (the Step-5 fa4 page serves their key
// side with reverse block lists). For query t, query head h, KV head g = h / G, routed
// keys R_t and the forward's outputs out and lse (natural log):
//   p_r  = exp(scale * q.k_r - lse)
//   D    = dO . out                 (equal to sum_r p_r dO.v_r)
//   ds_r = p_r (dO.v_r - D)
//   dq   = scale * sum_r ds_r k_r,   dk_r += scale * ds_r q,   dv_r += p_r dO
//
// This is the first, plain version: the contractions are per (key, head) vector
// products on the CUDA cores. A work item is (query, KV head, block of <= 16 query heads),
// one CTA of 4 warps; warp w owns the heads j = w (mod 4) of the block, so its dq rows
// are private (shared memory, no atomics). Routed rows are staged 16 at a time; for each
// row a warp sums its heads' dk/dv contributions in registers (lane l holds dims
// l, l+32, ...), the four warps meet in a shared-memory row, and the staged rows are
// flushed to the FP32 global accumulators with float4 atomics. No waits on other CTAs.
#include "irs_internal.h"
#include "irs_ptx.cuh"

namespace irs {

namespace {

constexpr int kBwdThreads = 128;
constexpr int kBwdMaxHB = 16;          // query heads per work item
constexpr int kBwdMaxDq = 576 / 32;    // key dims per lane
constexpr int kBwdMaxDv = 512 / 32;    // value dims per lane

struct BwdLayout {
  uint32_t ids, q, dO, dq, k, v, acc, misc, total;
};

__host__ __device__ inline uint32_t round16(uint32_t x) { return (x + 15u) & ~15u; }

// ids[W] | q[HB][Dqk] f32 | dO[HB][Dv] f32 | dq[HB][Dqk] f32 | K[NKC][Dqk] bf16 |
// V[NKC][Dv] bf16 (absent when values alias keys) | acc[NKC][Dqk + Dv] f32 | D[16] lse2[16] cnt[4]
__host__ __device__ inline BwdLayout bwd_layout(int Dqk, int Dv, int W, int HB, int v_alias, int nkc) {
  BwdLayout L{};
  uint32_t off = 0;
  L.ids = off; off += round16((uint32_t)W * 4u);
  L.q = off; off += (uint32_t)(HB * Dqk) * 4u;
  L.dO = off; off += (uint32_t)(HB * Dv) * 4u;
  L.dq = off; off += (uint32_t)(HB * Dqk) * 4u;
  L.k = off; off += (uint32_t)(nkc * Dqk) * 2u;
  L.v = off; off += v_alias ? 0u : (uint32_t)(nkc * Dv) * 2u;
  L.acc = off; off += (uint32_t)(nkc * (Dqk + Dv)) * 4u;
  L.misc = off; off += (16 + 16 + 4) * 4u;
  L.total = round16(off);
  return L;
}

__global__ void __launch_bounds__(kBwdThreads) attn_bwd_kernel(BwdArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const BwdLayout L = bwd_layout(a.Dqk, a.Dv, a.W, a.HB, a.v_alias, a.nkc);
  int32_t* ids = reinterpret_cast<int32_t*>(smem + L.ids);
  float* qs = reinterpret_cast<float*>(smem + L.q);
  float* dos = reinterpret_cast<float*>(smem + L.dO);
  float* dqs = reinterpret_cast<float*>(smem + L.dq);
  __nv_bfloat16* ks = reinterpret_cast<__nv_bfloat16*>(smem + L.k);
  __nv_bfloat16* vs = a.v_alias ? ks : reinterpret_cast<__nv_bfloat16*>(smem + L.v);
  float* acc = reinterpret_cast<float*>(smem + L.acc);
  float* Dh = reinterpret_cast<float*>(smem + L.misc);
  float* l2h = Dh + 16;
  int* wcnt = reinterpret_cast<int*>(l2h + 16);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Dqk = a.Dqk, Dv = a.Dv;
  const int nq = Dqk >> 5, nvd = Dv >> 5;
  const int vrow = a.v_alias ? Dqk : Dv;      // row stride of the staged values
  const int per_t = a.Hkv * a.nhb;
  const int t = (int)(blockIdx.x / (unsigned)per_t);
  const int rem = (int)(blockIdx.x % (unsigned)per_t);
  const int g = rem / a.nhb, hb = rem % a.nhb;
  const int h0 = g * a.G + hb * a.HB;
  const int nh = min(a.HB, a.G - hb * a.HB);

  // query rows, output gradients, D = dO.out and lse (base 2) of the block's heads
  for (int i = tid; i < nh * Dqk; i += kBwdThreads) {
    const int j = i / Dqk, d = i - j * Dqk;
    qs[i] = __bfloat162float(a.q[(int64_t)t * a.q_st + (int64_t)(h0 + j) * a.q_sh + d]);
    dqs[i] = 0.f;
  }
  const __nv_bfloat16* dO_t = a.dout + ((int64_t)t * a.Hq + h0) * Dv;
  const __nv_bfloat16* o_t = a.out + ((int64_t)t * a.Hq + h0) * Dv;
  for (int i = tid; i < nh * Dv; i += kBwdThreads) dos[i] = __bfloat162float(dO_t[i]);
  for (int j = warp; j < nh; j += 4) {
    float s = 0.f;
    for (int d = lane; d < Dv; d += 32)
      s = fmaf(__bfloat162float(dO_t[j * Dv + d]), __bfloat162float(o_t[j * Dv + d]), s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) {
      Dh[j] = s;
      l2h[j] = a.lse[(int64_t)t * a.Hq + h0 + j] * 1.4426950408889634f;
    }
  }

  // valid IDs of the route row, in slot order
  int n = 0;
  for (int base = 0; base < a.W; base += kBwdThreads) {
    const int i = base + tid;
    int id = -1;
    bool ok = false;
    if (i < a.W) {
      id = a.route[(int64_t)t * a.route_stride + i];
      ok = id >= 0 && id < a.Tk;
      if (!ok && id != -1 && g == 0 && hb == 0) record_error(a.err, IRS_DEVERR_ROUTE_ID);
    }
    const unsigned bal = __ballot_sync(0xffffffffu, ok);
    if (lane == 0) wcnt[warp] = __popc(bal);
    __syncthreads();
    int off = n;
    for (int w2 = 0; w2 < warp; ++w2) off += wcnt[w2];
    if (ok) ids[off + __popc(bal & ((1u << lane) - 1u))] = id;
    n += wcnt[0] + wcnt[1] + wcnt[2] + wcnt[3];
    __syncthreads();
  }

  const int kp = Dqk >> 3, vp = Dv >> 3;       // 16-byte pieces per staged row
  const int racc = Dqk + Dv;
  for (int c0 = 0; c0 < n; c0 += a.nkc) {
    const int nc = min(a.nkc, n - c0);
    for (int i = tid; i < nc * kp; i += kBwdThreads) {
      const int r = i / kp, pc = i - r * kp;
      const uint4* src = reinterpret_cast<const uint4*>(a.k + (int64_t)ids[c0 + r] * a.k_st + (int64_t)g * a.k_sh);
      reinterpret_cast<uint4*>(ks + r * Dqk)[pc] = src[pc];
    }
    if (!a.v_alias) {
      for (int i = tid; i < nc * vp; i += kBwdThreads) {
        const int r = i / vp, pc = i - r * vp;
        const uint4* src = reinterpret_cast<const uint4*>(a.v + (int64_t)ids[c0 + r] * a.v_st + (int64_t)g * a.v_sh);
        reinterpret_cast<uint4*>(vs + r * Dv)[pc] = src[pc];
      }
    }
    for (int i = tid; i < nc * racc; i += kBwdThreads) acc[i] = 0.f;
    __syncthreads();

    if (warp < nh) {                             // warp-uniform
      for (int r = 0; r < nc; ++r) {
        float kr[kBwdMaxDq], ak[kBwdMaxDq], vr[kBwdMaxDv], av[kBwdMaxDv];
#pragma unroll
        for (int i = 0; i < kBwdMaxDq; ++i) {
          kr[i] = i < nq ? __bfloat162float(ks[r * Dqk + lane + 32 * i]) : 0.f;
          ak[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < kBwdMaxDv; ++i) {
          vr[i] = i < nvd ? __bfloat162float(vs[r * vrow + lane + 32 * i]) : 0.f;
          av[i] = 0.f;
        }
        for (int j = warp; j < nh; j += 4) {
          const float* qj = qs + j * Dqk;
          const float* dj = dos + j * Dv;
          float s = 0.f, dp = 0.f;
#pragma unroll
          for (int i = 0; i < kBwdMaxDq; ++i)
            if (i < nq) s = fmaf(qj[lane + 32 * i], kr[i], s);
#pragma unroll
          for (int i = 0; i < kBwdMaxDv; ++i)
            if (i < nvd) dp = fmaf(dj[lane + 32 * i], vr[i], dp);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            s += __shfl_xor_sync(0xffffffffu, s, o);
            dp += __shfl_xor_sync(0xffffffffu, dp, o);
          }
          const float p = ex2_approx(fmaf(s, a.scale_log2, -l2h[j]));
          const float dsk = p * (dp - Dh[j]) * a.scale;
          float* dqj = dqs + j * Dqk;
#pragma unroll
          for (int i = 0; i < kBwdMaxDq; ++i) {
            if (i < nq) {
              dqj[lane + 32 * i] = fmaf(dsk, kr[i], dqj[lane + 32 * i]);
              ak[i] = fmaf(dsk, qj[lane + 32 * i], ak[i]);
            }
          }
#pragma unroll
          for (int i = 0; i < kBwdMaxDv; ++i)
            if (i < nvd) av[i] = fmaf(p, dj[lane + 32 * i], av[i]);
        }
        float* ar = acc + r * racc;
#pragma unroll
        for (int i = 0; i < kBwdMaxDq; ++i)
          if (i < nq) atomicAdd(&ar[lane + 32 * i], ak[i]);
#pragma unroll
        for (int i = 0; i < kBwdMaxDv; ++i)
          if (i < nvd) atomicAdd(&ar[Dqk + lane + 32 * i], av[i]);
      }
    }
    __syncthreads();

    // staged rows -> FP32 global accumulators; with a shared dk/dv buffer the value
    // gradient is added into the first Dv dims of the key row
    const int fq = Dqk >> 2, fv = a.dv_alias ? 0 : (Dv >> 2);
    for (int i = tid; i < nc * (fq + fv); i += kBwdThreads) {
      const int r = i / (fq + fv);
      int pc = i - r * (fq + fv);
      const float* ar = acc + r * racc;
      const int64_t row = (int64_t)ids[c0 + r] * a.Hkv + g;
      if (pc < fq) {
        float4 x = reinterpret_cast<const float4*>(ar)[pc];
        if (a.dv_alias && 4 * pc < Dv) {
          const float4 y = reinterpret_cast<const float4*>(ar + Dqk)[pc];
          x.x += y.x; x.y += y.y; x.z += y.z; x.w += y.w;
        }
        atomicAdd(reinterpret_cast<float4*>(a.dk + row * Dqk) + pc, x);
      } else {
        pc -= fq;
        atomicAdd(reinterpret_cast<float4*>(a.dv + row * Dv) + pc, reinterpret_cast<const float4*>(ar + Dqk)[pc]);
      }
    }
    __syncthreads();
  }

  float* dq_t = a.dq + ((int64_t)t * a.Hq + h0) * Dqk;
  for (int i = tid; i < nh * Dqk; i += kBwdThreads) dq_t[i] = dqs[i];
}

// ---------------------------------------------------------------------------------------
// Fast path for the GQA shapes (values not part of the key rows): dims known at compile
// time (NQ = Dqk/32, NV = Dv/32), lane l holds dims [l*NQ, (l+1)*NQ) of every key row and
// [l*NV, (l+1)*NV) of every value row. Each warp takes whole routed rows of a staged chunk
// and loops over the block's heads: s and dp by lane-local FMAs and a butterfly, then the
// row's dk/dv contributions summed in registers and added to the global accumulators with
// vector atomics (one per lane per row), and the heads' dq partials kept in registers.
// The four warps' dq partials meet once per work item. Per (row, head) about 50
// instructions, where the general kernel above spends several hundred on predicated
// 18-wide arrays and shared-memory read-modify-writes.
// ---------------------------------------------------------------------------------------
constexpr int kFastRows = 32;   // routed rows staged per chunk (8 per warp)

struct FastLayout {
  uint32_t ids, q, dO, dq, misc, k, v, total;
};

__host__ __device__ inline FastLayout fast_layout(int Dqk, int Dv, int W, int HB) {
  FastLayout L{};
  uint32_t off = 0;
  L.ids = off; off += round16((uint32_t)W * 4u);
  L.q = off; off += (uint32_t)(HB * Dqk) * 4u;
  L.dO = off; off += (uint32_t)(HB * Dv) * 4u;
  L.dq = off; off += (uint32_t)(HB * Dqk) * 4u;
  L.misc = off; off += (16 + 16 + 4) * 4u;
  L.k = off; off += (uint32_t)(kFastRows * Dqk) * 2u;
  L.v = off; off += (uint32_t)(kFastRows * Dv) * 2u;
  L.total = round16(off);
  return L;
}

template <int N>
__device__ __forceinline__ void ld_bf16n(const __nv_bfloat16* p, float (&x)[N]) {
#pragma unroll
  for (int i = 0; i < N; i += 2) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p + i));
    x[i] = f.x;
    x[i + 1] = f.y;
  }
}
template <int N>
__device__ __forceinline__ void ld_f32n(const float* p, float (&x)[N]) {
#pragma unroll
  for (int i = 0; i < N; i += 2) {
    const float2 f = *reinterpret_cast<const float2*>(p + i);
    x[i] = f.x;
    x[i + 1] = f.y;
  }
}
// x[0..N) added to p[0..N) (p 16-byte aligned when N % 4 == 0, else 8-byte aligned)
template <int N>
__device__ __forceinline__ void red_add_n(float* p, const float (&x)[N]) {
  if constexpr (N % 4 == 0) {
#pragma unroll
    for (int i = 0; i < N; i += 4)
      atomicAdd(reinterpret_cast<float4*>(p + i), make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]));
  } else {
#pragma unroll
    for (int i = 0; i < N; i += 2) atomicAdd(reinterpret_cast<float2*>(p + i), make_float2(x[i], x[i + 1]));
  }
}

template <int NQ, int NV, int NHB>
__global__ void __launch_bounds__(kBwdThreads) attn_bwd_fast_kernel(BwdArgs a) {
  constexpr int DQ = 32 * NQ, DV = 32 * NV;
  extern __shared__ __align__(16) uint8_t smem[];
  const FastLayout L = fast_layout(DQ, DV, a.W, a.HB);
  int32_t* ids = reinterpret_cast<int32_t*>(smem + L.ids);
  float* qs = reinterpret_cast<float*>(smem + L.q);
  float* dos = reinterpret_cast<float*>(smem + L.dO);
  float* dqr = reinterpret_cast<float*>(smem + L.dq);
  float* Dh = reinterpret_cast<float*>(smem + L.misc);
  float* l2h = Dh + 16;
  int* wcnt = reinterpret_cast<int*>(l2h + 16);
  __nv_bfloat16* ks = reinterpret_cast<__nv_bfloat16*>(smem + L.k);
  __nv_bfloat16* vs = reinterpret_cast<__nv_bfloat16*>(smem + L.v);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int per_t = a.Hkv * a.nhb;
  const int t = (int)(blockIdx.x / (unsigned)per_t);
  const int rem = (int)(blockIdx.x % (unsigned)per_t);
  const int g = rem / a.nhb, hb = rem % a.nhb;
  const int h0 = g * a.G + hb * a.HB;
  const int nh = min(a.HB, a.G - hb * a.HB);

  for (int i = tid; i < nh * DQ; i += kBwdThreads) {
    const int j = i / DQ, d = i - j * DQ;
    qs[i] = __bfloat162float(a.q[(int64_t)t * a.q_st + (int64_t)(h0 + j) * a.q_sh + d]);
    dqr[i] = 0.f;
  }
  const __nv_bfloat16* dO_t = a.dout + ((int64_t)t * a.Hq + h0) * DV;
  const __nv_bfloat16* o_t = a.out + ((int64_t)t * a.Hq + h0) * DV;
  for (int i = tid; i < nh * DV; i += kBwdThreads) dos[i] = __bfloat162float(dO_t[i]);
  for (int j = warp; j < nh; j += 4) {
    float s = 0.f;
    for (int d = lane; d < DV; d += 32)
      s = fmaf(__bfloat162float(dO_t[j * DV + d]), __bfloat162float(o_t[j * DV + d]), s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) {
      Dh[j] = s;
      l2h[j] = a.lse[(int64_t)t * a.Hq + h0 + j] * 1.4426950408889634f;
    }
  }
  // valid IDs of the route row, in slot order
  int n = 0;
  for (int base = 0; base < a.W; base += kBwdThreads) {
    const int i = base + tid;
    int id = -1;
    bool ok = false;
    if (i < a.W) {
      id = a.route[(int64_t)t * a.route_stride + i];
      ok = id >= 0 && id < a.Tk;
      if (!ok && id != -1 && g == 0 && hb == 0) record_error(a.err, IRS_DEVERR_ROUTE_ID);
    }
    const unsigned bal = __ballot_sync(0xffffffffu, ok);
    if (lane == 0) wcnt[warp] = __popc(bal);
    __syncthreads();
    int off = n;
    for (int w2 = 0; w2 < warp; ++w2) off += wcnt[w2];
    if (ok) ids[off + __popc(bal & ((1u << lane) - 1u))] = id;
    n += wcnt[0] + wcnt[1] + wcnt[2] + wcnt[3];
    __syncthreads();
  }

  float dqa[NHB][NQ];
#pragma unroll
  for (int j = 0; j < NHB; ++j)
#pragma unroll
    for (int i = 0; i < NQ; ++i) dqa[j][i] = 0.f;

  constexpr int kp = DQ / 8, vp = DV / 8;   // 16-byte pieces per staged row
  for (int c0 = 0; c0 < n; c0 += kFastRows) {
    const int nc = min(kFastRows, n - c0);
    for (int i = tid; i < nc * kp; i += kBwdThreads) {
      const int r = i / kp, pc = i - r * kp;
      const uint4* src = reinterpret_cast<const uint4*>(a.k + (int64_t)ids[c0 + r] * a.k_st + (int64_t)g * a.k_sh);
      reinterpret_cast<uint4*>(ks + r * DQ)[pc] = __ldg(src + pc);
    }
    for (int i = tid; i < nc * vp; i += kBwdThreads) {
      const int r = i / vp, pc = i - r * vp;
      const uint4* src = reinterpret_cast<const uint4*>(a.v + (int64_t)ids[c0 + r] * a.v_st + (int64_t)g * a.v_sh);
      reinterpret_cast<uint4*>(vs + r * DV)[pc] = __ldg(src + pc);
    }
    __syncthreads();
    for (int r = warp; r < nc; r += 4) {
      float kr[NQ], vr[NV], ak[NQ], av[NV];
      ld_bf16n<NQ>(ks + r * DQ + lane * NQ, kr);
      ld_bf16n<NV>(vs + r * DV + lane * NV, vr);
#pragma unroll
      for (int i = 0; i < NQ; ++i) ak[i] = 0.f;
#pragma unroll
      for (int i = 0; i < NV; ++i) av[i] = 0.f;
#pragma unroll
      for (int j = 0; j < NHB; ++j) {
        if (j < nh) {   // warp-uniform
          float q[NQ], d[NV];
          ld_f32n<NQ>(qs + j * DQ + lane * NQ, q);
          ld_f32n<NV>(dos + j * DV + lane * NV, d);
          float s = 0.f, dp = 0.f;
#pragma unroll
          for (int i = 0; i < NQ; ++i) s = fmaf(q[i], kr[i], s);
#pragma unroll
          for (int i = 0; i < NV; ++i) dp = fmaf(d[i], vr[i], dp);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            s += __shfl_xor_sync(0xffffffffu, s, o);
            dp += __shfl_xor_sync(0xffffffffu, dp, o);
          }
          const float p = ex2_approx(fmaf(s, a.scale_log2, -l2h[j]));
          const float dsk = p * (dp - Dh[j]) * a.scale;
#pragma unroll
          for (int i = 0; i < NQ; ++i) {
            dqa[j][i] = fmaf(dsk, kr[i], dqa[j][i]);
            ak[i] = fmaf(dsk, q[i], ak[i]);
          }
#pragma unroll
          for (int i = 0; i < NV; ++i) av[i] = fmaf(p, d[i], av[i]);
        }
      }
      const int64_t row = (int64_t)ids[c0 + r] * a.Hkv + g;
      red_add_n<NQ>(a.dk + row * DQ + lane * NQ, ak);
      red_add_n<NV>(a.dv + row * DV + lane * NV, av);
    }
    __syncthreads();   // the staged rows are reused by the next chunk
  }
  // the four warps' dq partials, then dq out
#pragma unroll
  for (int j = 0; j < NHB; ++j)
    if (j < nh)
#pragma unroll
      for (int i = 0; i < NQ; ++i) atomicAdd(&dqr[j * DQ + lane * NQ + i], dqa[j][i]);
  __syncthreads();
  float* dq_t = a.dq + ((int64_t)t * a.Hq + h0) * DQ;
  for (int i = tid; i < nh * DQ; i += kBwdThreads) dq_t[i] = dqr[i];
}

template <int NQ, int NV>
static bool launch_fast_nq(const BwdArgs& a, unsigned items, cudaStream_t stream, cudaError_t* e) {
  const size_t smem = fast_layout(32 * NQ, 32 * NV, a.W, a.HB).total;
  auto go = [&](auto kernel) {
    *e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (*e == cudaSuccess) {
      kernel<<<items, kBwdThreads, smem, stream>>>(a);
      *e = cudaGetLastError();
    }
    return true;
  };
  if (a.HB <= 4) return go(attn_bwd_fast_kernel<NQ, NV, 4>);
  if (a.HB <= 8) return go(attn_bwd_fast_kernel<NQ, NV, 8>);
  return go(attn_bwd_fast_kernel<NQ, NV, 16>);
}

// The fast kernel when the shape has an instantiation; false otherwise.
static bool launch_fast(const BwdArgs& a, unsigned items, cudaStream_t stream, cudaError_t* e) {
  if (a.v_alias || a.dv_alias || a.HB > 16) return false;
  if (fast_layout(a.Dqk, a.Dv, a.W, a.HB).total > 227u * 1024u) return false;
  switch (a.Dqk * 1000 + a.Dv) {
    case 64064: return launch_fast_nq<2, 2>(a, items, stream, e);
    case 64128: return launch_fast_nq<2, 4>(a, items, stream, e);
    case 128128: return launch_fast_nq<4, 4>(a, items, stream, e);
    case 128256: return launch_fast_nq<4, 8>(a, items, stream, e);
    case 192128: return launch_fast_nq<6, 4>(a, items, stream, e);
    default: return false;
  }
}

}  // namespace

size_t bwd_smem_bytes(const BwdArgs& a) {
  return bwd_layout(a.Dqk, a.Dv, a.W, a.HB, a.v_alias, a.nkc).total;
}

int bwd_pick_rows(const BwdArgs& a, size_t max_smem) {
  for (int nkc = 16; nkc >= 1; nkc >>= 1)
    if (bwd_layout(a.Dqk, a.Dv, a.W, a.HB, a.v_alias, nkc).total <= max_smem) return nkc;
  return 0;
}

int bwd_max_heads() { return kBwdMaxHB; }

cudaError_t configure_bwd_kernel(size_t smem) {
  return cudaFuncSetAttribute(attn_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream) {
  const long long items = (long long)a.T * a.Hkv * a.nhb;
  if (items <= 0) return cudaSuccess;
  cudaError_t e = cudaSuccess;
  if (launch_fast(a, (unsigned)items, stream, &e)) return e;
  attn_bwd_kernel<<<(unsigned)items, kBwdThreads, bwd_smem_bytes(a), stream>>>(a);
  return cudaGetLastError();
}

}  // namespace irs
