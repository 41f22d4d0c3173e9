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
// The FP32 CUDA-core kernels, and the dispatch (launch_bwd) among them and the tensor-core
// kernel of irs_bwd_tc.cu. A work item is (query, KV head, block of <= 16 query heads), one
// CTA of 4 warps; no kernel waits on other CTAs.
//   attn_bwd_kernel       the general kernel (latent rows, any shape): warp w owns the heads
//                         j = w (mod 4) of the block, so its dq rows are private; routed rows
//                         are staged 16 at a time, each warp sums its heads' dk/dv
//                         contributions in registers, the four warps meet in a shared row,
//                         and staged rows go to the FP32 accumulators by float4 atomics.
//   attn_bwd_fast_kernel  separate K and V of the common head dims: one routed row per warp,
//                         all heads reduced at once (see its own comment).
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
constexpr int kFastRows = 16;   // routed rows per staged chunk; two chunk buffers

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
  L.k = off; off += (uint32_t)(2 * kFastRows * Dqk) * 2u;
  L.v = off; off += (uint32_t)(2 * kFastRows * Dv) * 2u;
  L.total = round16(off);
  return L;
}

template <int N>
__device__ __forceinline__ void ld_bf16n(const __nv_bfloat16* p, float (&x)[N]) {
  if constexpr (N % 8 == 0) {
#pragma unroll
    for (int i = 0; i < N; i += 8) {
      const uint4 u = *reinterpret_cast<const uint4*>(p + i);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
        x[i + 2 * k] = f.x;
        x[i + 2 * k + 1] = f.y;
      }
    }
  } else if constexpr (N % 4 == 0) {
#pragma unroll
    for (int i = 0; i < N; i += 4) {
      const uint2 u = *reinterpret_cast<const uint2*>(p + i);
      const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
      const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
      x[i] = f0.x;
      x[i + 1] = f0.y;
      x[i + 2] = f1.x;
      x[i + 3] = f1.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < N; i += 2) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p + i));
      x[i] = f.x;
      x[i + 1] = f.y;
    }
  }
}
// The 2H dims of one lane, as H packed FP32 pairs, from a pair-interleaved row (pair i of
// lane l at float2 index i * 32 + l): each load of the warp reads 256 contiguous bytes.
template <int H>
__device__ __forceinline__ void ld_pairs(const float* p, int lane, uint64_t (&x)[H]) {
#pragma unroll
  for (int i = 0; i < H; ++i) x[i] = *reinterpret_cast<const uint64_t*>(p + (i * 32 + lane) * 2);
}
// 2H bf16 values as H packed FP32 pairs
template <int H>
__device__ __forceinline__ void ld_bf16_pairs(const __nv_bfloat16* p, uint64_t (&x)[H]) {
  float f[2 * H];
  ld_bf16n<2 * H>(p, f);
#pragma unroll
  for (int i = 0; i < H; ++i) x[i] = pack2(f[2 * i], f[2 * i + 1]);
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
// H packed pairs added to p[0..2H)
template <int H>
__device__ __forceinline__ void red_add_pairs(float* p, const uint64_t (&x)[H]) {
  float f[2 * H];
#pragma unroll
  for (int i = 0; i < H; ++i) {
    const float2 v = unpack2(x[i]);
    f[2 * i] = v.x;
    f[2 * i + 1] = v.y;
  }
  red_add_n<2 * H>(p, f);
}

// Per-lane sizes of the fast kernel: a routed row spreads over the 32 lanes of one warp.
template <int DQ, int DV, int NHB>
struct FastShape {
  static constexpr int NQ = DQ / 32, NV = DV / 32;   // dims per lane
  static constexpr int HQ = NQ / 2, HV = NV / 2;     // ... as packed FP32 pairs
  // small head blocks keep q and dO in registers for the whole CTA (they are the same for
  // every routed row); larger ones re-read them from shared memory per row
  static constexpr bool kQReg = NHB * (NQ + NV) <= 64;
  static constexpr int V = 2 * NHB;   // partial sums per row: s and dp of each head
  static constexpr int LV = NHB == 4 ? 3 : (NHB == 8 ? 4 : 5);   // log2(V)
};

// Head j's q and dO dims of this lane: from registers, or from the lane-interleaved rows.
template <bool kQReg, int RH, int HQ, int HV>
__device__ __forceinline__ void head_vectors(const uint64_t (&qr)[RH][HQ], const uint64_t (&dr)[RH][HV],
                                             const float* qs, const float* dos, int j, int lane, uint64_t (&q)[HQ],
                                             uint64_t (&d)[HV]) {
  if constexpr (kQReg) {
#pragma unroll
    for (int i = 0; i < HQ; ++i) q[i] = qr[j][i];
#pragma unroll
    for (int i = 0; i < HV; ++i) d[i] = dr[j][i];
  } else {
    ld_pairs<HQ>(qs + j * 64 * HQ, lane, q);
    ld_pairs<HV>(dos + j * 64 * HV, lane, d);
  }
}

// One CTA per (query, KV head, head block), 4 warps. The routed rows of the query are staged
// in chunks of kFastRows; each row goes to one warp, whose lane l holds the row's K and V dims
// [l*N, (l+1)*N) and, for every head, the matching q and dO dims. Per row and
// head: s = q.k and dp = dO.v (lane partial sums, reduced together), p = exp2(s*scale*log2e
// - lse*log2e), ds = p*(dp - D)*scale, then dq += ds*k in registers and ds*q, p*dO summed
// over the heads into the row's dk and dv with one vector atomic per 4 dims.
template <int DQ, int DV, int NHB>
__global__ void __launch_bounds__(kBwdThreads) attn_bwd_fast_kernel(BwdArgs a) {
  using Sh = FastShape<DQ, DV, NHB>;
  constexpr int NQ = Sh::NQ, NV = Sh::NV, HQ = Sh::HQ, HV = Sh::HV, V = Sh::V, LV = Sh::LV;
  constexpr bool kQReg = Sh::kQReg;
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

  // q and dO as FP32, pair-interleaved: dims (2i, 2i+1) of lane l's range [l*N, (l+1)*N) of
  // head j at float2 [j][i][l], so a warp reads each pair of all its lanes as 256 bytes
  for (int i = tid; i < nh * DQ; i += kBwdThreads) {
    const int j = i / DQ, d = i - j * DQ;
    qs[j * DQ + (((d % NQ) >> 1) * 32 + d / NQ) * 2 + (d & 1)] =
        __bfloat162float(a.q[(int64_t)t * a.q_st + (int64_t)(h0 + j) * a.q_sh + d]);
    dqr[i] = 0.f;
  }
  const __nv_bfloat16* dO_t = a.dout + ((int64_t)t * a.Hq + h0) * DV;
  const __nv_bfloat16* o_t = a.out + ((int64_t)t * a.Hq + h0) * DV;
  for (int i = tid; i < nh * DV; i += kBwdThreads) {
    const int j = i / DV, d = i - j * DV;
    dos[j * DV + (((d % NV) >> 1) * 32 + d / NV) * 2 + (d & 1)] = __bfloat162float(dO_t[i]);
  }
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
  __syncthreads();   // qs, dos, Dh and l2h complete even when the route row is empty

  // all arithmetic on packed FP32 pairs (fma.rn.f32x2: two FMAs per instruction); a zero
  // pair is the all-zero bit pattern
  uint64_t dqa[NHB][HQ];
#pragma unroll
  for (int j = 0; j < NHB; ++j)
#pragma unroll
    for (int i = 0; i < HQ; ++i) dqa[j][i] = 0ull;
  constexpr int RH = kQReg ? NHB : 1;
  uint64_t qr[RH][HQ], dr[RH][HV];
  if constexpr (kQReg) {
#pragma unroll
    for (int j = 0; j < NHB; ++j) {
#pragma unroll
      for (int i = 0; i < HQ; ++i) qr[j][i] = 0ull;
#pragma unroll
      for (int i = 0; i < HV; ++i) dr[j][i] = 0ull;
      if (j < nh) {
        ld_pairs<HQ>(qs + j * DQ, lane, qr[j]);
        ld_pairs<HV>(dos + j * DV, lane, dr[j]);
      }
    }
  }

  constexpr int kp = DQ / 8, vp = DV / 8;   // 16-byte pieces per staged row
  constexpr int SH = 5 - LV;                // after the reduction, 2^SH lanes share one sum
  const int vi = lane >> SH;                // ... namely s_vi (vi < NHB) or dp_(vi-NHB)
  // chunk c's K and V rows land in buffer c & 1 by cp.async, issued one chunk ahead
  auto stage = [&](int c0, int buf) {
    const int nc = min(kFastRows, n - c0);
    const uint32_t kb = smem_u32(ks + buf * kFastRows * DQ), vb = smem_u32(vs + buf * kFastRows * DV);
    for (int i = tid; i < nc * kp; i += kBwdThreads) {
      const int r = i / kp, pc = i - r * kp;
      const uint4* src = reinterpret_cast<const uint4*>(a.k + (int64_t)ids[c0 + r] * a.k_st + (int64_t)g * a.k_sh);
      cp_async_16(kb + (uint32_t)(r * DQ + pc * 8) * 2u, src + pc, 16);
    }
    for (int i = tid; i < nc * vp; i += kBwdThreads) {
      const int r = i / vp, pc = i - r * vp;
      const uint4* src = reinterpret_cast<const uint4*>(a.v + (int64_t)ids[c0 + r] * a.v_st + (int64_t)g * a.v_sh);
      cp_async_16(vb + (uint32_t)(r * DV + pc * 8) * 2u, src + pc, 16);
    }
    cp_async_commit();
  };
  if (n > 0) stage(0, 0);
  for (int c0 = 0, buf = 0; c0 < n; c0 += kFastRows, buf ^= 1) {
    const int nc = min(kFastRows, n - c0);
    if (c0 + kFastRows < n) {
      stage(c0 + kFastRows, buf ^ 1);   // buffer buf^1 was released by the last chunk's barrier
      cp_async_wait_pending(1);
    } else {
      cp_async_wait_pending(0);
    }
    __syncthreads();
    const __nv_bfloat16* kc = ks + buf * kFastRows * DQ;
    const __nv_bfloat16* vc = vs + buf * kFastRows * DV;
    for (int r = warp; r < nc; r += 4) {
      uint64_t kr[HQ], vr[HV], ak[HQ], av[HV];
      ld_bf16_pairs<HQ>(kc + r * DQ + lane * NQ, kr);
      ld_bf16_pairs<HV>(vc + r * DV + lane * NV, vr);
#pragma unroll
      for (int i = 0; i < HQ; ++i) ak[i] = 0ull;
#pragma unroll
      for (int i = 0; i < HV; ++i) av[i] = 0ull;
      // s_j and dp_j of every head as lane partial sums, then one transposed butterfly over
      // all V = 2*NHB values: at each of the first log2(V) steps a lane keeps half of its
      // values and swaps the other half with its partner, so it ends with one sum and 2^SH
      // lanes share it: V - 1 + SH shuffles for the row instead of 5 per value
      float x[V];
#pragma unroll
      for (int j = 0; j < NHB; ++j) {
        uint64_t s2 = 0ull, dp2 = 0ull;
        if (j < nh) {   // warp-uniform
          uint64_t q[HQ], d[HV];
          head_vectors<kQReg>(qr, dr, qs, dos, j, lane, q, d);
#pragma unroll
          for (int i = 0; i < HQ; ++i) s2 = ffma2(q[i], kr[i], s2);
#pragma unroll
          for (int i = 0; i < HV; ++i) dp2 = ffma2(d[i], vr[i], dp2);
        }
        const float2 sp = unpack2(s2), dpp = unpack2(dp2);
        x[j] = sp.x + sp.y;
        x[NHB + j] = dpp.x + dpp.y;
      }
#pragma unroll
      for (int k = 0; k < LV; ++k) {
        const int o = 16 >> k, m = V >> k;
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < m / 2; ++i) {
          const float send = upper ? x[i] : x[i + m / 2];
          const float keep = upper ? x[i + m / 2] : x[i];
          x[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
#pragma unroll
      for (int o = 16 >> LV; o > 0; o >>= 1) x[0] += __shfl_xor_sync(0xffffffffu, x[0], o);
      const float dp_mine = __shfl_sync(0xffffffffu, x[0], ((vi + NHB) << SH) | (lane & ((1 << SH) - 1)));
      float p_mine = 0.f, ds_mine = 0.f;
      if (vi < nh) {
        p_mine = ex2_approx(fmaf(x[0], a.scale_log2, -l2h[vi]));
        ds_mine = p_mine * (dp_mine - Dh[vi]) * a.scale;
      }
#pragma unroll
      for (int j = 0; j < NHB; ++j) {
        if (j < nh) {   // warp-uniform
          const float p = __shfl_sync(0xffffffffu, p_mine, j << SH);
          const float dsk = __shfl_sync(0xffffffffu, ds_mine, j << SH);
          const uint64_t p2 = pack2(p, p), ds2 = pack2(dsk, dsk);
          uint64_t q[HQ], d[HV];
          head_vectors<kQReg>(qr, dr, qs, dos, j, lane, q, d);
#pragma unroll
          for (int i = 0; i < HQ; ++i) {
            dqa[j][i] = ffma2(ds2, kr[i], dqa[j][i]);
            ak[i] = ffma2(ds2, q[i], ak[i]);
          }
#pragma unroll
          for (int i = 0; i < HV; ++i) av[i] = ffma2(p2, d[i], av[i]);
        }
      }
      const int64_t row = (int64_t)ids[c0 + r] * a.Hkv + g;
      red_add_pairs<HQ>(a.dk + row * DQ + lane * NQ, ak);
      red_add_pairs<HV>(a.dv + row * DV + lane * NV, av);
    }
    __syncthreads();   // buffer buf is refilled by the next iteration's prefetch
  }
  // the four warps' dq partials, then dq out
#pragma unroll
  for (int j = 0; j < NHB; ++j)
    if (j < nh)
#pragma unroll
      for (int i = 0; i < HQ; ++i) {
        const float2 v = unpack2(dqa[j][i]);
        atomicAdd(&dqr[j * DQ + lane * NQ + 2 * i], v.x);
        atomicAdd(&dqr[j * DQ + lane * NQ + 2 * i + 1], v.y);
      }
  __syncthreads();
  float* dq_t = a.dq + ((int64_t)t * a.Hq + h0) * DQ;
  for (int i = tid; i < nh * DQ; i += kBwdThreads) dq_t[i] = dqr[i];
}

template <int DQ, int DV>
static bool launch_fast_dims(const BwdArgs& a, unsigned items, cudaStream_t stream, cudaError_t* e) {
  const size_t smem = fast_layout(DQ, DV, a.W, a.HB).total;
  auto go = [&](auto kernel) {
    *e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (*e == cudaSuccess) {
      kernel<<<items, kBwdThreads, smem, stream>>>(a);
      *e = cudaGetLastError();
    }
    return true;
  };
  if (a.HB <= 4) return go(attn_bwd_fast_kernel<DQ, DV, 4>);
  if (a.HB <= 8) return go(attn_bwd_fast_kernel<DQ, DV, 8>);
  return go(attn_bwd_fast_kernel<DQ, DV, 16>);
}

// The fast kernel when the shape has an instantiation; false otherwise.
static bool launch_fast(const BwdArgs& a, unsigned items, cudaStream_t stream, cudaError_t* e) {
  if (a.v_alias || a.dv_alias || a.HB > 16) return false;
  if (fast_layout(a.Dqk, a.Dv, a.W, a.HB).total > 227u * 1024u) return false;
  switch (a.Dqk * 1000 + a.Dv) {
    case 64064: return launch_fast_dims<64, 64>(a, items, stream, e);
    case 64128: return launch_fast_dims<64, 128>(a, items, stream, e);
    case 128128: return launch_fast_dims<128, 128>(a, items, stream, e);
    case 128256: return launch_fast_dims<128, 256>(a, items, stream, e);
    case 192128: return launch_fast_dims<192, 128>(a, items, stream, e);
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
  // Tensor cores for blocks of 8 or more query heads; with fewer heads per routed row the
  // CUDA-core warp-per-row kernel is as fast (4 heads: 31.0 against 32.4 ms on the mid
  // workload) and takes over where it has an instantiation.
  const bool tc = bwd_tc_supported(a);
  if (tc && a.HB >= 8) return launch_bwd_tc(a, (unsigned)items, stream);
  if (launch_fast(a, (unsigned)items, stream, &e)) return e;
  if (tc) return launch_bwd_tc(a, (unsigned)items, stream);
  attn_bwd_kernel<<<(unsigned)items, kBwdThreads, bwd_smem_bytes(a), stream>>>(a);
  return cudaGetLastError();
}

}  // namespace irs
