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
  attn_bwd_kernel<<<(unsigned)items, kBwdThreads, bwd_smem_bytes(a), stream>>>(a);
  return cudaGetLastError();
}

}  // namespace irs
