// Gathered sparse GQA / latent attention forward on sm_103a (tcgen05 + TMEM).
//
// Semantics: QSA page (nemo_automodel.components.models.qwen3_8_flash_next.qsa,
// `gathered_qsa_gqa_attention`): query t, head h attends the keys/values of its KV
// head g = h / G at the global IDs of route row t; -1 slots are padding; softmax with
// a positive scale. Latent attention page (`cudnn_sparse_attention`): one latent KV
// head, keys are the full latent rows and values their first Dv dims.
//
// Design. A CTA owns a query row t (grid-stride over rows) and walks its KV heads and
// head blocks (<= 16 query heads of one KV head). The valid route IDs are compacted
// once per row into shared memory. Routed key/value rows stream through a ring of
// shared-memory stages with 16-byte cp.async (padding rows are zero-filled, never
// read); each chunk holds 128 keys in the SW128 atom layout. Per chunk:
//   S^T[128 keys, 16 heads]  = K_chunk . Q^T      (UMMA M=128, N=16, K=Dqk; TMEM)
//   online softmax over keys (lane = key; head maxima reduced across the 4 warps)
//   O^T[dv, 16 heads]       = V_chunk^T . P^T    (UMMA M=128 per 128 dv, N=16, K=128,
//                                                  V read MN-major straight from the
//                                                  gathered [key][dv] tile)
//   the running output (lane = dv) is rescaled and accumulated in registers.
// For latent attention the value tile is the gathered key tile itself.
#include "irs_internal.h"
#include "irs_ptx.cuh"

namespace irs {

constexpr int kAttnThreads = 128;
constexpr int kChunk = 128;   // keys per chunk (UMMA M of the score product)
constexpr int kNH = 16;       // head columns per work item (UMMA N)
constexpr int kMaxDvBlocks = 4;

struct AttnSmem {
  uint32_t k_stage, v_stage, q_off, p_off, idx_off, red_off, bar_off, total;
};

__host__ __device__ inline AttnSmem attn_smem_layout(int Dqk, int Dv, int W, int stages, int v_alias) {
  AttnSmem L{};
  L.k_stage = (uint32_t)kChunk * Dqk * 2;
  L.v_stage = v_alias ? 0u : (uint32_t)kChunk * Dv * 2;
  uint32_t off = (L.k_stage + L.v_stage) * stages;
  L.q_off = off;
  off += (uint32_t)kNH * Dqk * 2;
  off = (off + 1023u) & ~1023u;
  L.p_off = off;
  off += (uint32_t)kNH * kChunk * 2;
  L.idx_off = off;
  off += (uint32_t)W * 4;
  off = (off + 15u) & ~15u;
  L.red_off = off;
  off += 4 * kNH * 4 + 64;
  off = (off + 15u) & ~15u;
  L.bar_off = off;
  off += 64;
  L.total = off + 1024;   // alignment slack
  return L;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Issue the gathers of one chunk (keys [c*128, c*128+128) of the compacted row) into a stage.
__device__ __forceinline__ void issue_chunk(const AttnArgs& a, int g, int c, int nvalid, const int32_t* sIdx,
                                            uint8_t* sK, uint8_t* sV, int tid) {
  const int kc = a.Dqk >> 3;   // 16-byte chunks per key row
  const __nv_bfloat16* kbase = a.k + (long long)g * a.k_sh;
  const uint32_t dK = smem_u32(sK);
  for (int i = tid; i < kChunk * kc; i += kAttnThreads) {
    const int r = i / kc, j = i - r * kc;
    const int idx = c * kChunk + r;
    const int id = idx < nvalid ? sIdx[idx] : -1;
    const __nv_bfloat16* src = id >= 0 ? kbase + (long long)id * a.k_st + j * 8 : a.k;
    cp_async_16(dK + sw128_offset(r, j * 8, kChunk), src, id >= 0 ? 16u : 0u);
  }
  if (!a.v_alias) {
    const int vc = a.Dv >> 3;
    const __nv_bfloat16* vbase = a.v + (long long)g * a.v_sh;
    const uint32_t dV = smem_u32(sV);
    for (int i = tid; i < kChunk * vc; i += kAttnThreads) {
      const int r = i / vc, j = i - r * vc;
      const int idx = c * kChunk + r;
      const int id = idx < nvalid ? sIdx[idx] : -1;
      const __nv_bfloat16* src = id >= 0 ? vbase + (long long)id * a.v_st + j * 8 : a.v;
      cp_async_16(dV + sw128_offset(r, j * 8, kChunk), src, id >= 0 ? 16u : 0u);
    }
  }
}

__global__ void __launch_bounds__(kAttnThreads, 1) attn_fwd_kernel(AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const AttnSmem Lay = attn_smem_layout(a.Dqk, a.Dv, a.W, a.stages, a.v_alias);
  uint8_t* sQ = smem + Lay.q_off;
  uint8_t* sP = smem + Lay.p_off;
  int32_t* sIdx = reinterpret_cast<int32_t*>(smem + Lay.idx_off);
  float* sRed = reinterpret_cast<float*>(smem + Lay.red_off);        // [4 warps][16]
  int* sCnt = reinterpret_cast<int*>(sRed + 4 * kNH);                 // [4] + running
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + Lay.bar_off);    // [0] S done, [1] O done
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ST = a.stages;
  const uint32_t stage_bytes = Lay.k_stage + Lay.v_stage;
  const int ndvb = a.Dv / 128;
  constexpr uint32_t IDESC_S = idesc_bf16(kChunk, kNH, false, false);
  constexpr uint32_t IDESC_O = idesc_bf16(128, kNH, true, false);

  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tslot, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const uint32_t tS = tbase;                 // columns [0, 16)
  const uint32_t tO = tbase + kNH;           // columns [16, 16 + 16*ndvb)
  const uint32_t lane_addr = tmem_lane_base(warp);
  uint32_t ph_s = 0, ph_o = 0;

  for (long long t = blockIdx.x; t < a.T && !*abort_flag; t += gridDim.x) {
    // ---- compact the valid route IDs of row t ----
    const int32_t* rrow = a.route + t * a.route_stride;
    int running = 0;
    for (int base = 0; base < a.W; base += kAttnThreads) {
      const int i = base + tid;
      const int id = i < a.W ? __ldg(rrow + i) : -1;
      const bool ok = id >= 0 && id < a.Tk;
      if (i < a.W && id != -1 && !ok) record_error(a.err, IRS_DEVERR_ROUTE_ID);
      const uint32_t bal = __ballot_sync(0xffffffffu, ok);
      if (lane == 0) sCnt[warp] = __popc(bal);
      __syncthreads();
      int before = running;
      for (int w2 = 0; w2 < warp; ++w2) before += sCnt[w2];
      if (ok) sIdx[before + __popc(bal & ((1u << lane) - 1u))] = id;
      running += sCnt[0] + sCnt[1] + sCnt[2] + sCnt[3];
      __syncthreads();
    }
    const int nvalid = running;
    const int nchunks = (nvalid + kChunk - 1) / kChunk;

    for (int g = 0; g < a.Hkv && !*abort_flag; ++g) {
      for (int hb = 0; hb < a.nhb && !*abort_flag; ++hb) {
        const int h0 = g * a.G + hb * a.HB;
        const int nh = min(a.HB, a.G - hb * a.HB);
        // ---- Q tile (16 rows, zero beyond nh) in the SW128 K-major layout ----
        {
          const int qc = a.Dqk >> 3;
          for (int i = tid; i < kNH * qc; i += kAttnThreads) {
            const int r = i / qc, j = i - r * qc;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (r < nh) v = __ldg(reinterpret_cast<const uint4*>(a.q + t * a.q_st + (long long)(h0 + r) * a.q_sh + j * 8));
            *reinterpret_cast<uint4*>(sQ + sw128_offset(r, j * 8, kNH)) = v;
          }
        }
        if (nvalid == 0) {
          // reading: no valid key -> zeros and -inf
          for (int i = tid; i < nh * a.Dv; i += kAttnThreads) {
            const int h = i / a.Dv, dv = i - h * a.Dv;
            a.out[(t * a.Hq + h0 + h) * a.Dv + dv] = __float2bfloat16_rn(0.f);
          }
          if (a.lse != nullptr && tid < nh) a.lse[t * a.Hq + h0 + tid] = -INFINITY;
          __syncthreads();
          continue;
        }
        // ---- prologue: start the first ST chunks ----
        for (int c = 0; c < ST; ++c) {
          if (c < nchunks)
            issue_chunk(a, g, c, nvalid, sIdx, smem + (uint32_t)c * stage_bytes,
                        smem + (uint32_t)c * stage_bytes + Lay.k_stage, tid);
          cp_async_commit();
        }
        float m[kNH], l[kNH], acc[kMaxDvBlocks][kNH], alpha[kNH];
#pragma unroll
        for (int h = 0; h < kNH; ++h) {
          m[h] = -INFINITY;
          l[h] = 0.f;
#pragma unroll
          for (int b = 0; b < kMaxDvBlocks; ++b) acc[b][h] = 0.f;
        }
        for (int c = 0; c < nchunks; ++c) {
          const int st = c % ST;
          uint8_t* sK = smem + (uint32_t)st * stage_bytes;
          uint8_t* sV = a.v_alias ? sK : sK + Lay.k_stage;
          cp_async_wait_pending(ST - 1);
          fence_proxy_async_smem();
          __syncthreads();
          // ---- S^T = K . Q^T ----
          if (tid == 0) {
            tc_fence_after();
            const uint32_t kb = smem_u32(sK), qb = smem_u32(sQ);
            for (int ks = 0; ks < a.Dqk / 16; ++ks) {
              const uint64_t ad = sdesc_sw128(kb + (ks >> 2) * (kChunk * 128) + (ks & 3) * 32, 16, 1024);
              const uint64_t bd = sdesc_sw128(qb + (ks >> 2) * (kNH * 128) + (ks & 3) * 32, 16, 1024);
              umma_bf16(tS, ad, bd, IDESC_S, ks > 0);
            }
            umma_commit(&bar[0]);
          }
          const bool ok_s = mbar_wait(&bar[0], ph_s, abort_flag, a.err);
          ph_s ^= 1;
          tc_fence_after();
          float s[kNH];
          tmem_ld16(tS + lane_addr, s);
          tmem_ld_wait();
          const int key = c * kChunk + warp * 32 + lane;
          const bool kvalid = key < nvalid;
          // ---- online softmax (base-2 exponent domain) ----
#pragma unroll
          for (int h = 0; h < kNH; ++h) {
            s[h] = (kvalid && h < nh) ? s[h] * a.scale_log2 : -INFINITY;
            const float mx = warp_max(s[h]);
            if (lane == 0) sRed[warp * kNH + h] = mx;
          }
          if (__syncthreads_or(!ok_s)) break;   // every thread leaves together on a timeout
          float p[kNH];
#pragma unroll
          for (int h = 0; h < kNH; ++h) {
            const float cm = fmaxf(fmaxf(sRed[h], sRed[kNH + h]), fmaxf(sRed[2 * kNH + h], sRed[3 * kNH + h]));
            const float mn = fmaxf(m[h], cm);
            const float base = mn == -INFINITY ? 0.f : mn;
            alpha[h] = exp2f(m[h] - base);
            p[h] = exp2f(s[h] - base);
            l[h] = l[h] * alpha[h] + p[h];
            m[h] = mn;
          }
          // P (bf16) as the K-major B operand: row h, key column (warp*32 + lane)
          {
            const int r = warp * 32 + lane;
#pragma unroll
            for (int h = 0; h < kNH; ++h)
              *reinterpret_cast<__nv_bfloat16*>(sP + sw128_offset(h, r, kNH)) = __float2bfloat16_rn(p[h]);
          }
          tc_fence_before();
          fence_proxy_async_smem();
          __syncthreads();
          // ---- O^T_chunk = V^T . P^T ----
          if (tid == 0) {
            tc_fence_after();
            const uint32_t vb = smem_u32(sV), pb = smem_u32(sP);
            for (int b = 0; b < ndvb; ++b) {
              for (int ks = 0; ks < kChunk / 16; ++ks) {
                const uint64_t ad = sdesc_sw128(vb + (2 * b) * (kChunk * 128) + ks * 2048, kChunk * 128, 1024);
                const uint64_t bd = sdesc_sw128(pb + (ks >> 2) * (kNH * 128) + (ks & 3) * 32, 16, 1024);
                umma_bf16(tO + b * kNH, ad, bd, IDESC_O, ks > 0);
              }
            }
            umma_commit(&bar[1]);
          }
          const bool ok_o = mbar_wait(&bar[1], ph_o, abort_flag, a.err);
          ph_o ^= 1;
          tc_fence_after();
#pragma unroll
          for (int b = 0; b < kMaxDvBlocks; ++b) {
            if (b < ndvb) {
              float o[kNH];
              tmem_ld16(tO + b * kNH + lane_addr, o);
              tmem_ld_wait();
#pragma unroll
              for (int h = 0; h < kNH; ++h) acc[b][h] = acc[b][h] * alpha[h] + o[h];
            }
          }
          tc_fence_before();
          // every thread is done with this stage's smem and with S/O in TMEM
          if (__syncthreads_or(!ok_o)) break;
          // ---- refill the stage just consumed ----
          const int cn = c + ST;
          if (cn < nchunks)
            issue_chunk(a, g, cn, nvalid, sIdx, smem + (uint32_t)st * stage_bytes,
                        smem + (uint32_t)st * stage_bytes + Lay.k_stage, tid);
          cp_async_commit();
        }
        cp_async_wait_pending(0);
        if (*abort_flag) break;
        // ---- finalize: row sums across the 128 key lanes, normalise, store ----
#pragma unroll
        for (int h = 0; h < kNH; ++h) {
          const float sm = warp_sum(l[h]);
          if (lane == 0) sRed[warp * kNH + h] = sm;
        }
        __syncthreads();
        float inv[kNH];
#pragma unroll
        for (int h = 0; h < kNH; ++h) {
          const float tot = sRed[h] + sRed[kNH + h] + sRed[2 * kNH + h] + sRed[3 * kNH + h];
          inv[h] = tot > 0.f ? 1.f / tot : 0.f;
          l[h] = tot;
        }
        const int dvl = warp * 32 + lane;
#pragma unroll
        for (int b = 0; b < kMaxDvBlocks; ++b) {
          if (b < ndvb) {
#pragma unroll
            for (int h = 0; h < kNH; ++h)
              if (h < nh) a.out[(t * a.Hq + h0 + h) * a.Dv + b * 128 + dvl] = __float2bfloat16_rn(acc[b][h] * inv[h]);
          }
        }
        if (a.lse != nullptr && tid < kNH) {
          // lse = ln(2) * (m + log2(l)) with m in the base-2 domain
#pragma unroll
          for (int h = 0; h < kNH; ++h)
            if (h == tid && h < nh)
              a.lse[t * a.Hq + h0 + h] = l[h] > 0.f ? (m[h] + log2f(l[h])) * 0.69314718055994531f : -INFINITY;
        }
        __syncthreads();
      }
    }
  }
  cp_async_wait_pending(0);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 128);
  }
}

AttnPlan plan_attn(const AttnArgs& a, int num_sms) {
  AttnPlan p{};
  p.items = a.T;
  int st = 3;
  while (st > 1 && attn_smem_layout(a.Dqk, a.Dv, a.W, st, a.v_alias).total > 227 * 1024) --st;
  p.stages = st;
  p.smem = attn_smem_layout(a.Dqk, a.Dv, a.W, st, a.v_alias).total;
  const int per_sm = p.smem <= 113 * 1024 ? 2 : 1;
  const long long g = (long long)num_sms * per_sm;
  p.grid = (int)(p.items < g ? p.items : g);
  if (p.grid < 1) p.grid = 1;
  return p;
}

cudaError_t configure_attn_kernel(size_t smem) {
  return cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

cudaError_t launch_attn(const AttnArgs& a, const AttnPlan& p, cudaStream_t stream) {
  AttnArgs b = a;
  b.stages = p.stages;
  attn_fwd_kernel<<<p.grid, kAttnThreads, p.smem, stream>>>(b);
  return cudaGetLastError();
}

}  // namespace irs
