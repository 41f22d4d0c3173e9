// The indexer's projections on tcgen05: queries, raw keys and signed head weights from
// hidden states in one GEMM.
//
// QSA page (nemo_automodel.components.models.qwen3_8_flash_next.qsa, the indexer class):
// one fused projection produces the raw query/key layout [B, S, (H_index + 1) * D_index],
// split into queries [B, S, H_index, D_index] and raw keys [B, S, 1, D_index]. Step-5
// sparse page (nemo_automodel.components.models.step5.sparse, Step5IndexerWeightProjection):
// FP32 source weights matched by a BF16 projection give signed FP32 head weights. Here
// one bf16 weight matrix W [(Hi+1)*Di + Hi, H] holds all three: row n gives output
// column n; columns [0, Hi*Di) are the queries (head-major), [Hi*Di, (Hi+1)*Di) the raw
// keys, the last Hi the head weights. Products of bf16 values accumulate in FP32 in TMEM;
// queries and keys are rounded once to bf16 (nearest even), head weights stay FP32.
//
// Design: out[T, N] = X[T, H] . W[N, H]^T with UMMA M = 128 tokens, N = 256 output columns
// and K in 64-element SW128 atoms (both operands K-major, as they lie in memory). A
// persistent CTA per SM walks the output tiles (token tile major, so the CTAs in flight
// share their token tiles and the whole W in L2). Warp 0 issues the TMA copies of both
// operands into a 4-stage ring, warp 1 owns the tensor memory and issues the MMAs into one
// of two 256-column accumulators, and 8 epilogue warps (two per TMEM lane quarter, 128
// columns each) convert and store the previous tile while the next one accumulates. The
// MMA issue loop advances its ring stage and phase incrementally: tcgen05.mma blocks once
// the tensor pipe's short queue is full, so any latency between two atoms' MMAs idles the
// pipe. All cross-warp waits are bounded mbarrier waits.
#include "irs_internal.h"
#include "irs_ptx.cuh"

namespace irs {

namespace {

constexpr int kPM = 128;                     // tokens per tile (UMMA M)
constexpr int kPN = 256;                     // output columns per tile (UMMA N)
constexpr int kPStages = 4;
constexpr int kPEpi = 8;                     // epilogue warps
constexpr int kPThreads = 32 * (2 + kPEpi);
constexpr uint32_t kPAAtom = kPM * 128;      // 16 KB: 128 rows x 64 bf16
constexpr uint32_t kPBAtom = kPN * 128;      // 32 KB: 256 rows x 64 bf16
constexpr uint32_t kPStage = kPAAtom + kPBAtom;

struct ProjSmem {
  static constexpr uint32_t bar_off = kPStages * kPStage;
  // full[S], empty[S], t_full[2], t_empty[2], drain; then the TMEM slot and the abort word
  static constexpr uint32_t total = bar_off + (2 * kPStages + 5) * 8 + 16 + 1024;
};

// Query front half on one head row of the accumulator, read from tensor memory (the
// values rounded to bf16 first, as the unfused path's qI): RMSNorm then rotate-half RoPE,
// in FP32 with every operation rounded on its own, in the order of the indexer's
// front-half kernels (sum of squares in ascending dim order; IEEE division and square
// root; the rotation as separate products then a difference or sum), then one rounding to
// bf16. tcgen05.ld takes a run-time column, so the rotation pairs (d, d + rope_dims/2) are
// loaded where they lie. Warp-collective: every lane calls it; only rows < T store.
__device__ __forceinline__ float bf16r(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

template <int DI>
__device__ __forceinline__ void front_head(uint32_t taddr, const float* __restrict__ wt, float eps,
                                           const float* __restrict__ rope, int rope_dims, bool store,
                                           __nv_bfloat16* __restrict__ out) {
  float ss = 0.f;
#pragma unroll
  for (int c = 0; c < DI / 32; ++c) {
    float v[32];
    tmem_ld32(taddr + 32 * c, v);
    tmem_ld_wait_regs(v);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float x = bf16r(v[i]);
      ss = __fadd_rn(ss, __fmul_rn(x, x));
    }
  }
  const float r = __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)DI), eps));
  const int h = rope_dims >> 1;
  for (int d0 = 0; d0 < h; d0 += 8) {
    float a[8], b[8];
    tmem_ld8(taddr + d0, a);
    tmem_ld8(taddr + d0 + h, b);
    tmem_ld_wait_regs(a);   // waits, and keeps every use of a and b behind the wait
    tmem_ld_wait_regs(b);
    if (store) {
      __nv_bfloat162 p1[4], p2[4];
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        float o1[2], o2[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int d = d0 + i + k;
          const float y1 = __fmul_rn(__fdiv_rn(bf16r(a[i + k]), r), __ldg(wt + d));
          const float y2 = __fmul_rn(__fdiv_rn(bf16r(b[i + k]), r), __ldg(wt + d + h));
          const float cs = __ldg(rope + d), sn = __ldg(rope + h + d);
          o1[k] = __fsub_rn(__fmul_rn(y1, cs), __fmul_rn(y2, sn));
          o2[k] = __fadd_rn(__fmul_rn(y2, cs), __fmul_rn(y1, sn));
        }
        p1[i >> 1] = __floats2bfloat162_rn(o1[0], o1[1]);
        p2[i >> 1] = __floats2bfloat162_rn(o2[0], o2[1]);
      }
      *reinterpret_cast<uint4*>(out + d0) = *reinterpret_cast<const uint4*>(p1);
      *reinterpret_cast<uint4*>(out + d0 + h) = *reinterpret_cast<const uint4*>(p2);
    }
  }
  for (int d0 = rope_dims; d0 < DI; d0 += 8) {
    float a[8];
    tmem_ld8(taddr + d0, a);
    tmem_ld_wait_regs(a);
    if (store) {
      __nv_bfloat162 p[4];
#pragma unroll
      for (int i = 0; i < 8; i += 2)
        p[i >> 1] = __floats2bfloat162_rn(__fmul_rn(__fdiv_rn(bf16r(a[i]), r), __ldg(wt + d0 + i)),
                                          __fmul_rn(__fdiv_rn(bf16r(a[i + 1]), r), __ldg(wt + d0 + i + 1)));
      *reinterpret_cast<uint4*>(out + d0) = *reinterpret_cast<const uint4*>(p);
    }
  }
}

// Store one 8-column chunk of row `row` (global columns gcol .. gcol+7) where it belongs.
__device__ __forceinline__ void proj_store8(const ProjArgs& a, int row, int gcol, const float* v) {
  const int qd = a.Hi * a.Di;
  if (gcol + 8 <= qd) {
    __nv_bfloat162 p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    *reinterpret_cast<uint4*>(a.qI + (int64_t)row * qd + gcol) = *reinterpret_cast<const uint4*>(p);
  } else if (gcol >= qd && gcol + 8 <= qd + a.Di) {
    __nv_bfloat162 p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    *reinterpret_cast<uint4*>(a.kI + (int64_t)row * a.Di + (gcol - qd)) = *reinterpret_cast<const uint4*>(p);
  } else {
    // the head weights (FP32), and columns past the last one (skipped)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int n = gcol + i - qd - a.Di;
      if (n >= 0 && n < a.Hi) a.w[(int64_t)row * a.Hi + n] = v[i];
    }
  }
}

template <int FRONT_DI>   // 0: plain; 64 or 128: queries leave with the front half applied
__global__ void __launch_bounds__(kPThreads, 1)
    proj_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w, ProjArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + ProjSmem::bar_off);
  uint64_t* empty = full + kPStages;
  uint64_t* t_full = empty + kPStages;   // [2]
  uint64_t* t_empty = t_full + 2;        // [2]
  uint64_t* drain = t_empty + 2;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kPStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&t_full[i], 1); mbar_init(&t_empty[i], kPEpi); }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tslot, 2 * kPN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const int ntiles = a.tiles_m * a.tiles_n;
  const int katoms = (a.H + 63) / 64;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_map(&tm_x);
      tma_prefetch_map(&tm_w);
      int st = 0;
      uint32_t ph = 0;
      uint32_t issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
        const int m = tile / a.tiles_n, n = tile - m * a.tiles_n;
        for (int ka = 0; ka < katoms; ++ka, ++issued) {
          if (issued >= (uint32_t)kPStages && !mbar_wait(&empty[st], ph ^ 1u, abort_flag, a.err)) { ok = false; break; }
          uint8_t* dst = smem + (uint32_t)st * kPStage;
          mbar_arrive_expect_tx(&full[st], kPStage);
          tma_load_2d(dst, &tm_x, ka * 64, m * kPM, &full[st]);
          tma_load_2d(dst + kPAAtom, &tm_w, ka * 64, n * kPN, &full[st]);
          if (++st == kPStages) { st = 0; ph ^= 1u; }
        }
      }
      if (*abort_flag) {
        // let the copies still in flight land before the CTA leaves
        const uint32_t first = issued > (uint32_t)kPStages ? issued - kPStages : 0;
        for (uint32_t x = first; x < issued; ++x) {
          const unsigned long long t0 = globaltimer_ns();
          while (!mbar_try_wait(&full[x % kPStages], (x / kPStages) & 1) && globaltimer_ns() - t0 < kWaitLimitNs) {}
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t IDESC = idesc_bf16(kPM, kPN, false, false);
      const uint64_t a_desc0 = sdesc_sw128(smem_u32(smem), 16, 1024);
      const uint64_t b_desc0 = sdesc_sw128(smem_u32(smem + kPAAtom), 16, 1024);
      int st = 0;
      uint32_t ph = 0, tc = 0;
      bool alive = true;
      for (int tile = blockIdx.x; tile < ntiles && alive; tile += gridDim.x, ++tc) {
        const uint32_t buf = tc & 1u;
        if (tc >= 2 && !mbar_wait(&t_empty[buf], ((tc >> 1) - 1) & 1, abort_flag, a.err)) break;
        for (int ka = 0; ka < katoms; ++ka) {
          if (!mbar_wait(&full[st], ph, abort_flag, a.err)) { alive = false; break; }
          tc_fence_after();
          const uint64_t soff = (uint64_t)((st * kPStage) >> 4);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            umma_bf16(tbase + buf * kPN, a_desc0 + soff + (uint64_t)ks * 2, b_desc0 + soff + (uint64_t)ks * 2, IDESC,
                      (ka > 0 || ks > 0) ? 1u : 0u);
          umma_commit(&empty[st]);
          if (++st == kPStages) { st = 0; ph ^= 1u; }
        }
        if (!alive) break;
        umma_commit(&t_full[buf]);
      }
      // every issued MMA completes before the CTA releases its tensor memory
      umma_commit(drain);
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {}
    }
  } else {
    // ---------------- epilogue: warps 2..9 ----------------
    const int e = warp - 2;
    const int quarter = warp & 3;
    const int col0 = (e >> 2) * (kPN / 2);
    const uint32_t lane_addr = tmem_lane_base(warp);
    uint32_t tc = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++tc) {
      const int m = tile / a.tiles_n, n = tile - m * a.tiles_n;
      const uint32_t buf = tc & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait(&t_full[buf], (tc >> 1) & 1, abort_flag, a.err))) break;
      tc_fence_after();
      const int row = m * kPM + quarter * 32 + lane;
      if constexpr (FRONT_DI > 0) {
        const int gbase = n * kPN + col0;
        if (gbase + kPN / 2 <= a.Hi * a.Di) {
          // 128 query columns = 128 / Di whole heads of this token
          const bool live = row < a.T;
#pragma unroll 1
          for (int hd = 0; hd < (kPN / 2) / FRONT_DI; ++hd) {
            const int head = gbase / FRONT_DI + hd;
            front_head<FRONT_DI>(tbase + lane_addr + buf * kPN + col0 + hd * FRONT_DI, a.q_weight, a.eps,
                                 a.rope + (int64_t)(live ? row : 0) * a.rope_dims, a.rope_dims, live,
                                 a.qI + ((int64_t)(live ? row : 0) * a.Hi + head) * FRONT_DI);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&t_empty[buf]);
          continue;
        }
      }
#pragma unroll 1
      for (int c32 = 0; c32 < kPN / 2; c32 += 32) {
        float v[32];
        tmem_ld32(tbase + lane_addr + buf * kPN + col0 + c32, v);
        tmem_ld_wait_regs(v);
        const int gcol = n * kPN + col0 + c32;
        if (row < a.T && gcol < a.N) {
#pragma unroll
          for (int j = 0; j < 4; ++j) proj_store8(a, row, gcol + 8 * j, v + 8 * j);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&t_empty[buf]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 2 * kPN);
  }
}

}  // namespace

size_t proj_smem_bytes() { return ProjSmem::total; }

cudaError_t configure_proj_kernel() {
  cudaError_t e = cudaFuncSetAttribute(proj_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)ProjSmem::total);
  if (e != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(proj_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)ProjSmem::total)) != cudaSuccess)
    return e;
  return cudaFuncSetAttribute(proj_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ProjSmem::total);
}

cudaError_t launch_proj(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const ProjArgs& a, int num_sms,
                        cudaStream_t stream) {
  const int ntiles = a.tiles_m * a.tiles_n;
  const int grid = ntiles < num_sms ? ntiles : num_sms;
  if (a.q_weight == nullptr) proj_kernel<0><<<grid, kPThreads, ProjSmem::total, stream>>>(tm_x, tm_w, a);
  else if (a.Di == 64) proj_kernel<64><<<grid, kPThreads, ProjSmem::total, stream>>>(tm_x, tm_w, a);
  else proj_kernel<128><<<grid, kPThreads, ProjSmem::total, stream>>>(tm_x, tm_w, a);
  return cudaGetLastError();
}

}  // namespace irs
