// Sparse latent attention forward (one latent KV head, many query heads) on sm_103a.
//
// Semantics: latent attention page (`cudnn_sparse_attention`): every query head of query
// t attends the latent rows at the valid IDs of route row t; the keys are the full Dqk-dim
// latent rows and the values their first Dv dims; softmax with a positive scale, lse in
// natural log; a row without valid IDs gives zeros and lse = -inf.
//
// Why a kernel of its own. With 128 query heads, 576-dim keys and 512-dim values, every
// gathered 1152-byte row feeds 128 x (576 + 512) multiply-adds, so the work is balanced
// between HBM and the tensor cores and a row must be used by many heads while it sits in
// shared memory. The GQA kernel (<= 16 heads per pass, output folded in registers) would
// gather each row once per 16 heads. Here a work item is (query t, block of 64 heads):
//   * the 64 x Dqk query tile Q^T stays in shared memory for the whole route;
//   * routed rows arrive in 64-row stages (Dqk/64 SW128 atoms of 64 rows each);
//   * S^T = K.Q^T runs as M=128 (keys) x N=64 (heads): rows 64..127 read the next atom and
//     are ignored (a 64-row chunk keeps two stages in 227 KB);
//   * O^T = V^T.P^T (M=128 dv per block, N=64 heads, K=64 keys) accumulates in TMEM over
//     the whole route (4 blocks x 64 columns for Dv = 512); P is written key-major (one
//     128-byte row of 64 heads per key, read as an MN-major operand) over the last key
//     atom of the stage, which S no longer needs (so Dqk >= Dv + 64);
//   * row sums stay in FP32: each softmax thread (one key) accumulates its 64 unrounded
//     probabilities in its own TMEM row beside O^T, and the rows are summed over the keys
//     once per item;
//   * running maxima move only when a score exceeds them by more than 2^8 (base-2
//     scores). Each softmax thread checks its 64 scores against that bound and the two
//     softmax warps vote; only then (and at the start of an item) are the head maxima
//     reduced over the keys, and O^T and the row sums rescaled in TMEM. The maxima are
//     kept in TMEM beside the row sums, one copy per softmax lane: the hot path reads no
//     shared memory, whose load queue the producers' copies keep full.
// Consecutive items are the two head blocks of one query, so neighbouring CTAs gather
// the same rows and the second read is an L2 hit.
//
// Warp roles: 9 producer warps (route compaction, query tile and row gathers with 16-byte
// cp.async), an S issuer (also TMEM owner), an O issuer, and 4 softmax/correction warps
// (the two whose TMEM lane quarters hold keys 0..63 compute the softmax; all four rescale
// and store O). All waits are bounded mbarrier waits.
#include "irs_internal.h"
#include "irs_ptx.cuh"

namespace irs {

namespace {

constexpr int kMH = 64;                    // query heads per work item (UMMA N)
constexpr int kMK = 64;                    // keys per chunk
constexpr uint32_t kAtom = kMK * 128;      // one 64-dim SW128 atom of 64 rows: 8 KB
constexpr int kMlaStages = 2;
constexpr int kMlaPW = 9;                  // producer warps (288 threads: 4 rows of 72 pieces per pass)
constexpr int kMlaProducers = 32 * kMlaPW;
constexpr int kMlaThreads = 32 * (kMlaPW + 6);
constexpr float kRescaleLog2 = 8.f;
constexpr uint32_t kTmemCols = 512;        // S^T 2 x 64, O^T up to 4 x 64, row sums 64 columns
constexpr uint32_t kOCol = 2 * kMH;        // first O^T column
constexpr uint32_t kLCol = 6 * kMH;        // per-key FP32 row sums (lanes 0..63)
constexpr uint32_t kMCol = 7 * kMH;        // running head maxima, one copy per softmax lane

struct MlaLayout {
  uint32_t stage_bytes, q_off, idx_off, misc_off, bar_off, total;
};

__host__ __device__ inline MlaLayout mla_layout(int Dqk, int W) {
  MlaLayout L{};
  const uint32_t katoms = (uint32_t)Dqk / 64;
  L.stage_bytes = katoms * kAtom;
  L.q_off = L.stage_bytes * kMlaStages;
  L.idx_off = L.q_off + katoms * kAtom;
  L.misc_off = L.idx_off + (uint32_t)((W + 63) / 64) * 64 * 4;
  // m_run[64] alpha[64] red[2][64] | flagw[2][2] flag[2] nv[2] cnt[kMlaPW]
  L.bar_off = L.misc_off + (64 * 2 + 128) * 4 + (4 + 2 + 2 + 12) * 4;
  L.total = L.bar_off + 26 * 8 + 16;
  return L;
}

// transposed butterfly over 32 values per lane: at each step a lane keeps half of its
// values and swaps the other half with its partner, so lane L ends with the reduction of
// value L over the warp (31 shuffles instead of 5 x 32)
template <bool MAX>
__device__ __forceinline__ float mla_reduce32(const float (&x)[32], int lane) {
  float v[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const bool up = (lane & 16) != 0;
    const float send = up ? x[i] : x[i + 16];
    const float keep = up ? x[i + 16] : x[i];
    const float got = __shfl_xor_sync(0xffffffffu, send, 16);
    v[i] = MAX ? fmaxf(keep, got) : keep + got;
  }
#pragma unroll
  for (int lvl = 1; lvl < 5; ++lvl) {
    const int half = 16 >> lvl, o = 16 >> lvl;
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = up ? v[i] : v[i + half];
      const float keep = up ? v[i + half] : v[i];
      const float got = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  return v[0];
}

// S^T (+)= K.Q^T: A = stage (64-row atoms, rows 64..127 of the M=128 product fall in the
// next atom and are never read back), B = Q^T (64 head rows per atom).
template <int KA>
__device__ __forceinline__ void mla_issue_s(uint32_t d, uint32_t kb, uint32_t qb, uint32_t idesc) {
  const uint64_t a0 = sdesc_sw128(kb, 16, 1024), b0 = sdesc_sw128(qb, 16, 1024);
#pragma unroll
  for (int ks = 0; ks < 4 * KA; ++ks) {
    const uint64_t step = (uint64_t)(((ks >> 2) * kAtom + (ks & 3) * 32) >> 4);
    umma_bf16(d, a0 + step, b0 + step, idesc, ks > 0);
  }
}
__device__ __forceinline__ void mla_issue_s_any(int katoms, uint32_t d, uint32_t kb, uint32_t qb, uint32_t idesc) {
  switch (katoms) {
    case 2: mla_issue_s<2>(d, kb, qb, idesc); break;
    case 3: mla_issue_s<3>(d, kb, qb, idesc); break;
    case 4: mla_issue_s<4>(d, kb, qb, idesc); break;
    case 5: mla_issue_s<5>(d, kb, qb, idesc); break;
    case 6: mla_issue_s<6>(d, kb, qb, idesc); break;
    case 7: mla_issue_s<7>(d, kb, qb, idesc); break;
    case 8: mla_issue_s<8>(d, kb, qb, idesc); break;
    default: mla_issue_s<9>(d, kb, qb, idesc); break;
  }
}
// O^T (+)= V^T.P^T for NB blocks of 128 dv: A = V^T read MN-major from the stage (two
// 64-dv atoms per block, LBO = one atom), B = P stored key-major (64 key rows x 64 heads,
// MN-major operand).
template <int NB>
__device__ __forceinline__ void mla_issue_o(uint32_t d, uint32_t vb, uint32_t pb, uint32_t idesc, bool acc) {
  const uint64_t a0 = sdesc_sw128(vb, kAtom, 1024), b0 = sdesc_sw128(pb, kAtom, 1024);
#pragma unroll
  for (int blk = 0; blk < NB; ++blk) {
#pragma unroll
    for (int ks = 0; ks < kMK / 16; ++ks)
      umma_bf16(d + blk * kMH, a0 + (uint64_t)(((2 * blk) * kAtom + ks * 2048) >> 4),
                b0 + (uint64_t)((ks * 2048) >> 4), idesc, (acc || ks > 0) ? 1u : 0u);
  }
}
__device__ __forceinline__ void mla_issue_o_any(int ndvb, uint32_t d, uint32_t vb, uint32_t pb, uint32_t idesc,
                                                bool acc) {
  switch (ndvb) {
    case 1: mla_issue_o<1>(d, vb, pb, idesc, acc); break;
    case 2: mla_issue_o<2>(d, vb, pb, idesc, acc); break;
    case 3: mla_issue_o<3>(d, vb, pb, idesc, acc); break;
    default: mla_issue_o<4>(d, vb, pb, idesc, acc); break;
  }
}
// rows x kc 16-byte pieces into a tile of 64-row SW128 atoms (row stride `stride`
// elements; row r comes from base + ids[r] * stride, or base + r * stride without ids)
__device__ __forceinline__ void mla_copy_rows(uint32_t dst, const __nv_bfloat16* base, int64_t stride,
                                              const int32_t* ids, int rows, int kc, int ptid) {
  const int dr = kMlaProducers / kc;
  if (dr >= 1 && ptid < dr * kc) {
    const int j = ptid % kc;
    const uint32_t atom = (uint32_t)(j >> 3) * kAtom;
    const uint32_t jc = (uint32_t)(j & 7);
    const __nv_bfloat16* sj = base + j * 8;
#pragma unroll 4
    for (int r = ptid / kc; r < rows; r += dr) {
      const int64_t id = ids != nullptr ? (int64_t)ids[r] : (int64_t)r;
      cp_async_16(dst + atom + (uint32_t)r * 128 + ((jc ^ ((uint32_t)r & 7)) << 4), sj + id * stride, 16u);
    }
  }
}

__global__ void __launch_bounds__(kMlaThreads, 1) mla_fwd_kernel(AttnArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the layout leaves no slack for re-alignment: the dynamic window starts 1 KB aligned
  if ((smem_u32(smem) & 1023u) != 0) {
    if (tid == 0) record_error(a.err, IRS_DEVERR_TIMEOUT);
    return;
  }
  constexpr int kSW = kMlaPW;          // S issuer, TMEM owner
  constexpr int kOW = kMlaPW + 1;      // O issuer
  constexpr int kXW = kMlaPW + 2;      // first of the 4 softmax/correction warps
  const MlaLayout Ly = mla_layout(a.Dqk, a.W);
  const int katoms = a.Dqk >> 6;
  const int ndvb = a.Dv >> 7;
  const int kc = a.Dqk >> 3;
  const int nhb = a.Hq / kMH;
  const long long items = (long long)a.T * nhb;
  uint8_t* sQ = smem + Ly.q_off;
  int32_t* sIdx = reinterpret_cast<int32_t*>(smem + Ly.idx_off);
  float* m_run = reinterpret_cast<float*>(smem + Ly.misc_off);
  float* alpha = m_run + 64;
  float* red = alpha + 64;       // [2 softmax warps][64]
  int32_t* flagw = reinterpret_cast<int32_t*>(red + 128);   // [2 chunk parities][2 softmax warps]
  int32_t* flag = flagw + 4;                                // [2] chunk needs an O/l rescale
  int32_t* sNv = flag + 2;                                  // [2]
  int32_t* sCnt = sNv + 2;                                  // [kMlaPW]
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + Ly.bar_off);
  uint64_t* kv_full = bar;           // [2]
  uint64_t* kv_empty = bar + 2;      // [2]
  uint64_t* q_full = bar + 4;
  uint64_t* q_empty = bar + 5;
  uint64_t* idx_full = bar + 6;      // [2]
  uint64_t* idx_empty = bar + 8;     // [2]
  uint64_t* s_full = bar + 10;       // [2]
  uint64_t* s_empty = bar + 12;      // [2]
  uint64_t* p_full = bar + 14;       // [2]
  uint64_t* red_bar = bar + 16;
  uint64_t* red2_bar = bar + 17;
  uint64_t* stat_bar = bar + 18;
  uint64_t* corr_bar = bar + 19;
  uint64_t* fin_bar = bar + 22;
  uint64_t* o_full = bar + 20;
  uint64_t* o_free = bar + 21;
  uint64_t* drain = bar + 24;        // [2]: the S and O issuers' last products have completed
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 26);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  constexpr uint32_t IDESC_S = idesc_bf16(128, kMH, false, false);
  constexpr uint32_t IDESC_O = idesc_bf16(128, kMH, true, true);

  // ---- set-up: finite operand memory (S^T reads 64 rows past every atom), barriers, TMEM ----
  {
    uint4* z = reinterpret_cast<uint4*>(smem);
    for (uint32_t i = tid; i < Ly.idx_off / 16; i += kMlaThreads) z[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kv_full[i], kMlaProducers);
      mbar_init(&kv_empty[i], 1);
      mbar_init(&idx_full[i], 1);
      mbar_init(&idx_empty[i], 6);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 2);
      mbar_init(&p_full[i], 2);
    }
    mbar_init(q_full, kMlaProducers);
    mbar_init(q_empty, 1);
    mbar_init(red_bar, 4);
    mbar_init(red2_bar, 2);
    mbar_init(stat_bar, 1);
    mbar_init(corr_bar, 4);
    mbar_init(fin_bar, 2);
    mbar_init(o_full, 1);
    mbar_init(o_free, 4);
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kSW) {
    tmem_alloc(tslot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  if (warp < kMlaPW) {
    // =========================== producers ===========================
    const int ptid = tid;
    uint32_t n = 0, qi = 0, uq = 0;
    bool mine = true;
    for (long long it = blockIdx.x; it < items; it += gridDim.x, ++qi) {
      const long long t = it / nhb;
      const int h0 = (int)(it - t * nhb) * kMH;
      const int b = qi & 1;
      const bool ok = mine && (qi < 2 || mbar_wait(&idx_empty[b], ((qi >> 1) - 1) & 1, abort_flag, a.err));
      if (!named_bar_and(1, kMlaProducers, ok)) break;
      // ---- compact the valid IDs of route row t ----
      const int32_t* rrow = a.route + t * a.route_stride;
      int run = 0;
      for (int base = 0; base < a.W; base += 8 * kMlaProducers) {
        int ids[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int i = base + k * kMlaProducers + ptid;
          ids[k] = i < a.W ? __ldg(rrow + i) : -1;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (base + k * kMlaProducers >= a.W) break;
          const int i = base + k * kMlaProducers + ptid;
          const int id = ids[k];
          const bool okid = id >= 0 && id < a.Tk;
          if (i < a.W && id != -1 && !okid && h0 == 0) record_error(a.err, IRS_DEVERR_ROUTE_ID);
          const uint32_t bal = __ballot_sync(0xffffffffu, okid);
          if (lane == 0) sCnt[warp] = __popc(bal);
          named_bar_sync(1, kMlaProducers);
          int before = run;
          for (int w2 = 0; w2 < warp; ++w2) before += sCnt[w2];
          if (okid) sIdx[before + __popc(bal & ((1u << lane) - 1u))] = id;
          for (int w2 = 0; w2 < kMlaPW; ++w2) run += sCnt[w2];
          named_bar_sync(1, kMlaProducers);
        }
      }
      if (ptid == 0) sNv[b] = run;
      named_bar_sync(1, kMlaProducers);
      if (ptid == 0) mbar_arrive(&idx_full[b]);
      const int nv = run;
      if (nv == 0) continue;
      // ---- query tile of the 64 heads ----
      if (uq >= 1 && !mbar_wait(q_empty, (uq - 1) & 1, abort_flag, a.err)) mine = false;
      ++uq;
      if (!mine) continue;
      mla_copy_rows(smem_u32(sQ), a.q + t * a.q_st + (int64_t)h0 * a.q_sh, a.q_sh, nullptr, kMH, kc, ptid);
      cp_async_mbar_arrive_noinc(q_full);
      // ---- routed rows, 64 per stage ----
      const int nchunks = (nv + kMK - 1) / kMK;
      for (int c = 0; c < nchunks; ++c, ++n) {
        const int st = n & 1;
        if (n >= 2 && !mbar_wait(&kv_empty[st], ((n >> 1) - 1) & 1, abort_flag, a.err)) { mine = false; break; }
        mla_copy_rows(smem_u32(smem + st * Ly.stage_bytes), a.k, a.k_st, sIdx + c * kMK, min(kMK, nv - c * kMK), kc,
                      ptid);
        cp_async_mbar_arrive_noinc(&kv_full[st]);
      }
    }
    cp_async_wait_pending(0);
  } else if (warp == kSW) {
    // =========================== S issuer ===========================
    if (lane == 0) {
      uint32_t n = 0, qi = 0, uq = 0;
      bool alive = true;
      for (long long it = blockIdx.x; it < items && alive; it += gridDim.x, ++qi) {
        const int b = qi & 1;
        if (!mbar_wait(&idx_full[b], (qi >> 1) & 1, abort_flag, a.err)) break;
        const int nv = sNv[b];
        mbar_arrive(&idx_empty[b]);
        if (nv == 0) continue;
        if (!mbar_wait(q_full, uq & 1, abort_flag, a.err)) break;
        ++uq;
        const int nchunks = (nv + kMK - 1) / kMK;
        for (int c = 0; c < nchunks; ++c, ++n) {
          const int st = n & 1, sb = n & 1;
          if (!mbar_wait(&kv_full[st], (n >> 1) & 1, abort_flag, a.err)) { alive = false; break; }
          if (n >= 2 && !mbar_wait(&s_empty[sb], ((n >> 1) - 1) & 1, abort_flag, a.err)) { alive = false; break; }
          fence_proxy_async_smem();   // cp.async rows (generic proxy) -> UMMA reads
          tc_fence_after();
          mla_issue_s_any(katoms, tbase + sb * kMH, smem_u32(smem + st * Ly.stage_bytes), smem_u32(sQ), IDESC_S);
          umma_commit(&s_full[sb]);
        }
        if (alive) umma_commit(q_empty);
      }
      // every S product this thread issued completes before the CTA releases tensor memory
      umma_commit(&drain[0]);
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_try_wait(&drain[0], 0) && globaltimer_ns() - t0 < kWaitLimitNs) {}
    }
  } else if (warp == kOW) {
    // =========================== O issuer ===========================
    if (lane == 0) {
      uint32_t m = 0, qi = 0, uq = 0, kcorr = 0;
      bool alive = true;
      for (long long it = blockIdx.x; it < items && alive; it += gridDim.x, ++qi) {
        const int b = qi & 1;
        if (!mbar_wait(&idx_full[b], (qi >> 1) & 1, abort_flag, a.err)) break;
        const int nv = sNv[b];
        mbar_arrive(&idx_empty[b]);
        if (nv == 0) continue;
        // the O^T accumulator is overwritten by the first chunk: the previous item's
        // output must have been read out
        if (uq >= 1 && !mbar_wait(o_free, (uq - 1) & 1, abort_flag, a.err)) break;
        ++uq;
        const int nchunks = (nv + kMK - 1) / kMK;
        for (int c = 0; c < nchunks; ++c, ++m) {
          const int pb = m & 1;
          if (!mbar_wait(&p_full[pb], (m >> 1) & 1, abort_flag, a.err)) { alive = false; break; }
          if (flag[pb]) {
            if (!mbar_wait(corr_bar, kcorr & 1, abort_flag, a.err)) { alive = false; break; }
            ++kcorr;
          }
          tc_fence_after();
          const uint32_t stage = smem_u32(smem + (m & 1) * Ly.stage_bytes);
          const uint32_t pkeys = stage + (uint32_t)(katoms - 1) * kAtom;
          mla_issue_o_any(ndvb, tbase + kOCol, stage, pkeys, IDESC_O, c > 0);
          umma_commit(o_full);
          umma_commit(&kv_empty[m & 1]);
        }
      }
      umma_commit(&drain[1]);
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_try_wait(&drain[1], 0) && globaltimer_ns() - t0 < kWaitLimitNs) {}
    }
  } else {
    // =========================== softmax + correction ===========================
    const int q = warp & 3;                       // TMEM lane quarter
    const int lanerow = q * 32 + lane;            // key of S (q < 2), dv of O
    const uint32_t lane_addr = tmem_lane_base(warp);
    uint32_t n = 0, qi = 0, uq = 0, kslow = 0, kcorr = 0;
    for (long long it = blockIdx.x; it < items; it += gridDim.x, ++qi) {
      const long long t = it / nhb;
      const int h0 = (int)(it - t * nhb) * kMH;
      const int b = qi & 1;
      if (!mbar_wait(&idx_full[b], (qi >> 1) & 1, abort_flag, a.err)) break;
      const int nv = min(max(sNv[b], 0), a.W);
      __syncwarp();
      if (lane == 0) mbar_arrive(&idx_empty[b]);
      __nv_bfloat16* orow = a.out + (t * a.Hq + h0) * (int64_t)a.Dv;
      if (nv == 0) {
        // reading: a row without any valid key gives zeros and lse = -inf
        for (int blk = 0; blk < ndvb; ++blk)
          for (int h = 0; h < kMH; ++h) orow[(int64_t)h * a.Dv + blk * 128 + lanerow] = __float2bfloat16_rn(0.f);
        if (a.lse != nullptr && q == 0) {
          a.lse[t * a.Hq + h0 + lane] = -INFINITY;
          a.lse[t * a.Hq + h0 + lane + 32] = -INFINITY;
        }
        continue;
      }
      const int nchunks = (nv + kMK - 1) / kMK;
      for (int c = 0; c < nchunks; ++c, ++n) {
        const int sb = n & 1;
        const bool kvalid = c * kMK + lanerow < nv;
        const uint32_t sbuf = tbase + sb * kMH + lane_addr;
        uint8_t* prow = smem + (n & 1) * Ly.stage_bytes + (katoms - 1) * kAtom + lanerow * 128;
        // p = 2^(s - m) for this key's 64 heads, 16 at a time from TMEM (scores and maxima
        // stay there, so few registers are live; spills would queue behind the producers'
        // copies). The FP32 row sums in TMEM are set (mode 0), accumulated (1), or rescaled
        // and accumulated (2); P goes key-major over the last key atom of the stage (S of
        // this chunk is complete): row `lanerow`, 16-byte chunk j = heads 8j..8j+7 at chunk
        // position j ^ (row & 7). Returns the largest margin s - m over the heads.
        auto p_pass = [&](int mode) -> float {
          float dmax = -INFINITY;
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            float v[16], lp[16], mr[16];
            tmem_ld16(sbuf + qq * 16, v);
            tmem_ld16(tbase + kMCol + qq * 16 + lane_addr, mr);
            const uint32_t ta = tbase + kLCol + qq * 16 + lane_addr;
            if (mode != 0) tmem_ld16(ta, lp);
            tmem_ld_wait_regs(v);
            tmem_ld_wait_regs(mr);
            if (mode != 0) tmem_ld_wait_regs(lp);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float x = fmaf(v[i], a.scale_log2, -mr[i]);
              dmax = fmaxf(dmax, x);
              v[i] = kvalid ? ex2_approx(x) : 0.f;
            }
            // explicit (warp-uniform) branches keep the rare rescale factor loads off the
            // common path
            if (mode == 0) {
#pragma unroll
              for (int i = 0; i < 16; ++i) lp[i] = v[i];
            } else if (mode == 1) {
#pragma unroll
              for (int i = 0; i < 16; ++i) lp[i] += v[i];
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i) lp[i] = fmaf(lp[i], alpha[qq * 16 + i], v[i]);
            }
            tmem_st16(ta, lp);
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
              uint32_t pk[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 two = __floats2bfloat162_rn(v[8 * jj + 2 * e], v[8 * jj + 2 * e + 1]);
                pk[e] = *reinterpret_cast<const uint32_t*>(&two);
              }
              const int j = qq * 2 + jj;
              *reinterpret_cast<uint4*>(prow + ((j ^ (lanerow & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
            tmem_st_wait();   // lp's registers are reused by the next pass
          }
          return kvalid ? dmax : -INFINITY;
        };
        if (q < 2) {
          mbar_wait(&s_full[sb], (n >> 1) & 1, abort_flag, a.err);
          __syncwarp();   // converge after the polling wait: tcgen05.ld/st are warp-aligned
          tc_fence_after();
          // after the first chunk of a route, P and the row sums are computed at once with the
          // current maxima; the vote below keeps them unless some score passed its bound
          const bool ex = c == 0 || p_pass(1) > kRescaleLog2;   // c is warp-uniform
          const bool any = __any_sync(0xffffffffu, ex);
          if (lane == 0) flagw[sb * 2 + q] = any ? 1 : 0;
          __syncwarp();
        }
        // o_full completes once per chunk; a parity wait is only sound if every phase is
        // waited in order, before the next one can complete. Warps 2 and 3 wait for O of
        // the previous chunk here (O of this chunk needs their arrival below), warps 0 and 1
        // before they release this chunk's P.
        if (q >= 2 && c > 0) mbar_wait(o_full, (n - 1) & 1, abort_flag, a.err);
        if (lane == 0) mbar_arrive(red_bar);
        mbar_wait(red_bar, n & 1, abort_flag, a.err);
        __syncwarp();
        const bool slow = (flagw[sb * 2] | flagw[sb * 2 + 1]) != 0;
        if (slow) {
          if (q < 2 && c > 0) {
            // take the speculative p (at the old maxima, still in TMEM) back out of the sums
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
              float v[16], lp[16], mr[16];
              const uint32_t ta = tbase + kLCol + qq * 16 + lane_addr;
              tmem_ld16(sbuf + qq * 16, v);
              tmem_ld16(tbase + kMCol + qq * 16 + lane_addr, mr);
              tmem_ld16(ta, lp);
              tmem_ld_wait_regs(v);
              tmem_ld_wait_regs(mr);
              tmem_ld_wait_regs(lp);
#pragma unroll
              for (int i = 0; i < 16; ++i) lp[i] -= kvalid ? ex2_approx(fmaf(v[i], a.scale_log2, -mr[i])) : 0.f;
              tmem_st16(ta, lp);
              tmem_st_wait();
            }
          }
          // reduce the head maxima over the 64 keys; move those that grew past the bound
          if (q < 2) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              float v[32];
              tmem_ld32(sbuf + half * 32, v);
              tmem_ld_wait_regs(v);
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = kvalid ? v[i] * a.scale_log2 : -INFINITY;
              red[q * 64 + half * 32 + lane] = mla_reduce32<true>(v, lane);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(red2_bar);
          }
          if (q == 0) {
            mbar_wait(red2_bar, kslow & 1, abort_flag, a.err);
            bool need = false;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int h = lane + 32 * e;
              const float cm = fmaxf(red[h], red[64 + h]);
              float mn = cm, al = 1.f;
              if (c > 0) {
                const float mo = m_run[h];
                if (cm > mo + kRescaleLog2) {
                  al = ex2_approx(mo - cm);
                  need = true;
                } else {
                  mn = mo;
                }
              }
              m_run[h] = mn;
              alpha[h] = al;
            }
            need = __any_sync(0xffffffffu, need);
            if (lane == 0) flag[sb] = need ? 1 : 0;
            __syncwarp();
            if (lane == 0) mbar_arrive(stat_bar);
          } else {
            mbar_wait(stat_bar, kslow & 1, abort_flag, a.err);
          }
          __syncwarp();
          ++kslow;
          if (q < 2) {
            // every softmax lane keeps its own copy of the maxima in TMEM
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              float mr[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) mr[i] = m_run[half * 32 + i];
              tmem_st32(tbase + kMCol + half * 32 + lane_addr, mr);
              tmem_st_wait();
            }
            (void)p_pass(c == 0 ? 0 : (flag[sb] != 0 ? 2 : 1));
          }
        } else if (q == 0 && lane == 0) {
          flag[sb] = 0;
        }
        if (q < 2) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&s_empty[sb]);
          fence_proxy_async_smem();
          if (c > 0) mbar_wait(o_full, (n - 1) & 1, abort_flag, a.err);
          __syncwarp();
          if (lane == 0) mbar_arrive(&p_full[sb]);
        }
        if (slow && flag[sb]) {
          // O^T holds chunks 0..c-1 at the old maxima (all complete: waited above)
          __syncwarp();
          tc_fence_after();
          for (int blk = 0; blk < ndvb; ++blk)
            for (int half = 0; half < 2; ++half) {
              float v[32];
              const uint32_t ta = tbase + kOCol + blk * kMH + half * 32 + lane_addr;
              tmem_ld32(ta, v);
              tmem_ld_wait_regs(v);
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] *= alpha[half * 32 + i];
              tmem_st32(ta, v);
              tmem_st_wait();   // the registers are reused by the next load
            }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(corr_bar);
          mbar_wait(corr_bar, kcorr & 1, abort_flag, a.err);
          ++kcorr;
        }
      }
      // ---- epilogue: sum the per-key row sums over the 64 keys, then O^T / l -> out, lse ----
      if (q < 2) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float lp[32];
          tmem_ld32(tbase + kLCol + half * 32 + lane_addr, lp);
          tmem_ld_wait_regs(lp);
          red[q * 64 + half * 32 + lane] = mla_reduce32<false>(lp, lane);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(fin_bar);
      }
      mbar_wait(fin_bar, uq & 1, abort_flag, a.err);
      ++uq;
      mbar_wait(o_full, (n - 1) & 1, abort_flag, a.err);
      __syncwarp();
      tc_fence_after();
      if (a.lse != nullptr && q == 0) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int h = lane + 32 * e;
          const float l = red[h] + red[64 + h];
          a.lse[t * a.Hq + h0 + h] = l > 0.f ? (m_run[h] + log2f(l)) * 0.69314718055994531f : -INFINITY;
        }
      }
      for (int half = 0; half < 2; ++half) {
        float inv[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float l = red[half * 32 + i] + red[64 + half * 32 + i];
          inv[i] = l > 0.f ? 1.f / l : 0.f;
        }
        for (int blk = 0; blk < ndvb; ++blk) {
          float v[32];
          tmem_ld32(tbase + kOCol + blk * kMH + half * 32 + lane_addr, v);
          tmem_ld_wait_regs(v);
#pragma unroll
          for (int i = 0; i < 32; ++i)
            orow[(int64_t)(half * 32 + i) * a.Dv + blk * 128 + lanerow] = __float2bfloat16_rn(v[i] * inv[i]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kSW) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

}  // namespace

bool mla_supported(const AttnArgs& a) {
  return a.Hkv == 1 && a.v_alias && a.Hq % kMH == 0 && a.Dqk >= a.Dv + 64 && a.Dqk >= 128 && a.W <= 2048 &&
         mla_layout(a.Dqk, a.W).total <= 227u * 1024u;
}

size_t mla_smem_bytes(const AttnArgs& a) { return mla_layout(a.Dqk, a.W).total; }

cudaError_t configure_mla_kernel(size_t smem) {
  return cudaFuncSetAttribute(mla_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

cudaError_t launch_mla(const AttnArgs& a, int num_sms, cudaStream_t stream) {
  const long long items = (long long)a.T * (a.Hq / kMH);
  const int grid = (int)(items < num_sms ? items : num_sms);
  mla_fwd_kernel<<<grid, kMlaThreads, mla_layout(a.Dqk, a.W).total, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace irs
