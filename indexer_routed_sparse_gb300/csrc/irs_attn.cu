// Gathered sparse GQA attention forward on sm_103a (tcgen05 + TMEM; cp.async gathers, TMA row tiles).
//
// Semantics: QSA page (nemo_automodel.components.models.qwen3_8_flash_next.qsa,
// `gathered_qsa_gqa_attention`): query t, head h attends the keys/values of its KV
// head g = h / G at the global IDs of route row t; -1 slots are padding; softmax with
// a positive scale. Latent attention page (`cudnn_sparse_attention`): one latent KV
// head, keys are the full latent rows and values their first Dv dims.
//
// Design. A persistent CTA walks query rows t (grid-stride); for each row it walks its
// KV heads and head blocks (<= 16 query heads of one KV head, a "sub-item"). Warp roles:
//   producer warps (8, or 4 for the widest head/dv tiles): compact the valid route IDs of
//               the row into shared memory, then per sub-item copy the query tile and
//               gather the routed K/V rows with 16-byte cp.async into a ring of 128-key
//               stages (SW128 layout); completion reaches the stage's mbarrier by
//               cp.async-arrive. (Random 256-byte rows reach about 3x the L2 bandwidth
//               this way than with TMA gather4.) When the key/value rows exceed half the
//               L2 (variant RUNS), 64-slot groups of a route that hold 64 consecutive
//               tokens (a sliding window, whole 64-token blocks) load instead as one TMA
//               row tile per 64-dim atom, announced on the same barrier as transaction
//               bytes: far more bytes in flight for DRAM latency than the copies.
//   S warp      TMEM owner; issues S^T = K.Q^T (M=128 keys, N=16 heads, K=Dqk) as each
//               stage lands.
//   O warp      issues O^T = V^T.P^T (M=128 dv per block, N=16, K=128 keys; V read
//               MN-major from the gathered [key][dv] tile) as soon as a chunk's P is
//               written; its completion releases the stage. The thread that issues
//               tcgen05.mma runs in step with the tensor pipe (its waits, fences and
//               commits leave the pipe idle), so two issuers keep it fed. Each product is
//               a fully unrolled run of tcgen05.mma with descriptors formed as base plus a
//               constant (a run-time trip count doubles the cost per instruction).
//   4 softmax warps, one key (for S) / one dv (for O) per thread: an online softmax in
//               base 2 with head maxima exchanged through shared memory, P written as the
//               bf16 B operand, then the previous chunk's output rescaled and accumulated
//               in registers; at the end normalised and stored.
// S, P and O are double-buffered, so S of chunk n+1 and O of chunk n run on the tensor
// cores while the softmax warps work on chunk n, and the producer runs ahead across
// sub-items and rows. All cross-warp waits are bounded mbarrier waits.
#include "irs_internal.h"
#include "irs_ptx.cuh"

namespace irs {

// Warps: PW producer warps, the S issuer, the O issuer, then 4 softmax warps (32*(PW+6) threads).
__host__ __device__ constexpr int attn_threads(int pw) { return 32 * (pw + 6); }
constexpr int kChunk = 128;   // keys per chunk (UMMA M of the score product)
constexpr int kNH = 16;       // head columns per sub-item (UMMA N)
constexpr int kMaxDvBlocks = 4;

struct AttnLayout {
  uint32_t k_bytes, v_bytes, stage_bytes, idx_words;
  uint32_t q_off, p_off, idx_off, nv_off, run_off, red_off, fin_off, bar_off, total;
};

__host__ __device__ inline AttnLayout attn_layout(int Dqk, int Dv, int W, int stages, int v_alias) {
  AttnLayout L{};
  L.k_bytes = (uint32_t)kChunk * Dqk * 2;
  L.v_bytes = v_alias ? 0u : (uint32_t)kChunk * Dv * 2;
  L.stage_bytes = L.k_bytes + L.v_bytes;
  L.idx_words = (uint32_t)((W + kChunk - 1) / kChunk) * kChunk;
  uint32_t off = L.stage_bytes * stages;
  L.q_off = off;
  off += 2u * kNH * Dqk * 2;
  off = (off + 1023u) & ~1023u;
  L.p_off = off;
  off += 2u * kNH * kChunk * 2;
  L.idx_off = off;
  off += L.idx_words * 4;   // one buffer: only the producer reads the IDs
  L.nv_off = off;
  off += 16 + 32;           // sNv[2] and the producer's per-warp counts
  L.red_off = off;
  off += 2 * 4 * kNH * 4;
  L.fin_off = off;
  off += 2 * 4 * kNH * 4;
  L.bar_off = off;
  off += 40 * 8 + 16;
  L.run_off = off;
  off += L.idx_words / 64 * 4;   // per 64-slot group: 1 = 64 consecutive token IDs
  L.total = off + 1024;   // alignment slack
  return L;
}

// Reduce NH per-lane values over the warp with op in a transposed butterfly: at each of the
// first log2(NH) steps a lane keeps half of its values and swaps the other half with its
// partner, so NH values take NH-1 + (5 - log2 NH) shuffles instead of 5*NH. On return
// lane L holds the reduction of value head_of(L); lanes with the low (5 - log2 NH) bits
// clear own the result.
template <int NH>
__device__ __forceinline__ constexpr int log2_nh() { return NH == 4 ? 2 : (NH == 8 ? 3 : 4); }
template <int NH>
__device__ __forceinline__ int transposed_head(int lane) {
  int h = 0;
#pragma unroll
  for (int lvl = 0; lvl < log2_nh<NH>(); ++lvl)
    if (lane & (16 >> lvl)) h += NH >> (lvl + 1);
  return h;
}
template <int NH, bool MAX>
__device__ __forceinline__ float warp_reduce_transposed(const float (&x)[NH], int lane) {
  float v[NH];
#pragma unroll
  for (int h = 0; h < NH; ++h) v[h] = x[h];
#pragma unroll
  for (int lvl = 0; lvl < log2_nh<NH>(); ++lvl) {
    const int half = NH >> (lvl + 1), o = 16 >> lvl;
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = up ? v[i] : v[i + half];
      const float keep = up ? v[i + half] : v[i];
      const float got = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  float r = v[0];
#pragma unroll
  for (int o = 16 >> log2_nh<NH>(); o > 0; o >>= 1) {
    const float got = __shfl_xor_sync(0xffffffffu, r, o);
    r = MAX ? fmaxf(r, got) : r + got;
  }
  return r;
}

template <int NH>
__device__ __forceinline__ void tmem_ld_nh(uint32_t taddr, float (&v)[NH]) {
  if constexpr (NH == 4) tmem_ld4(taddr, v);
  else if constexpr (NH == 8) tmem_ld8(taddr, v);
  else tmem_ld16(taddr, v);
}

// Gather `rows` routed rows of kc 16-byte pieces each into a SW128 operand tile with
// 16-byte cp.async, spread over the PT producer threads. When a second tile (V) has the
// same row width, both are gathered in the same pass so each row index is read once.
// ids[r] are valid row indices.
template <int PT>
__device__ __forceinline__ void gather_rows(uint32_t dst, const __nv_bfloat16* src, int64_t row_stride,
                                            uint32_t dst2, const __nv_bfloat16* src2, int64_t row_stride2,
                                            const int32_t* ids, int rows, int kc, int ptid) {
  const int dr = PT / kc;   // rows per pass
  if (dr >= 2) {
    // each thread keeps one 16-byte column j and walks rows r0, r0+dr, ...; the last
    // PT - dr*kc threads stay idle
    if (ptid >= dr * kc) return;
    const int j = ptid % kc;
    int r = ptid / kc;
    const __nv_bfloat16* sj = src + j * 8;
    const __nv_bfloat16* sj2 = src2 + j * 8;
    if ((dr & 7) == 0) {
      // rows step by a multiple of 8: the swizzled chunk position is fixed
      const uint32_t off = sw128_offset(r, j * 8, kChunk);
      uint32_t d = dst + off, d2 = dst2 + off;
      if (src2 != nullptr) {
#pragma unroll 4
        for (; r < rows; r += dr, d += dr * 128, d2 += dr * 128) {
          const int64_t id = ids[r];
          cp_async_16(d, sj + id * row_stride, 16u);
          cp_async_16(d2, sj2 + id * row_stride2, 16u);
        }
      } else {
#pragma unroll 4
        for (; r < rows; r += dr, d += dr * 128) cp_async_16(d, sj + (int64_t)ids[r] * row_stride, 16u);
      }
    } else {
      const uint32_t atom = (uint32_t)(j >> 3) * (kChunk * 128);
      const uint32_t jc = (uint32_t)(j & 7);
#pragma unroll 4
      for (; r < rows; r += dr) {
        const int64_t id = ids[r];
        const uint32_t off = atom + (uint32_t)r * 128 + ((jc ^ ((uint32_t)r & 7)) << 4);
        cp_async_16(dst + off, sj + id * row_stride, 16u);
        if (src2 != nullptr) cp_async_16(dst2 + off, sj2 + id * row_stride2, 16u);
      }
    }
    return;
  }
  int r = ptid / kc, j = ptid - (ptid / kc) * kc;
  const int dj = PT - dr * kc;
  while (r < rows) {
    const int64_t id = ids[r];
    const uint32_t off = sw128_offset(r, j * 8, kChunk);
    cp_async_16(dst + off, src + id * row_stride + j * 8, 16u);
    if (src2 != nullptr) cp_async_16(dst2 + off, src2 + id * row_stride2 + j * 8, 16u);
    r += dr;
    j += dj;
    if (j >= kc) { j -= kc; ++r; }
  }
}

// S^T (+)= K.Q^T over KA SW128 atoms of Dqk (4 k-steps of 16 per atom). Descriptors are
// one base descriptor plus a compile-time start-address step (the 14-bit start field cannot
// carry: shared addresses stay below 256 KB).
template <int KA>
__device__ __forceinline__ void issue_scores(uint32_t d, uint32_t kb, uint32_t qb, uint32_t idesc) {
  const uint64_t a0 = sdesc_sw128(kb, 16, 1024), b0 = sdesc_sw128(qb, 16, 1024);
#pragma unroll
  for (int ks = 0; ks < 4 * KA; ++ks)
    umma_bf16(d, a0 + (uint64_t)(((ks >> 2) * (kChunk * 128) + (ks & 3) * 32) >> 4),
              b0 + (uint64_t)(((ks >> 2) * (kNH * 128) + (ks & 3) * 32) >> 4), idesc, ks > 0);
}
__device__ __forceinline__ void issue_scores_any(int katoms, uint32_t d, uint32_t kb, uint32_t qb, uint32_t idesc) {
  switch (katoms) {
    case 1: issue_scores<1>(d, kb, qb, idesc); break;
    case 2: issue_scores<2>(d, kb, qb, idesc); break;
    case 3: issue_scores<3>(d, kb, qb, idesc); break;
    case 4: issue_scores<4>(d, kb, qb, idesc); break;
    case 5: issue_scores<5>(d, kb, qb, idesc); break;
    case 6: issue_scores<6>(d, kb, qb, idesc); break;
    case 7: issue_scores<7>(d, kb, qb, idesc); break;
    case 8: issue_scores<8>(d, kb, qb, idesc); break;
    default: issue_scores<9>(d, kb, qb, idesc); break;
  }
}
// O^T = V^T.P^T for NB blocks of 128 dv (V MN-major: two 64-dv atoms of 128 key rows
// per block; P K-major: 16 head rows of 128 keys).
template <int NB>
__device__ __forceinline__ void issue_output(uint32_t d, uint32_t vb, uint32_t pb, uint32_t idesc) {
  const uint64_t a0 = sdesc_sw128(vb, kChunk * 128, 1024), b0 = sdesc_sw128(pb, 16, 1024);
#pragma unroll
  for (int blk = 0; blk < NB; ++blk) {
#pragma unroll
    for (int ks = 0; ks < kChunk / 16; ++ks)
      umma_bf16(d + blk * kNH, a0 + (uint64_t)(((2 * blk) * (kChunk * 128) + ks * 2048) >> 4),
                b0 + (uint64_t)(((ks >> 2) * (kNH * 128) + (ks & 3) * 32) >> 4), idesc, ks > 0);
  }
}
__device__ __forceinline__ void issue_output_any(int ndvb, uint32_t d, uint32_t vb, uint32_t pb, uint32_t idesc) {
  switch (ndvb) {
    case 1: issue_output<1>(d, vb, pb, idesc); break;
    case 2: issue_output<2>(d, vb, pb, idesc); break;
    case 3: issue_output<3>(d, vb, pb, idesc); break;
    default: issue_output<4>(d, vb, pb, idesc); break;
  }
}

struct AttnBars {
  uint64_t* kv_full;
  uint64_t* kv_empty;
  uint64_t* q_full;    // [2]
  uint64_t* q_empty;   // [2]
  uint64_t* idx_full;  // [2]
  uint64_t* idx_empty; // [2]
  uint64_t* s_full;    // [2]
  uint64_t* s_empty;   // [2]
  uint64_t* p_full;    // [2] (a P buffer is free again once O of its chunk is done: o_full)
  uint64_t* o_full;    // [2]
  uint64_t* o_empty;   // [2]
  uint64_t* red;       // [2] chunk-max exchange among the softmax warps
  uint64_t* fin;       // [2] row-sum exchange
};

template <int NH, int DVB, int PW, bool RUNS>
__global__ void __launch_bounds__(attn_threads(PW), 1) attn_fwd_kernel(const __grid_constant__ AttnMaps maps, AttnArgs a) {
  constexpr int kThreads = attn_threads(PW);
  constexpr int kProducerThreads = 32 * PW;
  constexpr int kSWarp = PW;       // TMEM owner, issues the S products
  constexpr int kOWarp = PW + 1;   // issues the O products
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int ST = a.stages;
  const AttnLayout Ly = attn_layout(a.Dqk, a.Dv, a.W + a.window, ST, a.v_alias);
  uint8_t* sQ = smem + Ly.q_off;                                  // [2][16 rows x Dqk]
  uint8_t* sP = smem + Ly.p_off;                                  // [2][16 rows x 128 keys]
  int32_t* sIdx = reinterpret_cast<int32_t*>(smem + Ly.idx_off);  // [idx_words] (producer only)
  int32_t* sNv = reinterpret_cast<int32_t*>(smem + Ly.nv_off);    // [2]
  int32_t* sCnt = sNv + 4;                                        // [PW] producer warp counts
  int32_t* sRun = reinterpret_cast<int32_t*>(smem + Ly.run_off);  // [idx_words / 64]
  float* sRed = reinterpret_cast<float*>(smem + Ly.red_off);      // [2][4][16]
  float* sFin = reinterpret_cast<float*>(smem + Ly.fin_off);      // [2][4][16]
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + Ly.bar_off);
  AttnBars B;
  B.kv_full = bar;
  B.kv_empty = bar + ST;
  B.q_full = bar + 2 * ST;
  B.q_empty = B.q_full + 2;
  B.idx_full = B.q_empty + 2;
  B.idx_empty = B.idx_full + 2;
  B.s_full = B.idx_empty + 2;
  B.s_empty = B.s_full + 2;
  B.p_full = B.s_empty + 2;
  B.o_full = B.p_full + 2;
  B.o_empty = B.o_full + 2;
  B.red = B.o_empty + 2;
  B.fin = B.red + 2;
  uint64_t* drain = B.fin + 2;   // [2]: the S and O issuers' last products have completed
  uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int katoms = a.Dqk >> 6;
  const int ndvb = a.Dv >> 7;
  const int qc = a.Dqk >> 3;
  const int n_sub = a.ng * a.nhb;   // sub-items per row
  constexpr uint32_t IDESC_S = idesc_bf16(kChunk, kNH, false, false);
  constexpr uint32_t IDESC_O = idesc_bf16(128, kNH, true, false);

  // ---- set-up: zero the operand buffers (stale rows must stay finite), barriers, TMEM ----
  {
    uint4* z = reinterpret_cast<uint4*>(smem);
    const uint32_t nz = Ly.idx_off / 16;
    for (uint32_t i = tid; i < nz; i += kThreads) z[i] = make_uint4(0, 0, 0, 0);
    if (tid < 2) sNv[tid] = 0;
    fence_proxy_async_smem();
  }
  if (tid == 0) {
    // kv_full: one cp.async arrival per producer thread (TMA tiles add transaction bytes)
    for (int s = 0; s < ST; ++s) { mbar_init(&B.kv_full[s], kProducerThreads); mbar_init(&B.kv_empty[s], 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B.q_full[i], kProducerThreads);
      mbar_init(&B.q_empty[i], 1);
      mbar_init(&B.idx_full[i], 1);
      mbar_init(&B.idx_empty[i], 6);
      mbar_init(&B.s_full[i], 1);
      mbar_init(&B.s_empty[i], 4);
      mbar_init(&B.p_full[i], 4);
      mbar_init(&B.o_full[i], 1);
      mbar_init(&B.o_empty[i], 4);
      mbar_init(&B.red[i], 4);
      mbar_init(&B.fin[i], 4);
      mbar_init(&drain[i], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kSWarp) {
    tmem_alloc(tslot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  if (warp < PW) {
    // =========================== producer (warps 0..PW-1) ===========================
    // The producer threads agree (named_bar_and) once per row; inside a row each thread
    // waits for its stages on its own, so warps run ahead of one another. A thread whose
    // wait gave up stops issuing and carries that into the next agreement.
    const int ptid = tid;
    uint32_t n = 0, u = 0, qi = 0;
    int pst = 0;          // n % ST
    uint32_t pph = 0;     // (n / ST) & 1
    bool mine = true;
    for (long long t = blockIdx.x; t < a.T; t += gridDim.x, ++qi) {
      const int b = qi & 1;
      const bool ok = mine && (qi < 2 || mbar_wait(&B.idx_empty[b], ((qi >> 1) - 1) & 1, abort_flag, a.err));
      if (!named_bar_and(1, kProducerThreads, ok)) break;
      // ---- the window's tokens first (no route reads), then the valid IDs of route row t
      //      below the window (8 loads in flight per thread) ----
      const int32_t* rrow = a.route + t * a.route_stride;
      int run = 0;
      int lo_w = -1;   // route IDs at or above this are inside the window: skipped
      if (a.window > 0) {
        int lo_d = 0, hi_d = a.ndocs - 1;   // document of t: largest d with cu[d] <= t
        while (lo_d < hi_d) {
          const int mid = (lo_d + hi_d + 1) >> 1;
          if (__ldg(a.cu + mid) <= t) lo_d = mid; else hi_d = mid - 1;
        }
        lo_w = (int)t - a.window + 1;
        const int lo = max(max(__ldg(a.cu + lo_d), lo_w), 0);
        run = max(0, (int)t - lo + 1);
        for (int i = ptid; i < run; i += kProducerThreads) sIdx[i] = lo + i;
      }
      for (int base = 0; base < a.W; base += 8 * kProducerThreads) {
        int ids[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int i = base + k * kProducerThreads + ptid;
          ids[k] = i < a.W ? __ldg(rrow + i) : -1;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (base + k * kProducerThreads >= a.W) break;
          const int i = base + k * kProducerThreads + ptid;
          const int id = ids[k];
          const bool inrange = id >= 0 && id < a.Tk;
          if (i < a.W && id != -1 && !inrange && a.flag_routes) record_error(a.err, IRS_DEVERR_ROUTE_ID);
          const bool okid = inrange && (a.window == 0 || id < lo_w);
          const uint32_t bal = __ballot_sync(0xffffffffu, okid);
          if (lane == 0) sCnt[warp] = __popc(bal);
          named_bar_sync(1, kProducerThreads);
          int before = run;
          for (int w2 = 0; w2 < warp; ++w2) before += sCnt[w2];
          if (okid) sIdx[before + __popc(bal & ((1u << lane) - 1u))] = id;
          for (int w2 = 0; w2 < PW; ++w2) run += sCnt[w2];
          named_bar_sync(1, kProducerThreads);
        }
      }
      if (ptid == 0) sNv[b] = run;
      named_bar_sync(1, kProducerThreads);
      if (ptid == 0) mbar_arrive(&B.idx_full[b]);
      const int nv = run;
      if (nv == 0) continue;
      // 64-slot groups holding 64 consecutive token IDs (e.g. a sliding window, or whole
      // 64-token blocks) are loaded as one TMA tile per 64-dim atom instead of 16-byte copies
      // (bit g of runmask; the same for every KV head and head block of the row)
      uint64_t runmask = 0;
      if (RUNS) {
        const int ngrp = nv >> 6;
        for (int gi = ptid; gi < ngrp; gi += kProducerThreads) sRun[gi] = 1;
        named_bar_sync(1, kProducerThreads);
        for (int i = ptid; i < (ngrp << 6); i += kProducerThreads)
          if ((i & 63) != 0 && sIdx[i] != sIdx[i - 1] + 1) sRun[i >> 6] = 0;
        named_bar_sync(1, kProducerThreads);
        for (int gi = 0; gi < ngrp; ++gi) runmask |= (uint64_t)(sRun[gi] != 0) << gi;
      }
      const int nchunks = (nv + kChunk - 1) / kChunk;
      for (int sub = 0; sub < n_sub && mine; ++sub, ++u) {
        const int g = sub / a.nhb, hb = sub - g * a.nhb;
        const int h0 = (a.g0 + g) * a.G + hb * a.HB;
        const int nh = min(a.HB, a.G - hb * a.HB);
        const int qb = u & 1;
        if (u >= 2 && !mbar_wait(&B.q_empty[qb], ((u >> 1) - 1) & 1, abort_flag, a.err)) { mine = false; break; }
        const uint32_t q_dst = smem_u32(sQ + qb * (kNH * a.Dqk * 2));
        for (int i = ptid; i < nh * qc; i += kProducerThreads) {
          const int r = i / qc, j = i - r * qc;
          cp_async_16(q_dst + sw128_offset(r, j * 8, kNH), a.q + t * a.q_st + (long long)(h0 + r) * a.q_sh + j * 8, 16u);
        }
        cp_async_mbar_arrive_noinc(&B.q_full[qb]);
        const __nv_bfloat16* kbase = a.k + (long long)(a.g0 + g) * a.k_sh;
        const __nv_bfloat16* vbase = a.v + (long long)(a.g0 + g) * a.v_sh;
        for (int c = 0; c < nchunks; ++c, ++n) {
          // stage n % ST and the parity of use n / ST - 1, kept incrementally (no division)
          const int st = pst;
          const uint32_t par = pph ^ 1u;
          if (++pst == ST) { pst = 0; pph ^= 1u; }
          if ((int)n >= ST && !mbar_wait(&B.kv_empty[st], par, abort_flag, a.err)) { mine = false; break; }
          const int rows = min(kChunk, nv - c * kChunk);
          const int32_t* ids = sIdx + c * kChunk;
          uint8_t* stage = smem + (uint32_t)st * Ly.stage_bytes;
          // halves of the chunk that are runs of 64 consecutive rows: TMA tiles
          const bool run0 = RUNS && ((runmask >> (2 * c)) & 1u) != 0;
          const bool run1 = RUNS && rows == kChunk && ((runmask >> (2 * c + 1)) & 1u) != 0;
          if (!run0 && !run1) {
            if (a.v_alias) {
              gather_rows<kProducerThreads>(smem_u32(stage), kbase, a.k_st, 0, nullptr, 0, ids, rows, qc, ptid);
            } else if (a.Dv == a.Dqk) {
              gather_rows<kProducerThreads>(smem_u32(stage), kbase, a.k_st, smem_u32(stage + Ly.k_bytes), vbase,
                                            a.v_st, ids, rows, qc, ptid);
            } else {
              gather_rows<kProducerThreads>(smem_u32(stage), kbase, a.k_st, 0, nullptr, 0, ids, rows, qc, ptid);
              gather_rows<kProducerThreads>(smem_u32(stage + Ly.k_bytes), vbase, a.v_st, 0, nullptr, 0, ids, rows,
                                            a.Dv >> 3, ptid);
            }
          } else if constexpr (RUNS) {
            if (ptid == 0) {
              // the bytes are announced before the tiles are issued and before this thread's
              // own arrival, so the phase cannot complete without them
              const uint32_t half_bytes = 64u * 128u * (uint32_t)(katoms + (a.v_alias ? 0 : a.Dv >> 6));
              mbar_expect_tx(&B.kv_full[st], ((run0 ? 1u : 0u) + (run1 ? 1u : 0u)) * half_bytes);
#pragma unroll 1
              for (int h = 0; h < 2; ++h) {
                if (!(h == 0 ? run0 : run1)) continue;
                const int y = ids[64 * h];
                for (int at = 0; at < katoms; ++at)
                  tma_load_2d(stage + at * (kChunk * 128) + h * 8192, &maps.k[g], at * 64, y, &B.kv_full[st]);
                if (!a.v_alias)
                  for (int at = 0; at < (a.Dv >> 6); ++at)
                    tma_load_2d(stage + Ly.k_bytes + at * (kChunk * 128) + h * 8192, &maps.v[g], at * 64, y,
                                &B.kv_full[st]);
              }
            }
            // the half that is not a run, by 16-byte copies
            const int r_lo = run0 ? 64 : 0, gr = (run1 ? 64 : rows) - r_lo;
            if (gr > 0) {
              const uint32_t roff = (uint32_t)r_lo * 128u;   // row offset inside every 128-row atom
              const int32_t* gids = ids + r_lo;
              if (a.v_alias) {
                gather_rows<kProducerThreads>(smem_u32(stage) + roff, kbase, a.k_st, 0, nullptr, 0, gids, gr, qc,
                                              ptid);
              } else if (a.Dv == a.Dqk) {
                gather_rows<kProducerThreads>(smem_u32(stage) + roff, kbase, a.k_st,
                                              smem_u32(stage + Ly.k_bytes) + roff, vbase, a.v_st, gids, gr, qc, ptid);
              } else {
                gather_rows<kProducerThreads>(smem_u32(stage) + roff, kbase, a.k_st, 0, nullptr, 0, gids, gr, qc,
                                              ptid);
                gather_rows<kProducerThreads>(smem_u32(stage + Ly.k_bytes) + roff, vbase, a.v_st, 0, nullptr, 0, gids,
                                              gr, a.Dv >> 3, ptid);
              }
            }
          }
          cp_async_mbar_arrive_noinc(&B.kv_full[st]);
        }
      }
    }
    cp_async_wait_pending(0);   // nothing of this CTA's gathers is in flight when it leaves
    if (RUNS && ptid == 0 && *abort_flag) {
      // a wait gave up: let the row tiles this thread issued for the last stages land (their
      // phases may also miss arrivals of threads that stopped, hence the short bound)
      for (uint32_t x = n > (uint32_t)ST ? n - ST : 0; x < n; ++x) {
        const unsigned long long t0 = globaltimer_ns();
        while (!mbar_try_wait(&B.kv_full[x % ST], (x / ST) & 1) && globaltimer_ns() - t0 < 50000000ull) {}
      }
    }
  } else if (warp == kSWarp) {
    // =========================== S issuer ===========================
    // The issuing thread runs in step with the tensor pipe, so S and O products come from
    // two warps: each one's waits, fences and commits overlap the other's MMAs, and O of a
    // chunk never queues behind S of a chunk whose stage has not landed.
    if (lane == 0) {
      uint32_t n = 0, u = 0, qi = 0;
      int sst = 0;          // n % ST
      uint32_t sph = 0;     // (n / ST) & 1
      bool alive = true;
      for (long long t = blockIdx.x; t < a.T && alive; t += gridDim.x, ++qi) {
        const int b = qi & 1;
        if (!mbar_wait(&B.idx_full[b], (qi >> 1) & 1, abort_flag, a.err)) { alive = false; break; }
        const int nv = sNv[b];
        mbar_arrive(&B.idx_empty[b]);
        if (nv == 0) continue;
        const int nchunks = (nv + kChunk - 1) / kChunk;
        for (int sub = 0; sub < n_sub && alive; ++sub, ++u) {
          const int qb = u & 1;
          if (!mbar_wait(&B.q_full[qb], (u >> 1) & 1, abort_flag, a.err)) { alive = false; break; }
          const uint32_t qbase = smem_u32(sQ + qb * (kNH * a.Dqk * 2));
          for (int c = 0; c < nchunks; ++c, ++n) {
            const int st = sst, sb = n & 1;
            const uint32_t par = sph;
            if (++sst == ST) { sst = 0; sph ^= 1u; }
            if (!mbar_wait(&B.kv_full[st], par, abort_flag, a.err)) { alive = false; break; }
            if (n >= 2 && !mbar_wait(&B.s_empty[sb], ((n >> 1) - 1) & 1, abort_flag, a.err)) { alive = false; break; }
            fence_proxy_async_smem();   // gathered rows (generic-proxy writes) -> UMMA reads
            tc_fence_after();
            issue_scores_any(katoms, tbase + sb * kNH, smem_u32(smem + (uint32_t)st * Ly.stage_bytes), qbase, IDESC_S);
            umma_commit(&B.s_full[sb]);
            if (c == nchunks - 1) umma_commit(&B.q_empty[qb]);
          }
        }
      }
      // every S product this thread issued completes before the CTA releases tensor memory
      umma_commit(&drain[0]);
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_try_wait(&drain[0], 0) && globaltimer_ns() - t0 < kWaitLimitNs) {}
    }
  } else if (warp == kOWarp) {
    // =========================== O issuer ===========================
    // O of chunk m goes once its P is written and the O buffer it reuses has been read;
    // its completion frees the P buffer and the K/V stage.
    if (lane == 0) {
      uint32_t m = 0, qi = 0;
      int ost = 0;          // m % ST
      bool alive = true;
      for (long long t = blockIdx.x; t < a.T && alive; t += gridDim.x, ++qi) {
        const int b = qi & 1;
        if (!mbar_wait(&B.idx_full[b], (qi >> 1) & 1, abort_flag, a.err)) { alive = false; break; }
        const int nv = sNv[b];
        mbar_arrive(&B.idx_empty[b]);
        if (nv == 0) continue;
        const int total = ((nv + kChunk - 1) / kChunk) * n_sub;
        for (int j = 0; j < total; ++j, ++m) {
          const int pb = m & 1;
          if (!mbar_wait(&B.p_full[pb], (m >> 1) & 1, abort_flag, a.err)) { alive = false; break; }
          if (m >= 2 && !mbar_wait(&B.o_empty[pb], ((m >> 1) - 1) & 1, abort_flag, a.err)) { alive = false; break; }
          tc_fence_after();
          const int ost_m = ost;
          if (++ost == ST) ost = 0;
          const uint8_t* stage = smem + (uint32_t)ost_m * Ly.stage_bytes;
          const uint32_t vb = smem_u32(a.v_alias ? stage : stage + Ly.k_bytes);
          issue_output_any(ndvb, tbase + 32 + pb * (kNH * kMaxDvBlocks), vb, smem_u32(sP + pb * (kNH * kChunk * 2)),
                           IDESC_O);
          umma_commit(&B.o_full[pb]);
          umma_commit(&B.kv_empty[ost_m]);
        }
      }
      umma_commit(&drain[1]);
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_try_wait(&drain[1], 0) && globaltimer_ns() - t0 < kWaitLimitNs) {}
    }
  } else {
    // =========================== softmax + correction (warps PW+1 .. PW+4) ===========================
    const int sw = warp - (PW + 2);
    const int lanerow = (warp & 3) * 32 + lane;      // TMEM lane: key of S, dv of O
    const uint32_t lane_addr = tmem_lane_base(warp);
    uint32_t n = 0, u = 0, qi = 0;
    for (long long t = blockIdx.x; t < a.T; t += gridDim.x, ++qi) {
      const int b = qi & 1;
      mbar_wait(&B.idx_full[b], (qi >> 1) & 1, abort_flag, a.err);
      const int nv = min(max(sNv[b], 0), a.W + a.window);
      __syncwarp();
      if (lane == 0) mbar_arrive(&B.idx_empty[b]);
      const int nchunks = (nv + kChunk - 1) / kChunk;
      if (nv == 0) {
        // reading: a row without any valid key gives zeros and lse = -inf
        for (int sub = 0; sub < n_sub; ++sub) {
          const int g = sub / a.nhb, hb = sub - g * a.nhb;
          const int h0 = (a.g0 + g) * a.G + hb * a.HB;
          const int nh = min(a.HB, a.G - hb * a.HB);
          __nv_bfloat16* orow = a.out + (t * a.Hq + h0) * (long long)a.Dv;
          for (int blk = 0; blk < ndvb; ++blk)
            for (int h = 0; h < nh; ++h) orow[(long long)h * a.Dv + blk * 128 + lanerow] = __float2bfloat16_rn(0.f);
          if (a.lse != nullptr && lanerow < nh) a.lse[t * a.Hq + h0 + lanerow] = -INFINITY;
        }
        continue;
      }
      for (int sub = 0; sub < n_sub; ++sub, ++u) {
        const int g = sub / a.nhb, hb = sub - g * a.nhb;
        const int h0 = (a.g0 + g) * a.G + hb * a.HB;
        const int nh = min(a.HB, a.G - hb * a.HB);
        __nv_bfloat16* orow = a.out + (t * a.Hq + h0) * (long long)a.Dv;
        float m[NH], l[NH], al[NH], alp[NH], acc[DVB][NH];
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          m[h] = -INFINITY;
          l[h] = 0.f;
          al[h] = 1.f;
          alp[h] = 1.f;
#pragma unroll
          for (int blk = 0; blk < DVB; ++blk) acc[blk][h] = 0.f;
        }
        // acc <- acc * alp + O of chunk mm (alp: rescale factor of chunk mm)
        auto correct = [&](uint32_t mm) {
          const int ob = mm & 1;
          mbar_wait(&B.o_full[ob], (mm >> 1) & 1, abort_flag, a.err);
          __syncwarp();   // converge after the polling wait: tcgen05.ld is warp-aligned
          tc_fence_after();
#pragma unroll
          for (int blk = 0; blk < DVB; ++blk)
            if (blk < ndvb) {
              float o[NH];
              tmem_ld_nh<NH>(tbase + 32 + ob * (kNH * kMaxDvBlocks) + blk * kNH + lane_addr, o);
              tmem_ld_wait_regs(o);
#pragma unroll
              for (int h = 0; h < NH; ++h) acc[blk][h] = fmaf(acc[blk][h], alp[h], o[h]);
            }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&B.o_empty[ob]);
        };
        for (int c = 0; c < nchunks; ++c, ++n) {
          const int sb = n & 1;
          mbar_wait(&B.s_full[sb], (n >> 1) & 1, abort_flag, a.err);
          __syncwarp();
          tc_fence_after();
          float s[NH];
          tmem_ld_nh<NH>(tbase + sb * kNH + lane_addr, s);
          tmem_ld_wait_regs(s);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&B.s_empty[sb]);
          const bool kvalid = c * kChunk + lanerow < nv;
          float* red = sRed + sb * (4 * kNH);
#pragma unroll
          for (int h = 0; h < NH; ++h) s[h] = (kvalid && h < nh) ? s[h] * a.scale_log2 : -INFINITY;
          {
            const float mx = warp_reduce_transposed<NH, true>(s, lane);
            if ((lane & ((32 >> log2_nh<NH>()) - 1)) == 0) red[sw * kNH + transposed_head<NH>(lane)] = mx;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&B.red[sb]);
          mbar_wait(&B.red[sb], (n >> 1) & 1, abort_flag, a.err);
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            const float cm = fmaxf(fmaxf(red[h], red[kNH + h]), fmaxf(red[2 * kNH + h], red[3 * kNH + h]));
            const float mn = fmaxf(m[h], cm);
            const float base = mn == -INFINITY ? 0.f : mn;
            al[h] = ex2_approx(m[h] - base);
            s[h] = ex2_approx(s[h] - base);   // p
            l[h] = fmaf(l[h], al[h], s[h]);
            m[h] = mn;
          }
          // P buffer sb was last read by O of chunk n-2, whose completion this warp has
          // already seen (o_full) when it folded that chunk in
          uint8_t* pdst = sP + sb * (kNH * kChunk * 2);
#pragma unroll
          for (int h = 0; h < NH; ++h)
            *reinterpret_cast<__nv_bfloat16*>(pdst + sw128_offset(h, lanerow, kNH)) = __float2bfloat16_rn(s[h]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&B.p_full[sb]);
          // P of this chunk is out; now fold in the previous chunk's output, which ran on
          // the tensor cores meanwhile, with the rescale factor that belongs to it
          if (c > 0) correct(n - 1);
#pragma unroll
          for (int h = 0; h < NH; ++h) alp[h] = al[h];
        }
        correct(n - 1);
        // ---- finalize: row sums over the 128 key lanes, normalise, store ----
        const int fb = u & 1;
        float* fin = sFin + fb * (4 * kNH);
        {
          const float sm = warp_reduce_transposed<NH, false>(l, lane);
          if ((lane & ((32 >> log2_nh<NH>()) - 1)) == 0) fin[sw * kNH + transposed_head<NH>(lane)] = sm;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.fin[fb]);
        mbar_wait(&B.fin[fb], (u >> 1) & 1, abort_flag, a.err);
        float inv[NH], tot[NH];
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          tot[h] = fin[h] + fin[kNH + h] + fin[2 * kNH + h] + fin[3 * kNH + h];
          inv[h] = tot[h] > 0.f ? 1.f / tot[h] : 0.f;
        }
#pragma unroll
        for (int blk = 0; blk < DVB; ++blk)
          if (blk < ndvb) {
#pragma unroll
            for (int h = 0; h < NH; ++h)
              if (h < nh) orow[(long long)h * a.Dv + blk * 128 + lanerow] = __float2bfloat16_rn(acc[blk][h] * inv[h]);
          }
        if (a.lse != nullptr && lanerow < nh) {
#pragma unroll
          for (int h = 0; h < NH; ++h)
            if (h == lanerow)
              a.lse[t * a.Hq + h0 + h] = tot[h] > 0.f ? (m[h] + log2f(tot[h])) * 0.69314718055994531f : -INFINITY;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kSWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, 256);
  }
}

AttnPlan plan_attn(const AttnArgs& a, int num_sms) {
  AttnPlan p{};
  p.items = a.T;
  int st = 4;
  while (st > 1 && attn_layout(a.Dqk, a.Dv, a.W + a.window, st, a.v_alias).total > 227 * 1024) --st;
  p.stages = st;
  p.smem = attn_layout(a.Dqk, a.Dv, a.W + a.window, st, a.v_alias).total;
  p.grid = (int)(a.T < num_sms ? a.T : num_sms);
  if (p.grid < 1) p.grid = 1;
  p.nh_class = a.HB <= 4 ? 4 : (a.HB <= 8 ? 8 : 16);
  return p;
}

// Producer warps by softmax register need: a warp scheduler holds 16K registers, so with
// 14 warps (4 on some schedulers) a thread gets at most 128, with 12 warps 168.
template <int NH, int DVB>
constexpr int producer_warps() { return NH * DVB <= 8 ? 8 : (NH * DVB <= 32 ? 6 : 4); }

template <int NH, int DVB>
static cudaError_t attn_attr(size_t smem) {
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<NH, DVB, producer_warps<NH, DVB>(), false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(attn_fwd_kernel<NH, DVB, producer_warps<NH, DVB>(), true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

cudaError_t configure_attn_kernel(size_t smem) {
  cudaError_t e = cudaSuccess;
  for (cudaError_t x : {attn_attr<4, 1>(smem), attn_attr<4, 2>(smem), attn_attr<4, 4>(smem), attn_attr<8, 1>(smem),
                        attn_attr<8, 2>(smem), attn_attr<8, 4>(smem), attn_attr<16, 1>(smem), attn_attr<16, 2>(smem),
                        attn_attr<16, 4>(smem)})
    if (x != cudaSuccess) e = x;
  return e;
}

// The row-tile path is a separate instantiation: its code in the producer loop costs the
// all-copy path a few percent even when no chunk takes it.
template <int NH, int DVB>
static void launch_variant(const AttnMaps& maps, const AttnArgs& b, const AttnPlan& p, cudaStream_t stream) {
  constexpr int PW = producer_warps<NH, DVB>();
  if (b.tile_runs)
    attn_fwd_kernel<NH, DVB, PW, true><<<p.grid, attn_threads(PW), p.smem, stream>>>(maps, b);
  else
    attn_fwd_kernel<NH, DVB, PW, false><<<p.grid, attn_threads(PW), p.smem, stream>>>(maps, b);
}

cudaError_t launch_attn(const AttnMaps& maps, const AttnArgs& a, const AttnPlan& p, cudaStream_t stream) {
  AttnArgs b = a;
  b.stages = p.stages;
  const int dvb = (a.Dv + 127) / 128 <= 1 ? 1 : ((a.Dv + 127) / 128 <= 2 ? 2 : 4);
  switch (p.nh_class * 10 + dvb) {
    case 41: launch_variant<4, 1>(maps, b, p, stream); break;
    case 42: launch_variant<4, 2>(maps, b, p, stream); break;
    case 44: launch_variant<4, 4>(maps, b, p, stream); break;
    case 81: launch_variant<8, 1>(maps, b, p, stream); break;
    case 82: launch_variant<8, 2>(maps, b, p, stream); break;
    case 84: launch_variant<8, 4>(maps, b, p, stream); break;
    case 161: launch_variant<16, 1>(maps, b, p, stream); break;
    case 162: launch_variant<16, 2>(maps, b, p, stream); break;
    default: launch_variant<16, 4>(maps, b, p, stream); break;
  }
  return cudaGetLastError();
}

}  // namespace irs
