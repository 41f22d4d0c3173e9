// Sparse attention backward over routed keys on the tensor cores (tcgen05 + TMEM), for
// separate K and V of GQA shapes.
//
// Semantics: latent attention page (`_CudnnSparseAttention.backward`): the BF16 output
// gradient is mapped to gradients of the query and of the gathered K/V rows; the GQA routes
// of the QSA page get the same gradients. For query t, query head h, KV head g = h / G,
// routed keys R_t and the forward's outputs out and lse (natural log):
//   p_r  = exp(scale * q.k_r - lse),   D = dO . out,   ds_r = scale * p_r (dO.v_r - D)
//   dq   = sum_r ds_r k_r,   dk_r += ds_r q,   dv_r += p_r dO
//
// Design. A work item is (query t, KV head g, block of <= 16 query heads): one CTA. Its
// routed keys go in chunks of 128 through a two-stage ring (16-byte cp.async gathers into
// SW128 tiles), and every contraction runs on the tensor cores with FP32 accumulators in TMEM:
//   S^T  = K.Q^T, dP^T = V.dO^T        M = 128 keys, N = 16 heads (K = Dqk, Dv)
//   dV   = P^T.dO, dK = dS^T.Q         M = 128 keys, N = Dv, Dqk, K = 16 heads (dO, Q MN-major)
//   dQ^T += K^T.dS^T                   M = 128 dims per block, N = 16 heads, K = 128 keys
//                                      (K MN-major from the stage), accumulated over chunks
// P and dS are formed per key row from the known lse (no online softmax) and rounded to bf16
// as operands, as the forward rounds P. Each chunk's dK and dV rows are added to the FP32
// global accumulators with float4 reductions by their own warps while the next chunk's
// scores are computed; dQ leaves TMEM once, at the end.
// S^T and dP^T are double-buffered in TMEM; the scores of chunk c+1 are issued before the
// gradient products of chunk c when its rows have landed, so P and dS of the next chunk
// are formed while the current chunk's dK/dV rows drain.
// Warps: 0-5 gather, 6 issues the products (TMEM owner), 7..10 form P and dS (one key per
// thread), 11..14 drain dK/dV (one key per thread) and then dQ (one dim per thread); each
// group of four covers the four TMEM lane quarters. Waits are bounded; after one gives up,
// each role stops and the CTA drains its tensor-core work and copies before it releases
// TMEM.
#include "irs_internal.h"
#include "irs_ptx.cuh"

namespace irs {
namespace {

constexpr int kTcThreads = 480;      // 15 warps (<= 136 registers per thread)
constexpr int kGatherThreads = 192;  // warps 0..5
constexpr int kMmaWarp = 6;
constexpr int kDrainWarp0 = 11;      // warps 7..10 form P and dS; 11..14 drain dK / dV rows, then dQ
constexpr int kTcKeys = 128;   // routed keys per chunk
constexpr int kTcHeads = 16;   // head rows of the Q and dO tiles
constexpr int kTrRows = 16;    // rows a drain warp transposes at a time
constexpr int kTrPitch = 36;   // floats per transposed row: 32 + 4, so 16 rows' float4 writes spread over the banks

struct TcLayout {
  uint32_t stage_bytes, q_off, do_off, pt_off, dst_off, dsh_off, pbuf_bytes, ids_off, tr_off, misc_off, bar_off, total;
  int npb;   // P / dS tile sets: 2 where shared memory allows
};

__host__ __device__ inline TcLayout tc_layout_n(int Dqk, int Dv, int W, int npb) {
  TcLayout L{};
  L.npb = npb;
  L.stage_bytes = (uint32_t)kTcKeys * (uint32_t)(Dqk + Dv) * 2u;   // K atoms, then V atoms
  uint32_t off = 2u * L.stage_bytes;
  L.q_off = off;
  off += (uint32_t)Dqk * kTcHeads * 2u;   // Q: 16 rows per 64-dim atom
  L.do_off = off;
  off += (uint32_t)Dv * kTcHeads * 2u;    // dO
  // per P / dS set: P^T and dS^T (128 key rows, columns 0..15 used), dS (16 head rows of
  // 128 keys, two 64-key atoms)
  L.pbuf_bytes = 2u * kTcKeys * 128u + 2u * kTcHeads * 128u;
  L.pt_off = off;
  L.dst_off = off + kTcKeys * 128u;
  L.dsh_off = off + 2u * kTcKeys * 128u;
  off += L.pbuf_bytes * (uint32_t)npb;
  L.ids_off = off;
  off += ((uint32_t)W * 4u + 15u) & ~15u;
  L.tr_off = off;
  off += 4u * kTrRows * kTrPitch * 4u;    // per drain warp: 16 rows x 32 columns (padded)
  L.misc_off = off;
  off += 48u * 4u;                        // D, lse (base 2), warp counts
  L.bar_off = off;
  off += 20u * 8u + 16u;                  // 19 barriers, TMEM slot, abort word
  L.total = off + 1024u;                  // alignment slack
  return L;
}
// Two P / dS sets when they fit: P and dS of chunk c+1 are then written while the products
// of chunk c still read the other set.
__host__ __device__ inline TcLayout tc_layout(int Dqk, int Dv, int W) {
  const TcLayout two = tc_layout_n(Dqk, Dv, W, 2);
  return two.total <= 227u * 1024u ? two : tc_layout_n(Dqk, Dv, W, 1);
}

// D[128 keys x 16 heads] = X.Y^T over KA 64-dim atoms: X a staged K or V tile (128-row
// atoms), Y the 16-row Q or dO tile, both K-major.
template <int KA>
__device__ __forceinline__ void rows_by_heads(uint32_t d, uint32_t xb, uint32_t yb, uint32_t idesc) {
  const uint64_t a0 = sdesc_sw128(xb, 16, 1024), b0 = sdesc_sw128(yb, 16, 1024);
#pragma unroll
  for (int ks = 0; ks < 4 * KA; ++ks)
    umma_bf16(d, a0 + (uint64_t)(((ks >> 2) * (kTcKeys * 128) + (ks & 3) * 32) >> 4),
              b0 + (uint64_t)(((ks >> 2) * (kTcHeads * 128) + (ks & 3) * 32) >> 4), idesc, ks > 0);
}
__device__ __forceinline__ void rows_by_heads_any(int atoms, uint32_t d, uint32_t xb, uint32_t yb, uint32_t idesc) {
  switch (atoms) {
    case 1: rows_by_heads<1>(d, xb, yb, idesc); break;
    case 2: rows_by_heads<2>(d, xb, yb, idesc); break;
    case 3: rows_by_heads<3>(d, xb, yb, idesc); break;
    default: rows_by_heads<4>(d, xb, yb, idesc); break;
  }
}
// D[128 keys x N dims] = A.B: A a 128-row tile of 16 head columns (P^T or dS^T, one K
// step), B the 16-row dO or Q tile read MN-major (64-dim atoms of 16 rows, 2 KB apart).
__device__ __forceinline__ void rows_by_dims(uint32_t d, uint32_t ab, uint32_t bb, uint32_t idesc) {
  umma_bf16(d, sdesc_sw128(ab, 16, 1024), sdesc_sw128(bb, kTcHeads * 128, 1024), idesc, 0u);
}
// dQ^T[128 dims x 16 heads] (+)= K^T.dS^T for one 128-dim block: K read MN-major from the
// stage (64-dim atoms of 128 key rows, 16 KB apart), dS the 16-row K-major tile of 128 keys.
__device__ __forceinline__ void dq_block(uint32_t d, uint32_t kb, uint32_t dsb, uint32_t idesc, bool accumulate) {
  const uint64_t a0 = sdesc_sw128(kb, kTcKeys * 128, 1024), b0 = sdesc_sw128(dsb, 16, 1024);
#pragma unroll
  for (int ks = 0; ks < kTcKeys / 16; ++ks)
    umma_bf16(d, a0 + (uint64_t)((ks * 2048) >> 4),
              b0 + (uint64_t)(((ks >> 2) * (kTcHeads * 128) + (ks & 3) * 32) >> 4), idesc,
              (accumulate || ks > 0) ? 1u : 0u);
}

// Adds 32 columns [col0, col0+32) of this warp's 32 rows (lane l holds row l's values in
// x) to the global rows dst + (cids[l] * hkv + g) * ld (rows l < nrows only), through the
// warp's shared tile: 16 rows at a time are written row-wise, then read so that each float4
// reduction instruction covers 4 rows x 128 contiguous bytes (8 lanes per row) instead of
// 32 rows x 16 bytes.
__device__ __forceinline__ void drain_cols(float* tr, const float (&x)[32], int lane, float* dst, int64_t ld, int col0,
                                           const int32_t* cids, int nrows, int hkv, int g) {
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    __syncwarp();
    if ((lane >> 4) == half) {
      float* trow = tr + (lane & 15) * kTrPitch;
#pragma unroll
      for (int i = 0; i < 32; i += 4) *reinterpret_cast<float4*>(trow + i) = make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]);
    }
    __syncwarp();
#pragma unroll
    for (int s = 0; s < kTrRows / 4; ++s) {
      const int rr = 4 * s + (lane >> 3), cc = 4 * (lane & 7);
      const int row = 16 * half + rr;
      if (row < nrows) {
        const float4 v = *reinterpret_cast<const float4*>(tr + rr * kTrPitch + cc);
        const int64_t grow = (int64_t)cids[row] * hkv + g;
        atomicAdd(reinterpret_cast<float4*>(dst + grow * ld + col0 + cc), v);
      }
    }
  }
}

__global__ void __launch_bounds__(kTcThreads, 1) attn_bwd_tc_kernel(BwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int DQ = a.Dqk, DV = a.Dv;
  const TcLayout L = tc_layout(DQ, DV, a.W);
  int32_t* ids = reinterpret_cast<int32_t*>(smem + L.ids_off);
  float* Dh = reinterpret_cast<float*>(smem + L.misc_off);
  float* l2h = Dh + 16;
  int* wcnt = reinterpret_cast<int*>(l2h + 16);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  uint64_t* kv_full = bar;        // [2]
  uint64_t* kv_empty = bar + 2;   // [2]
  uint64_t* qd_full = bar + 4;
  uint64_t* sd_full = bar + 5;    // [2]
  uint64_t* sd_empty = bar + 7;   // [2]
  uint64_t* dv_full = bar + 9;     // dV rows of the chunk are in TMEM
  uint64_t* dv_empty = bar + 10;   // ... and have been read
  uint64_t* dk_full = bar + 11;
  uint64_t* dk_empty = bar + 12;
  uint64_t* dq_full = bar + 13;
  uint64_t* drain = bar + 14;
  uint64_t* p_full = bar + 15;     // [2]: P / dS set written
  uint64_t* p_empty = bar + 17;    // [2]: ... and read by the products
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 19);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int per_t = a.Hkv * a.nhb;
  const int t = (int)(blockIdx.x / (unsigned)per_t);
  const int rem = (int)(blockIdx.x % (unsigned)per_t);
  const int g = rem / a.nhb, hb = rem % a.nhb;
  const int h0 = g * a.G + hb * a.HB;
  const int nh = min(a.HB, a.G - hb * a.HB);
  const int qa = DQ >> 6, va = DV >> 6, nqb = (DQ + 127) >> 7;
  // TMEM columns: S^T / dP^T of buffer b at 32b / 32b+16, dQ^T blocks at 64 + 16 blk,
  // dV rows at 96, dK rows at 96 + Dv
  const uint32_t tcols = 96u + (uint32_t)(DV + DQ) <= 256u ? 256u : 512u;
  const uint32_t TC_DQ = 64u, TC_DV = 96u, TC_DK = 96u + (uint32_t)DV;

  // ---- set-up: zero the operand tiles (head rows past nh, unused columns and rows past a
  //      partial chunk are read by the products and must stay finite), barriers ----
  {
    uint4* z = reinterpret_cast<uint4*>(smem);
    for (uint32_t i = tid; i < L.ids_off / 16u; i += kTcThreads) z[i] = make_uint4(0, 0, 0, 0);
  }
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kv_full[i], kGatherThreads);
      mbar_init(&kv_empty[i], 1);
      mbar_init(&sd_full[i], 1);
      mbar_init(&sd_empty[i], 4);
    }
    mbar_init(qd_full, kGatherThreads);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&p_full[i], 4);
      mbar_init(&p_empty[i], 1);
    }
    mbar_init(dv_full, 1);
    mbar_init(dv_empty, 4);
    mbar_init(dk_full, 1);
    mbar_init(dk_empty, 4);
    mbar_init(dq_full, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // D = dO . out (from the bf16 forward output) and the base-2 lse, per head
  const __nv_bfloat16* dO_t = a.dout + ((int64_t)t * a.Hq + h0) * DV;
  const __nv_bfloat16* o_t = a.out + ((int64_t)t * a.Hq + h0) * DV;
  for (int j = warp; j < nh; j += kTcThreads / 32) {
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
  // the valid IDs of the route row, in slot order (all of this thread's loads issued first)
  constexpr int kIdsPerThread = (4096 + kTcThreads - 1) / kTcThreads;
  int idv[kIdsPerThread];
#pragma unroll
  for (int k = 0; k < kIdsPerThread; ++k) {
    const int i = k * kTcThreads + tid;
    idv[k] = i < a.W ? __ldg(a.route + (int64_t)t * a.route_stride + i) : -1;
  }
  int n = 0;
#pragma unroll
  for (int k = 0; k < kIdsPerThread; ++k) {
    if (k * kTcThreads >= a.W) break;   // uniform
    const int i = k * kTcThreads + tid;
    const int id = idv[k];
    bool ok = false;
    if (i < a.W) {
      ok = id >= 0 && id < a.Tk;
      if (!ok && id != -1 && g == 0 && hb == 0) record_error(a.err, IRS_DEVERR_ROUTE_ID);
    }
    const unsigned bal = __ballot_sync(0xffffffffu, ok);
    if (lane == 0) wcnt[warp] = __popc(bal);
    __syncthreads();
    int off = n;
    for (int w2 = 0; w2 < warp; ++w2) off += wcnt[w2];
    if (ok) ids[off + __popc(bal & ((1u << lane) - 1u))] = id;
    for (int w2 = 0; w2 < kTcThreads / 32; ++w2) n += wcnt[w2];
    __syncthreads();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tslot, tcols);
    tmem_relinquish();
  }
  fence_proxy_async_smem();   // the zeroed tiles (generic writes) before tensor-core reads
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const int nchunks = (n + kTcKeys - 1) / kTcKeys;
  uint8_t* sQ = smem + L.q_off;
  uint8_t* sdO = smem + L.do_off;

  if (n == 0) {
    // no valid key: dq is zero
    float* dq_t = a.dq + ((int64_t)t * a.Hq + h0) * DQ;
    for (int i = tid; i < nh * DQ; i += kTcThreads) dq_t[i] = 0.f;
  } else if (warp < kGatherThreads / 32) {
    // =========================== gathers (warps 0-5) ===========================
    // each thread copies one fixed 16-byte column of every rpi-th row: no division per copy
    const int ptid = tid;
    const int qc = DQ >> 3, vc = DV >> 3;   // 16-byte pieces per row
    const int rpk = kGatherThreads / qc, rpv = kGatherThreads / vc;   // rows per pass
    const int rk = ptid / qc, jk = ptid - rk * qc, rv = ptid / vc, jv = ptid - rv * vc;
    for (int r = rk; r < nh && rk < rpk; r += rpk)
      cp_async_16(smem_u32(sQ) + sw128_offset(r, jk * 8, kTcHeads),
                  a.q + (int64_t)t * a.q_st + (int64_t)(h0 + r) * a.q_sh + jk * 8, 16u);
    for (int r = rv; r < nh && rv < rpv; r += rpv)
      cp_async_16(smem_u32(sdO) + sw128_offset(r, jv * 8, kTcHeads), dO_t + (int64_t)r * DV + jv * 8, 16u);
    cp_async_mbar_arrive_noinc(qd_full);
    const __nv_bfloat16* kbase = a.k + (int64_t)g * a.k_sh + jk * 8;
    const __nv_bfloat16* vbase = a.v + (int64_t)g * a.v_sh + jv * 8;
    for (int c = 0; c < nchunks; ++c) {
      const int st = c & 1;
      if (c >= 2 && !mbar_wait(&kv_empty[st], ((c >> 1) - 1) & 1, abort_flag, a.err)) break;
      const int rows = min(kTcKeys, n - c * kTcKeys);
      const int32_t* cids = ids + c * kTcKeys;
      const uint32_t kb = smem_u32(smem + (uint32_t)st * L.stage_bytes);
      const uint32_t vb = kb + (uint32_t)qa * (kTcKeys * 128u);
      if (rk < rpk)
        for (int r = rk; r < rows; r += rpk)
          cp_async_16(kb + sw128_offset(r, jk * 8, kTcKeys), kbase + (int64_t)cids[r] * a.k_st, 16u);
      if (rv < rpv)
        for (int r = rv; r < rows; r += rpv)
          cp_async_16(vb + sw128_offset(r, jv * 8, kTcKeys), vbase + (int64_t)cids[r] * a.v_st, 16u);
      cp_async_mbar_arrive_noinc(&kv_full[st]);
    }
    cp_async_wait_pending(0);   // nothing of this CTA's gathers is in flight when it leaves
  } else if (warp == kMmaWarp) {
    // =========================== products ===========================
    if (lane == 0) {
      const uint32_t IDESC_RH = idesc_bf16(kTcKeys, kTcHeads, false, false);
      const uint32_t IDESC_DV = idesc_bf16(kTcKeys, DV, false, true);
      const uint32_t IDESC_DK = idesc_bf16(kTcKeys, DQ, false, true);
      const uint32_t IDESC_DQ = idesc_bf16(128, kTcHeads, true, false);
      const uint32_t qb = smem_u32(sQ), dob = smem_u32(sdO);
      const uint32_t ptb0 = smem_u32(smem + L.pt_off), dstb0 = smem_u32(smem + L.dst_off);
      const uint32_t dshb0 = smem_u32(smem + L.dsh_off);
      // S^T and dP^T of chunk c into TMEM buffer c & 1
      auto scores = [&](int c) -> bool {
        const int st = c & 1, sb = c & 1;
        if (!mbar_wait(&kv_full[st], (c >> 1) & 1, abort_flag, a.err)) return false;
        if (c >= 2 && !mbar_wait(&sd_empty[sb], ((c >> 1) - 1) & 1, abort_flag, a.err)) return false;
        fence_proxy_async_smem();   // gathered rows (generic-proxy writes) -> tensor-core reads
        tc_fence_after();
        const uint32_t kb = smem_u32(smem + (uint32_t)st * L.stage_bytes);
        const uint32_t vb = kb + (uint32_t)qa * (kTcKeys * 128u);
        rows_by_heads_any(qa, tbase + 32u * (uint32_t)sb, kb, qb, IDESC_RH);         // S^T
        rows_by_heads_any(va, tbase + 32u * (uint32_t)sb + 16u, vb, dob, IDESC_RH);  // dP^T
        umma_commit(&sd_full[sb]);
        return true;
      };
      bool alive = mbar_wait(qd_full, 0, abort_flag, a.err) && scores(0);
      for (int c = 0; c < nchunks && alive; ++c) {
        const int st = c & 1;
        // the next chunk's scores go first only when its rows have already landed: waiting
        // for them here would hold back this chunk's products, whose completion frees the
        // stage the chunk after next is gathered into
        const bool early = c + 1 < nchunks && mbar_test(&kv_full[(c + 1) & 1], ((c + 1) >> 1) & 1);
        if (early && !scores(c + 1)) break;
        // P / dS set pb of chunk c (use c / npb of that set)
        const int pb = c % L.npb, pu = c / L.npb;
        const uint32_t ptb = ptb0 + (uint32_t)pb * L.pbuf_bytes, dstb = dstb0 + (uint32_t)pb * L.pbuf_bytes;
        const uint32_t dshb = dshb0 + (uint32_t)pb * L.pbuf_bytes;
        if (!mbar_wait(&p_full[pb], pu & 1, abort_flag, a.err)) break;
        // dV, then dK, each as soon as the drain warps have read the previous chunk's rows:
        // the next dV product runs while the last dK rows drain
        if (c > 0 && !mbar_wait(dv_empty, (c - 1) & 1, abort_flag, a.err)) break;
        tc_fence_after();
        rows_by_dims(tbase + TC_DV, ptb, dob, IDESC_DV);    // dV rows
        umma_commit(dv_full);
        if (c > 0 && !mbar_wait(dk_empty, (c - 1) & 1, abort_flag, a.err)) break;
        tc_fence_after();
        rows_by_dims(tbase + TC_DK, dstb, qb, IDESC_DK);    // dK rows
        umma_commit(dk_full);
        const uint32_t kb = smem_u32(smem + (uint32_t)st * L.stage_bytes);
        for (int b = 0; b < nqb; ++b)                      // dQ^T, over all chunks
          dq_block(tbase + TC_DQ + 16u * (uint32_t)b, kb + (uint32_t)b * (2u * kTcKeys * 128u), dshb, IDESC_DQ, c > 0);
        umma_commit(&kv_empty[st]);
        umma_commit(&p_empty[pb]);
        if (c == nchunks - 1) umma_commit(dq_full);
        if (c + 1 < nchunks && !early && !scores(c + 1)) break;
      }
      // every product this thread issued completes before the CTA releases tensor memory
      umma_commit(drain);
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {}
    }
  } else if (warp < kDrainWarp0) {
    // =========================== P and dS, one key per thread ===========================
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_addr = tmem_lane_base(warp);
    uint8_t* pt_row0 = smem + L.pt_off + r * 128;
    uint8_t* dst_row0 = smem + L.dst_off + r * 128;
    uint8_t* dsh0 = smem + L.dsh_off;
    for (int c = 0; c < nchunks; ++c) {
      const int sb = c & 1;
      const bool ok = mbar_wait(&sd_full[sb], (c >> 1) & 1, abort_flag, a.err);
      __syncwarp();   // converge after the polling wait: tcgen05.ld is warp-aligned
      if (!ok) break;
      tc_fence_after();
      float s[16], dp[16];
      tmem_ld16(tbase + 32u * (uint32_t)sb + lane_addr, s);
      tmem_ld16(tbase + 32u * (uint32_t)sb + 16u + lane_addr, dp);
      tmem_ld_wait_regs(s);
      tmem_ld_wait_regs(dp);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sd_empty[sb]);
      const bool valid = c * kTcKeys + r < n;
      uint32_t pw[8], dw[8];
#pragma unroll
      for (int h = 0; h < 16; h += 2) {
        float p2[2], d2[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int hh = h + e;
          const bool on = valid && hh < nh;
          const float p = on ? ex2_approx(fmaf(s[hh], a.scale_log2, -l2h[hh])) : 0.f;
          p2[e] = p;
          d2[e] = on ? p * (dp[hh] - Dh[hh]) * a.scale : 0.f;
        }
        const __nv_bfloat162 pp = __floats2bfloat162_rn(p2[0], p2[1]);
        const __nv_bfloat162 dd = __floats2bfloat162_rn(d2[0], d2[1]);
        pw[h >> 1] = *reinterpret_cast<const uint32_t*>(&pp);
        dw[h >> 1] = *reinterpret_cast<const uint32_t*>(&dd);
      }
      const int pb = c % L.npb, pu = c / L.npb;   // P / dS set, and its use count
      if (pu > 0 && !mbar_wait(&p_empty[pb], (pu - 1) & 1, abort_flag, a.err)) break;   // its last products read
      uint8_t* pt_row = pt_row0 + pb * L.pbuf_bytes;
      uint8_t* dst_row = dst_row0 + pb * L.pbuf_bytes;
      uint8_t* dsh = dsh0 + pb * L.pbuf_bytes;
      *reinterpret_cast<uint4*>(pt_row + ((0 ^ (r & 7)) << 4)) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
      *reinterpret_cast<uint4*>(pt_row + ((1 ^ (r & 7)) << 4)) = make_uint4(pw[4], pw[5], pw[6], pw[7]);
      *reinterpret_cast<uint4*>(dst_row + ((0 ^ (r & 7)) << 4)) = make_uint4(dw[0], dw[1], dw[2], dw[3]);
      *reinterpret_cast<uint4*>(dst_row + ((1 ^ (r & 7)) << 4)) = make_uint4(dw[4], dw[5], dw[6], dw[7]);
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        const uint32_t w = dw[h >> 1];
        const unsigned short bits = (h & 1) ? (unsigned short)(w >> 16) : (unsigned short)(w & 0xFFFFu);
        *reinterpret_cast<unsigned short*>(dsh + sw128_offset(h, r, kTcHeads)) = bits;
      }
      fence_proxy_async_smem();   // generic-proxy tile writes -> tensor-core reads
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[pb]);
    }
  } else {
    // ============ dK / dV rows to the accumulators, then dQ (one key / dim per thread) ============
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_addr = tmem_lane_base(warp);
    float* tr = reinterpret_cast<float*>(smem + L.tr_off) + (warp - kDrainWarp0) * (kTrRows * kTrPitch);
    bool alive = true;
    // the rows of one product (columns col .. col+ncols of TMEM) to dst
    auto drain_rows = [&](uint64_t* full, uint64_t* empty, int c, uint32_t col, int ncols, float* dst) -> bool {
      const bool ok = mbar_wait(full, c & 1, abort_flag, a.err);
      __syncwarp();
      if (!ok) return false;
      tc_fence_after();
      // this warp's 32 keys: slots kbase .. kbase+31 of the compacted route row
      const int kbase = c * kTcKeys + (warp & 3) * 32;
      const int nrows = min(32, n - kbase);
      for (int j = 0; j < ncols / 32; ++j) {
        float v[32];
        tmem_ld32(tbase + col + 32u * (uint32_t)j + lane_addr, v);
        tmem_ld_wait_regs(v);
        drain_cols(tr, v, lane, dst, ncols, 32 * j, ids + kbase, nrows, a.Hkv, g);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(empty);
      return true;
    };
    for (int c = 0; c < nchunks; ++c) {
      if (!drain_rows(dv_full, dv_empty, c, TC_DV, DV, a.dv) || !drain_rows(dk_full, dk_empty, c, TC_DK, DQ, a.dk)) {
        alive = false;
        break;
      }
    }
    if (alive) {
      const bool ok = mbar_wait(dq_full, 0, abort_flag, a.err);
      __syncwarp();
      if (ok) {
        tc_fence_after();
        float* dq_t = a.dq + ((int64_t)t * a.Hq + h0) * DQ;
        for (int b = 0; b < nqb; ++b) {
          float v[16];
          tmem_ld16(tbase + TC_DQ + 16u * (uint32_t)b + lane_addr, v);
          tmem_ld_wait_regs(v);
          const int d = 128 * b + r;
          if (d < DQ)
#pragma unroll
            for (int h = 0; h < 16; ++h)
              if (h < nh) dq_t[(int64_t)h * DQ + d] = v[h];
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, tcols);
  }
}

}  // namespace

bool bwd_tc_supported(const BwdArgs& a) {
  if (a.v_alias || a.dv_alias || a.HB > kTcHeads) return false;
  if (a.Dqk % 64 != 0 || a.Dv % 64 != 0 || a.Dqk > 256 || a.Dv > 256) return false;
  if (96 + a.Dv + a.Dqk > 512) return false;   // TMEM: two S/dP buffers, dQ blocks, dV, dK
  return tc_layout(a.Dqk, a.Dv, a.W).total <= 227u * 1024u;
}

cudaError_t launch_bwd_tc(const BwdArgs& a, unsigned items, cudaStream_t stream) {
  const size_t smem = tc_layout(a.Dqk, a.Dv, a.W).total;
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  attn_bwd_tc_kernel<<<items, kTcThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace irs
