// Compressed-block indexer on sm_103a: document layout, FP32 block mean-pool,
// tensor-core weighted-ReLU scoring, per-query radix top-k, bitmap packing and route
// expansion, plus the sliding-window route composition.
//
// Definitions follow the QSA page (nemo_automodel.components.models.qwen3_8_flash_next.qsa:
// `select_qsa_token_ids`, `Qwen3_8_FlashNextQSAIndexer`, `_forward_packed`) and the Step-5
// sparse page (nemo_automodel.components.models.step5.sparse: `indexer_score_tile`,
// `pack_region_bitmap`).
#include "irs_internal.h"
#include "irs_ptx.cuh"

namespace irs {

// =====================================================================================
// a1: document layout. One CTA validates cu_seqlens and writes, per document, the first
// pooled-block row and the first score tile. meta[0] = 1 when the layout is valid.
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
    if (!ok) record_error(err, IRS_DEVERR_CU_SEQLENS);
  }
}

// Document containing token t: largest d with cu[d] <= t (cu strictly increasing).
__device__ __forceinline__ int find_doc(const int32_t* __restrict__ cu, int ndocs, int t) {
  int lo = 0, hi = ndocs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Largest d in [0, n) with off[d] <= x (off non-decreasing, off[0] = 0 <= x).
__device__ __forceinline__ int find_le(const int32_t* __restrict__ off, int n, int x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// =====================================================================================
// a2: block mean-pool. Thread = (pooled block, 8 consecutive dims). FP32 sequential sum
// over the c rows in token order, one IEEE division by c, then round-to-nearest-even
// to bf16 (the scoring operand).
// =====================================================================================
__global__ void __launch_bounds__(256) pool_kernel(const __nv_bfloat16* __restrict__ kI,
                                                   const int32_t* __restrict__ cu, int ndocs, int Di, int c,
                                                   const int32_t* __restrict__ meta,
                                                   const int32_t* __restrict__ blk_off,
                                                   __nv_bfloat16* __restrict__ kbar) {
  if (meta[0] != 1) return;
  const int nblk = meta[1];
  const int chunks = Di >> 3;
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int gb = (int)(gid / chunks);
  const int ch = (int)(gid % chunks);
  if (gb >= nblk) return;
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
  uint4 o;
  __nv_bfloat162* q = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    q[i] = __floats2bfloat162_rn(__fdiv_rn(acc[2 * i], fc), __fdiv_rn(acc[2 * i + 1], fc));
  reinterpret_cast<uint4*>(kbar + (long long)gb * Di)[ch] = o;
}

// =====================================================================================
// a3: weighted-ReLU block scores on tcgen05.
//
// One CTA scores one tile of QT consecutive sparse queries of one document against all
// their visible blocks. The contraction runs transposed: the UMMA's M = 128 pooled key
// blocks (one per TMEM lane), N = QT*Hi = 256 (query, head) columns, K = Di. The query
// tile (B operand) stays in shared memory; 128-block key tiles (A operand) stream through
// a TMA ring. Two TMEM accumulators (2 x 256 columns) let the epilogue of tile j overlap
// the MMAs of tile j+1. The epilogue thread of lane b reads its 256 columns and reduces
// each query's heads in order: s = sum_h w[t,h] * max(acc, 0) (FP32 FMA chain).
//
// Warps: 0 = TMA producer, 1 = TMEM owner + MMA issuer, 2..17 = epilogue (four warps per
// TMEM lane quarter, each taking a quarter of the 256 columns, or whole queries if Hi > 64).
// =====================================================================================
constexpr int kScoreThreads = 576;   // producer, MMA, 16 epilogue warps
constexpr int kScoreN = 256;          // (query, head) columns per tile
constexpr int kScoreM = 128;          // key blocks per tile

struct ScoreArgs {
  const float* w;
  const int32_t* cu;
  const int32_t* blk_off;
  const int32_t* tile_off;
  const int32_t* meta;
  float* scores;
  int64_t ldS;
  int32_t* err;
  int ndocs, T, Hi, c, kb, QT, tau_sparse, stages;
};

__device__ __forceinline__ int rot_tile(int j, int jrot, int nbt) {
  const int r = j + jrot;
  return r >= nbt ? r - nbt : r;
}

__device__ __forceinline__ float w4f(const float4* w4, int k) {
  const float4 v = w4[k >> 2];
  return (k & 3) == 0 ? v.x : ((k & 3) == 1 ? v.y : ((k & 3) == 2 ? v.z : v.w));
}

template <int DI, int HI>
__global__ void __launch_bounds__(kScoreThreads, 1)
    score_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k, ScoreArgs a) {
  constexpr int KATOMS = DI / 64;
  constexpr uint32_t A_ATOM = kScoreM * 128;            // bytes per 64-dim atom of a key tile
  constexpr uint32_t A_STAGE = KATOMS * A_ATOM;
  constexpr uint32_t B_ATOM = kScoreN * 128;
  constexpr uint32_t B_BYTES = KATOMS * B_ATOM;
  constexpr uint32_t IDESC = idesc_bf16(kScoreM, kScoreN, false, false);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sB = smem;
  uint8_t* sA = smem + B_BYTES;
  const int ST = a.stages;
  float* sW = reinterpret_cast<float*>(sA + (size_t)ST * A_STAGE);
  int* sNvis = reinterpret_cast<int*>(sW + kScoreN);                 // [QT] visible blocks per query
  uint64_t* full = reinterpret_cast<uint64_t*>(sNvis + kScoreN);
  uint64_t* empty = full + ST;
  uint64_t* bfull = empty + ST;
  uint64_t* tfull = bfull + 1;
  uint64_t* tempty = tfull + 2;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

  if (a.meta[0] != 1) return;
  const int ntiles = a.meta[2];
  if ((int)blockIdx.x >= ntiles) return;
  // heaviest tiles (largest visible prefix) first
  const int tile = ntiles - 1 - (int)blockIdx.x;
  const int d = find_le(a.tile_off, a.ndocs, tile);
  const int s_doc = a.cu[d];
  const int L = a.cu[d + 1] - s_doc;
  const int tau0 = a.tau_sparse + (tile - a.tile_off[d]) * a.QT;
  const int nq = min(a.QT, L - tau0);
  const int t0 = s_doc + tau0;
  const int nvis_last = (tau0 + nq) / a.c;
  const int nbt = (nvis_last + kScoreM - 1) / kScoreM;
  // CTAs start at different key tiles so that concurrent CTAs do not all read the same
  // 32 KB of pooled keys from L2 at the same moment
  const int jrot = (int)(blockIdx.x % (unsigned)max(nbt, 1));
  const int blk0 = a.blk_off[d];
  constexpr int Hi = HI;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // per-tile head weights (columns of the accumulator are (query, head) = row-major [QT][Hi])
  for (int i = tid; i < kScoreN; i += kScoreThreads) {
    const long long gi = (long long)t0 * Hi + i;
    sW[i] = (i < a.QT * Hi && gi < (long long)a.T * Hi) ? a.w[gi] : 0.f;
    sNvis[i] = i < nq ? (tau0 + i + 1) / a.c : 0;   // rows past the document see nothing
  }
  if (tid == 0) {
    for (int s = 0; s < ST; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    mbar_init(bfull, 1);
    mbar_init(&tfull[0], 1); mbar_init(&tfull[1], 1);
    mbar_init(&tempty[0], 16); mbar_init(&tempty[1], 16);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tslot, 2 * kScoreN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      tma_prefetch_map(&tm_q);
      tma_prefetch_map(&tm_k);
      mbar_arrive_expect_tx(bfull, B_BYTES);
      for (int ka = 0; ka < KATOMS; ++ka) tma_load_2d(sB + ka * B_ATOM, &tm_q, ka * 64, t0 * Hi, bfull);
      int issued = 0;
      for (int j = 0; j < nbt; ++j) {
        const int s = j % ST;
        if (j >= ST && !mbar_wait(&empty[s], ((j / ST) - 1) & 1, abort_flag, a.err)) break;
        mbar_arrive_expect_tx(&full[s], A_STAGE);
        const int bt = rot_tile(j, jrot, nbt);
        for (int ka = 0; ka < KATOMS; ++ka)
          tma_load_2d(sA + (size_t)s * A_STAGE + ka * A_ATOM, &tm_k, ka * 64, blk0 + bt * kScoreM, &full[s]);
        issued = j + 1;
      }
      if (*abort_flag) {
        // let copies already in flight land before the CTA leaves
        for (int j = max(0, issued - ST); j < issued; ++j) {
          const unsigned long long t_0 = globaltimer_ns();
          while (!mbar_try_wait(&full[j % ST], (j / ST) & 1) && globaltimer_ns() - t_0 < kWaitLimitNs) {}
        }
        const unsigned long long t_1 = globaltimer_ns();
        while (!mbar_try_wait(bfull, 0) && globaltimer_ns() - t_1 < kWaitLimitNs) {}
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      if (mbar_wait(bfull, 0, abort_flag, a.err)) {
        for (int j = 0; j < nbt; ++j) {
          const int s = j % ST, buf = j & 1;
          if (j >= 2 && !mbar_wait(&tempty[buf], ((j >> 1) - 1) & 1, abort_flag, a.err)) break;
          if (!mbar_wait(&full[s], (j / ST) & 1, abort_flag, a.err)) break;
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + (size_t)s * A_STAGE);
          const uint32_t b_base = smem_u32(sB);
#pragma unroll
          for (int ks = 0; ks < DI / 16; ++ks) {
            const uint64_t ad = sdesc_sw128(a_base + (ks >> 2) * A_ATOM + (ks & 3) * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(b_base + (ks >> 2) * B_ATOM + (ks & 3) * 32, 16, 1024);
            umma_bf16(tbase + buf * kScoreN, ad, bd, IDESC, ks > 0);
          }
          umma_commit(&empty[s]);
          umma_commit(&tfull[buf]);
        }
      }
    }
  } else {
    // ---------------- epilogue: warps 2..17 ----------------
    const int quarter = warp & 3;
    const int part = (warp - 2) >> 2;
    // each warp takes kHalfCols consecutive columns; a query's Hi columns stay in one warp
    constexpr int kHalfCols = HI > 64 ? HI : 64;
    const int col0 = part * kHalfCols;
    const bool active = col0 < kScoreN;
    const uint32_t lane_addr = tmem_lane_base(warp);
    for (int j = 0; j < nbt; ++j) {
      const int buf = j & 1;
      // one decision per warp, taken after every lane's wait: tcgen05.ld is warp-aligned
      if (!__all_sync(0xffffffffu, mbar_wait(&tfull[buf], (j >> 1) & 1, abort_flag, a.err))) break;
      tc_fence_after();
      if (active) {
        const int blk = rot_tile(j, jrot, nbt) * kScoreM + quarter * 32 + lane;
        float carry = 0.f;
#pragma unroll 1
        for (int cc = col0; cc < col0 + kHalfCols; cc += 64) {
          float v2[2][32];
          tmem_ld32(tbase + lane_addr + buf * kScoreN + cc, v2[0]);
          if (kHalfCols > 32) tmem_ld32(tbase + lane_addr + buf * kScoreN + cc + 32, v2[1]);
          tmem_ld_wait_regs(v2[0]);
          tmem_ld_wait_regs(v2[1]);
#pragma unroll
          for (int half2 = 0; half2 < 2; ++half2) {
          if (half2 == 1 && kHalfCols <= 32) break;
          const int ccx = cc + 32 * half2;
          const float* v = v2[half2];
          const float4* w4 = reinterpret_cast<const float4*>(sW + ccx);
          // per query: 4 interleaved FMA chains over its heads (h mod 4), then combined;
          // prod[q0] holds the sum of the group of columns starting at q0
          float prod[32];
          constexpr int G = HI < 32 ? HI : 32;        // columns of one query inside this chunk
          constexpr int CH = G < 4 ? G : 4;           // independent chains per query
#pragma unroll
          for (int q0 = 0; q0 < 32; q0 += G) {
            float acc4[CH];
#pragma unroll
            for (int cidx = 0; cidx < CH; ++cidx) acc4[cidx] = 0.f;
#pragma unroll
            for (int k = 0; k < G; ++k) acc4[k % CH] = fmaf(w4f(w4, q0 + k), fmaxf(v[q0 + k], 0.f), acc4[k % CH]);
            float sum = acc4[0];
#pragma unroll
            for (int cidx = 1; cidx < CH; ++cidx) sum += acc4[cidx];
            prod[q0] = sum;
          }
          if constexpr (HI <= 32) {
#pragma unroll
            for (int k = 0; k < 32; k += HI) {
              const int qi = (ccx + k) / HI;
              if (blk < sNvis[qi]) a.scores[(long long)(t0 + qi) * a.ldS + blk] = prod[k];
            }
          } else {
            carry += prod[0];
            if (((ccx + 32) & (HI - 1)) == 0) {
              const int qi = ccx / HI;
              if (blk < sNvis[qi]) a.scores[(long long)(t0 + qi) * a.ldS + blk] = carry;
              carry = 0.f;
            }
          }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 2 * kScoreN);
  }
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
  int32_t* out = a.route + (long long)t * W;

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
  int32_t* out = a.route + (long long)t * W;
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

// Launch the top-k + expansion for every row: the register variant when the longest row
// has at most 2048 visible blocks, else the shared-memory variant.
static cudaError_t launch_topk(const TopkArgs& ta, int kb, cudaStream_t stream, size_t cta_smem) {
  const int nv = ta.nvis_cap;
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
template <int DI>
static cudaError_t launch_score_di(int Hi, int grid, size_t smem, cudaStream_t st, const CUtensorMap& tq,
                                   const CUtensorMap& tk, const ScoreArgs& sa) {
  switch (Hi) {
    case 1: score_kernel<DI, 1><<<grid, kScoreThreads, smem, st>>>(tq, tk, sa); break;
    case 2: score_kernel<DI, 2><<<grid, kScoreThreads, smem, st>>>(tq, tk, sa); break;
    case 4: score_kernel<DI, 4><<<grid, kScoreThreads, smem, st>>>(tq, tk, sa); break;
    case 8: score_kernel<DI, 8><<<grid, kScoreThreads, smem, st>>>(tq, tk, sa); break;
    case 16: score_kernel<DI, 16><<<grid, kScoreThreads, smem, st>>>(tq, tk, sa); break;
    case 32: score_kernel<DI, 32><<<grid, kScoreThreads, smem, st>>>(tq, tk, sa); break;
    case 64: score_kernel<DI, 64><<<grid, kScoreThreads, smem, st>>>(tq, tk, sa); break;
    case 128: score_kernel<DI, 128><<<grid, kScoreThreads, smem, st>>>(tq, tk, sa); break;
    default: score_kernel<DI, 256><<<grid, kScoreThreads, smem, st>>>(tq, tk, sa); break;
  }
  return cudaGetLastError();
}

static cudaError_t launch_score(int Di, int Hi, int grid, size_t smem, cudaStream_t st, const CUtensorMap& tq,
                                const CUtensorMap& tk, const ScoreArgs& sa) {
  return Di == 64 ? launch_score_di<64>(Hi, grid, smem, st, tq, tk, sa)
                  : launch_score_di<128>(Hi, grid, smem, st, tq, tk, sa);
}

IndexPlan plan_index(int T, int Hi, int Di, int c, int budget, int ndocs, int max_doc_len, bool with_scores) {
  IndexPlan p{};
  p.kb = budget / c;
  p.QT = kScoreN / Hi;
  p.tau_sparse = (p.kb + 1) * c - 1;
  p.nblk_cap = T / c > 0 ? T / c : 1;
  p.ldS = max_doc_len / c > 0 ? max_doc_len / c : 1;
  p.score_tiles_cap = (T + p.QT - 1) / p.QT + ndocs;
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
  p.ws_bytes = (off + 255) / 256 * 256;
  p.stages = Di == 64 ? 6 : 4;
  const size_t b_bytes = (size_t)kScoreN * Di * 2;
  const size_t a_bytes = (size_t)p.stages * kScoreM * Di * 2;
  p.score_smem = 1024 + b_bytes + a_bytes + kScoreN * 8 + (2 * p.stages + 5) * 8 + 16;
  p.topk_smem = topk_smem_bytes(p.ldS, p.kb);
  return p;
}

size_t topk_smem_bytes(int nvis_cap, int kb) {
  const size_t nw = (size_t)(nvis_cap + 31) / 32;
  return (size_t)nvis_cap * 4 + nw * 4 * 3 + (size_t)kb * 4 + 16;
}

cudaError_t launch_index(const IndexPlan& p, const __nv_bfloat16* qI, const __nv_bfloat16* kI, const float* w,
                         const int32_t* cu, int ndocs, int max_doc_len, int T, int Hi, int Di, int c, int budget,
                         int32_t* route, float* scores, int64_t ldS, uint8_t* ws, int32_t* err,
                         const CUtensorMap& tm_q, const CUtensorMap& tm_k, cudaStream_t stream) {
  int32_t* meta = reinterpret_cast<int32_t*>(ws + p.off_meta);
  int32_t* blk_off = reinterpret_cast<int32_t*>(ws + p.off_blk);
  int32_t* tile_off = reinterpret_cast<int32_t*>(ws + p.off_tile);
  __nv_bfloat16* kbar = reinterpret_cast<__nv_bfloat16*>(ws + p.off_kbar);

  layout_kernel<<<1, 1024, 0, stream>>>(cu, ndocs, T, c, p.tau_sparse, p.QT, max_doc_len, meta, blk_off, tile_off,
                                        err);
  {
    const long long threads = (long long)p.nblk_cap * (Di / 8);
    const int grid = (int)((threads + 255) / 256);
    pool_kernel<<<grid, 256, 0, stream>>>(kI, cu, ndocs, Di, c, meta, blk_off, kbar);
  }
  ScoreArgs sa{w, cu, blk_off, tile_off, meta, scores, ldS, err, ndocs, T, Hi, c, p.kb, p.QT, p.tau_sparse,
               p.stages};
  const cudaError_t le = launch_score(Di, Hi, p.score_tiles_cap, p.score_smem, stream, tm_q, tm_k, sa);
  if (le != cudaSuccess) return le;
  TopkArgs ta{scores, ldS, cu, meta, route, err, ndocs, T, c, budget, max_doc_len, (int)p.ldS};
  return launch_topk(ta, p.kb, stream, p.topk_smem);
}

cudaError_t launch_topk_from_scores(const float* scores, int64_t ldS, const int32_t* cu, int ndocs, int max_doc_len,
                                    int T, int c, int budget, int32_t* route, int32_t* err, cudaStream_t stream) {
  const int nvis_cap = max_doc_len / c > 0 ? max_doc_len / c : 1;
  TopkArgs ta{scores, ldS, cu, nullptr, route, err, ndocs, T, c, budget, max_doc_len, nvis_cap};
  return launch_topk(ta, budget / c, stream, topk_smem_bytes(nvis_cap, budget / c));
}

cudaError_t launch_compose_window(const int32_t* route, int W, const int32_t* cu, int ndocs, int T, int window,
                                  int32_t* out, int32_t* err, cudaStream_t stream) {
  compose_window_kernel<<<T, 128, 0, stream>>>(route, W, cu, ndocs, T, window, out, err);
  return cudaGetLastError();
}

template <int DI, int HI>
static cudaError_t score_attr(size_t smem) {
  return cudaFuncSetAttribute(score_kernel<DI, HI>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

template <int DI>
static cudaError_t score_attr_all(size_t smem) {
  cudaError_t e = cudaSuccess;
  for (cudaError_t x : {score_attr<DI, 1>(smem), score_attr<DI, 2>(smem), score_attr<DI, 4>(smem),
                        score_attr<DI, 8>(smem), score_attr<DI, 16>(smem), score_attr<DI, 32>(smem),
                        score_attr<DI, 64>(smem), score_attr<DI, 128>(smem), score_attr<DI, 256>(smem)})
    if (x != cudaSuccess) e = x;
  return e;
}

cudaError_t configure_score_kernels(size_t smem) {
  cudaError_t e = score_attr_all<64>(smem);
  if (e != cudaSuccess) return e;
  return score_attr_all<128>(smem);
}

cudaError_t configure_topk_kernel(size_t smem) {
  return cudaFuncSetAttribute(topk_expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

}  // namespace irs
