// The persistent block-score kernel of the indexer (weighted-ReLU scores on tcgen05).
// Included by irs_index.cu and by the two translation units that instantiate the kernel
// for Di = 64 and Di = 128 (compiled in parallel).
//
// Definitions follow the QSA page (nemo_automodel.components.models.qwen3_8_flash_next.qsa:
// `select_qsa_token_ids`, `Qwen3_8_FlashNextQSAIndexer`) and the Step-5 sparse page
// (nemo_automodel.components.models.step5.sparse: `indexer_score_tile`, `pack_region_bitmap`).
#pragma once

#include "irs_internal.h"
#include "irs_ptx.cuh"

namespace irs {

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
// a3: weighted-ReLU block scores on tcgen05, one persistent kernel.
//
// Work: tiles of QT = 256/Hi consecutive sparse queries of one document, heaviest first
// (later tiles of a document see more blocks); CTAs take tiles from a device counter.
//
// The contraction runs transposed: UMMA M = 128 pooled key blocks (one TMEM lane each),
// N = QT*Hi = 256 (query, head) columns, K = Di. The query tile (B operand, TMA) is
// double-buffered across tiles, so the next tile's queries load while the current one's
// key tiles run; key tiles (A operand) stream through a TMA ring of 64-dim atoms; two TMEM
// accumulators (2 x 256 columns) let the epilogue of one key tile overlap the MMAs of the
// next. The epilogue thread of lane b reduces each query's heads in order,
// s = sum_h w[t,h] * max(acc, 0) (FP32 FMA chains), and writes row t of the FP32 scores.
//
// Warps: 0 scheduler + TMA producer, 1 TMEM owner + MMA issuer, 2..17 epilogue (four per
// TMEM lane quarter, 64 columns each). The producer only issues copies (it fetches the
// next tile's id one tile ahead); each epilogue warp loads the head weights of its own
// columns, so no global-load latency sits between two tiles' key copies. Every cross-warp
// wait is a bounded mbarrier wait.
// =====================================================================================
constexpr int kIdxThreads = 576;      // producer, MMA issuer, 16 epilogue warps
constexpr int kIdxN = 256;           // (query, head) columns per tile
constexpr int kIdxM = 128;           // key blocks per key tile
constexpr int kEpiWarp0 = 2;
constexpr int kNumEpi = 16;
constexpr int kTileSlots = 4;
constexpr int kIdxAtom = kIdxM * 128;   // bytes of one 64-dim atom of a key tile
enum { kTileSparse = 0, kTileStop = 2 };

struct TileInfo {
  int kind, t0, n, s_doc, tau0, nbt, blk0, jrot;
};

struct IndexArgs {
  const float* w;
  const int32_t* cu;
  const int32_t* blk_off;
  const int32_t* tile_off;
  int32_t* meta;      // [0] layout valid, [1] pooled blocks, [2] score tiles, [3] tile counter
  float* scores;      // row t at t * ldS
  int64_t ldS;
  int32_t* err;
  int ndocs, T, c, QT, tau_sparse, stages;
  int64_t w_ts;       // elements between the head weights of consecutive tokens (Hi, or G*Hi
                      // for per-group weights, w already offset to the group)
  int q_y0;           // first of the token's query rows in tm_q (g*Hi for group g)
};

__device__ __forceinline__ int rot_tile(int j, int jrot, int nbt) {
  const int r = j + jrot;
  return r >= nbt ? r - nbt : r;
}

static __device__ TileInfo decode_tile(const IndexArgs& a, int id, int nsparse) {
  TileInfo ti{};
  ti.kind = kTileStop;
  if (id < nsparse) {
    const int tile = nsparse - 1 - id;   // later tiles of a document see more blocks: heaviest first
    const int d = find_le(a.tile_off, a.ndocs, tile);
    const int s = a.cu[d], L = a.cu[d + 1] - s;
    ti.kind = kTileSparse;
    ti.s_doc = s;
    ti.tau0 = a.tau_sparse + (tile - a.tile_off[d]) * a.QT;
    ti.n = min(a.QT, L - ti.tau0);
    ti.t0 = s + ti.tau0;
    ti.nbt = ((ti.tau0 + ti.n) / a.c + kIdxM - 1) / kIdxM;
    ti.blk0 = a.blk_off[d];
    // tiles start at different key tiles, so concurrent CTAs of one document do not all
    // read the same pooled keys from L2 at the same moment
    ti.jrot = id % max(ti.nbt, 1);
  }
  return ti;
}

__device__ __forceinline__ float w4f(const float4* w4, int k) {
  const float4 v = w4[k >> 2];
  return (k & 3) == 0 ? v.x : ((k & 3) == 1 ? v.y : ((k & 3) == 2 ? v.z : v.w));
}

// Shared-memory layout of the score kernel for Di of bf16 (F8 = false: 64 elements per
// 128-byte atom row) or of E4M3 (F8 = true: 128 elements per row) operands.
template <int DI, bool F8 = false>
struct IdxSmem {
  static constexpr int kAtomElems = F8 ? 128 : 64;
  static constexpr uint32_t kBAtom = kIdxN * 128;
  static constexpr uint32_t kBBytes = (DI / kAtomElems) * kBAtom;
  static constexpr uint32_t b_off = 0;                                   // [2] query tiles
  static constexpr uint32_t a_off = 2 * kBBytes;                         // [stages] key atoms
  // [16 epilogue warps][64] fp32: each warp's copy of its columns' head weights
  __host__ __device__ static uint32_t w_off(int st) { return a_off + (uint32_t)st * kIdxAtom; }
  // [2 buffers][4 lane quarters][4 column blocks][32 lanes] fp32 partial sums
  __host__ __device__ static uint32_t part_off(int st) { return w_off(st) + kNumEpi * 64 * 4; }
  __host__ __device__ static uint32_t tile_off(int st) { return part_off(st) + 2 * 512 * 4; }
  __host__ __device__ static uint32_t bar_off(int st) { return tile_off(st) + kTileSlots * sizeof(TileInfo); }
  __host__ __device__ static uint32_t total(int st) { return bar_off(st) + (2 * st + 17) * 8 + 16 + 1024; }
};

template <bool F8>
__device__ __forceinline__ void umma_op(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  if constexpr (F8) umma_f8(d, a, b, idesc, acc);
  else umma_bf16(d, a, b, idesc, acc);
}

template <int DI, int HI, bool F8>
__global__ void __launch_bounds__(kIdxThreads, 1)
    score_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       IndexArgs a) {
  using L = IdxSmem<DI, F8>;
  constexpr int AE = L::kAtomElems;   // elements per 128-byte row of an atom
  constexpr int KATOMS = DI / AE;
  constexpr uint32_t IDESC = F8 ? idesc_e4m3(kIdxM, kIdxN) : idesc_bf16(kIdxM, kIdxN, false, false);
  constexpr int kColsPerWarp = kIdxN / 4;

  extern __shared__ uint8_t smem_raw[];
  // aligned by pointer arithmetic on the __shared__ array, so that accesses through these
  // pointers compile to shared-memory instructions
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int S = a.stages;
  uint8_t* sB = smem + L::b_off;
  uint8_t* sA = smem + L::a_off;
  float* sW = reinterpret_cast<float*>(smem + L::w_off(S));
  float* sPart = reinterpret_cast<float*>(smem + L::part_off(S));
  TileInfo* sTile = reinterpret_cast<TileInfo*>(smem + L::tile_off(S));
  uint64_t* a_full = reinterpret_cast<uint64_t*>(smem + L::bar_off(S));
  uint64_t* a_empty = a_full + S;
  uint64_t* b_full = a_empty + S;        // [2]
  uint64_t* b_empty = b_full + 2;        // [2]
  uint64_t* t_full = b_empty + 2;        // [2]
  uint64_t* t_empty = t_full + 2;        // [2]
  uint64_t* tile_full = t_empty + 2;     // [4]
  uint64_t* tile_empty = tile_full + 4;  // [4]
  uint64_t* drain = tile_empty + 4;      // [1]
  uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

  if (a.meta[0] != 1) return;   // malformed cu_seqlens: reported by the layout kernel
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) { mbar_init(&a_full[s], 1); mbar_init(&a_empty[s], 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&b_full[i], 1);                // the query tile's TMA
      mbar_init(&b_empty[i], 1);               // the last MMA of the tile
      mbar_init(&t_full[i], 1);
      mbar_init(&t_empty[i], kNumEpi);
    }
    for (int i = 0; i < kTileSlots; ++i) {
      mbar_init(&tile_full[i], 1);
      mbar_init(&tile_empty[i], 1 + kNumEpi);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tslot, 2 * kIdxN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  if (warp == 0) {
    // ---------------- scheduler + TMA producer (whole warp; lane 0 issues) ----------------
    const int nsparse = a.meta[2];
    if (lane == 0) { tma_prefetch_map(&tm_q); tma_prefetch_map(&tm_k); }
    uint32_t i = 0, nb = 0, at = 0;
    int pst = 0;          // ring stage of atom `at`
    uint32_t pph = 0;     // (at / S) & 1
    // the next tile's id is fetched one tile ahead, so the counter's round trip overlaps
    // the current tile's loads
    int next_id = 0;
    if (lane == 0) next_id = atomicAdd(&a.meta[3], 1);
    while (true) {
      const int slot = i & (kTileSlots - 1);
      if (i >= kTileSlots &&
          !__all_sync(0xffffffffu, mbar_wait(&tile_empty[slot], ((i / kTileSlots) - 1) & 1, abort_flag, a.err)))
        break;
      const int id = __shfl_sync(0xffffffffu, next_id, 0);
      const TileInfo ti = decode_tile(a, id, nsparse);
      if (lane == 0) sTile[slot] = ti;
      __syncwarp();
      if (lane == 0) mbar_arrive(&tile_full[slot]);
      ++i;
      if (ti.kind == kTileStop) break;
      if (lane == 0) next_id = atomicAdd(&a.meta[3], 1);
      const int bs = nb & 1;
      if (nb >= 2 && !__all_sync(0xffffffffu, mbar_wait(&b_empty[bs], ((nb >> 1) - 1) & 1, abort_flag, a.err)))
        break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&b_full[bs], L::kBBytes);
        // tm_q: 3-D [T][rows per token][Di], box {64, Hi, QT}: the tile's (query, head) rows
        for (int ka = 0; ka < KATOMS; ++ka)
          tma_load_3d(sB + bs * L::kBBytes + ka * L::kBAtom, &tm_q, ka * AE, a.q_y0, ti.t0, &b_full[bs]);
      }
      ++nb;
      bool ok = true;
      if (lane == 0) {
        for (int j = 0; j < ti.nbt && ok; ++j) {
          const int bt = rot_tile(j, ti.jrot, ti.nbt);
          for (int ka = 0; ka < KATOMS; ++ka, ++at) {
            if (at >= (uint32_t)S && !mbar_wait(&a_empty[pst], pph ^ 1u, abort_flag, a.err)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&a_full[pst], kIdxAtom);
            tma_load_2d(sA + (size_t)pst * kIdxAtom, &tm_k, ka * AE, ti.blk0 + bt * kIdxM, &a_full[pst]);
            if (++pst == S) { pst = 0; pph ^= 1u; }
          }
        }
      }
      if (!__shfl_sync(0xffffffffu, (int)ok, 0)) break;
    }
    if (lane == 0 && *abort_flag) {
      // let the copies still in flight land before the CTA leaves
      const uint32_t first = at > (uint32_t)S ? at - S : 0;
      for (uint32_t x = first; x < at; ++x) {
        const unsigned long long t0 = globaltimer_ns();
        while (!mbar_try_wait(&a_full[x % S], (x / S) & 1) && globaltimer_ns() - t0 < kWaitLimitNs) {}
      }
      for (uint32_t x = nb > 2 ? nb - 2 : 0; x < nb; ++x) {
        const unsigned long long t0 = globaltimer_ns();
        while (!mbar_try_wait(&b_full[x & 1], (x >> 1) & 1) && globaltimer_ns() - t0 < kWaitLimitNs) {}
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    // tcgen05.mma blocks once the tensor pipe's short queue is full, so whatever this
    // thread does between two atoms' MMAs shows up as idle pipe time: the ring stage and
    // its phase advance incrementally (no division by the runtime stage count) and the
    // descriptors are a base plus an offset.
    if (lane == 0) {
      uint32_t i = 0, nb = 0, kt = 0;
      int st = 0;
      uint32_t aph = 0;   // phase parity of the ring's current pass
      const uint64_t a_desc0 = sdesc_sw128(smem_u32(sA), 16, 1024);
      const uint64_t b_desc0 = sdesc_sw128(smem_u32(sB), 16, 1024);
      bool alive = true;
      while (alive) {
        const int slot = i & (kTileSlots - 1);
        if (!mbar_wait(&tile_full[slot], (i / kTileSlots) & 1, abort_flag, a.err)) break;
        const TileInfo ti = sTile[slot];
        mbar_arrive(&tile_empty[slot]);
        ++i;
        if (ti.kind == kTileStop) break;
        const int bs = nb & 1;
        if (!mbar_wait(&b_full[bs], (nb >> 1) & 1, abort_flag, a.err)) break;
        const uint64_t b_desc = b_desc0 + (uint64_t)((bs * L::kBBytes) >> 4);
        for (int j = 0; j < ti.nbt && alive; ++j, ++kt) {
          const int buf = kt & 1;
          if (kt >= 2 && !mbar_wait(&t_empty[buf], ((kt >> 1) - 1) & 1, abort_flag, a.err)) { alive = false; break; }
          // each atom's MMAs go out as soon as it has landed; the stages are released
          // together at the end of the key tile, so no commit sits between two atoms' MMAs
          int sts[KATOMS];
#pragma unroll
          for (int ka = 0; ka < KATOMS; ++ka) {
            sts[ka] = st;
            if (!mbar_wait(&a_full[st], aph, abort_flag, a.err)) { alive = false; break; }
            if (++st == S) { st = 0; aph ^= 1u; }
            tc_fence_after();
            const uint64_t ad = a_desc0 + (uint64_t)((sts[ka] * kIdxAtom) >> 4);
            const uint64_t bd = b_desc + (uint64_t)((ka * L::kBAtom) >> 4);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              umma_op<F8>(tbase + buf * kIdxN, ad + (uint64_t)((ks * 32) >> 4), bd + (uint64_t)((ks * 32) >> 4), IDESC,
                        (ka > 0 || ks > 0) ? 1u : 0u);
          }
          if (!alive) break;
#pragma unroll
          for (int ka = 0; ka < KATOMS; ++ka) umma_commit(&a_empty[sts[ka]]);
          if (!alive) break;
          umma_commit(&t_full[buf]);
        }
        if (!alive) break;
        umma_commit(&b_empty[bs]);
        ++nb;
      }
      // every issued MMA completes before the CTA releases its tensor memory
      umma_commit(drain);
      const unsigned long long t0 = globaltimer_ns();
      while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {}
    }
  } else {
    // ---------------- epilogue: warps 2..17 ----------------
    const int e = warp - kEpiWarp0;
    const int quarter = warp & 3;
    const int col0 = (e >> 2) * kColsPerWarp;
    const uint32_t lane_addr = tmem_lane_base(warp);
    uint32_t i = 0, kt = 0;
    bool alive = true;
    while (alive) {
      const int slot = i & (kTileSlots - 1);
      if (!__all_sync(0xffffffffu, mbar_wait(&tile_full[slot], (i / kTileSlots) & 1, abort_flag, a.err))) break;
      const TileInfo ti = sTile[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&tile_empty[slot]);
      ++i;
      if (ti.kind == kTileStop) break;
      {
        // this warp's head weights (its 64 columns; zero past the last token), loaded before
        // the first wait on the MMA so that their latency overlaps it
        float* wt = sW + e * kColsPerWarp;
        {
          float wv[kColsPerWarp / 32];
#pragma unroll
          for (int k = 0; k < kColsPerWarp / 32; ++k) {
            const int col = col0 + k * 32 + lane;
            const long long tq = (long long)ti.t0 + col / HI;
            wv[k] = tq < a.T ? __ldg(a.w + tq * a.w_ts + (col % HI)) : 0.f;
          }
          __syncwarp();   // the previous tile's reads of wt are done
#pragma unroll
          for (int k = 0; k < kColsPerWarp / 32; ++k) wt[k * 32 + lane] = wv[k];
          __syncwarp();
        }
        for (int j = 0; j < ti.nbt; ++j, ++kt) {
          const int buf = kt & 1;
          // one decision per warp, taken after every lane's wait: tcgen05.ld is warp-aligned
          if (!__all_sync(0xffffffffu, mbar_wait(&t_full[buf], (kt >> 1) & 1, abort_flag, a.err))) {
            alive = false;
            break;
          }
          tc_fence_after();
          const int blk = rot_tile(j, ti.jrot, ti.nbt) * kIdxM + quarter * 32 + lane;
          // query q of the tile sees block blk iff (blk+1)*c - 1 <= tau0 + q
          const int qmin = (blk + 1) * a.c - 1 - ti.tau0;
          float carry = 0.f;
          float v[2][32];
          tmem_ld32(tbase + lane_addr + buf * kIdxN + col0, v[0]);
          tmem_ld32(tbase + lane_addr + buf * kIdxN + col0 + 32, v[1]);
          tmem_ld_wait_regs(v[0]);
          tmem_ld_wait_regs(v[1]);
#pragma unroll
          for (int c4 = 0; c4 < 2; ++c4) {
            const int ccx = col0 + 32 * c4;
            const float4* w4 = reinterpret_cast<const float4*>(wt + 32 * c4);
            // per query: 4 interleaved FMA chains over its heads (h mod 4), then combined;
            // prod[q0] holds the sum of the group of columns starting at q0
            float prod[32];
            constexpr int G = HI < 32 ? HI : 32;   // columns of one query inside this chunk
            constexpr int CH = G < 4 ? G : 4;      // independent chains per query
#pragma unroll
            for (int q0 = 0; q0 < 32; q0 += G) {
              if constexpr (G >= 4) {
                // two packed chains (heads 4j, 4j+1 and 4j+2, 4j+3): one f32x2 FMA per two
                // columns after the scalar ReLU
                uint64_t acc2[2] = {0ull, 0ull};
#pragma unroll
                for (int k = 0; k < G; k += 4) {
                  const float4 wq = w4[(q0 + k) >> 2];
                  acc2[0] = ffma2(pack2(wq.x, wq.y), pack2(fmaxf(v[c4][q0 + k], 0.f), fmaxf(v[c4][q0 + k + 1], 0.f)),
                                  acc2[0]);
                  acc2[1] = ffma2(pack2(wq.z, wq.w),
                                  pack2(fmaxf(v[c4][q0 + k + 2], 0.f), fmaxf(v[c4][q0 + k + 3], 0.f)), acc2[1]);
                }
                const float2 a0 = unpack2(acc2[0]), a1 = unpack2(acc2[1]);
                prod[q0] = (a0.x + a1.x) + (a0.y + a1.y);
              } else {
                float acc4[CH];
#pragma unroll
                for (int x = 0; x < CH; ++x) acc4[x] = 0.f;
#pragma unroll
                for (int k = 0; k < G; ++k)
                  acc4[k % CH] = fmaf(w4f(w4, q0 + k), fmaxf(v[c4][q0 + k], 0.f), acc4[k % CH]);
                float sum = acc4[0];
#pragma unroll
                for (int x = 1; x < CH; ++x) sum += acc4[x];
                prod[q0] = sum;
              }
            }
            if constexpr (HI <= 32) {
#pragma unroll
              for (int k = 0; k < 32; k += HI) {
                const int qi = (ccx + k) / HI;
                if (qi >= qmin && qi < ti.n) a.scores[(int64_t)(ti.t0 + qi) * a.ldS + blk] = prod[k];
              }
            } else {
              carry += prod[0];
              if constexpr (HI <= kColsPerWarp) {
                if (((ccx + 32) & (HI - 1)) == 0) {
                  const int qi = ccx / HI;
                  if (qi >= qmin && qi < ti.n) a.scores[(int64_t)(ti.t0 + qi) * a.ldS + blk] = carry;
                  carry = 0.f;
                }
              }
            }
          }
          if constexpr (HI > kColsPerWarp) {
            // a query spans HI/64 warps of this lane quarter: each leaves its partial sum, and
            // the warp holding the query's first columns adds them in column order
            constexpr int WPQ = HI / kColsPerWarp;
            float* part = sPart + (kt & 1) * 512 + quarter * 128;
            const int cb = col0 / kColsPerWarp;
            part[cb * 32 + lane] = carry;
            named_bar_sync(1 + quarter, 128);
            if (cb % WPQ == 0) {
              float sum = part[cb * 32 + lane];
#pragma unroll
              for (int x = 1; x < WPQ; ++x) sum += part[(cb + x) * 32 + lane];
              const int qi = col0 / HI;
              if (qi >= qmin && qi < ti.n) a.scores[(int64_t)(ti.t0 + qi) * a.ldS + blk] = sum;
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&t_empty[buf]);
        }
        if (!alive) break;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 2 * kIdxN);
  }
}

// Host side of the translation units that instantiate the kernel.
template <int DI, bool F8>
static cudaError_t launch_score_di(int Hi, int grid, size_t smem, cudaStream_t st, const CUtensorMap& tq,
                                   const CUtensorMap& tk, const IndexArgs& ia) {
  switch (Hi) {
    case 1: score_kernel<DI, 1, F8><<<grid, kIdxThreads, smem, st>>>(tq, tk, ia); break;
    case 2: score_kernel<DI, 2, F8><<<grid, kIdxThreads, smem, st>>>(tq, tk, ia); break;
    case 4: score_kernel<DI, 4, F8><<<grid, kIdxThreads, smem, st>>>(tq, tk, ia); break;
    case 8: score_kernel<DI, 8, F8><<<grid, kIdxThreads, smem, st>>>(tq, tk, ia); break;
    case 16: score_kernel<DI, 16, F8><<<grid, kIdxThreads, smem, st>>>(tq, tk, ia); break;
    case 32: score_kernel<DI, 32, F8><<<grid, kIdxThreads, smem, st>>>(tq, tk, ia); break;
    case 64: score_kernel<DI, 64, F8><<<grid, kIdxThreads, smem, st>>>(tq, tk, ia); break;
    case 128: score_kernel<DI, 128, F8><<<grid, kIdxThreads, smem, st>>>(tq, tk, ia); break;
    default: score_kernel<DI, 256, F8><<<grid, kIdxThreads, smem, st>>>(tq, tk, ia); break;
  }
  return cudaGetLastError();
}

template <int DI, int HI, bool F8>
static cudaError_t score_attr(size_t smem) {
  return cudaFuncSetAttribute(score_kernel<DI, HI, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

template <int DI, bool F8>
static cudaError_t score_attr_all(size_t smem) {
  cudaError_t e = cudaSuccess;
  for (cudaError_t x : {score_attr<DI, 1, F8>(smem), score_attr<DI, 2, F8>(smem), score_attr<DI, 4, F8>(smem),
                        score_attr<DI, 8, F8>(smem), score_attr<DI, 16, F8>(smem), score_attr<DI, 32, F8>(smem),
                        score_attr<DI, 64, F8>(smem), score_attr<DI, 128, F8>(smem), score_attr<DI, 256, F8>(smem)})
    if (x != cudaSuccess) e = x;
  return e;
}

cudaError_t launch_score_64(int Hi, int grid, size_t smem, cudaStream_t st, const CUtensorMap& tq, const CUtensorMap& tk,
                            const IndexArgs& ia);
cudaError_t launch_score_128(int Hi, int grid, size_t smem, cudaStream_t st, const CUtensorMap& tq,
                             const CUtensorMap& tk, const IndexArgs& ia);
cudaError_t configure_score_64(size_t smem);
cudaError_t configure_score_128(size_t smem);
// E4M3 operands (Di = 128 only)
cudaError_t launch_score_e4m3(int Hi, int grid, size_t smem, cudaStream_t st, const CUtensorMap& tq,
                              const CUtensorMap& tk, const IndexArgs& ia);
cudaError_t configure_score_e4m3(size_t smem);

}  // namespace irs
