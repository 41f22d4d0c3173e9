"""Plain CPU oracle for indexer-routed sparse GQA attention.

TEST INFRASTRUCTURE. Only the tests, the smoke check of ``__graft_entry__`` and
the CPU-baseline / reference leg of ``bench.py`` may import or run this module.
The CUDA library never calls it and it never calls the CUDA library: the two
share no code. It is slow on purpose: every step is the plain definition,
evaluated in float64 (except where the method itself fixes FP32), one query row
at a time.

Sources (NVIDIA NeMo AutoModel API reference pages):

* "nemo_automodel.components.models.qwen3_8_flash_next.qsa" (the QSA page):
  - ``Qwen3_8_FlashNextQSAIndexer`` class description: the raw index keys
    [B,S,1,D_index] are pooled by an FP32 mean over each whole run of
    ``compress_ratio`` consecutive keys, giving [B, floor(S/c), 1, D_index]; a
    route row has budget + c - 1 entries ([B, S, budget + c - 1]).
  - ``select_qsa_token_ids`` description: the query at position t can see
    floor((t+1)/c) whole blocks, each scored as a head sum of
    ReLU(q_h . k_block); the budget/c highest-scoring blocks turn into their
    token IDs, followed by the 0..c-1 tokens of the query's unfinished block;
    unused slots hold -1.
  - ``_forward_packed`` description: for packed documents the pooling runs
    start over in each document, a query sees only its own document, and IDs
    are positions in the flattened sequence (document start + local offset).
  - the same class description: the pooled keys then get K RMSNorm and
    group-start RoPE; ``apply_qsa_rope``: per-token rotary values cat(cos, sin)
    over the first D_rope dims, the remaining dims unchanged.
  - ``gathered_qsa_gqa_attention`` / ``_gathered_qsa_gqa_attention_chunk``:
    grouped queries [B,Q,Hkv,G,D] attend K/V [B,S,Hkv,D] at the listed global
    IDs; -1 marks invalid slots; the default scale is 1/sqrt(D).
* "nemo_automodel.components.models.step5.sparse" (the Step-5 sparse page):
  ``indexer_score_tile`` fuses weighted-ReLU scoring with FP32 per-head weights
  into an FP32 score tile (per KV group, with signed weights and E4M3-rounded
  operands); ``Step5SparseIndexer.forward`` returns region IDs per KV group;
  ``pack_region_bitmap`` packs selected region IDs into 32-bit words.
* "nemo_automodel.components.models.step5.fa4" (``heads_per_group``):
  consecutive query heads share one KV group.
* "nemo_automodel.components.models.common.cudnn_sparse_attention":
  latent attention, q [Tq,H,576], kv_latent [Tk,1,576], values are the first
  512 latent dims, int32 indices with -1 invalid; ``_CudnnSparseAttention``
  pairs the forward with a backward that maps the BF16 output gradient to the
  query and latent-KV gradients.

Readings where the pages are silent or loose (each one is listed in the design
notes of the repository):

* R1  The FP32 block mean is rounded once to bf16 (round to nearest even)
      before it is used as a scoring operand (the scores are tensor-core dot
      products of bf16 operands).
* R2  Each block scores sum_h w[t,h] * ReLU(q[t,h] . k~[b]) with no extra
      1/sqrt(D) factor: a caller who wants one folds it into w.
* R3  Top-k ties go to the lower block index; -0.0 equals +0.0.
* R4  A route row has fixed sections: slots [0, budget) hold the selected blocks
      in ascending block order, c tokens each, then -1; slots
      [budget, budget+c-1) hold the incomplete-block tail tokens, then -1.
* R5  When (tau+1) % c == 0 the query's own block is complete and competes in
      the top-k like any other block; the tail is then empty.
* R6  Unstated softmax scales are 1/sqrt(D_qk).
* R7  A row with no valid route entry produces out = 0 and lse = -inf.
* R14 RoPE (``apply_qsa_rope``, rotary values stored as cat(cos, sin)) rotates
      the pairs (d, d + D_rope/2) of the first D_rope dims (rotate-half).
* R15 Front half: keys get K RMSNorm and the rotary values of their block's first
      token; queries get RMSNorm per head and those of their own token; the
      transform is evaluated in FP32 (sum of squares in ascending dim order, no
      fused multiply-add) and rounded once to bf16.
* R16 E4M3 operands (Step-5): queries are rounded bf16 -> E4M3 and pooled keys
      FP32 -> bf16 -> E4M3, ties to even, saturating past 448.
* R17 Learned-logit summaries (Step-5): the page gives the inputs (keys and
      per-dimension compression logits shaped like them), FP32 arithmetic and the
      two roundings, not the formula. Read plainly: per region and dim, the
      softmax of the logits over the region's c tokens weights the keys, in FP32
      (max subtracted, sequential sums in token order, one division), then bf16,
      then E4M3. The exponential is `exp_f32`, a stated FP32 evaluation, so that
      the codes it decides are reproducible.
* R18 Indexer projections: one bf16 weight matrix W [(Hi+1)*Di + Hi, H]; output
      columns [0, Hi*Di) are the queries (head-major), then the raw keys, then the
      Hi signed head weights; exact dot products rounded once, to bf16 (queries,
      keys) or FP32 (head weights).
* The FP32 mean is a sequential FP32 sum over the c rows of the block in
  ascending token order, followed by one IEEE division by c.
* Route entries outside [0, Tk) are padding.
"""
from __future__ import annotations

import math

import numpy as np

# --------------------------------------------------------------------------------------
# bf16 helpers (bit patterns are numpy uint16)
# --------------------------------------------------------------------------------------


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns, as float64."""
    u = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Nearest bf16 value of each float32 in `x`, ties to even mantissa (reading R1).

    Written from the definition: the two bf16 neighbours of x are the float32
    patterns with the low 16 bits cleared (toward zero) and that plus one bf16
    ulp (away from zero); pick the nearer one in exact float64 arithmetic, and
    on a tie the one whose last kept mantissa bit is 0. Returns float32 values.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32)
    lo_bits = bits & np.uint32(0xFFFF0000)
    hi_bits = lo_bits + np.uint32(0x10000)
    lo = lo_bits.view(np.float32).astype(np.float64)
    hi = hi_bits.view(np.float32).astype(np.float64)
    xv = x.astype(np.float64)
    d_lo = np.abs(xv - lo)
    d_hi = np.abs(hi - xv)
    lo_even = ((lo_bits >> np.uint32(16)) & np.uint32(1)) == 0
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & lo_even)
    return np.where(pick_lo, lo_bits, hi_bits).view(np.float32)


# --------------------------------------------------------------------------------------
# a1: document layout (QSA page, `_forward_packed`: cu_seqlens strictly increasing,
# from 0 up to T)
# --------------------------------------------------------------------------------------


def doc_bounds(cu_seqlens: np.ndarray, T: int) -> tuple[np.ndarray, np.ndarray]:
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    if cu.ndim != 1 or cu.shape[0] < 2:
        raise ValueError("cu_seqlens must be 1-D with at least two entries")
    if cu[0] != 0 or cu[-1] != T or np.any(cu[1:] <= cu[:-1]):
        raise ValueError("cu_seqlens must be strictly increasing from 0 to T")
    return cu[:-1].copy(), cu[1:].copy()


def doc_of_token(cu_seqlens: np.ndarray, t: int) -> int:
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    return int(np.searchsorted(cu, t, side="right") - 1)


# --------------------------------------------------------------------------------------
# a2: block mean-pool (QSA page, indexer class description)
# --------------------------------------------------------------------------------------


def pool_doc(kI_doc_f32: np.ndarray, c: int) -> np.ndarray:
    """FP32 means of the complete consecutive groups of `c` rows of one document.

    Each block is summed row by row in ascending token order in float32, then
    divided once by c in float32. Returns float32 [floor(L/c), Di].
    """
    L, Di = kI_doc_f32.shape
    nb = L // c
    x = np.asarray(kI_doc_f32, dtype=np.float32)
    acc = np.zeros((nb, Di), dtype=np.float32)
    for j in range(c):                               # row j of every block, in token order
        acc = (acc + x[j: nb * c: c]).astype(np.float32)
    return (acc / np.float32(c)).astype(np.float32)


def pool_keys(kI_bits: np.ndarray, cu_seqlens: np.ndarray, c: int) -> tuple[np.ndarray, np.ndarray]:
    """Pooled keys of every document, concatenated; and the per-document block offsets."""
    T = kI_bits.shape[0]
    starts, ends = doc_bounds(cu_seqlens, T)
    kI = bf16_to_f32(kI_bits)
    blocks = []
    blk_off = [0]
    for s, e in zip(starts, ends):
        p = pool_doc(kI[s:e], c)
        blocks.append(p)
        blk_off.append(blk_off[-1] + p.shape[0])
    Di = kI_bits.shape[1]
    kbar = np.concatenate(blocks, axis=0) if blocks else np.zeros((0, Di), np.float32)
    return kbar, np.asarray(blk_off, dtype=np.int64)


# --------------------------------------------------------------------------------------
# a0: the indexer's projections (QSA page, indexer class: one fused projection gives the
# raw query/key layout [B, S, (H_index + 1) * D_index], split into queries
# [B, S, H_index, D_index] and raw keys [B, S, 1, D_index]; Step-5 sparse page,
# `Step5IndexerWeightProjection`: FP32 source weights, a BF16 projection, signed FP32 head
# weights). Reading R18: one bf16 weight matrix W [(Hi+1)*Di + Hi, H], row n giving output
# column n; columns [0, Hi*Di) are the queries (head-major), [Hi*Di, (Hi+1)*Di) the raw
# keys, the last Hi the head weights. Each output is the exact dot product of the bf16
# operands, rounded once: to bf16 for queries and keys, to FP32 for the head weights.
# --------------------------------------------------------------------------------------


def round_f64_to_bf16(x: np.ndarray) -> np.ndarray:
    """Nearest bf16 value of each float64, ties to even, in one rounding (no detour through
    float32). bf16 keeps 8 significant bits: with |x| = m * 2^e, 0.5 <= m < 1, its spacing
    is 2^(e-8). Returns float64 (normal magnitudes; the projection's outputs are)."""
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(np.abs(x))
    q = np.ldexp(1.0, e - 8)
    return np.copysign(np.round(np.abs(x) / q) * q, x)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of float64 values that are exact in bf16."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float32))
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def project_indexer(hidden_bits: np.ndarray, W_bits: np.ndarray, Hi: int, Di: int):
    """Indexer inputs from hidden states (reading R18): hidden [T, H] and W
    [(Hi+1)*Di + Hi, H] bf16 bits. Returns qI bits [T, Hi, Di], kI bits [T, Di] (bf16) and
    w float32 [T, Hi]. The dot products are taken in float64 (a library matmul of exact
    bf16 values; its rounding error is below 2^-40 of the terms' magnitude here)."""
    T, H = hidden_bits.shape
    N = W_bits.shape[0]
    if N != (Hi + 1) * Di + Hi or W_bits.shape[1] != H:
        raise ValueError("W must be [(Hi+1)*Di + Hi, H]")
    y = bf16_to_f64(hidden_bits) @ bf16_to_f64(W_bits).T
    qk = f64_to_bf16_bits(round_f64_to_bf16(y[:, :(Hi + 1) * Di]))
    qI = np.ascontiguousarray(qk[:, :Hi * Di].reshape(T, Hi, Di))
    kI = np.ascontiguousarray(qk[:, Hi * Di:])
    w = y[:, (Hi + 1) * Di:].astype(np.float32)
    return qI, kI, w


# --------------------------------------------------------------------------------------
# a2'' (next): indexer front half (QSA page, indexer class: the FP32 group means get K
# RMSNorm and group-start RoPE; `apply_qsa_rope`: the rotary values of a token are
# cat(cos, sin) over the first D_rope dims, the other dims pass through). Readings: the
# rotation pairs dims d and d + D_rope/2 (rotate-half, R14); queries get RMSNorm per head
# and the rotary values of their own token; a pooled key gets those of its block's first
# token; the transform is evaluated in FP32, the precision of the kernels that round its
# result to the bf16 scoring operand, with the sum of squares in ascending dim order and
# every operation rounded to float32 (no fused multiply-add), then rounded once to bf16
# (R15; the pooled mean follows the same rule, R1).
# --------------------------------------------------------------------------------------


def rms_norm(x: np.ndarray, weight: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis in float32: ss = sum of x_d * x_d in ascending d,
    r = sqrt(ss / D + eps), y_d = (x_d / r) * weight_d, each operation rounded to float32."""
    x = np.asarray(x, dtype=np.float32)
    D = x.shape[-1]
    ss = np.zeros(x.shape[:-1], dtype=np.float32)
    for d in range(D):
        ss = (ss + (x[..., d] * x[..., d]).astype(np.float32)).astype(np.float32)
    r = np.sqrt(((ss / np.float32(D)).astype(np.float32) + np.float32(eps)).astype(np.float32)).astype(np.float32)
    return ((x / r[..., None]).astype(np.float32) * np.asarray(weight, dtype=np.float32)).astype(np.float32)


def apply_rope(x: np.ndarray, rope: np.ndarray) -> np.ndarray:
    """Rotate the first D_rope dims of x [..., D] by rope [..., D_rope] = cat(cos, sin), in
    float32. With h = D_rope / 2, dims d and d + h (d < h) form one pair:
    (x_d, x_{d+h}) -> (x_d cos_d - x_{d+h} sin_d, x_{d+h} cos_d + x_d sin_d),
    each product and each sum rounded to float32. rope broadcasts against x's leading axes
    (one row per token for all heads)."""
    y = np.array(x, dtype=np.float32, copy=True)
    r = np.asarray(rope, dtype=np.float32)
    h = r.shape[-1] // 2
    cos, sin = r[..., :h], r[..., h:2 * h]
    x1 = y[..., :h].copy()
    x2 = y[..., h:2 * h].copy()
    y[..., :h] = (x1 * cos).astype(np.float32) - (x2 * sin).astype(np.float32)
    y[..., h:2 * h] = (x2 * cos).astype(np.float32) + (x1 * sin).astype(np.float32)
    return y


def block_start_tokens(cu_seqlens: np.ndarray, T: int, c: int) -> np.ndarray:
    """Global index of the first token of every pooled block, in `pool_keys` order."""
    starts, ends = doc_bounds(cu_seqlens, T)
    out = [s + c * np.arange((e - s) // c, dtype=np.int64) for s, e in zip(starts, ends)]
    return np.concatenate(out) if out else np.zeros(0, np.int64)


def front_keys(kI_bits, cu_seqlens, c: int, k_weight, eps: float, rope) -> tuple[np.ndarray, np.ndarray]:
    """Pooled index keys after K RMSNorm and group-start RoPE, as bf16 values (float64),
    and the per-document block offsets."""
    T = kI_bits.shape[0]
    kbar, blk_off = pool_keys(kI_bits, cu_seqlens, c)
    first = block_start_tokens(cu_seqlens, T, c)
    y = apply_rope(rms_norm(kbar, k_weight, eps), np.asarray(rope)[first])
    return round_to_bf16(y).astype(np.float64), blk_off


def front_query_row(qI_t_bits, q_weight, eps: float, rope_t) -> np.ndarray:
    """Index queries of one token [Hi, Di] after per-head RMSNorm and the token's RoPE,
    as bf16 values (float64)."""
    y = apply_rope(rms_norm(bf16_to_f32(qI_t_bits), q_weight, eps), rope_t)
    return round_to_bf16(y).astype(np.float64)


# --------------------------------------------------------------------------------------
# a3: visibility and block scores (QSA page `select_qsa_token_ids`; Step-5 sparse page
# `indexer_score_tile` for the per-head FP32 weights)
# --------------------------------------------------------------------------------------


def visible_blocks(tau: int, c: int) -> int:
    """Complete blocks visible to a query at document-local position tau."""
    return (tau + 1) // c


def block_scores(qI_t: np.ndarray, w_t: np.ndarray, ktilde: np.ndarray) -> np.ndarray:
    """score[b] = sum_h w[h] * ReLU(sum_d qI[h,d] * k~[b,d]), float64, rounded once to float32.

    qI_t: float64 [Hi, Di]; w_t: float64 [Hi]; ktilde: float64 [n, Di] (bf16 values).
    """
    dots = qI_t @ ktilde.T                      # [Hi, n]
    relu = np.maximum(dots, 0.0)
    s = w_t @ relu                              # [n]
    return s.astype(np.float32)


# --------------------------------------------------------------------------------------
# a4: top-k (reading R3) and a5: bitmap + expansion (reading R4)
# --------------------------------------------------------------------------------------


def select_top(scores_f32: np.ndarray, kb: int) -> np.ndarray:
    """Indices of the kb largest scores, ties to the lower index, in ascending order."""
    s = np.asarray(scores_f32, dtype=np.float32).astype(np.float64)
    n = s.shape[0]
    if n <= kb:
        return np.arange(n, dtype=np.int64)
    order = np.lexsort((np.arange(n), -s))     # primary: score descending; then index ascending
    return np.sort(order[:kb])


def pack_bitmap(selected: np.ndarray, nblocks: int) -> np.ndarray:
    """32-bit words, bit (b % 32) of word b // 32 set for each selected block b."""
    words = np.zeros((nblocks + 31) // 32, dtype=np.uint32)
    for b in selected:
        words[b // 32] |= np.uint32(1) << np.uint32(b % 32)
    return words


def unpack_bitmap(words: np.ndarray, nblocks: int) -> np.ndarray:
    out = []
    for b in range(nblocks):
        if (int(words[b // 32]) >> (b % 32)) & 1:
            out.append(b)
    return np.asarray(out, dtype=np.int64)


def expand_route(doc_start: int, tau: int, c: int, budget: int, selected: np.ndarray) -> np.ndarray:
    """One route row [budget + c - 1] in global token IDs (reading R4)."""
    W = budget + c - 1
    row = np.full(W, -1, dtype=np.int32)
    slot = 0
    for b in selected:
        for j in range(c):
            row[slot] = doc_start + int(b) * c + j
            slot += 1
    nv = visible_blocks(tau, c)
    tail = (tau + 1) % c
    for j in range(tail):
        row[budget + j] = doc_start + nv * c + j
    return row


def route_row(doc_start: int, tau: int, c: int, budget: int, scores_f32) -> np.ndarray:
    """Route of one query from its block scores (None when every visible block is taken)."""
    kb = budget // c
    nv = visible_blocks(tau, c)
    if nv <= kb:
        selected = np.arange(nv, dtype=np.int64)
    else:
        selected = select_top(scores_f32, kb)
        selected = unpack_bitmap(pack_bitmap(selected, nv), nv)
    return expand_route(doc_start, tau, c, budget, selected)


def index_routes(qI_bits, kI_bits, w, cu_seqlens, c: int, budget: int, rows=None,
                 want_scores: bool = False, ldS: int | None = None, front: dict | None = None,
                 operands: str = "bf16", logits=None):
    """Indexer routes (and optionally FP32 block scores) for the requested rows.

    qI_bits [T, Hi, Di] bf16 bits, kI_bits [T, Di] bf16 bits, w [T, Hi] float32,
    cu_seqlens int [ndocs+1]. Returns int32 routes [len(rows), budget + c - 1];
    with want_scores also float32 scores [len(rows), ldS] (NaN where not scored:
    a row is scored only when more than budget/c blocks are visible).
    front: optional indexer front half, a dict with q_weight [Di], k_weight [Di], eps and
    rope [T, D_rope] (per-token cat(cos, sin)); the queries and pooled keys are then
    normalised and rotated before scoring (`front_query_row`, `front_keys`).
    operands: "bf16", or "e4m3" for the Step-5 scoring operands: the bf16 queries and
    bf16 pooled keys are further rounded to FP8 E4M3 values (`round_to_e4m3`).
    logits: optional Step-5 compression logits, bf16 bits shaped like kI_bits; the block
    keys are then the learned-logit summaries (`region_summaries_e4m3`) instead of the
    means, and `operands` decides only whether the queries are rounded to E4M3.
    """
    if logits is not None and front is not None:
        raise ValueError("learned-logit summaries take the keys as given (no front half)")
    if operands not in ("bf16", "e4m3"):
        raise ValueError("operands must be 'bf16' or 'e4m3'")
    if budget % c != 0 or budget <= 0 or c <= 0:
        raise ValueError("budget must be a positive multiple of c")
    T = qI_bits.shape[0]
    starts, ends = doc_bounds(cu_seqlens, T)
    rows = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    kb = budget // c
    W = budget + c - 1
    if logits is not None:
        ktilde, blk_off = region_summaries_e4m3(kI_bits, logits, cu_seqlens, c)
    elif front is None:
        kbar, blk_off = pool_keys(kI_bits, cu_seqlens, c)
        ktilde = round_to_bf16(kbar).astype(np.float64)
    else:
        ktilde, blk_off = front_keys(kI_bits, cu_seqlens, c, front["k_weight"], front["eps"], front["rope"])
    if operands == "e4m3":
        ktilde = round_to_e4m3(ktilde)
    if ldS is None:
        ldS = int(np.max(ends - starts)) // c
    routes = np.full((rows.shape[0], W), -1, dtype=np.int32)
    scores = np.full((rows.shape[0], max(ldS, 1)), np.nan, dtype=np.float32) if want_scores else None
    for i, t in enumerate(rows):
        d = doc_of_token(cu_seqlens, int(t))
        s = int(starts[d])
        tau = int(t) - s
        nv = visible_blocks(tau, c)
        sc = None
        if nv > kb:
            kt = ktilde[blk_off[d]: blk_off[d] + nv]
            q_t = (bf16_to_f64(qI_bits[t]) if front is None else
                   front_query_row(qI_bits[t], front["q_weight"], front["eps"], np.asarray(front["rope"])[t]))
            if operands == "e4m3":
                q_t = round_to_e4m3(q_t)
            sc = block_scores(q_t, np.asarray(w[t], dtype=np.float64), kt)
            if want_scores:
                scores[i, :nv] = sc
        routes[i] = route_row(s, tau, c, budget, sc)
    return (routes, scores) if want_scores else routes


def routes_from_scores(scores: np.ndarray, cu_seqlens, T: int, c: int, budget: int, rows=None) -> np.ndarray:
    """Routes from given float32 scores [T, ldS] (entries [0, nvis) of sparse rows are read)."""
    starts, _ = doc_bounds(cu_seqlens, T)
    rows = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    kb = budget // c
    out = np.full((rows.shape[0], budget + c - 1), -1, dtype=np.int32)
    for i, t in enumerate(rows):
        d = doc_of_token(cu_seqlens, int(t))
        s = int(starts[d])
        tau = int(t) - s
        nv = visible_blocks(tau, c)
        sc = scores[t, :nv] if nv > kb else None
        out[i] = route_row(s, tau, c, budget, sc)
    return out


# --------------------------------------------------------------------------------------
# Step-5 variants (Step-5 sparse page): `indexer_score_tile` scores
# [batch, groups, queries, regions] from queries [..., groups, heads, dim] and signed FP32
# head weights [..., groups, heads] against shared region summaries, and
# `Step5SparseIndexer.forward` returns region IDs per KV group; its scoring operands are
# bf16 queries and summaries whose values were rounded to FP8 E4M3.
# --------------------------------------------------------------------------------------


def round_to_e4m3(x: np.ndarray) -> np.ndarray:
    """Nearest FP8 E4M3 value of each element (1 sign, 4 exponent bits with bias 7, 3
    mantissa bits: normals 2^-6 .. 448, subnormals k * 2^-9), ties to even. Magnitudes
    past 448 saturate (reading R16). Returns float64."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, ex = np.frexp(a)                               # a = m * 2^ex, 0.5 <= m < 1 (ex = 0 for 0)
    e = np.maximum(ex.astype(np.float64) - 1.0, -6.0)  # exponent of the leading bit; subnormal floor
    quantum = np.exp2(e - 3.0)                        # spacing of E4M3 values at that exponent
    q = np.minimum(np.round(a / quantum) * quantum, 448.0)   # numpy rounds halves to even
    return np.copysign(q, x)


# --------------------------------------------------------------------------------------
# Step-5 learned-logit region summaries (Step-5 sparse page: `project_keys` returns the
# index keys and per-dimension compression logits shaped like them; `gather_region_payload`
# takes both; `_summarize_region_payload` turns them into region summaries in FP32 and
# keeps both roundings, BF16 then FP8 E4M3; `indexer_score_tile` scores the
# "E4M3-rounded BF16 region summaries [batch, regions, dim]"; `region_metadata` resets the
# regions at every document boundary). Reading R17.
# --------------------------------------------------------------------------------------

# Natural-log constants as the float32 nearest to their exact values, and the Taylor
# coefficients (ln 2)^k / k! of 2^f = e^(f ln 2), k = 0..7, each the float32 nearest to it.
_LOG2E_F32 = np.float32(1.0 / math.log(2.0))
_EXP2_TAYLOR_F32 = [np.float32(math.log(2.0) ** k / math.factorial(k)) for k in range(8)]


def exp_f32(x: np.ndarray) -> np.ndarray:
    """e^x for float32 x <= 0 in float32 arithmetic, every operation rounded to nearest
    (reading R17). Cody and Waite's range reduction (Software Manual for the Elementary
    Functions, 1980) to base 2: t = x * log2(e), n = rint(t) (ties to even), f = t - n
    (exact, |f| <= 1/2); 2^f from its degree-7 Taylor polynomial in Horner form, no fused
    multiply-add; the result p * 2^n (exact). For t < -125 the result is 0: e^x < 2^-125
    there, and the scaled result stays a normal float32 otherwise."""
    x = np.asarray(x, dtype=np.float32)
    with np.errstate(over="ignore"):                  # x * log2(e) may round to -inf: flushed below
        t = (x * _LOG2E_F32).astype(np.float32)
    under = t < np.float32(-125.0)
    t = np.where(under, np.float32(0.0), t).astype(np.float32)
    n = np.rint(t).astype(np.float32)
    f = (t - n).astype(np.float32)
    p = np.full_like(f, _EXP2_TAYLOR_F32[7])
    for k in range(6, -1, -1):
        p = ((p * f).astype(np.float32) + _EXP2_TAYLOR_F32[k]).astype(np.float32)
    y = np.ldexp(p, n.astype(np.int32)).astype(np.float32)
    return np.where(under, np.float32(0.0), y).astype(np.float32)


def summarize_doc(k_doc_bits: np.ndarray, z_doc_bits: np.ndarray, c: int) -> np.ndarray:
    """FP32 learned-logit summaries of the complete runs of c tokens of one document
    (reading R17): per region and dim d, the softmax over the region's tokens of the
    compression logits z[., d] weights the keys k[., d].

    m_d = max_j z[j,d]; e_j = exp_f32(z[j,d] - m_d) (the difference rounded to float32);
    s_d and n_d are sequential float32 sums over j in token order of e_j and of
    e_j * k[j,d] (the product rounded first); summary_d = n_d / s_d (one float32 division).
    Returns float32 [floor(L/c), Di].
    """
    L, Di = k_doc_bits.shape
    nb = L // c
    k = bf16_to_f32(k_doc_bits)[: nb * c].reshape(nb, c, Di)
    z = bf16_to_f32(z_doc_bits)[: nb * c].reshape(nb, c, Di)
    m = z.max(axis=1)
    s = np.zeros((nb, Di), dtype=np.float32)
    num = np.zeros((nb, Di), dtype=np.float32)
    for j in range(c):
        e = exp_f32((z[:, j] - m).astype(np.float32))
        s = (s + e).astype(np.float32)
        num = (num + (e * k[:, j]).astype(np.float32)).astype(np.float32)
    return (num / s).astype(np.float32)


def region_summaries(kI_bits, z_bits, cu_seqlens, c: int) -> tuple[np.ndarray, np.ndarray]:
    """Summaries of every document's regions, concatenated (float32, before rounding), and
    the per-document region offsets. Regions start over at each document."""
    T = kI_bits.shape[0]
    starts, ends = doc_bounds(cu_seqlens, T)
    parts, offs = [], [0]
    for s, e in zip(starts, ends):
        sm = summarize_doc(kI_bits[s:e], z_bits[s:e], c)
        parts.append(sm)
        offs.append(offs[-1] + sm.shape[0])
    Di = kI_bits.shape[1]
    out = np.concatenate(parts, axis=0) if parts else np.zeros((0, Di), np.float32)
    return out, np.asarray(offs, dtype=np.int64)


def region_summaries_e4m3(kI_bits, z_bits, cu_seqlens, c: int) -> tuple[np.ndarray, np.ndarray]:
    """The summaries as the scorer sees them: FP32 -> bf16 -> E4M3 (float64 values)."""
    sm, offs = region_summaries(kI_bits, z_bits, cu_seqlens, c)
    return round_to_e4m3(round_to_bf16(sm).astype(np.float64)), offs


def index_routes_grouped(qI_bits, kI_bits, w, cu_seqlens, c: int, budget: int, rows=None,
                         operands: str = "bf16", logits=None) -> np.ndarray:
    """Per-KV-group routes int32 [len(rows), G, budget + c - 1].

    qI_bits [T, G, Hi, Di], w [T, G, Hi] (signed allowed): the heads and weights of group g
    score the shared pooled keys and group g selects its own blocks, each group exactly as
    `index_routes` does for one.
    """
    G = qI_bits.shape[1]
    return np.stack([index_routes(qI_bits[:, g], kI_bits, np.asarray(w)[:, g], cu_seqlens, c, budget, rows=rows,
                                  operands=operands, logits=logits) for g in range(G)], axis=1)


def attention_grouped(q_bits, k_bits, v_bits, routes_g, scale: float, rows=None):
    """Sparse attention with per-KV-group routes [T, Hkv, W]: the query heads of KV head g
    attend the IDs of routes_g[t, g]. Returns out float32 [len(rows), Hq, Dv], lse float32."""
    T, Hq, _ = q_bits.shape
    Tk, Hkv, _ = k_bits.shape
    Dv = v_bits.shape[2]
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    if not scale > 0:
        raise ValueError("scale must be positive")
    G = Hq // Hkv
    rows = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.zeros((rows.shape[0], Hq, Dv), dtype=np.float32)
    lse = np.zeros((rows.shape[0], Hq), dtype=np.float32)
    for i, t in enumerate(rows):
        for g in range(Hkv):
            ids = np.asarray(routes_g[t, g], dtype=np.int64)
            ids = ids[(ids >= 0) & (ids < Tk)]
            hs = slice(g * G, (g + 1) * G)
            o, l = attend_row(bf16_to_f64(q_bits[t, hs]), bf16_to_f64(k_bits[ids, g:g + 1]),
                              bf16_to_f64(v_bits[ids, g:g + 1]), scale, 1)
            out[i, hs] = o.astype(np.float32)
            lse[i, hs] = l.astype(np.float32)
    return out, lse


# --------------------------------------------------------------------------------------
# a5': sliding window in front of the indexer route (Step-5 layers page: attention is
# windowed or CSA-selected; the windowed workload uses both)
# --------------------------------------------------------------------------------------


def compose_window(routes: np.ndarray, cu_seqlens, T: int, window: int, rows=None) -> np.ndarray:
    """[window causal tokens t-window+1..t (-1 before the document start)] ++ the
    indexer route with every ID already inside the window replaced by -1.

    `routes` is the full indexer route tensor [T, W]; `rows` selects output rows.
    """
    starts, _ = doc_bounds(cu_seqlens, T)
    rows = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    W = routes.shape[1]
    out = np.full((rows.shape[0], window + W), -1, dtype=np.int32)
    for i, t in enumerate(rows):
        d = doc_of_token(cu_seqlens, int(t))
        s = int(starts[d])
        lo = int(t) - window + 1
        for j in range(window):
            tok = lo + j
            out[i, j] = tok if tok >= s else -1
        r = routes[t]
        for j in range(W):
            out[i, window + j] = r[j] if r[j] < lo else -1
    return out


# --------------------------------------------------------------------------------------
# a6: gathered sparse GQA attention (QSA page `gathered_qsa_gqa_attention`; latent
# attention page for the MLA case)
# --------------------------------------------------------------------------------------


def kv_group(h: int, Hq: int, Hkv: int) -> int:
    """KV head of query head h: consecutive query heads share one KV group."""
    return h // (Hq // Hkv)


def attend_row(q_t: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float, Hkv: int):
    """One query row over its gathered keys.

    q_t float64 [Hq, Dqk]; K float64 [n, Hkv, Dqk]; V float64 [n, Hkv, Dv].
    Returns out float64 [Hq, Dv], lse float64 [Hq] (natural log).
    """
    Hq = q_t.shape[0]
    Dv = V.shape[2]
    n = K.shape[0]
    out = np.zeros((Hq, Dv), dtype=np.float64)
    lse = np.full(Hq, -np.inf, dtype=np.float64)
    if n == 0:
        return out, lse                          # reading R7
    for h in range(Hq):
        g = kv_group(h, Hq, Hkv)
        s = scale * (K[:, g, :] @ q_t[h])        # [n]
        m = np.max(s)
        p = np.exp(s - m)
        l = np.sum(p)
        out[h] = (p @ V[:, g, :]) / l
        lse[h] = m + math.log(l)
    return out, lse


def attention(q_bits, k_bits, v_bits, routes, scale: float, rows=None):
    """Sparse attention of the requested rows.

    q_bits [T, Hq, Dqk], k_bits [Tk, Hkv, Dqk], v_bits [Tk, Hkv, Dv] (bf16 bits),
    routes int32 [T, W] global key IDs (anything outside [0, Tk) is padding).
    Returns out float32 [len(rows), Hq, Dv] and lse float32 [len(rows), Hq].
    """
    T, Hq, _ = q_bits.shape
    Tk, Hkv, _ = k_bits.shape
    Dv = v_bits.shape[2]
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    if not scale > 0:
        raise ValueError("scale must be positive")
    rows = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.zeros((rows.shape[0], Hq, Dv), dtype=np.float32)
    lse = np.zeros((rows.shape[0], Hq), dtype=np.float32)
    for i, t in enumerate(rows):
        ids = np.asarray(routes[t], dtype=np.int64)
        ids = ids[(ids >= 0) & (ids < Tk)]
        K = bf16_to_f64(k_bits[ids])
        V = bf16_to_f64(v_bits[ids])
        o, l = attend_row(bf16_to_f64(q_bits[t]), K, V, scale, Hkv)
        out[i] = o.astype(np.float32)
        lse[i] = l.astype(np.float32)
    return out, lse


def latent_attention(q_bits, kv_bits, routes, scale: float, Dv: int = 512, rows=None):
    """Latent (MLA) attention: keys are the full latent rows, values their first Dv dims."""
    return attention(q_bits, kv_bits, kv_bits[:, :, :Dv], routes, scale, rows=rows)


# --------------------------------------------------------------------------------------
# a7: backward of the gathered sparse attention (latent attention page,
# `_CudnnSparseAttention.backward`: the BF16 output gradient is mapped to gradients of
# the query and of the gathered K/V rows; the FA4 page's reverse block lists serve the
# same key-side gradients for GQA)
# --------------------------------------------------------------------------------------


def attend_row_grad(q_t: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float, Hkv: int,
                    dO_t: np.ndarray):
    """Gradients of sum(out_t * dO_t) for one query row over its gathered keys.

    q_t float64 [Hq, Dqk]; K float64 [n, Hkv, Dqk]; V float64 [n, Hkv, Dv];
    dO_t float64 [Hq, Dv]. With p[h] = softmax over r of scale * K[r,g] . q[h] and
    out[h] = sum_r p[h,r] V[r,g] (g the KV group of h):
      dV[r,g] = sum over h in g of p[h,r] dO[h]
      dp[h,r] = dO[h] . V[r,g]
      ds[h,r] = p[h,r] (dp[h,r] - sum_r' p[h,r'] dp[h,r'])    (softmax Jacobian)
      dq[h]   = scale * sum_r ds[h,r] K[r,g]
      dK[r,g] = scale * sum over h in g of ds[h,r] q[h]
    Returns dq [Hq, Dqk], dK [n, Hkv, Dqk], dV [n, Hkv, Dv]. A row without keys has a
    constant output (reading R7), so all of its gradients are zero.
    """
    Hq, Dqk = q_t.shape
    n = K.shape[0]
    Dv = V.shape[2]
    dq = np.zeros((Hq, Dqk), dtype=np.float64)
    dK = np.zeros((n, Hkv, Dqk), dtype=np.float64)
    dV = np.zeros((n, Hkv, Dv), dtype=np.float64)
    if n == 0:
        return dq, dK, dV
    for h in range(Hq):
        g = kv_group(h, Hq, Hkv)
        s = scale * (K[:, g, :] @ q_t[h])        # [n]
        e = np.exp(s - np.max(s))
        p = e / np.sum(e)
        dV[:, g, :] += np.outer(p, dO_t[h])
        dp = V[:, g, :] @ dO_t[h]                # [n]
        ds = p * (dp - np.sum(p * dp))
        dq[h] = scale * (ds @ K[:, g, :])
        dK[:, g, :] += scale * np.outer(ds, q_t[h])
    return dq, dK, dV


def attention_bwd(q_bits, k_bits, v_bits, routes, scale: float, dout_bits, rows=None):
    """Backward of `attention` for the loss sum(out * dout).

    dout_bits bf16 bits [T, Hq, Dv]. The key and value gradients of every routed ID are
    summed over the requested rows. Returns dq float32 [len(rows), Hq, Dqk], dk float32
    [Tk, Hkv, Dqk] and dv float32 [Tk, Hkv, Dv], accumulated in float64.
    """
    T, Hq, Dqk = q_bits.shape
    Tk, Hkv, _ = k_bits.shape
    Dv = v_bits.shape[2]
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    if not scale > 0:
        raise ValueError("scale must be positive")
    rows = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    dq = np.zeros((rows.shape[0], Hq, Dqk), dtype=np.float64)
    dk = np.zeros((Tk, Hkv, Dqk), dtype=np.float64)
    dv = np.zeros((Tk, Hkv, Dv), dtype=np.float64)
    for i, t in enumerate(rows):
        ids = np.asarray(routes[t], dtype=np.int64)
        ids = ids[(ids >= 0) & (ids < Tk)]
        gq, gK, gV = attend_row_grad(bf16_to_f64(q_bits[t]), bf16_to_f64(k_bits[ids]),
                                     bf16_to_f64(v_bits[ids]), scale, Hkv, bf16_to_f64(dout_bits[t]))
        dq[i] = gq
        np.add.at(dk, ids, gK)
        np.add.at(dv, ids, gV)
    return dq.astype(np.float32), dk.astype(np.float32), dv.astype(np.float32)


def latent_attention_bwd(q_bits, kv_bits, routes, scale: float, dout_bits, Dv: int = 512, rows=None):
    """Backward of `latent_attention`: the latent rows are both the keys and (by their
    first Dv dims) the values, so their gradient is the key gradient plus the value
    gradient on those dims. Returns dq [len(rows), Hq, Dqk] and dkv [Tk, 1, Dqk]."""
    dq, dk, dv = attention_bwd(q_bits, kv_bits, kv_bits[:, :, :Dv], routes, scale, dout_bits, rows=rows)
    dkv = dk.astype(np.float64)
    dkv[:, :, :Dv] += dv
    return dq, dkv.astype(np.float32)
