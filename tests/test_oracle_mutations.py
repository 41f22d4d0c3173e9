"""Plant plausible mistakes in the CPU oracle and check that some pin catches each.

Every mutation replaces one oracle function for the duration of a test
(monkeypatch on the oracle module; the oracle looks its helpers up at call time).
"""
import math

import numpy as np
import pytest

import oracle_pins
from oracle import irs_oracle as O


def _select_top_high_ties(scores_f32, kb):
    s = np.asarray(scores_f32, dtype=np.float32).astype(np.float64)
    n = s.shape[0]
    if n <= kb:
        return np.arange(n)
    order = np.lexsort((-np.arange(n), -s))
    return np.sort(order[:kb])


def _select_top_smallest(scores_f32, kb):
    s = np.asarray(scores_f32, dtype=np.float32).astype(np.float64)
    n = s.shape[0]
    if n <= kb:
        return np.arange(n)
    return np.sort(np.lexsort((np.arange(n), s))[:kb])


def _scores_no_relu(qI_t, w_t, kt):
    return (w_t @ (qI_t @ kt.T)).astype(np.float32)


def _scores_no_weight(qI_t, w_t, kt):
    return np.maximum(qI_t @ kt.T, 0.0).sum(axis=0).astype(np.float32)


def _scores_max_heads(qI_t, w_t, kt):
    return (w_t[:, None] * np.maximum(qI_t @ kt.T, 0.0)).max(axis=0).astype(np.float32)


def _expand_no_tail(doc_start, tau, c, budget, selected):
    row = np.full(budget + c - 1, -1, dtype=np.int32)
    slot = 0
    for b in selected:
        for j in range(c):
            row[slot] = doc_start + int(b) * c + j
            slot += 1
    return row


def _expand_tail_shift(doc_start, tau, c, budget, selected):
    row = _expand_no_tail(doc_start, tau, c, budget, selected)
    nv = O.visible_blocks(tau, c)
    for j in range((tau + 1) % c):
        row[budget + j] = doc_start + nv * c + j + 1
    return row


def _expand_global_ids_missing_offset(doc_start, tau, c, budget, selected):
    row = np.full(budget + c - 1, -1, dtype=np.int32)
    slot = 0
    for b in selected:
        for j in range(c):
            row[slot] = int(b) * c + j
            slot += 1
    nv = O.visible_blocks(tau, c)
    for j in range((tau + 1) % c):
        row[budget + j] = nv * c + j
    return row


def _pool_no_div(x, c):
    L, Di = x.shape
    nb = L // c
    acc = np.zeros((nb, Di), np.float32)
    for j in range(c):
        acc = (acc + x[j: nb * c: c]).astype(np.float32)
    return acc


def _pool_strided(x, c):
    L, Di = x.shape
    nb = L // c
    acc = np.zeros((nb, Di), np.float32)
    for j in range(c):
        acc = (acc + x[j * nb:(j + 1) * nb]).astype(np.float32)
    return (acc / np.float32(c)).astype(np.float32)


def _pool_ignores_docs(kI_bits, cu_seqlens, c):
    T = kI_bits.shape[0]
    kbar = O.pool_doc(O.bf16_to_f32(kI_bits), c)
    offs = [0]
    cu = np.asarray(cu_seqlens, np.int64)
    for d in range(cu.shape[0] - 1):
        offs.append(int(cu[d + 1]) // c)
    return kbar, np.asarray(offs, np.int64)


def _round_truncate(x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)


def _attend_no_scale(q_t, K, V, scale, Hkv):
    return _REAL_ATTEND(q_t, K, V, 1.0, Hkv)


def _attend_lse_no_max(q_t, K, V, scale, Hkv):
    out, lse = _REAL_ATTEND(q_t, K, V, scale, Hkv)
    if K.shape[0] == 0:
        return out, lse
    Hq = q_t.shape[0]
    G = Hq // Hkv
    for h in range(Hq):
        s = scale * (K[:, h // G, :] @ q_t[h])
        lse[h] = math.log(np.sum(np.exp(s - np.max(s))))
    return out, lse


def _compose_shifted(routes, cu_seqlens, T, window, rows=None):
    out = _REAL_COMPOSE(routes, cu_seqlens, T, window, rows)
    out[:, :window] = np.where(out[:, :window] >= 0, out[:, :window] - 1, -1)
    return out


def _row_grad_variant(centre=True, dk_scale=True, normalise=True, key_group=None):
    """attend_row_grad with one planted mistake (the flags select which)."""
    def grad(q_t, K, V, scale, Hkv, dO_t):
        Hq, Dqk = q_t.shape
        n = K.shape[0]
        dq = np.zeros((Hq, Dqk))
        dK = np.zeros((n, Hkv, Dqk))
        dV = np.zeros((n, Hkv, V.shape[2]))
        if n == 0:
            return dq, dK, dV
        for h in range(Hq):
            g = h // (Hq // Hkv)
            gk = g if key_group is None else key_group(h, Hq, Hkv)
            s = scale * (K[:, g, :] @ q_t[h])
            e = np.exp(s - np.max(s))
            p = e / np.sum(e)
            dV[:, g, :] += np.outer(p if normalise else e, dO_t[h])
            dp = V[:, g, :] @ dO_t[h]
            ds = p * (dp - np.sum(p * dp)) if centre else p * dp
            dq[h] = scale * (ds @ K[:, g, :])
            dK[:, gk, :] += (scale if dk_scale else 1.0) * np.outer(ds, q_t[h])
        return dq, dK, dV
    return grad


def _bwd_scatter_overwrites(q_bits, k_bits, v_bits, routes, scale, dout_bits, rows=None):
    T, Hq, Dqk = q_bits.shape
    Tk, Hkv, _ = k_bits.shape
    dq = np.zeros((T, Hq, Dqk))
    dk = np.zeros((Tk, Hkv, Dqk))
    dv = np.zeros((Tk, Hkv, v_bits.shape[2]))
    for t in range(T):
        ids = np.asarray(routes[t], np.int64)
        ids = ids[(ids >= 0) & (ids < Tk)]
        gq, gK, gV = O.attend_row_grad(O.bf16_to_f64(q_bits[t]), O.bf16_to_f64(k_bits[ids]),
                                       O.bf16_to_f64(v_bits[ids]), scale, Hkv, O.bf16_to_f64(dout_bits[t]))
        dq[t] = gq
        dk[ids] = gK
        dv[ids] = gV
    return dq.astype(np.float32), dk.astype(np.float32), dv.astype(np.float32)


def _latent_bwd_no_value_grad(q_bits, kv_bits, routes, scale, dout_bits, Dv=512, rows=None):
    dq, dk, _ = O.attention_bwd(q_bits, kv_bits, kv_bits[:, :, :Dv], routes, scale, dout_bits, rows=rows)
    return dq, dk


def _rope_interleaved(x, rope):
    y = np.array(x, dtype=np.float64, copy=True)
    r = np.asarray(rope, dtype=np.float64)
    h = r.shape[-1] // 2
    cos, sin = r[..., :h], r[..., h:2 * h]
    x1 = y[..., 0:2 * h:2].copy()
    x2 = y[..., 1:2 * h:2].copy()
    y[..., 0:2 * h:2] = x1 * cos - x2 * sin
    y[..., 1:2 * h:2] = x2 * cos + x1 * sin
    return y


def _rope_sign_flipped(x, rope):
    r = np.array(rope, dtype=np.float64, copy=True)
    h = r.shape[-1] // 2
    r[..., h:2 * h] *= -1.0
    return _REAL_ROPE(x, r)


def _rms_norm_no_eps(x, weight, eps):
    return _REAL_RMS(x, weight, 0.0)


def _rms_norm_mean_abs(x, weight, eps):
    x = np.asarray(x, dtype=np.float32)
    return (x / (np.mean(np.abs(x), axis=-1, keepdims=True) + np.float32(eps)) * np.asarray(weight, np.float32)
            ).astype(np.float32)


def _block_end_tokens(cu_seqlens, T, c):
    return _REAL_STARTS(cu_seqlens, T, c) + (c - 1)


def _block_starts_without_doc_offset(cu_seqlens, T, c):
    starts, ends = O.doc_bounds(cu_seqlens, T)
    return np.concatenate([c * np.arange((e - s) // c, dtype=np.int64) for s, e in zip(starts, ends)])


def _front_query_without_norm(qI_t_bits, q_weight, eps, rope_t):
    return O.round_to_bf16(O.apply_rope(O.bf16_to_f32(qI_t_bits), rope_t)).astype(np.float64)


def _e4m3_variant(subnormals=True, ties_even=True, mant_bits=3):
    def rnd(x):
        x = np.asarray(x, dtype=np.float64)
        a = np.abs(x)
        _, ex = np.frexp(a)
        e = np.maximum(ex.astype(np.float64) - 1.0, -6.0)
        quantum = np.exp2(e - mant_bits)
        r = np.round(a / quantum) if ties_even else np.floor(a / quantum + 0.5)
        q = np.minimum(r * quantum, 448.0)
        if not subnormals:
            q = np.where(a < 2.0 ** -6, 0.0, q)
        return np.copysign(q, x)
    return rnd


def _grouped_routes_shared_weights(qI_bits, kI_bits, w, cu_seqlens, c, budget, rows=None, operands="bf16"):
    G = qI_bits.shape[1]
    return np.stack([O.index_routes(qI_bits[:, g], kI_bits, np.asarray(w)[:, 0], cu_seqlens, c, budget, rows=rows,
                                    operands=operands) for g in range(G)], axis=1)


def _grouped_routes_first_group(qI_bits, kI_bits, w, cu_seqlens, c, budget, rows=None, operands="bf16"):
    r = O.index_routes(qI_bits[:, 0], kI_bits, np.asarray(w)[:, 0], cu_seqlens, c, budget, rows=rows,
                       operands=operands)
    return np.repeat(r[:, None], qI_bits.shape[1], axis=1)


def _grouped_attention_group0(q_bits, k_bits, v_bits, routes_g, scale, rows=None):
    return _REAL_GROUPED_ATTN(q_bits, k_bits, v_bits, np.repeat(routes_g[:, :1], routes_g.shape[1], axis=1), scale,
                              rows)


def _exp_variant(coef3_div=6, log2e=True):
    def ex(x):
        x = np.asarray(x, dtype=np.float32)
        with np.errstate(over="ignore"):
            t = (x * np.float32(1.0 / math.log(2.0) if log2e else math.log(2.0))).astype(np.float32)
        under = t < -125
        t = np.where(under, np.float32(0.0), t).astype(np.float32)
        n = np.rint(t).astype(np.float32)
        f = (t - n).astype(np.float32)
        cf = [np.float32(math.log(2.0) ** k / math.factorial(k)) for k in range(8)]
        cf[3] = np.float32(math.log(2.0) ** 3 / coef3_div)
        p = np.full_like(f, cf[7])
        for k in range(6, -1, -1):
            p = ((p * f).astype(np.float32) + cf[k]).astype(np.float32)
        return np.where(under, np.float32(0.0), np.ldexp(p, n.astype(np.int32))).astype(np.float32)
    return ex


def _summary_variant(weights="softmax", normalise=True, sign=1.0):
    def summ(k_doc_bits, z_doc_bits, c):
        L, Di = k_doc_bits.shape
        nb = L // c
        k = O.bf16_to_f32(k_doc_bits)[: nb * c].reshape(nb, c, Di).astype(np.float64)
        z = sign * O.bf16_to_f32(z_doc_bits)[: nb * c].reshape(nb, c, Di).astype(np.float64)
        if weights == "mean":
            e = np.ones_like(z)
        elif weights == "over_dims":
            e = np.exp(z - z.max(axis=2, keepdims=True))
            e = e / e.sum(axis=2, keepdims=True) * e.sum(axis=1, keepdims=True)
        else:
            e = np.exp(z - z.max(axis=1, keepdims=True))
        num = (e * k).sum(axis=1)
        return (num / e.sum(axis=1) if normalise else num).astype(np.float32)
    return summ


def _summaries_ignore_docs(kI_bits, z_bits, cu_seqlens, c):
    sm = O.summarize_doc(kI_bits, z_bits, c)
    offs = [0] + [int(v) // c for v in np.asarray(cu_seqlens, np.int64)[1:]]
    return sm, np.asarray(offs, np.int64)


def _summaries_one_rounding(kI_bits, z_bits, cu_seqlens, c):
    sm, offs = O.region_summaries(kI_bits, z_bits, cu_seqlens, c)
    return O.round_to_e4m3(sm.astype(np.float64)), offs


def _round_via_f32(x):
    return O.round_to_bf16(np.asarray(x, np.float64).astype(np.float32)).astype(np.float64)


def _project_variant(keys_first=False, weights_bf16=False):
    def proj(hidden_bits, W_bits, Hi, Di):
        T = hidden_bits.shape[0]
        y = O.bf16_to_f64(hidden_bits) @ O.bf16_to_f64(W_bits).T
        qk = O.f64_to_bf16_bits(O.round_f64_to_bf16(y[:, :(Hi + 1) * Di]))
        if keys_first:
            kI, qI = qk[:, :Di], qk[:, Di:].reshape(T, Hi, Di)
        else:
            qI, kI = qk[:, :Hi * Di].reshape(T, Hi, Di), qk[:, Hi * Di:]
        w = y[:, (Hi + 1) * Di:]
        w = (O.round_f64_to_bf16(w) if weights_bf16 else w).astype(np.float32)
        return np.ascontiguousarray(qI), np.ascontiguousarray(kI), w
    return proj


_REAL_ATTEND = O.attend_row
_REAL_GROUPED_ATTN = O.attention_grouped
_REAL_COMPOSE = O.compose_window
_REAL_ROPE = O.apply_rope
_REAL_RMS = O.rms_norm
_REAL_STARTS = O.block_start_tokens

MUTATIONS = {
    "visibility_off_by_one": ("visible_blocks", lambda tau, c: tau // c),
    "visibility_one_extra": ("visible_blocks", lambda tau, c: (tau + 1) // c + 1 if tau > 0 else 0),
    "ties_to_higher_index": ("select_top", _select_top_high_ties),
    "smallest_instead_of_largest": ("select_top", _select_top_smallest),
    "missing_relu": ("block_scores", _scores_no_relu),
    "missing_head_weights": ("block_scores", _scores_no_weight),
    "max_over_heads": ("block_scores", _scores_max_heads),
    "missing_tail": ("expand_route", _expand_no_tail),
    "tail_shifted": ("expand_route", _expand_tail_shift),
    "local_ids_not_global": ("expand_route", _expand_global_ids_missing_offset),
    "pool_without_division": ("pool_doc", _pool_no_div),
    "pool_wrong_grouping": ("pool_doc", _pool_strided),
    "pool_ignores_documents": ("pool_keys", _pool_ignores_docs),
    "bf16_truncation": ("round_to_bf16", _round_truncate),
    "kv_group_modulo": ("kv_group", lambda h, Hq, Hkv: h % Hkv),
    "scale_ignored": ("attend_row", _attend_no_scale),
    "lse_missing_max": ("attend_row", _attend_lse_no_max),
    "window_shifted": ("compose_window", _compose_shifted),
    "bwd_softmax_not_centred": ("attend_row_grad", _row_grad_variant(centre=False)),
    "bwd_dk_without_scale": ("attend_row_grad", _row_grad_variant(dk_scale=False)),
    "bwd_dv_unnormalised": ("attend_row_grad", _row_grad_variant(normalise=False)),
    "bwd_dk_group_modulo": ("attend_row_grad", _row_grad_variant(key_group=lambda h, Hq, Hkv: h % Hkv)),
    "bwd_scatter_overwrites": ("attention_bwd", _bwd_scatter_overwrites),
    "bwd_latent_drops_value_grad": ("latent_attention_bwd", _latent_bwd_no_value_grad),
    "rope_interleaved_pairs": ("apply_rope", _rope_interleaved),
    "rope_sign_flipped": ("apply_rope", _rope_sign_flipped),
    "rms_norm_without_eps": ("rms_norm", _rms_norm_no_eps),
    "rms_norm_mean_abs": ("rms_norm", _rms_norm_mean_abs),
    "rope_at_block_end": ("block_start_tokens", _block_end_tokens),
    "rope_block_start_without_doc_offset": ("block_start_tokens", _block_starts_without_doc_offset),
    "front_query_without_norm": ("front_query_row", _front_query_without_norm),
    "e4m3_flushes_subnormals": ("round_to_e4m3", _e4m3_variant(subnormals=False)),
    "e4m3_ties_away_from_zero": ("round_to_e4m3", _e4m3_variant(ties_even=False)),
    "e4m3_four_mantissa_bits": ("round_to_e4m3", _e4m3_variant(mant_bits=4)),
    "e4m3_not_applied": ("round_to_e4m3", lambda x: np.asarray(x, dtype=np.float64)),
    "grouped_routes_shared_weights": ("index_routes_grouped", _grouped_routes_shared_weights),
    "grouped_routes_first_group_only": ("index_routes_grouped", _grouped_routes_first_group),
    "grouped_attention_first_group_routes": ("attention_grouped", _grouped_attention_group0),
    "exp_wrong_cubic_term": ("exp_f32", _exp_variant(coef3_div=3)),
    "exp_ln2_for_log2e": ("exp_f32", _exp_variant(log2e=False)),
    "summary_mean_weights": ("summarize_doc", _summary_variant(weights="mean")),
    "summary_softmax_over_dims": ("summarize_doc", _summary_variant(weights="over_dims")),
    "summary_unnormalised": ("summarize_doc", _summary_variant(normalise=False)),
    "summary_negated_logits": ("summarize_doc", _summary_variant(sign=-1.0)),
    "summaries_ignore_documents": ("region_summaries", _summaries_ignore_docs),
    "summaries_one_rounding": ("region_summaries_e4m3", _summaries_one_rounding),
    "bf16_rounding_via_float32": ("round_f64_to_bf16", _round_via_f32),
    "projection_keys_first": ("project_indexer", _project_variant(keys_first=True)),
    "projection_weights_rounded_to_bf16": ("project_indexer", _project_variant(weights_bf16=True)),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(O, attr, fn)
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(O)
        except Exception:
            return
    pytest.fail(f"no pin caught the planted mistake {name!r}")
