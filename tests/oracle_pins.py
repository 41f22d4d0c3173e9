"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each ``pin_*`` takes the oracle module ``O`` and raises ``AssertionError`` when
the oracle disagrees with what the reference pages or mathematics fix:
hand-worked examples from the pages' rules (tests/golden), brute-force
enumeration, closed forms, library routines (torch SDPA, torch's bf16 cast,
numpy's bit packing) and invariants. ``test_oracle_pins`` runs them on the real
oracle; ``test_oracle_mutations`` plants mistakes in the oracle and checks that
some pin fails.
"""
from __future__ import annotations

import itertools
import math
import os
from fractions import Fraction

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------------------
# helpers (no method arithmetic beyond what each pin states)
# --------------------------------------------------------------------------------------


def exact_bf16_bits(values) -> np.ndarray:
    """bf16 bits of values that are exactly representable (fixtures)."""
    x = np.asarray(values, dtype=np.float32)
    bits = x.view(np.uint32)
    assert np.all(bits & np.uint32(0xFFFF) == 0), "fixture value not exact in bf16"
    return (bits >> np.uint32(16)).astype(np.uint16)


def torch_bf16_bits(x_f32: np.ndarray) -> np.ndarray:
    """Library rounding: torch's float32 -> bfloat16 cast (round to nearest even)."""
    t = torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(bits) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).view(
        torch.bfloat16).to(torch.float64).numpy()


def parse_fixture(name: str) -> list[tuple[str, list[str]]]:
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out.append((key, vals))
    return out


def doc_start_of(cu, t):
    cu = list(int(x) for x in cu)
    for d in range(len(cu) - 1):
        if cu[d] <= t < cu[d + 1]:
            return cu[d], cu[d + 1]
    raise AssertionError("token outside documents")


def small_case(seed: int, T: int, Hq: int, Hkv: int, Dqk: int, Dv: int, Hi: int, Di: int,
               doc_lens, w_kind="uniform"):
    import irs_synth

    return irs_synth.custom(T, Hq, Hkv, Dqk, Dv, Hi, Di, c=4, budget=8, doc_lens=doc_lens, seed=seed,
                            w_kind=w_kind)


# --------------------------------------------------------------------------------------
# golden, hand-worked examples
# --------------------------------------------------------------------------------------


def pin_golden_two_docs(O):
    recs = parse_fixture("route_two_docs.txt")
    d = {}
    routes_by_budget = {}
    budget = None
    for key, vals in recs:
        if key == "budget":
            budget = int(vals[0])
            routes_by_budget[budget] = {}
        elif key == "route":
            routes_by_budget[budget][int(vals[0])] = [int(v) for v in vals[1:]]
        else:
            d[key] = vals
    c = int(d["c"][0])
    cu = np.asarray([int(v) for v in d["cu_seqlens"]], dtype=np.int32)
    k0 = [float(v) for v in d["kI0"]]
    k1 = [float(v) for v in d["kI1"]]
    T = len(k0)
    kI = exact_bf16_bits(np.stack([k0, k1], axis=1))
    qI = exact_bf16_bits(np.tile(np.asarray([[[1.0, 0.0]]], np.float32), (T, 1, 1)))
    w = np.ones((T, 1), dtype=np.float32)
    for b, expect in routes_by_budget.items():
        got = O.index_routes(qI, kI, w, cu, c, b)
        for t, row in expect.items():
            assert got[t].tolist() == row, f"budget {b} t {t}: {got[t].tolist()} != {row}"
        assert got.shape == (T, b + c - 1)


def pin_golden_head_weights(O):
    recs = dict((k, v) for k, v in parse_fixture("route_head_weights.txt") if k != "route")
    routes = {int(v[0]): [int(x) for x in v[1:]] for k, v in parse_fixture("route_head_weights.txt")
              if k == "route"}
    c = int(recs["c"][0])
    budget = int(recs["budget"][0])
    cu = np.asarray([int(v) for v in recs["cu_seqlens"]], dtype=np.int32)
    kI = exact_bf16_bits(np.asarray([float(v) for v in recs["kI_rows"]], np.float32).reshape(-1, 2))
    T = kI.shape[0]
    w = np.tile(np.asarray([[float(v) for v in recs["w"]]], np.float32), (T, 1))
    qI = exact_bf16_bits(np.tile(np.asarray([[[1.0, 0.0], [0.0, 1.0]]], np.float32), (T, 1, 1)))
    got, scores = O.index_routes(qI, kI, w, cu, c, budget, want_scores=True)
    for t, row in routes.items():
        assert got[t].tolist() == row, f"t {t}: {got[t].tolist()} != {row}"
    t_s = int(recs["scores_at"][0])
    expect = [float(v) for v in recs["scores_at"][1:]]
    assert scores[t_s, :len(expect)].tolist() == expect


# --------------------------------------------------------------------------------------
# top-k: brute force over all subsets
# --------------------------------------------------------------------------------------


def brute_force_topk(scores, kb):
    """Max-sum subset of size kb; among equal sums the lexicographically smallest sorted tuple."""
    n = len(scores)
    if n <= kb:
        return tuple(range(n))
    best, best_sum = None, None
    for sub in itertools.combinations(range(n), kb):
        s = math.fsum(float(scores[i]) for i in sub)   # exact: few float32 terms
        if best is None or s > best_sum or (s == best_sum and sub < best):
            best, best_sum = sub, s
    return best


def pin_topk_bruteforce(O):
    rng = np.random.default_rng(123)
    for trial in range(200):
        n = int(rng.integers(1, 13))
        kb = int(rng.integers(1, 5))
        if trial % 3 == 0:
            s = rng.choice(np.asarray([0.0, -0.0, 0.5, 1.0, 2.0], np.float32), size=n).astype(np.float32)
        else:
            s = rng.standard_normal(n).astype(np.float32)
        got = tuple(int(x) for x in O.select_top(s, kb))
        assert got == brute_force_topk(s, kb), (s, kb, got)


def pin_routes_from_scores_bruteforce(O):
    """Whole route rows from given scores: blocks = brute-force argmax set, tail per the page."""
    rng = np.random.default_rng(7)
    c, budget = 2, 6          # kb = 3
    cu = np.asarray([0, 13, 24], np.int32)
    T = 24
    ldS = 6
    scores = rng.choice(np.asarray([0.0, 1.0, 2.0, 3.0], np.float32), size=(T, ldS)).astype(np.float32)
    got = O.routes_from_scores(scores, cu, T, c, budget)
    kb = budget // c
    for t in range(T):
        s, _ = doc_start_of(cu, t)
        tau = t - s
        nv = (tau + 1) // c
        blocks = brute_force_topk(scores[t, :nv], kb) if nv > kb else tuple(range(nv))
        expect_ids = sorted(s + b * c + j for b in blocks for j in range(c))
        row = got[t]
        assert row[:len(expect_ids)].tolist() == expect_ids, (t, row)
        assert np.all(row[len(expect_ids):budget] == -1)
        tail = [s + nv * c + j for j in range((tau + 1) % c)]
        assert row[budget:budget + len(tail)].tolist() == tail
        assert np.all(row[budget + len(tail):] == -1)


# --------------------------------------------------------------------------------------
# route invariants on random multi-document inputs
# --------------------------------------------------------------------------------------


def check_route_invariants(routes, cu, c, budget, rows=None):
    T = routes.shape[0] if rows is None else None
    rows = range(routes.shape[0]) if rows is None else rows
    kb = budget // c
    assert routes.shape[1] == budget + c - 1
    for i, t in enumerate(rows):
        row = routes[i]
        s, e = doc_start_of(cu, t)
        tau = t - s
        nv = (tau + 1) // c
        valid = row[row >= 0]
        assert np.all((valid >= s) & (valid <= t)), f"t {t}: route leaves [doc start, t]"
        assert len(set(valid.tolist())) == valid.shape[0], "duplicate IDs"
        assert valid.shape[0] == min(nv, kb) * c + (tau + 1) % c, f"t {t}: valid count"
        blk = row[:budget]
        bv = blk[blk >= 0]
        assert bv.shape[0] == min(nv, kb) * c
        assert np.all(blk[bv.shape[0]:] == -1), "block section not a valid prefix"
        starts = bv[::c]
        assert np.all((starts - s) % c == 0), "block not c-aligned to the document start"
        assert np.all(np.diff(starts) > 0), "blocks not ascending"
        for j in range(c):
            assert np.all(bv[j::c] == starts + j), "block not expanded to c consecutive tokens"
        assert np.all(starts + c - 1 < s + nv * c), "block not complete or not visible"
        tail = row[budget:]
        ntail = (tau + 1) % c
        assert tail[:ntail].tolist() == list(range(s + nv * c, t + 1)), "tail tokens"
        assert np.all(tail[ntail:] == -1)
    return T


def pin_route_invariants(O):
    for seed, lens in ((1, [37, 5, 64, 22]), (2, [128]), (3, [1, 2, 3, 4, 50, 3])):
        T = sum(lens)
        for c, budget in ((4, 8), (4, 16), (1, 3), (3, 9)):
            wl = small_case(seed, T, 2, 1, 8, 8, 3, 8, lens)
            r = O.index_routes(wl.arrays["qI"], wl.arrays["kI"], wl.arrays["w"], wl.cu_seqlens, c, budget)
            check_route_invariants(r, wl.cu_seqlens, c, budget)


def pin_dense_budget_routes(O):
    """budget >= document length: every causal token of the document is routed."""
    lens = [19, 33, 12]
    T = sum(lens)
    wl = small_case(5, T, 2, 1, 8, 8, 2, 8, lens)
    for c in (1, 2, 4):
        budget = 36 if c != 1 else 34
        budget -= budget % c
        r = O.index_routes(wl.arrays["qI"], wl.arrays["kI"], wl.arrays["w"], wl.cu_seqlens, c, budget)
        for t in range(T):
            s, _ = doc_start_of(wl.cu_seqlens, t)
            v = np.sort(r[t][r[t] >= 0])
            assert v.tolist() == list(range(s, t + 1)), (c, t)


# --------------------------------------------------------------------------------------
# block scores: closed forms and symmetries
# --------------------------------------------------------------------------------------


def pin_score_closed_form(O):
    """One-hot index query and weight: score_b = w * ReLU(bf16(mean of block column d0))."""
    rng = np.random.default_rng(11)
    T, Hi, Di, c = 40, 3, 8, 4
    kI_vals = (rng.integers(-64, 64, size=(T, Di)) / 8.0).astype(np.float32)   # block sums exact
    kI = exact_bf16_bits(kI_vals)
    cu = np.asarray([0, 17, 40], np.int32)
    for h0, d0 in ((0, 3), (2, 7), (1, 0)):
        qI_vals = np.zeros((T, Hi, Di), np.float32)
        qI_vals[:, h0, d0] = 1.0
        qI_vals[:, (h0 + 1) % Hi, :] = 0.0
        w = np.zeros((T, Hi), np.float32)
        w[:, h0] = 0.75
        _, sc = O.index_routes(exact_bf16_bits(qI_vals), kI, w, cu, c, 4, want_scores=True)
        for t in range(T):
            s, _ = doc_start_of(cu, t)
            nv = (t - s + 1) // c
            if nv <= 1:
                continue
            for b in range(nv):
                m = sum(Fraction(float(kI_vals[s + b * c + j, d0])) for j in range(c)) / c
                mb = bits_to_f64(torch_bf16_bits(np.asarray([float(m)], np.float32)))[0]
                assert sc[t, b] == np.float32(0.75 * max(mb, 0.0)), (t, b, sc[t, b], mb)


def pin_score_symmetries(O):
    wl = small_case(9, 48, 2, 1, 8, 8, 4, 16, [48])
    qI, kI, w, cu = wl.arrays["qI"], wl.arrays["kI"], wl.arrays["w"], wl.cu_seqlens
    c, budget = 4, 4
    _, s0 = O.index_routes(qI, kI, w, cu, c, budget, want_scores=True)
    # permuting index heads together with their weights leaves scores unchanged
    perm_h = np.asarray([2, 0, 3, 1])
    _, s1 = O.index_routes(qI[:, perm_h], kI, w[:, perm_h], cu, c, budget, want_scores=True)
    np.testing.assert_allclose(s1, s0, rtol=1e-6, atol=0)
    # permuting feature dims of queries and keys together leaves scores unchanged
    perm_d = np.random.default_rng(0).permutation(16)
    _, s2 = O.index_routes(qI[:, :, perm_d], kI[:, perm_d], w, cu, c, budget, want_scores=True)
    np.testing.assert_allclose(s2, s0, rtol=1e-6, atol=0)
    # doubling the weights doubles the scores exactly
    _, s3 = O.index_routes(qI, kI, (w * np.float32(2)).astype(np.float32), cu, c, budget, want_scores=True)
    np.testing.assert_array_equal(s3, s0 * np.float32(2))


def pin_bf16_rounding(O):
    rng = np.random.default_rng(3)
    x = rng.standard_normal(20000).astype(np.float32) * np.float32(10.0)
    # exact ties: low 16 bits == 0x8000, both parities of the last kept bit, both signs
    base = rng.standard_normal(4000).astype(np.float32).view(np.uint32) & np.uint32(0xFFFF0000)
    ties = (base | np.uint32(0x8000)).view(np.float32)
    ties_odd = ((base | np.uint32(0x10000)) | np.uint32(0x8000)).view(np.float32)
    x = np.concatenate([x, ties, ties_odd, -ties])
    got = O.round_to_bf16(x).view(np.uint32) >> np.uint32(16)
    ref = torch_bf16_bits(x).astype(np.uint32)
    np.testing.assert_array_equal(got, ref)


def pin_pool_mean(O):
    rng = np.random.default_rng(5)
    lens = [7, 13, 9]
    T, Di = sum(lens), 6
    cu = np.asarray([0, 7, 20, 29], np.int32)
    vals = rng.standard_normal((T, Di)).astype(np.float32)
    kI = torch_bf16_bits(vals)
    kf = bits_to_f64(kI)
    for c in (1, 2, 3, 4):
        kbar, blk_off = O.pool_keys(kI, cu, c)
        assert blk_off.tolist() == [0] + list(np.cumsum([L // c for L in lens]))
        for d, L in enumerate(lens):
            s = int(cu[d])
            for b in range(L // c):
                got = kbar[blk_off[d] + b]
                exact = [sum(Fraction(float(kf[s + b * c + j, i])) for j in range(c)) / c for i in range(Di)]
                for i in range(Di):
                    e = float(exact[i])
                    mag = float(sum(abs(Fraction(float(kf[s + b * c + j, i]))) for j in range(c)) / c)
                    assert abs(float(got[i]) - e) <= (c + 1) * 2.0 ** -24 * c * mag + 1e-38, (c, d, b, i)
    # a constant group pools exactly to the constant
    kc = exact_bf16_bits(np.full((8, 2), 1.5, np.float32))
    kbar, _ = O.pool_keys(kc, np.asarray([0, 8], np.int32), 4)
    assert np.all(kbar == np.float32(1.5))


def pin_bitmap(O):
    rng = np.random.default_rng(2)
    for n in (1, 31, 32, 33, 100):
        sel = np.sort(rng.choice(n, size=min(n, 7), replace=False))
        words = O.pack_bitmap(sel, n)
        flags = np.zeros(((n + 31) // 32) * 32, np.uint8)
        flags[sel] = 1
        ref = np.packbits(flags, bitorder="little").view(np.uint8)
        ref_words = np.frombuffer(ref.tobytes(), dtype="<u4")
        np.testing.assert_array_equal(words, ref_words)
        np.testing.assert_array_equal(O.unpack_bitmap(words, n), sel)


# --------------------------------------------------------------------------------------
# attention: library routine (torch SDPA) on the same gathered sets, and invariants
# --------------------------------------------------------------------------------------


def sdpa_masked(q_bits, k_bits, v_bits, routes, scale):
    """Reference: dense SDPA over all keys with a boolean mask built from the routes."""
    q = torch.from_numpy(bits_to_f64(q_bits))           # [T, Hq, D]
    k = torch.from_numpy(bits_to_f64(k_bits))           # [Tk, Hkv, D]
    v = torch.from_numpy(bits_to_f64(v_bits))
    T, Hq, _ = q.shape
    Tk, Hkv, _ = k.shape
    G = Hq // Hkv
    allowed = torch.zeros(T, Tk, dtype=torch.bool)
    for t in range(T):
        ids = [int(x) for x in routes[t] if 0 <= int(x) < Tk]
        allowed[t, ids] = True
    kk = k.repeat_interleave(G, dim=1).permute(1, 0, 2)    # [Hq, Tk, D]
    vv = v.repeat_interleave(G, dim=1).permute(1, 0, 2)
    qq = q.permute(1, 0, 2)                                 # [Hq, T, D]
    out = torch.nn.functional.scaled_dot_product_attention(
        qq, kk, vv, attn_mask=allowed.unsqueeze(0), scale=scale)
    scores = (qq @ kk.transpose(1, 2)) * scale
    scores = scores.masked_fill(~allowed.unsqueeze(0), float("-inf"))
    lse = torch.logsumexp(scores, dim=-1)                   # [Hq, T]
    return out.permute(1, 0, 2).numpy(), lse.T.numpy()


def pin_attention_vs_sdpa(O):
    import irs_synth

    for seed, (Hq, Hkv, Dqk, Dv), lens in ((1, (4, 2, 16, 8), [40]), (2, (6, 3, 8, 16), [10, 25, 15]),
                                            (3, (4, 1, 24, 24), [3, 47])):
        T = sum(lens)
        wl = irs_synth.custom(T, Hq, Hkv, Dqk, Dv, 2, 8, 4, 8, doc_lens=lens, seed=seed)
        rng = np.random.default_rng(seed)
        routes = irs_synth.random_routes(rng, T, T, 12, wl.cu_seqlens)
        scale = 0.3
        out, lse = O.attention(wl.arrays["q"], wl.arrays["k"], wl.arrays["v"], routes, scale)
        ref_o, ref_l = sdpa_masked(wl.arrays["q"], wl.arrays["k"], wl.arrays["v"], routes, scale)
        np.testing.assert_allclose(out, ref_o, rtol=1e-5, atol=1e-6)
        np.testing.assert_allclose(lse, ref_l, rtol=1e-5, atol=1e-6)


def pin_dense_causal_attention(O):
    """budget >= document length: indexer routes + attention == dense causal varlen GQA."""
    import irs_synth

    lens = [24, 9, 31]
    T = sum(lens)
    wl = irs_synth.custom(T, 4, 2, 16, 16, 2, 8, 4, 32, doc_lens=lens, seed=4)
    r = O.index_routes(wl.arrays["qI"], wl.arrays["kI"], wl.arrays["w"], wl.cu_seqlens, 4, 32)
    out, lse = O.attention(wl.arrays["q"], wl.arrays["k"], wl.arrays["v"], r, 0.25)
    q = torch.from_numpy(bits_to_f64(wl.arrays["q"]))
    k = torch.from_numpy(bits_to_f64(wl.arrays["k"])).repeat_interleave(2, dim=1)
    v = torch.from_numpy(bits_to_f64(wl.arrays["v"])).repeat_interleave(2, dim=1)
    cu = wl.cu_seqlens
    for d in range(len(lens)):
        s, e = int(cu[d]), int(cu[d + 1])
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[s:e].permute(1, 0, 2), k[s:e].permute(1, 0, 2), v[s:e].permute(1, 0, 2),
            is_causal=True, scale=0.25).permute(1, 0, 2).numpy()
        np.testing.assert_allclose(out[s:e], ref, rtol=1e-5, atol=1e-6)


def pin_attention_invariants(O):
    import irs_synth

    T, Hq, Hkv, D = 24, 4, 2, 16
    wl = irs_synth.custom(T, Hq, Hkv, D, D, 2, 8, 4, 8, seed=8)
    rng = np.random.default_rng(8)
    routes = irs_synth.random_routes(rng, T, T, 10, wl.cu_seqlens)
    q, k, v = wl.arrays["q"], wl.arrays["k"], wl.arrays["v"]
    scale = 1.0 / math.sqrt(D)
    out, lse = O.attention(q, k, v, routes, scale)
    # softmax weights sum to one: all-ones values give all-ones output
    ones = exact_bf16_bits(np.ones_like(bits_to_f64(v), dtype=np.float32))
    o1, _ = O.attention(q, k, ones, routes, scale)
    np.testing.assert_allclose(o1, 1.0, rtol=0, atol=1e-6)
    # moving, adding or removing -1 slots changes nothing
    r2 = np.full((T, 17), -1, np.int32)
    for t in range(T):
        vals = routes[t][routes[t] >= 0]
        slots = np.sort(rng.choice(17, size=vals.shape[0], replace=False))
        r2[t, slots] = vals
    o2, l2 = O.attention(q, k, v, r2, scale)
    np.testing.assert_allclose(o2, out, rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(l2, lse, rtol=1e-6, atol=1e-7)
    # permuting the valid IDs changes nothing
    r3 = routes[:, rng.permutation(routes.shape[1])]
    o3, _ = O.attention(q, k, v, r3, scale)
    np.testing.assert_allclose(o3, out, rtol=1e-6, atol=1e-7)
    # a single valid ID: out is that value row, lse = scale * q . k
    r4 = np.full((T, 5), -1, np.int32)
    r4[:, 3] = np.arange(T) // 2
    o4, l4 = O.attention(q, k, v, r4, scale)
    qf, kf, vf = bits_to_f64(q), bits_to_f64(k), bits_to_f64(v)
    G = Hq // Hkv
    for t in range(T):
        j = t // 2
        for h in range(Hq):
            g = h // G
            np.testing.assert_allclose(o4[t, h], vf[j, g], rtol=0, atol=1e-7)
            np.testing.assert_allclose(l4[t, h], scale * qf[t, h] @ kf[j, g], rtol=1e-6, atol=1e-6)
    # no valid ID at all: zeros and -inf (reading R7)
    r5 = np.full((T, 4), -1, np.int32)
    o5, l5 = O.attention(q, k, v, r5, scale)
    assert np.all(o5 == 0) and np.all(np.isneginf(l5))


def pin_latent_attention(O):
    import irs_synth

    rng = np.random.default_rng(6)
    q = torch_bf16_bits(rng.standard_normal((6, 4, 64)).astype(np.float32))
    kv = torch_bf16_bits(rng.standard_normal((200, 1, 64)).astype(np.float32))
    r = irs_synth.latent_routes(rng, 6, 200, 16)
    out, lse = O.latent_attention(q, kv, r, 0.125, Dv=48)
    ref_o, ref_l = sdpa_masked(q, kv, kv[:, :, :48], r, 0.125)
    np.testing.assert_allclose(out, ref_o, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(lse, ref_l, rtol=1e-5, atol=1e-6)


# --------------------------------------------------------------------------------------
# a7: attention backward
# --------------------------------------------------------------------------------------


def route_mask(routes, T, Tk):
    allowed = torch.zeros(T, Tk, dtype=torch.bool)
    for t in range(T):
        ids = [int(x) for x in routes[t] if 0 <= int(x) < Tk]
        allowed[t, ids] = True
    return allowed


def sdpa_backward(q, k, v, allowed, scale, dout):
    """Library reference: torch autograd through dense SDPA with the route mask.

    q [T, Hq, D], k [Tk, Hkv, D], v [Tk, Hkv, Dv]: float64 tensors that are, or are
    views of, leaves with requires_grad; the KV heads are repeated for their query
    heads, so autograd sums each group's gradient. Backpropagates sum(out * dout).
    """
    G = q.shape[1] // k.shape[1]
    kk = k.repeat_interleave(G, dim=1).permute(1, 0, 2)
    vv = v.repeat_interleave(G, dim=1).permute(1, 0, 2)
    out = torch.nn.functional.scaled_dot_product_attention(
        q.permute(1, 0, 2), kk, vv, attn_mask=allowed.unsqueeze(0), scale=scale)
    (out.permute(1, 0, 2) * dout).sum().backward()


def random_bf16(rng, shape):
    return torch_bf16_bits(rng.standard_normal(shape).astype(np.float32))


def pin_attention_bwd_vs_autograd(O):
    import irs_synth

    for seed, (Hq, Hkv, Dqk, Dv), lens in ((11, (4, 2, 16, 8), [40]), (12, (6, 3, 8, 16), [10, 25, 15]),
                                            (13, (4, 1, 24, 24), [3, 47])):
        T = sum(lens)
        wl = irs_synth.custom(T, Hq, Hkv, Dqk, Dv, 2, 8, 4, 8, doc_lens=lens, seed=seed)
        rng = np.random.default_rng(seed)
        routes = irs_synth.random_routes(rng, T, T, 12, wl.cu_seqlens)
        dout = random_bf16(rng, (T, Hq, Dv))
        scale = 0.3
        dq, dk, dv = O.attention_bwd(wl.arrays["q"], wl.arrays["k"], wl.arrays["v"], routes, scale, dout)
        q = torch.from_numpy(bits_to_f64(wl.arrays["q"])).requires_grad_(True)
        k = torch.from_numpy(bits_to_f64(wl.arrays["k"])).requires_grad_(True)
        v = torch.from_numpy(bits_to_f64(wl.arrays["v"])).requires_grad_(True)
        sdpa_backward(q, k, v, route_mask(routes, T, T), scale, torch.from_numpy(bits_to_f64(dout)))
        np.testing.assert_allclose(dq, q.grad.numpy(), rtol=1e-5, atol=1e-6)
        np.testing.assert_allclose(dk, k.grad.numpy(), rtol=1e-5, atol=1e-6)
        np.testing.assert_allclose(dv, v.grad.numpy(), rtol=1e-5, atol=1e-6)


def pin_latent_attention_bwd(O):
    """The latent rows are one leaf used as keys and, by their first Dv dims, as values."""
    import irs_synth

    rng = np.random.default_rng(16)
    Tq, H, D, Dv, Tk = 6, 4, 64, 48, 200
    q_bits = random_bf16(rng, (Tq, H, D))
    kv_bits = random_bf16(rng, (Tk, 1, D))
    r = irs_synth.latent_routes(rng, Tq, Tk, 16)
    dout = random_bf16(rng, (Tq, H, Dv))
    dq, dkv = O.latent_attention_bwd(q_bits, kv_bits, r, 0.125, dout, Dv=Dv)
    q = torch.from_numpy(bits_to_f64(q_bits)).requires_grad_(True)
    lat = torch.from_numpy(bits_to_f64(kv_bits)).requires_grad_(True)
    sdpa_backward(q, lat, lat[:, :, :Dv], route_mask(r, Tq, Tk), 0.125, torch.from_numpy(bits_to_f64(dout)))
    np.testing.assert_allclose(dq, q.grad.numpy(), rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(dkv, lat.grad.numpy(), rtol=1e-5, atol=1e-6)


def pin_attention_bwd_finite_diff(O):
    """Central differences of the oracle's own forward (pinned to SDPA above) along
    random directions agree with its gradients."""
    rng = np.random.default_rng(17)
    Hq, Hkv, n, D, Dv, scale = 4, 2, 5, 6, 3, 0.7
    q = rng.standard_normal((Hq, D))
    K = rng.standard_normal((n, Hkv, D))
    V = rng.standard_normal((n, Hkv, Dv))
    dO = rng.standard_normal((Hq, Dv))
    gq, gK, gV = O.attend_row_grad(q, K, V, scale, Hkv, dO)

    def f(qq, KK, VV):
        return float(np.sum(O.attend_row(qq, KK, VV, scale, Hkv)[0] * dO))

    eps = 1e-5
    for _ in range(4):
        uq, uK, uV = rng.standard_normal(q.shape), rng.standard_normal(K.shape), rng.standard_normal(V.shape)
        for grad, u, bump in ((gq, uq, lambda e, u=uq: (q + e * u, K, V)),
                              (gK, uK, lambda e, u=uK: (q, K + e * u, V)),
                              (gV, uV, lambda e, u=uV: (q, K, V + e * u))):
            fd = (f(*bump(eps)) - f(*bump(-eps))) / (2 * eps)
            assert abs(fd - float(np.sum(grad * u))) <= 1e-7 * max(1.0, abs(fd)), (fd, float(np.sum(grad * u)))


def pin_attention_bwd_invariants(O):
    import irs_synth

    T, Hq, Hkv, D, Dv = 24, 4, 2, 16, 8
    wl = irs_synth.custom(T, Hq, Hkv, D, Dv, 2, 8, 4, 8, seed=18)
    rng = np.random.default_rng(18)
    routes = irs_synth.random_routes(rng, T, T, 10, wl.cu_seqlens)
    q, k, v = wl.arrays["q"], wl.arrays["k"], wl.arrays["v"]
    dout = random_bf16(rng, (T, Hq, Dv))
    dO = bits_to_f64(dout)
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(D)
    dq, dk, dv = O.attention_bwd(q, k, v, routes, scale, dout)
    # softmax is shift-invariant in the keys: each row's key gradients sum to zero
    tot = dk.astype(np.float64).sum(axis=0)
    assert np.all(np.abs(tot) <= 1e-5 * np.abs(dk).astype(np.float64).sum(axis=0) + 1e-7), tot
    # the weights of a row sum to one: its value gradients add up to the group's dO
    want = dO.reshape(T, Hkv, G, Dv).sum(axis=(0, 2))
    np.testing.assert_allclose(dv.astype(np.float64).sum(axis=0), want, rtol=1e-5, atol=1e-5)
    # moving, adding or removing -1 slots, or permuting the IDs, changes nothing
    r2 = np.full((T, 17), -1, np.int32)
    for t in range(T):
        vals = routes[t][routes[t] >= 0]
        r2[t, np.sort(rng.choice(17, size=vals.shape[0], replace=False))] = rng.permutation(vals)
    for got, ref in zip(O.attention_bwd(q, k, v, r2, scale, dout), (dq, dk, dv)):
        np.testing.assert_allclose(got, ref, rtol=1e-6, atol=1e-7)
    # one key per row: the output is that value row whatever q and k are
    r4 = np.full((T, 5), -1, np.int32)
    r4[:, 2] = np.arange(T) // 2
    dq4, dk4, dv4 = O.attention_bwd(q, k, v, r4, scale, dout)
    assert np.all(dq4 == 0) and np.all(dk4 == 0)
    want4 = np.zeros((T, Hkv, Dv))
    for t in range(T):
        want4[t // 2] += dO[t].reshape(Hkv, G, Dv).sum(axis=1)
    np.testing.assert_allclose(dv4, want4, rtol=1e-6, atol=1e-6)
    # rows without keys have a constant output: no gradient anywhere
    z = O.attention_bwd(q, k, v, np.full((T, 3), -1, np.int32), scale, dout)
    assert all(np.all(x == 0) for x in z)


# --------------------------------------------------------------------------------------
# indexer front half: RMSNorm, RoPE, group start
# --------------------------------------------------------------------------------------


def pin_rms_norm_vs_torch(O):
    """The float32 evaluation against torch's float64 rms_norm of the same float32 inputs:
    within the rounding of a 64-term float32 sum, a square root, a division and a product."""
    rng = np.random.default_rng(31)
    x = rng.standard_normal((5, 3, 64)).astype(np.float32)
    w = rng.uniform(0.5, 1.5, 64).astype(np.float32)
    for eps in (1e-6, 0.1):
        ref = torch.nn.functional.rms_norm(torch.from_numpy(x.astype(np.float64)), (64,),
                                           torch.from_numpy(w.astype(np.float64)), eps).numpy()
        got = O.rms_norm(x, w, eps)
        assert got.dtype == np.float32
        np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-6)


def pin_rope_golden(O):
    recs = parse_fixture("rope_rotate_half.txt")
    assert recs[0][0] == "rope"
    rope = np.asarray([float(v) for v in recs[0][1]])
    pairs = recs[1:]
    assert len(pairs) % 2 == 0 and len(pairs) >= 4
    for (kx, xs), (ko, outs) in zip(pairs[0::2], pairs[1::2]):
        assert kx == "x" and ko == "out"
        got = O.apply_rope(np.asarray([float(v) for v in xs]), rope)
        np.testing.assert_array_equal(got, np.asarray([float(v) for v in outs]))


def pin_rope_rotation(O):
    """Each pair (x_d, x_{d+h}) is the complex number x_d + i x_{d+h} times e^(i theta_d)
    (numpy complex arithmetic); the inverse rotation restores x; dot products of rotated
    vectors depend only on the position difference."""
    rng = np.random.default_rng(32)
    D, Dr = 16, 8
    h = Dr // 2
    x = rng.standard_normal((3, D))
    theta = rng.uniform(-np.pi, np.pi, (3, h))
    rope = np.concatenate([np.cos(theta), np.sin(theta)], axis=-1)
    x = x.astype(np.float32)
    rope = rope.astype(np.float32)
    got = O.apply_rope(x, rope)
    xd, cd, sd = x.astype(np.float64), rope[:, :h].astype(np.float64), rope[:, h:].astype(np.float64)
    z = (xd[:, :h] + 1j * xd[:, h:Dr]) * (cd + 1j * sd)
    np.testing.assert_allclose(got[:, :h], z.real, rtol=0, atol=2e-6)
    np.testing.assert_allclose(got[:, h:Dr], z.imag, rtol=0, atol=2e-6)
    np.testing.assert_array_equal(got[:, Dr:], x[:, Dr:])
    inv = np.concatenate([rope[:, :h], -rope[:, h:]], axis=-1)
    np.testing.assert_allclose(O.apply_rope(got, inv), x, rtol=0, atol=4e-6)
    freq = 1.0 / (10000.0 ** (np.arange(h) / h))

    def table(p):
        return np.concatenate([np.cos(p * freq), np.sin(p * freq)])

    q, k = rng.standard_normal(D), rng.standard_normal(D)
    a = O.apply_rope(q, table(7.0)) @ O.apply_rope(k, table(3.0))
    b = O.apply_rope(q, table(104.0)) @ O.apply_rope(k, table(100.0))
    assert abs(a - b) <= 2e-5 * max(1.0, abs(a)), (a, b)
    # one table row rotates all heads of a token alike
    xh = rng.standard_normal((2, 3, D))
    rows = np.concatenate([np.cos(theta[:2]), np.sin(theta[:2])], axis=-1)
    per_head = O.apply_rope(xh, rows[:, None, :])
    for hd in range(3):
        np.testing.assert_array_equal(per_head[:, hd], O.apply_rope(xh[:, hd], rows))


def pin_front_keys_group_start(O):
    """The rotary values of exactly one token rotate by 90 degrees (cos 0, sin 1): only the
    pooled key whose block starts at that token turns, and by an exact swap with negation."""
    import irs_synth

    T, c, Di = 40, 4, 8
    cu = np.asarray([0, 13, 40], np.int32)
    rng = np.random.default_rng(33)
    kI = irs_synth.f32_to_bf16_bits(rng.standard_normal((T, Di)).astype(np.float32))
    ident = np.tile(np.asarray([1.0, 1.0, 0.0, 0.0]), (T, 1))
    ones = np.ones(Di)
    base, off = O.front_keys(kI, cu, c, ones, 1e-6, ident)
    for tok, doc, blk in ((17, 1, 1), (8, 0, 2)):              # first token of block 1 of doc 1, block 2 of doc 0
        rope = ident.copy()
        rope[tok] = [0.0, 0.0, 1.0, 1.0]
        got, off2 = O.front_keys(kI, cu, c, ones, 1e-6, rope)
        np.testing.assert_array_equal(off2, off)
        row = int(off[doc]) + blk
        want = base.copy()
        want[row, 0], want[row, 1], want[row, 2], want[row, 3] = (-base[row, 2], -base[row, 3], base[row, 0],
                                                                  base[row, 1])
        np.testing.assert_array_equal(got, want)
    # a token that starts no block (the second of a block, or past the last whole block) changes nothing
    for tok in (18, 37, 12):
        rope = ident.copy()
        rope[tok] = [0.0, 0.0, 1.0, 1.0]
        np.testing.assert_array_equal(O.front_keys(kI, cu, c, ones, 1e-6, rope)[0], base)


def pin_front_scores_closed_form(O):
    """Constant keys a and one-hot queries b e_d, unit norm weights, eps 0, identity
    rotary values: every normalised key dim is 1 and each query head becomes
    sign(b) sqrt(Di) e_d, so every block scores sqrt(Di) * sum over heads with b > 0 of w."""
    T, Hi, Di, c, budget = 24, 4, 16, 4, 4
    kI = exact_bf16_bits(np.full((T, Di), 0.5, np.float32))
    qv = np.zeros((T, Hi, Di), np.float32)
    rng = np.random.default_rng(34)
    sign = np.where(rng.random((T, Hi)) < 0.5, -1.0, 1.0)
    for t in range(T):
        for h in range(Hi):
            qv[t, h, (t + 3 * h) % Di] = sign[t, h] * (0.25 * (1 + h))
    qI = exact_bf16_bits(qv)
    w = rng.random((T, Hi), dtype=np.float32)
    front = dict(q_weight=np.ones(Di), k_weight=np.ones(Di), eps=0.0, rope=np.tile([1.0, 0.0], (T, 1)))
    cu = np.asarray([0, T], np.int32)
    _, sc = O.index_routes(qI, kI, w, cu, c, budget, want_scores=True, front=front)
    for t in range(T):
        nv = (t + 1) // c
        if nv <= budget // c:
            continue
        want = np.float32(4.0 * np.sum(w[t].astype(np.float64) * (sign[t] > 0)))
        np.testing.assert_array_equal(sc[t, :nv], np.full(nv, want, np.float32))


# --------------------------------------------------------------------------------------
# Step-5 variants: E4M3 operands, per-KV-group routes
# --------------------------------------------------------------------------------------


def torch_e4m3(x) -> np.ndarray:
    """Library rounding: torch's float32 -> float8_e4m3fn cast (in-range values)."""
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()


def pin_e4m3_vs_torch(O):
    # every finite E4M3 value is its own rounding
    codes = torch.arange(256, dtype=torch.int16).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    codes = codes[np.isfinite(codes)]
    np.testing.assert_array_equal(O.round_to_e4m3(codes), codes)
    # random magnitudes from the subnormals to the top of the range, and exact halfway points
    rng = np.random.default_rng(35)
    x = (rng.standard_normal(20000) * np.exp2(rng.uniform(-12, 8.5, 20000))).astype(np.float32)
    x = x[np.abs(x) <= 448]
    pos = np.sort(codes[codes > 0])
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    for v in (x, mids, -mids):
        np.testing.assert_array_equal(O.round_to_e4m3(v.astype(np.float64)), torch_e4m3(v))


def pin_e4m3_scores(O):
    """Constant keys a and one-hot queries b: the score is w * ReLU(e4m3(b) * e4m3(bf16(a)))
    with torch's casts; bf16 operands give w * ReLU(b * bf16(a))."""
    T, Hi, Di, c, budget = 20, 2, 8, 4, 4
    a = np.float32(0.3)
    kI = torch_bf16_bits(np.full((T, Di), a, np.float32))
    rng = np.random.default_rng(36)
    qv = np.zeros((T, Hi, Di), np.float32)
    bvals = np.asarray([0.71875, -1.3125], np.float32)            # exact in bf16, not in E4M3
    for t in range(T):
        for h in range(Hi):
            qv[t, h, (t + h) % Di] = bvals[h]
    qI = exact_bf16_bits(qv)
    w = rng.random((T, Hi), dtype=np.float32)
    cu = np.asarray([0, T], np.int32)
    abf = bits_to_f64(torch_bf16_bits(np.asarray([a])))[0]
    for operands, qk in (("e4m3", torch_e4m3(bvals) * torch_e4m3(np.asarray([abf]))[0]),
                         ("bf16", bvals.astype(np.float64) * abf)):
        _, sc = O.index_routes(qI, kI, w, cu, c, budget, want_scores=True, operands=operands)
        for t in range(T):
            nv = (t + 1) // c
            if nv <= budget // c:
                continue
            want = np.float32(np.sum(w[t].astype(np.float64) * np.maximum(qk, 0.0)))
            np.testing.assert_array_equal(sc[t, :nv], np.full(nv, want, np.float32))


def pin_grouped_routes(O):
    """Group g has two heads reading key dims g and g + 1 (one-hot queries) with its own
    weights, one of them negative: its blocks are the brute-force top-k of
    w0 ReLU(mean_g) + w1 ReLU(mean_{g+1}). Keys are multiples of 1/4 and the weights
    binary fractions, so means and scores are exact. Identical groups reproduce the
    shared routes."""
    T, G, Di, c, budget = 30, 3, 4, 2, 6
    kb = budget // c
    rng = np.random.default_rng(37)
    kv = rng.integers(-16, 17, size=(T, Di)).astype(np.float32) / 4
    kI = exact_bf16_bits(kv)
    qv = np.zeros((T, G, 2, Di), np.float32)
    for g in range(G):
        qv[:, g, 0, g] = 1.0
        qv[:, g, 1, (g + 1) % Di] = 1.0
    qI = exact_bf16_bits(qv)
    wg = np.asarray([[0.5, 2.0], [1.0, 1.5], [1.5, -1.0]], np.float32)
    w = np.tile(wg[None], (T, 1, 1))
    cu = np.asarray([0, 11, T], np.int32)
    got = O.index_routes_grouped(qI, kI, w, cu, c, budget)
    assert got.shape == (T, G, budget + c - 1)
    for t in range(T):
        s, _ = doc_start_of(cu, t)
        nv = (t - s + 1) // c
        for g in range(G):
            sc = []
            for b in range(nv):
                m = kv[s + b * c: s + b * c + c].astype(np.float64).mean(axis=0)
                sc.append(wg[g, 0] * max(0.0, m[g]) + wg[g, 1] * max(0.0, m[(g + 1) % Di]))
            blocks = brute_force_topk(np.asarray(sc, np.float32), kb) if nv > kb else tuple(range(nv))
            ids = sorted(s + b * c + j for b in blocks for j in range(c))
            assert got[t, g, :len(ids)].tolist() == ids, (t, g)
            assert np.all(got[t, g, len(ids):budget] == -1)
    same = O.index_routes_grouped(np.repeat(qI[:, :1], G, axis=1), kI, np.repeat(w[:, :1], G, axis=1), cu, c, budget)
    shared = O.index_routes(qI[:, 0], kI, w[:, 0], cu, c, budget)
    for g in range(G):
        np.testing.assert_array_equal(same[:, g], shared)


def pin_grouped_attention(O):
    """Per-group routes against SDPA with a per-head mask; identical groups reduce to the
    shared-route attention."""
    import irs_synth

    T, Hq, Hkv, D = 30, 6, 3, 16
    wl = irs_synth.custom(T, Hq, Hkv, D, D, 2, 8, 4, 8, doc_lens=[12, 18], seed=38)
    q, k, v = wl.arrays["q"], wl.arrays["k"], wl.arrays["v"]
    rng = np.random.default_rng(38)
    rg = np.stack([irs_synth.random_routes(rng, T, T, 9, wl.cu_seqlens) for _ in range(Hkv)], axis=1)
    out, lse = O.attention_grouped(q, k, v, rg, 0.25)
    G = Hq // Hkv
    mask = torch.zeros(Hq, T, T, dtype=torch.bool)
    for t in range(T):
        for h in range(Hq):
            ids = [int(x) for x in rg[t, h // G] if 0 <= int(x) < T]
            mask[h, t, ids] = True
    qq = torch.from_numpy(bits_to_f64(q)).permute(1, 0, 2)
    kk = torch.from_numpy(bits_to_f64(k)).repeat_interleave(G, dim=1).permute(1, 0, 2)
    vv = torch.from_numpy(bits_to_f64(v)).repeat_interleave(G, dim=1).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=0.25)
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), rtol=1e-5, atol=1e-6)
    sc = (qq @ kk.transpose(1, 2) * 0.25).masked_fill(~mask, float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(sc, dim=-1).T.numpy(), rtol=1e-5, atol=1e-6)
    r1 = rg[:, 0]
    o1, l1 = O.attention_grouped(q, k, v, np.repeat(r1[:, None], Hkv, axis=1), 0.25)
    o2, l2 = O.attention(q, k, v, r1, 0.25)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def pin_window_compose(O):
    rng = np.random.default_rng(4)
    cu = np.asarray([0, 30, 100], np.int32)
    T, c, budget, window = 100, 4, 16, 8
    import irs_synth

    wl = irs_synth.custom(T, 2, 1, 8, 8, 2, 8, c, budget, doc_lens=[30, 70], seed=4)
    r = O.index_routes(wl.arrays["qI"], wl.arrays["kI"], wl.arrays["w"], cu, c, budget)
    comp = O.compose_window(r, cu, T, window)
    assert comp.shape == (T, window + budget + c - 1)
    for t in range(T):
        s, _ = doc_start_of(cu, t)
        win = comp[t, :window]
        expect = [x if x >= s else -1 for x in range(t - window + 1, t + 1)]
        assert win.tolist() == expect
        allv = comp[t][comp[t] >= 0]
        assert len(set(allv.tolist())) == allv.shape[0], "duplicate after composition"
        assert set(allv.tolist()) == set(x for x in range(max(s, t - window + 1), t + 1)) | set(
            x for x in r[t].tolist() if x >= 0), "union of window and route"
    del rng


def pin_exp_f32(O):
    """exp_f32 against the library exponential: e^0 = 1 exactly; relative error within the
    range reduction's rounding (|t| * 2^-24 twice, scaled by ln 2) plus 8 float32 ulps for the
    polynomial; 0 where e^x < 2^-125 (the stated flush)."""
    assert O.exp_f32(np.float32(0.0)) == np.float32(1.0)
    x = np.concatenate([np.linspace(-86.0, 0.0, 40001), -np.geomspace(1e-7, 1.0, 2001)]).astype(np.float32)
    got = O.exp_f32(x).astype(np.float64)
    ref = np.asarray([math.exp(float(v)) for v in x])
    t = np.abs(x.astype(np.float64)) / math.log(2.0)
    bound = (2.0 * t * 2.0 ** -24 * math.log(2.0) + 8.0 * 2.0 ** -24) * ref
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) / bound))
    far = np.asarray([-88.0, -90.0, -200.0, -3.0e38], np.float32)
    np.testing.assert_array_equal(O.exp_f32(far), np.zeros(4, np.float32))
    assert math.exp(-87.0) < 2.0 ** -125


def _regions_fixture(rng, lens, Di):
    T = sum(lens)
    cu = np.asarray([0] + list(np.cumsum(lens)), np.int32)
    k = torch_bf16_bits(rng.standard_normal((T, Di)).astype(np.float32))
    return T, cu, k


def pin_summaries_uniform_logits(O):
    """Logits equal across a region's tokens give equal softmax weights: the summary is the
    mean of the region's keys (exact rational mean, one rounding; keys on a 2^-4 grid so that
    every FP32 partial sum is exact), then torch's bf16 and E4M3 casts. The pair
    (1.0625, 1.0703125) averages to a bf16 tie that rounds down onto an E4M3 tie: rounding
    twice gives 1.0 where one rounding would give 1.125."""
    rng = np.random.default_rng(40)
    lens, Di = [9, 6, 11], 5
    T = sum(lens)
    cu = np.asarray([0] + list(np.cumsum(lens)), np.int32)
    kv = (np.round(rng.uniform(-6, 6, (T, Di)) * 16) / 16).astype(np.float32)
    kv[0, 0], kv[1, 0] = 1.0625, 1.0703125
    k = exact_bf16_bits(kv)
    for c in (2, 3, 4):
        zr = rng.standard_normal((T // c + len(lens), Di)).astype(np.float32)
        z = np.zeros((T, Di), np.float32)
        starts = [int(v) for v in cu[:-1]]
        ridx = 0
        for s, L in zip(starts, lens):
            for b in range(L // c):
                z[s + b * c: s + b * c + c] = zr[ridx]
                ridx += 1
            z[s + (L // c) * c: s + L] = rng.standard_normal((L % c, Di))   # tails take no part
        sm, offs = O.region_summaries(k, torch_bf16_bits(z), cu, c)
        assert offs.tolist() == [0] + list(np.cumsum([L // c for L in lens]))
        want = []
        for s, L in zip(starts, lens):
            for b in range(L // c):
                want.append([np.float32(sum(Fraction(float(kv[s + b * c + j, i])) for j in range(c)) / c)
                             for i in range(Di)])
        want = np.asarray(want, np.float32)
        np.testing.assert_array_equal(sm, want)
        q, _ = O.region_summaries_e4m3(k, torch_bf16_bits(z), cu, c)
        np.testing.assert_array_equal(q, torch_e4m3(bits_to_f64(torch_bf16_bits(want))))
        if c == 2:
            assert q[0, 0] == 1.0


def pin_summaries_one_hot_logits(O):
    """One token per (region, dim) has logit 0 and the others -200: its softmax weight is 1
    and the others' e^-200 flush to 0, so the summary is that token's key in that dim,
    exactly; E4M3 rounding as torch's cast."""
    rng = np.random.default_rng(41)
    lens, Di, c = [13, 10], 7, 4
    T, cu, k = _regions_fixture(rng, lens, Di)
    kf = bits_to_f64(k)
    z = np.full((T, Di), -200.0, np.float32)
    want = []
    for s, L in zip(cu[:-1], lens):
        for b in range(L // c):
            pick = rng.integers(0, c, Di)
            z[s + b * c + pick, np.arange(Di)] = 0.0
            want.append(kf[s + b * c + pick, np.arange(Di)])
    sm, _ = O.region_summaries(k, exact_bf16_bits(z), cu, c)
    np.testing.assert_array_equal(sm.astype(np.float64), np.asarray(want))
    q, _ = O.region_summaries_e4m3(k, exact_bf16_bits(z), cu, c)
    np.testing.assert_array_equal(q, torch_e4m3(np.asarray(want, np.float32)))


def pin_summaries_softmax_fp64(O):
    """Random logits against the softmax-weighted sum in float64 (library exp): agreement
    within the FP32 evaluation's error, |x| * 2^-22 relative for the weights plus c + 2 ulps
    of the sums; tokens of a document's last incomplete region change nothing."""
    rng = np.random.default_rng(42)
    lens, Di = [11, 5, 14], 6
    T, cu, k = _regions_fixture(rng, lens, Di)
    kf = bits_to_f64(k)
    z = torch_bf16_bits((rng.standard_normal((T, Di)) * 3).astype(np.float32))
    zf = bits_to_f64(z)
    for c in (2, 5):
        sm, offs = O.region_summaries(k, z, cu, c)
        r = 0
        for s, L in zip(cu[:-1], lens):
            for b in range(L // c):
                zz = zf[s + b * c: s + b * c + c]
                kk = kf[s + b * c: s + b * c + c]
                x = zz - zz.max(axis=0)
                p = np.exp(x) / np.exp(x).sum(axis=0)
                ref = (p * kk).sum(axis=0)
                mag = (p * np.abs(kk)).sum(axis=0)
                tol = mag * (np.abs(x).max(axis=0) * 2.0 ** -22 + (c + 2) * 2.0 ** -23) + 1e-30
                assert np.all(np.abs(sm[r].astype(np.float64) - ref) <= tol), (c, r)
                r += 1
        assert r == sm.shape[0]
        # the incomplete tail of every document takes no part
        k2, z2 = k.copy(), z.copy()
        for s, L in zip(cu[:-1], lens):
            tail = slice(int(s) + (L // c) * c, int(s) + L)
            k2[tail] ^= np.uint16(0x1234)
            z2[tail] ^= np.uint16(0x0101)
        np.testing.assert_array_equal(O.region_summaries(k2, z2, cu, c)[0], sm)


def pin_summaries_two_tokens(O):
    """c = 2 with logits (0, -a): the summary is (k0 + e^-a k1) / (1 + e^-a)."""
    rng = np.random.default_rng(43)
    T, Di, c = 16, 8, 2
    cu = np.asarray([0, T], np.int32)
    k = torch_bf16_bits(rng.standard_normal((T, Di)).astype(np.float32))
    kf = bits_to_f64(k)
    a = bits_to_f64(torch_bf16_bits(rng.uniform(0.0, 4.0, (T // 2, Di)).astype(np.float32)))
    z = np.zeros((T, Di), np.float32)
    z[1::2] = -a
    sm, _ = O.region_summaries(k, exact_bf16_bits(z), cu, c)
    e = np.exp(-a)
    ref = (kf[0::2] + e * kf[1::2]) / (1.0 + e)
    tol = (np.abs(kf[0::2]) + np.abs(kf[1::2])) * 2.0 ** -20
    assert np.all(np.abs(sm.astype(np.float64) - ref) <= tol)


def pin_summary_scores(O):
    """One-hot queries read dim d of the summaries; one-hot logits make the summary of block
    b in dim d the key of one chosen token: each score is then sum_h w_h ReLU(b_h e4m3(k)) with
    torch's casts, rounded once to FP32 (bf16 queries; E4M3 queries round b_h too)."""
    rng = np.random.default_rng(44)
    lens, Hi, Di, c, budget = [14, 18], 2, 8, 2, 2
    T, cu, k = _regions_fixture(rng, lens, Di)
    kf = bits_to_f64(k)
    z = np.full((T, Di), -200.0, np.float32)
    pick = rng.integers(0, c, (T // c + 2, Di))
    chosen = {}
    r = 0
    for s, L in zip(cu[:-1], lens):
        for b in range(L // c):
            z[s + b * c + pick[r], np.arange(Di)] = 0.0
            chosen[(int(s), b)] = kf[s + b * c + pick[r], np.arange(Di)]
            r += 1
    bvals = np.asarray([0.71875, -1.3125], np.float32)
    qv = np.zeros((T, Hi, Di), np.float32)
    dims = rng.integers(0, Di, (T, Hi))
    for t in range(T):
        for h in range(Hi):
            qv[t, h, dims[t, h]] = bvals[h]
    qI = exact_bf16_bits(qv)
    w = rng.standard_normal((T, Hi)).astype(np.float32)
    for operands in ("bf16", "e4m3"):
        bq = torch_e4m3(bvals) if operands == "e4m3" else bvals.astype(np.float64)
        _, sc = O.index_routes(qI, k, w, cu, c, budget, want_scores=True, operands=operands,
                               logits=exact_bf16_bits(z))
        for t in range(T):
            d = int(np.searchsorted(cu, t, side="right") - 1)
            s = int(cu[d])
            nv = (t - s + 1) // c
            if nv <= budget // c:
                continue
            for b in range(nv):
                kk = torch_e4m3(chosen[(s, b)].astype(np.float32))
                want = np.float32(sum(float(w[t, h]) * max(bq[h] * kk[dims[t, h]], 0.0) for h in range(Hi)))
                assert sc[t, b] == want, (operands, t, b)


def pin_round_f64_to_bf16(O):
    """Direct float64 -> bf16 rounding: equals torch's cast on values exact in float32 (where
    no double rounding can occur), and the hand-worked cases where float64 bits below float32
    precision decide a tie (1 + 2^-8 is a tie, rounded to even 1.0; 1 + 2^-8 + 2^-40 is
    above it, 1 + 2^-7)."""
    rng = np.random.default_rng(50)
    x = (rng.standard_normal(20000) * np.exp2(rng.uniform(-20, 20, 20000))).astype(np.float32).astype(np.float64)
    ties = (np.arange(0, 128, dtype=np.float64) * 2.0 + 1.0) * 2.0 ** -8 + 1.0   # 1 + odd * 2^-8: halfway cases
    for v in (x, ties[ties < 2.0], -ties[ties < 2.0]):
        want = torch.from_numpy(v).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
        np.testing.assert_array_equal(O.round_f64_to_bf16(v), want)
    cases = {1.0 + 2.0 ** -8: 1.0, 1.0 + 2.0 ** -8 + 2.0 ** -40: 1.0 + 2.0 ** -7,
             1.0 + 3 * 2.0 ** -8 - 2.0 ** -40: 1.0 + 2.0 ** -7, -(2.0 + 2.0 ** -7 + 2.0 ** -45): -(2.0 + 2.0 ** -6)}
    for v, want in cases.items():
        assert O.round_f64_to_bf16(np.asarray([v]))[0] == want, (v, want)


def _projection_fixture(Hi=3, Di=8, H=16, T=12, seed=51):
    rng = np.random.default_rng(seed)
    N = (Hi + 1) * Di + Hi
    # weights: small integers times 2^-3 (exact in bf16); row n gets a value that encodes n
    Wv = (rng.integers(-8, 9, (N, H)) / 8.0).astype(np.float32)
    return rng, T, H, Hi, Di, N, Wv


def pin_projection_one_hot(O):
    """One-hot hidden rows pick one column of W: qI[t, h, d] = W[h*Di + d, j], kI[t, d] =
    W[Hi*Di + d, j], w[t, h] = W[(Hi+1)*Di + h, j], all exact (head-major queries, then keys,
    then head weights)."""
    rng, T, H, Hi, Di, N, Wv = _projection_fixture()
    j = rng.integers(0, H, T)
    hid = np.zeros((T, H), np.float32)
    hid[np.arange(T), j] = 1.0
    qI, kI, w = O.project_indexer(exact_bf16_bits(hid), exact_bf16_bits(Wv), Hi, Di)
    for t in range(T):
        col = Wv[:, j[t]]
        np.testing.assert_array_equal(bits_to_f64(qI[t]), col[:Hi * Di].reshape(Hi, Di).astype(np.float64))
        np.testing.assert_array_equal(bits_to_f64(kI[t]), col[Hi * Di:(Hi + 1) * Di].astype(np.float64))
        np.testing.assert_array_equal(w[t], col[(Hi + 1) * Di:])


def pin_projection_sums(O):
    """Two-hot hidden rows (a at column i, b at column j, exact in bf16): every output is
    a*W[n, i] + b*W[n, j], computed here in exact rationals; queries and keys are that sum
    rounded once to bf16 (torch's cast of the exact value, which these sums keep exact in
    float32), head weights the sum itself."""
    rng, T, H, Hi, Di, N, Wv = _projection_fixture(seed=52)
    hid = np.zeros((T, H), np.float32)
    ii = rng.integers(0, H // 2, T)
    jj = rng.integers(H // 2, H, T)
    av = np.asarray([1.0, -1.5, 0.375, 3.0], np.float32)[rng.integers(0, 4, T)]
    bv = np.asarray([1.0, 2.5, -0.75, 0.0078125], np.float32)[rng.integers(0, 4, T)]
    hid[np.arange(T), ii] = av
    hid[np.arange(T), jj] = bv
    qI, kI, w = O.project_indexer(exact_bf16_bits(hid), exact_bf16_bits(Wv), Hi, Di)
    for t in range(T):
        exact = [Fraction(float(av[t])) * Fraction(float(Wv[n, ii[t]])) + Fraction(float(bv[t])) * Fraction(float(Wv[n, jj[t]]))
                 for n in range(N)]
        ex = np.asarray([float(e) for e in exact])
        qk = torch.from_numpy(ex[:(Hi + 1) * Di].astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
        np.testing.assert_array_equal(bits_to_f64(qI[t]).ravel(), qk[:Hi * Di])
        np.testing.assert_array_equal(bits_to_f64(kI[t]), qk[Hi * Di:])
        np.testing.assert_array_equal(w[t].astype(np.float64), ex[(Hi + 1) * Di:])


ALL_PINS = [
    pin_golden_two_docs,
    pin_golden_head_weights,
    pin_topk_bruteforce,
    pin_routes_from_scores_bruteforce,
    pin_route_invariants,
    pin_dense_budget_routes,
    pin_score_closed_form,
    pin_score_symmetries,
    pin_bf16_rounding,
    pin_pool_mean,
    pin_bitmap,
    pin_attention_vs_sdpa,
    pin_dense_causal_attention,
    pin_attention_invariants,
    pin_latent_attention,
    pin_window_compose,
    pin_attention_bwd_vs_autograd,
    pin_latent_attention_bwd,
    pin_attention_bwd_finite_diff,
    pin_attention_bwd_invariants,
    pin_rms_norm_vs_torch,
    pin_rope_golden,
    pin_rope_rotation,
    pin_front_keys_group_start,
    pin_front_scores_closed_form,
    pin_e4m3_vs_torch,
    pin_e4m3_scores,
    pin_grouped_routes,
    pin_grouped_attention,
    pin_exp_f32,
    pin_summaries_uniform_logits,
    pin_summaries_one_hot_logits,
    pin_summaries_softmax_fp64,
    pin_summaries_two_tokens,
    pin_summary_scores,
    pin_round_f64_to_bf16,
    pin_projection_one_hot,
    pin_projection_sums,
]
