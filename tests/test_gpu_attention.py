"""Sparse attention on the GPU (through the C ABI) against the CPU oracle."""
import math

import numpy as np
import pytest
import torch

import irs_synth
import parity
from oracle import irs_oracle as O

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module")
def irs():
    import indexer_routed_sparse_gb300 as m

    m.lib()
    return m


def attend(irs, q, k, v, routes, scale):
    qd = torch.from_numpy(q).view(torch.bfloat16).to(DEV) if isinstance(q, np.ndarray) else q
    kd = torch.from_numpy(k).view(torch.bfloat16).to(DEV) if isinstance(k, np.ndarray) else k
    vd = torch.from_numpy(v).view(torch.bfloat16).to(DEV) if isinstance(v, np.ndarray) else v
    rd = torch.from_numpy(np.ascontiguousarray(routes)).to(DEV)
    out, lse = irs.sparse_gqa_attn_fwd(qd, kd, vd, rd, scale)
    irs.check_device_errors(DEV)
    return out, lse


def test_tiny_with_oracle_routes_all_rows(irs):
    wl = irs_synth.make("tiny")
    a = wl.arrays
    routes = O.index_routes(a["qI"], a["kI"], a["w"], wl.cu_seqlens, wl.c, wl.budget)
    out, lse = attend(irs, a["q"], a["k"], a["v"], routes, wl.scale)
    ref_o, ref_l = O.attention(a["q"], a["k"], a["v"], routes, wl.scale)
    parity.check_attention(out, lse, ref_o, ref_l, np.arange(wl.T))


@pytest.mark.parametrize("name", ["mid", "packed", "windowed"])
def test_full_size_sampled_rows(irs, name):
    wl = irs_synth.make(name)
    a = wl.arrays
    rows = parity.sample_rows(wl, 192, seed=2)
    W = wl.route_width
    routes = parity.window_like_routes(wl.T, wl.Tk, W, wl.cu_seqlens)
    rng = np.random.default_rng(7)
    sub = irs_synth.random_routes(rng, wl.T, wl.Tk, W, wl.cu_seqlens, frac_invalid=0.1) if wl.T <= 2048 else None
    if sub is None:
        # random document-confined routes for the sampled rows only
        cu = np.asarray(wl.cu_seqlens, np.int64)
        for t in rows:
            s = int(cu[np.searchsorted(cu, t, side="right") - 1])
            n_av = int(t) - s + 1
            n = min(W, n_av)
            ids = s + rng.choice(n_av, size=n, replace=False)
            row = np.full(W, -1, np.int32)
            row[rng.permutation(W)[:n]] = ids
            routes[t] = row
    else:
        routes = sub
    out, lse = attend(irs, a["q"], a["k"], a["v"], routes, wl.scale)
    ref_o, ref_l = O.attention(a["q"], a["k"], a["v"], routes, wl.scale, rows=rows)
    parity.check_attention(out, lse, ref_o, ref_l, rows)


def test_latent_full_size_sampled_rows(irs):
    wl = irs_synth.make("latent")
    a = wl.arrays
    rows = parity.sample_rows(wl, 96, seed=3)
    kv = torch.from_numpy(a["kv"]).view(torch.bfloat16).to(DEV)
    q = torch.from_numpy(a["q"]).view(torch.bfloat16).to(DEV)
    out, lse = attend(irs, q, kv, kv[:, :, :512], a["route"], wl.scale)
    ref_o, ref_l = O.latent_attention(a["q"], a["kv"], a["route"], wl.scale, Dv=512, rows=rows)
    parity.check_attention(out, lse, ref_o, ref_l, rows)


def test_latent_small_all_rows(irs):
    wl = irs_synth.make("latent", small=True)
    a = wl.arrays
    kv = torch.from_numpy(a["kv"]).view(torch.bfloat16).to(DEV)
    q = torch.from_numpy(a["q"]).view(torch.bfloat16).to(DEV)
    out, lse = attend(irs, q, kv, kv[:, :, :512], a["route"], wl.scale)
    rows = np.arange(0, wl.T, 7)
    ref_o, ref_l = O.latent_attention(a["q"], a["kv"], a["route"], wl.scale, Dv=512, rows=rows)
    parity.check_attention(out, lse, ref_o, ref_l, rows)


@pytest.mark.parametrize("Hq,Dqk,Dv,W,holes,boost", [
    (64, 576, 512, 300, True, 1.0),     # one 64-head block, -1 holes, rows without keys
    (128, 192, 128, 129, False, 1.0),   # narrow latent rows, W one past two 64-key chunks
    (128, 576, 256, 700, True, 1.0),    # two dv blocks
    (64, 576, 512, 600, False, 12.0),   # later keys' non-value dims 12x larger: maxima move, O is rescaled
])
def test_latent_kernel_shapes(irs, Hq, Dqk, Dv, W, holes, boost):
    """One latent KV head whose rows are the keys and, by their first Dv dims, the values."""
    T, Tk = 96, 1200
    rng = np.random.default_rng(Hq * 7 + W)
    q = irs_synth.f32_to_bf16_bits(rng.standard_normal((T, Hq, Dqk), dtype=np.float32))
    kvf = rng.standard_normal((Tk, 1, Dqk), dtype=np.float32)
    kvf[Tk // 2:, :, Dv:] *= boost   # scores grow along the route; values keep their scale
    kv = irs_synth.f32_to_bf16_bits(kvf)
    routes = np.full((T, W), -1, np.int32)
    for t in range(T):
        if t % 17 == 5:
            continue                                   # a row without any valid slot
        n = int(rng.integers(1, W + 1))
        ids = np.sort(rng.choice(Tk, size=n, replace=False)).astype(np.int32)
        slots = np.sort(rng.permutation(W)[:n]) if holes else np.arange(n)
        routes[t, slots] = ids
    kvd = torch.from_numpy(kv).view(torch.bfloat16).to(DEV)
    scale = 1.0 / math.sqrt(Dqk)
    out, lse = attend(irs, q, kvd, kvd[:, :, :Dv], routes, scale)
    ref_o, ref_l = O.latent_attention(q, kv, routes, scale, Dv=Dv)
    parity.check_attention(out, lse, ref_o, ref_l, np.arange(T))
    assert torch.all(out[5] == 0) and torch.all(torch.isneginf(lse[5]))


@pytest.mark.parametrize("Hq,Hkv,Dqk,Dv,alias,Tk", [
    (8, 2, 192, 128, False, 98304),    # separate value rows, Dqk != Dv (126 MB of K/V)
    (8, 2, 128, 128, False, 98304),    # K and V gathered in one pass where copied (100 MB)
    (4, 1, 256, 128, True, 196608),    # values are the first Dv dims of the key rows (100 MB)
])
def test_consecutive_runs_and_copies(irs, Hq, Hkv, Dqk, Dv, alias, Tk):
    """Routes mixing 64-key runs of consecutive tokens with scattered keys: each 128-key
    chunk has both halves runs, one or the other, or none, plus a partial last chunk and -1
    holes between runs. The K/V sets exceed half the L2, which selects the attention
    variant that loads runs as TMA row tiles (the others by 16-byte copies)."""
    T, W = 40, 700
    rng = np.random.default_rng(Dqk + Tk)
    q = irs_synth.f32_to_bf16_bits(rng.standard_normal((T, Hq, Dqk), dtype=np.float32))
    k = irs_synth.f32_to_bf16_bits(rng.standard_normal((Tk, Hkv, Dqk), dtype=np.float32))
    v = None if alias else irs_synth.f32_to_bf16_bits(rng.standard_normal((Tk, Hkv, Dv), dtype=np.float32))
    routes = np.full((T, W), -1, np.int32)
    for t in range(T):
        pieces = []
        for half in range(10):
            kind = (t + half) % 4
            if kind == 3:
                continue
            if kind < 2:                                    # a run of 64 consecutive tokens
                start = int(rng.integers(0, Tk - 64))
                pieces.append(np.arange(start, start + 64))
            else:                                           # 64 scattered tokens
                pieces.append(rng.choice(Tk, 64, replace=False))
        ids = np.concatenate(pieces + [rng.choice(Tk, t % 37, replace=False)])
        _, first = np.unique(ids, return_index=True)        # distinct IDs, first occurrence order
        ids = ids[np.sort(first)][:W - 20]
        slots = np.arange(len(ids)) + np.minimum(np.arange(len(ids)) // 200, 20)   # a few holes
        routes[t, slots] = ids.astype(np.int32)
    scale = 1.0 / math.sqrt(Dqk)
    kd = torch.from_numpy(k).view(torch.bfloat16).to(DEV)
    if alias:
        out, lse = attend(irs, q, kd, kd[:, :, :Dv], routes, scale)
        ref_o, ref_l = O.attention(q, k, k[:, :, :Dv], routes, scale)
    else:
        out, lse = attend(irs, q, kd, v, routes, scale)
        ref_o, ref_l = O.attention(q, k, v, routes, scale)
    parity.check_attention(out, lse, ref_o, ref_l, np.arange(T))


@pytest.mark.parametrize("Hq,Hkv,Dqk,Dv,W", [
    (4, 4, 64, 128, 1),        # G = 1, a single slot
    (32, 1, 128, 128, 300),    # G = 32: two head blocks per KV head
    (8, 2, 192, 256, 129),     # Dqk != Dv, two dv blocks, W one past a chunk
    (6, 2, 128, 128, 4096),    # G = 3 (padded), widest route
    (16, 16, 384, 256, 64),    # wide head dims without aliasing (one smem stage)
])
def test_shapes(irs, Hq, Hkv, Dqk, Dv, W):
    T = 200
    wl = irs_synth.custom(T, Hq, Hkv, Dqk, Dv, 2, 64, 4, 8, doc_lens=[70, 130], seed=Hq + W)
    a = wl.arrays
    rng = np.random.default_rng(W)
    routes = irs_synth.random_routes(rng, T, T, W, wl.cu_seqlens, frac_invalid=0.2)
    scale = 1.0 / math.sqrt(Dqk)
    out, lse = attend(irs, a["q"], a["k"], a["v"], routes, scale)
    ref_o, ref_l = O.attention(a["q"], a["k"], a["v"], routes, scale)
    parity.check_attention(out, lse, ref_o, ref_l, np.arange(T))


def test_empty_rows_and_out_of_range_ids(irs):
    T = 64
    wl = irs_synth.custom(T, 4, 2, 128, 128, 2, 64, 4, 8, seed=9)
    a = wl.arrays
    routes = np.full((T, 20), -1, np.int32)
    routes[1::2, 3] = np.arange(1, T, 2)                   # one key on odd rows, none on even rows
    routes[5, 7] = 10 * T                                  # out of range: padding + device flag
    routes[9, 0] = -7                                      # negative but not -1: padding + flag
    qd = torch.from_numpy(a["q"]).view(torch.bfloat16).to(DEV)
    kd = torch.from_numpy(a["k"]).view(torch.bfloat16).to(DEV)
    vd = torch.from_numpy(a["v"]).view(torch.bfloat16).to(DEV)
    irs.read_device_errors(DEV)
    out, lse = irs.sparse_gqa_attn_fwd(qd, kd, vd, torch.from_numpy(routes).to(DEV), wl.scale)
    assert irs.read_device_errors(DEV) & irs.DEVERR_ROUTE_ID
    ref_o, ref_l = O.attention(a["q"], a["k"], a["v"], routes, wl.scale)
    parity.check_attention(out, lse, ref_o, ref_l, np.arange(T))
    assert torch.all(out[0::2] == 0) and torch.all(torch.isneginf(lse[0::2]))


def test_strided_query_view(irs):
    T, Hq, Hkv, D = 96, 8, 2, 128
    wl = irs_synth.custom(T, Hq, Hkv, D, D, 2, 64, 4, 8, seed=4)
    a = wl.arrays
    big = torch.zeros(T, Hq + 3, D + 64, dtype=torch.bfloat16, device=DEV)
    big[:, 1:Hq + 1, 32:32 + D] = torch.from_numpy(a["q"]).view(torch.bfloat16).to(DEV)
    qv = big[:, 1:Hq + 1, 32:32 + D]
    rng = np.random.default_rng(1)
    routes = irs_synth.random_routes(rng, T, T, 50, wl.cu_seqlens)
    kd = torch.from_numpy(a["k"]).view(torch.bfloat16).to(DEV)
    vd = torch.from_numpy(a["v"]).view(torch.bfloat16).to(DEV)
    out, lse = irs.sparse_gqa_attn_fwd(qv, kd, vd, torch.from_numpy(routes).to(DEV), wl.scale)
    ref_o, ref_l = O.attention(a["q"], a["k"], a["v"], routes, wl.scale)
    parity.check_attention(out, lse, ref_o, ref_l, np.arange(T))


@pytest.mark.parametrize("name,nrows", [("mid", 128), ("packed", 256), ("windowed", 256)])
def test_end_to_end(irs, name, nrows):
    """Indexer -> (sliding window) -> attention, all on the GPU at full size.

    The oracle computes its own routes and attention for sampled rows (document starts
    and ends, tau in 0..c, the sparse boundary, random rows). Every sampled route row must
    equal the oracle's or differ only at an oracle near-tie of the kb-th score. Attention
    is then checked on every sampled row against the oracle's attention over the oracle's
    routes: the GPU attention runs again on a route tensor whose sampled rows are the
    oracle's, and rows whose routes already agreed must give bit-identical output in both
    GPU calls. On the windowed workload the attention kernel adds the 512-token window
    itself (the oracle composes it into the route), and the sampled rows are the real
    window-plus-64-token-block rows (Hq 64, Hkv 4, Dqk 192, Dv 128), whose K/V exceed half
    the L2, so they take the TMA row-tile path."""
    wl = irs_synth.make(name)
    a = wl.arrays
    t = irs_synth.as_torch(wl, device=DEV)
    route_idx = irs.sparse_index_score_topk(t["qI"], t["kI"], t["w"], t["cu_seqlens"], wl.c, wl.budget,
                                            max_doc_len=wl.max_doc_len)
    # the windowed workload attends its window in the attention kernel (no composed route)
    route = route_idx
    win = dict(window=wl.window, cu_seqlens=t["cu_seqlens"]) if wl.window else {}
    out, lse = irs.sparse_gqa_attn_fwd(t["q"], t["k"], t["v"], route, wl.scale, **win)
    irs.check_device_errors(DEV)
    rows = parity.sample_rows(wl, nrows, seed=5)
    idx = torch.as_tensor(rows, device=DEV)
    ldS = max(1, wl.max_doc_len // wl.c)
    ref_ri, ref_s = O.index_routes(a["qI"], a["kI"], a["w"], wl.cu_seqlens, wl.c, wl.budget, rows=rows,
                                   want_scores=True, ldS=ldS)
    g_ri = route_idx[idx].cpu().numpy()
    parity.check_routes_e2e(g_ri, ref_ri, ref_s, wl, rows)
    same = np.all(g_ri == ref_ri, axis=1)
    assert same.mean() >= 0.9, f"only {same.mean():.2%} of the sampled route rows agree"
    if wl.window:
        full_ri = np.full((wl.T, ref_ri.shape[1]), -1, np.int32)
        full_ri[rows] = ref_ri
        ref_r = O.compose_window(full_ri, wl.cu_seqlens, wl.T, wl.window, rows=rows)
    else:
        ref_r = ref_ri
    full = np.full((wl.T, ref_r.shape[1]), -1, np.int32)
    full[rows] = ref_r
    ref_o, ref_l = O.attention(a["q"], a["k"], a["v"], full, wl.scale, rows=rows)
    route2 = route.clone()
    route2[idx] = torch.from_numpy(ref_ri).to(DEV)
    out2, lse2 = irs.sparse_gqa_attn_fwd(t["q"], t["k"], t["v"], route2, wl.scale, **win)
    irs.check_device_errors(DEV)
    same_idx = torch.as_tensor(rows[same], device=DEV)
    assert torch.equal(out[same_idx], out2[same_idx]) and torch.equal(lse[same_idx], lse2[same_idx])
    parity.check_attention(out2, lse2, ref_o, ref_l, rows)


@pytest.mark.parametrize("case", ["windowed_small", "multi_doc", "window_wider_than_route", "g1_dv256",
                                  "g16_d192_docs"])
def test_window_in_the_kernel_equals_composed_route(irs, case):
    """The windowed attention entry point against composing the window into the route and
    attending that: the same keys in the same order, so the outputs agree bit for bit; and
    both against the oracle on sampled rows. The shapes cover ragged tails, windows that
    start at document starts (a one-token document included), G = 1, 4 and 16, Dqk 64 to
    192, Dv = 256 and a window wider than the route."""
    if case == "windowed_small":
        wl = irs_synth.make("windowed", small=True)
        a = wl.arrays
        t = irs_synth.as_torch(wl, device=DEV)
        route = irs.sparse_index_score_topk(t["qI"], t["kI"], t["w"], t["cu_seqlens"], wl.c, wl.budget,
                                            max_doc_len=wl.max_doc_len)
        window, cu, scale = wl.window, t["cu_seqlens"], wl.scale
        q, k, v = t["q"], t["k"], t["v"]
        cu_h = wl.cu_seqlens
    else:
        shapes = {  # T, Hq, Hkv, Dqk, Dv, doc lengths, route width, window
            "multi_doc": (700, 8, 2, 128, 128, [5, 300, 395], 40, 64),
            "window_wider_than_route": (700, 8, 2, 128, 128, [700], 7, 200),
            "g1_dv256": (300, 2, 2, 64, 256, [170, 130], 24, 100),
            "g16_d192_docs": (400, 32, 2, 192, 128, [90, 1, 309], 30, 130),
        }
        T, Hq, Hkv, Dqk, Dv, lens, W, window = shapes[case]
        wl = irs_synth.custom(T, Hq, Hkv, Dqk, Dv, 2, 64, 4, 8, doc_lens=lens, seed=len(lens) + 40)
        a = wl.arrays
        rng = np.random.default_rng(5)
        route = torch.from_numpy(irs_synth.random_routes(rng, T, T, W, wl.cu_seqlens, frac_invalid=0.2)).to(DEV)
        cu_h = wl.cu_seqlens
        cu = torch.from_numpy(cu_h).to(DEV)
        scale = wl.scale
        q, k, v = (torch.from_numpy(a[x]).view(torch.bfloat16).to(DEV) for x in ("q", "k", "v"))
    comp = irs.compose_window_routes(route, cu, window)
    o1, l1 = irs.sparse_gqa_attn_fwd(q, k, v, comp, scale)
    o2, l2 = irs.sparse_gqa_attn_fwd(q, k, v, route, scale, window=window, cu_seqlens=cu)
    irs.check_device_errors(DEV)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    rows = parity.sample_rows(wl, 96, seed=9)
    ref_comp = O.compose_window(route.cpu().numpy(), cu_h, wl.T, window)
    ref_o, ref_l = O.attention(a["q"], a["k"], a["v"], ref_comp, scale, rows=rows)
    parity.check_attention(o2, l2, ref_o, ref_l, rows)
