"""Indexer on the GPU (through the C ABI) against the CPU oracle."""
import numpy as np
import pytest
import torch

import irs_synth
import parity
from oracle import irs_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def irs():
    import indexer_routed_sparse_gb300 as m

    m.lib()
    return m


def run_index(irs, wl, with_scores=True):
    dev = torch.device("cuda", 0)
    t = irs_synth.as_torch(wl, device=dev)
    ld = max(1, wl.max_doc_len // wl.c)
    scores = torch.full((wl.T, ld), float("nan"), dtype=torch.float32, device=dev) if with_scores else None
    route = irs.sparse_index_score_topk(t["qI"], t["kI"], t["w"], t["cu_seqlens"], wl.c, wl.budget,
                                        max_doc_len=wl.max_doc_len, scores_out=scores)
    irs.check_device_errors(dev)
    return t, route, scores


def full_check(irs, wl, rows=None):
    a = wl.arrays
    t, route, scores = run_index(irs, wl)
    rows = np.arange(wl.T) if rows is None else rows
    ref_r, ref_s = O.index_routes(a["qI"], a["kI"], a["w"], wl.cu_seqlens, wl.c, wl.budget, rows=rows,
                                  want_scores=True, ldS=max(1, wl.max_doc_len // wl.c))
    idx = torch.as_tensor(rows, device=route.device)
    g_routes = route[idx].cpu().numpy()
    g_scores = scores[idx].cpu().numpy()
    parity.check_scores(g_scores, ref_s, wl, rows)
    ndiff = parity.check_routes_e2e(g_routes, ref_r, ref_s, wl, rows)
    # routes from the oracle's own FP32 scores must match bit for bit
    full_scores = np.zeros((wl.T, ref_s.shape[1]), np.float32)
    full_scores[rows] = np.nan_to_num(ref_s, nan=0.0)
    s_dev = torch.from_numpy(full_scores).to(route.device)
    r2 = irs.topk_from_scores(s_dev, t["cu_seqlens"], wl.c, wl.budget, max_doc_len=wl.max_doc_len)
    irs.check_device_errors(route.device)
    ref_r2 = O.routes_from_scores(full_scores, wl.cu_seqlens, wl.T, wl.c, wl.budget, rows=rows)
    np.testing.assert_array_equal(r2[idx].cpu().numpy(), ref_r2)
    return ndiff


def test_tiny_all_rows(irs):
    wl = irs_synth.make("tiny")
    ndiff = full_check(irs, wl)
    assert ndiff <= 2


@pytest.mark.parametrize("name", ["mid", "packed", "windowed"])
def test_small_variants_all_rows(irs, name):
    wl = irs_synth.make(name, small=True)
    full_check(irs, wl)


def test_mid_full_size_all_rows(irs):
    wl = irs_synth.make("mid")
    ndiff = full_check(irs, wl)
    assert ndiff <= 10


@pytest.mark.parametrize("name", ["packed", "windowed"])
def test_full_size_sampled_rows(irs, name):
    wl = irs_synth.make(name)
    rows = parity.sample_rows(wl, 384, seed=1)
    full_check(irs, wl, rows)


@pytest.mark.parametrize("shape", [
    dict(Hi=1, Di=64, c=1, budget=5, doc_lens=[1, 2, 3, 40, 7, 300]),
    dict(Hi=2, Di=128, c=3, budget=9, doc_lens=[100, 33, 250]),
    dict(Hi=8, Di=64, c=4, budget=4, doc_lens=[513]),
    dict(Hi=32, Di=128, c=2, budget=64, doc_lens=[700, 1]),
    dict(Hi=256, Di=64, c=4, budget=16, doc_lens=[129, 64]),
    dict(Hi=4, Di=64, c=4, budget=4096, doc_lens=[300, 200]),        # every row dense
    dict(Hi=16, Di=128, c=16, budget=32, doc_lens=[1000, 17, 15]),
])
def test_edge_shapes(irs, shape):
    lens = shape.pop("doc_lens")
    T = sum(lens)
    wl = irs_synth.custom(T, 2, 1, 64, 128, doc_lens=lens, seed=len(lens) + T, **shape)
    full_check(irs, wl)


def test_signed_weights_and_ties(irs):
    # signed head weights (Step-5 pages) and many exact-zero scores (ReLU) -> ties at zero
    wl = irs_synth.custom(600, 2, 1, 64, 128, Hi=4, Di=64, c=4, budget=32, doc_lens=[600], seed=5, w_kind="signed")
    full_check(irs, wl)
    wl2 = irs_synth.custom(400, 2, 1, 64, 128, Hi=1, Di=64, c=2, budget=16, doc_lens=[400], seed=6, w_kind="ones")
    full_check(irs, wl2)


def test_scores_scratch_in_workspace_gives_same_routes(irs):
    wl = irs_synth.make("mid", small=True)
    _, r1, _ = run_index(irs, wl, with_scores=True)
    _, r2, _ = run_index(irs, wl, with_scores=False)
    assert torch.equal(r1, r2)


def test_window_composition(irs):
    wl = irs_synth.make("windowed", small=True)
    t, route, _ = run_index(irs, wl, with_scores=False)
    comp = irs.compose_window_routes(route, t["cu_seqlens"], wl.window)
    irs.check_device_errors(route.device)
    r_h = route.cpu().numpy()
    ref = O.compose_window(r_h, wl.cu_seqlens, wl.T, wl.window)   # same input routes on both sides
    np.testing.assert_array_equal(comp.cpu().numpy(), ref)


def test_window_composition_multi_doc(irs):
    cu = np.asarray([0, 5, 700, 1000], np.int32)
    rng = np.random.default_rng(3)
    routes = irs_synth.random_routes(rng, 1000, 1000, 40, cu)
    dev = torch.device("cuda", 0)
    comp = irs.compose_window_routes(torch.from_numpy(routes).to(dev), torch.from_numpy(cu).to(dev), 64)
    np.testing.assert_array_equal(comp.cpu().numpy(), O.compose_window(routes, cu, 1000, 64))


def test_malformed_cu_seqlens_sets_the_device_flag(irs):
    wl = irs_synth.custom(256, 2, 1, 64, 128, Hi=4, Di=64, c=4, budget=16, doc_lens=[100, 156], seed=1)
    dev = torch.device("cuda", 0)
    t = irs_synth.as_torch(wl, device=dev)
    bad = torch.tensor([0, 200, 150, 256], dtype=torch.int32, device=dev)   # not increasing
    irs.read_device_errors(dev)
    irs.sparse_index_score_topk(t["qI"], t["kI"], t["w"], bad, wl.c, wl.budget, ndocs=3, max_doc_len=200)
    assert irs.read_device_errors(dev) & irs.DEVERR_CU_SEQLENS
    # the context is still usable afterwards
    run_index(irs, wl)


@pytest.mark.parametrize("budget", [64, 256])
@pytest.mark.parametrize("kind", ["constant", "two_values", "signed_zero", "negative", "wide_range"])
def test_topk_degenerate_scores_bit_exact(irs, kind, budget):
    """Ties everywhere, -0/+0, negative and widely spread scores: routes equal the oracle's
    (kb 32: the warp-per-row variant, its bit-serial path where many keys tie; kb 128: the
    register variant)."""
    rng = np.random.default_rng(len(kind))
    cu = np.asarray([0, 700, 2000], np.int32)
    T, c = 2000, 2
    ld = 1300 // c
    if kind == "constant":
        sc = np.full((T, ld), 0.75, np.float32)
    elif kind == "two_values":
        sc = rng.choice(np.asarray([1.0, 2.0], np.float32), size=(T, ld))
    elif kind == "signed_zero":
        sc = rng.choice(np.asarray([0.0, -0.0, 1e-30], np.float32), size=(T, ld))
    elif kind == "negative":
        sc = -rng.random((T, ld), dtype=np.float32)
    else:
        sc = (rng.standard_normal((T, ld)) * np.exp(rng.uniform(-30, 30, (T, ld)))).astype(np.float32)
    dev = torch.device("cuda", 0)
    r = irs.topk_from_scores(torch.from_numpy(sc).to(dev), torch.from_numpy(cu).to(dev), c, budget)
    irs.check_device_errors(dev)
    np.testing.assert_array_equal(r.cpu().numpy(), O.routes_from_scores(sc, cu, T, c, budget))


@pytest.mark.parametrize("c, budget, lens", [
    (64, 1024, [2048]),                          # kb 16, rows up to 32 blocks (lanes without keys)
    (4, 64, [1000, 24, 3000]),                   # kb 16, up to 750 blocks (KPL 32), a short document
    (2, 2, [4100]),                              # kb 1, up to 2050 blocks (KPL 64)
    (8, 256, [2048, 777]),                       # kb 32, up to 256 blocks (KPL 8)
    (1, 20, [400, 1700]),                        # kb 20, up to 1700 blocks, c = 1
    (3, 48, [1500]),                             # kb 16, c not a power of two
])
def test_topk_warp_variant_bit_exact(irs, c, budget, lens):
    """The warp-per-row top-k (kb <= 32) on continuous scores, where the candidate ranking
    decides, with a few rows of tied top scores mixed in (the bit-serial path): routes equal
    the oracle's selection from the same FP32 scores."""
    rng = np.random.default_rng(c * 1000 + budget)
    T = sum(lens)
    cu = np.zeros(len(lens) + 1, np.int32)
    cu[1:] = np.cumsum(lens)
    ld = max(lens) // c
    sc = rng.standard_normal((T, ld)).astype(np.float32)
    sc[::7, : ld // 2] = 3.0                      # many keys tied at the top of every 7th row
    sc[1::11] = np.abs(sc[1::11])                 # some rows of positive scores only
    dev = torch.device("cuda", 0)
    r = irs.topk_from_scores(torch.from_numpy(sc).to(dev), torch.from_numpy(cu).to(dev), c, budget)
    irs.check_device_errors(dev)
    np.testing.assert_array_equal(r.cpu().numpy(), O.routes_from_scores(sc, cu, T, c, budget))
