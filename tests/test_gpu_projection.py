"""The indexer's projections on the GPU (one tcgen05 GEMM, through the C ABI) against the CPU
oracle's `project_indexer` (QSA page, indexer class: the fused [(H_index+1)*D_index]
projection; Step-5 sparse page, `Step5IndexerWeightProjection`: signed FP32 head weights).

The kernel sums bf16 products in FP32, the oracle takes the exact dot product; both round
once. So every output must lie within half a bf16 (or FP32) spacing of the exact value plus
the FP32 accumulation bound 2 H 2^-24 sum_k |x_k w_k|; a bf16 output differs from the
oracle's rounding only where the exact value lies within that bound of a rounding midpoint
(about 0.2% of them at H = 4096), and never by more than one spacing."""
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


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits)).view(torch.bfloat16).to(DEV)


def check_projection(hidden, weight, Hi, Di, qI, kI, w):
    x = O.bf16_to_f64(hidden)
    W = O.bf16_to_f64(weight)
    y = x @ W.T
    acc = 2.0 * x.shape[1] * 2.0 ** -24 * (np.abs(x) @ np.abs(W).T)
    ref_q, ref_k, ref_w = O.project_indexer(hidden, weight, Hi, Di)
    T = x.shape[0]
    for name, got_bits, ref_bits, cols in (("qI", qI, ref_q, slice(0, Hi * Di)), ("kI", kI, ref_k, slice(Hi * Di, (Hi + 1) * Di))):
        g = O.bf16_to_f64(got_bits.reshape(T, -1))
        ex = y[:, cols]
        _, e = np.frexp(np.abs(ex))
        half_ulp = np.ldexp(1.0, e - 9)
        err = np.abs(g - ex)
        assert np.all(err <= half_ulp + acc[:, cols] + 1e-30), (name, float((err / (half_ulp + acc[:, cols])).max()))
        flips = np.count_nonzero(got_bits.reshape(T, -1) != ref_bits.reshape(T, -1))
        # about 2e-3 at H = 4096 (FP32 sum error ~ 4e-6 against a bf16 half-spacing of
        # 2e-3 near 1); a wrong rounding mode would flip about half of them
        assert flips <= max(2, 1e-2 * g.size), (name, flips, g.size)
    ex = y[:, (Hi + 1) * Di:]
    err = np.abs(w.astype(np.float64) - ex)
    assert np.all(err <= acc[:, (Hi + 1) * Di:] + np.abs(ex) * 2.0 ** -24 + 1e-30)
    np.testing.assert_allclose(w, ref_w, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("T, H, Hi, Di", [
    (300, 192, 4, 64),        # ragged token tile, three K steps, one output tile
    (1000, 512, 32, 128),     # 17 output tiles, keys and head weights in the last
    (257, 64, 1, 128),        # one K step, one head
    (129, 1000, 2, 64),       # H not a multiple of 64 (the last K step is zero-filled)
    (4096, 4096, 32, 128),    # the windowed workload's indexer width, hidden size 4096
])
def test_projection_matches_oracle(irs, T, H, Hi, Di):
    hidden, weight = irs_synth.projection_inputs(T, H, Hi, Di, seed=T + H)
    qI, kI, w = irs.indexer_projection(_dev(hidden), _dev(weight), Hi, Di)
    irs.check_device_errors(DEV)
    check_projection(hidden, weight, Hi, Di, _bits(qI), _bits(kI), w.cpu().numpy())


def test_projection_feeds_the_indexer(irs):
    """Projection, then the indexer on its outputs, all on the GPU: the routes equal the
    oracle's indexer run on the projected values (checked above against the oracle's
    projection), except at near-ties."""
    T, H, Hi, Di, c, budget = 2048, 256, 16, 128, 4, 256
    hidden, weight = irs_synth.projection_inputs(T, H, Hi, Di, seed=7)
    qI, kI, w = irs.indexer_projection(_dev(hidden), _dev(weight), Hi, Di)
    cu = torch.tensor([0, 1000, T], dtype=torch.int32, device=DEV)
    ld = 1048 // c
    scores = torch.full((T, ld), float("nan"), dtype=torch.float32, device=DEV)
    route = irs.sparse_index_score_topk(qI, kI, w, cu, c, budget, max_doc_len=1048, scores_out=scores)
    irs.check_device_errors(DEV)
    qb, kb, wf = _bits(qI), _bits(kI), w.cpu().numpy()
    check_projection(hidden, weight, Hi, Di, qb, kb, wf)
    wl = irs_synth.custom(T, 2, 1, 64, 128, Hi=Hi, Di=Di, c=c, budget=budget, doc_lens=[1000, 1048], seed=1)
    wl.arrays.update(qI=qb, kI=kb, w=wf)
    rows = np.arange(T)
    ref_r, ref_s = O.index_routes(qb, kb, wf, wl.cu_seqlens, c, budget, want_scores=True, ldS=ld)
    parity.check_scores(scores.cpu().numpy(), ref_s, wl, rows)
    parity.check_routes_e2e(route.cpu().numpy(), ref_r, ref_s, wl, rows)


def _front_dev(T, Di, rope_dims, seed):
    fr = irs_synth.front_half_inputs(T, Di, rope_dims, np.asarray([0, T], np.int32), seed=seed)
    front = {"q_weight": torch.from_numpy(fr["q_weight"]).to(DEV), "k_weight": torch.from_numpy(fr["k_weight"]).to(DEV),
             "eps": fr["eps"], "rope": torch.from_numpy(np.ascontiguousarray(fr["rope"])).to(DEV) if rope_dims else None}
    return fr, front


@pytest.mark.parametrize("Di, rope_dims, Hi", [(128, 64, 8), (128, 128, 4), (64, 32, 8), (64, 0, 2)])
def test_fused_query_front_half_is_bit_exact(irs, Di, rope_dims, Hi):
    """The projection with the queries' RMSNorm + RoPE in its epilogue: its queries equal
    the oracle's front transform of the unfused projection's bf16 queries bit for bit; the
    raw keys and head weights equal the unfused call's."""
    T, H = 777, 320
    hidden, weight = irs_synth.projection_inputs(T, H, Hi, Di, seed=Di + rope_dims)
    fr, front = _front_dev(T, Di, rope_dims, seed=3)
    raw = irs.indexer_projection(_dev(hidden), _dev(weight), Hi, Di)
    fused = irs.indexer_projection(_dev(hidden), _dev(weight), Hi, Di, front=front)
    irs.check_device_errors(DEV)
    assert torch.equal(fused[1], raw[1]) and torch.equal(fused[2], raw[2])
    raw_q = _bits(raw[0])
    rope = np.asarray(fr["rope"])
    want = np.stack([O.f64_to_bf16_bits(O.front_query_row(raw_q[t], fr["q_weight"], fr["eps"], rope[t]))
                     for t in range(T)])
    np.testing.assert_array_equal(_bits(fused[0]), want)


def test_fused_pipeline_equals_the_unfused_one(irs):
    """Projection with the fused query front half, then the indexer with the keys' front half
    only, gives the same scores and routes, bit for bit, as the plain projection followed by
    the indexer's full front half."""
    T, H, Hi, Di, c, budget = 2048, 256, 16, 128, 4, 256
    hidden, weight = irs_synth.projection_inputs(T, H, Hi, Di, seed=11)
    _, front = _front_dev(T, Di, 64, seed=12)
    cu = torch.tensor([0, 1000, T], dtype=torch.int32, device=DEV)
    ld = 1048 // c
    qI, kI, w = irs.indexer_projection(_dev(hidden), _dev(weight), Hi, Di)
    s_u = torch.full((T, ld), float("nan"), dtype=torch.float32, device=DEV)
    r_u = irs.sparse_index_score_topk(qI, kI, w, cu, c, budget, max_doc_len=1048, scores_out=s_u, front=front)
    qf, kf, wf = irs.indexer_projection(_dev(hidden), _dev(weight), Hi, Di, front=front)
    s_f = torch.full((T, ld), float("nan"), dtype=torch.float32, device=DEV)
    r_f = irs.sparse_index_score_topk(qf, kf, wf, cu, c, budget, max_doc_len=1048, scores_out=s_f, front=front,
                                      queries_ready=True)
    irs.check_device_errors(DEV)
    assert torch.equal(r_f, r_u)
    assert torch.equal(torch.nan_to_num(s_f, nan=-7.0), torch.nan_to_num(s_u, nan=-7.0))
