"""Step-5 per-KV-group selection and attention on the GPU (through the C ABI) against the
CPU oracle (Step-5 sparse page, `Step5SparseIndexer.forward`: region IDs per KV group;
`indexer_score_tile`: one score per group with that group's signed FP32 head weights)."""
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


def _grouped_inputs(T, G, Hi, Di, c, budget, doc_lens, seed, w_kind="signed"):
    rng = np.random.default_rng(seed)
    qI = irs_synth.f32_to_bf16_bits(rng.standard_normal((T, G, Hi, Di), dtype=np.float32))
    kI = irs_synth.f32_to_bf16_bits(rng.standard_normal((T, Di), dtype=np.float32))
    if w_kind == "signed":
        w = (rng.random((T, G, Hi), dtype=np.float32) * np.float32(2) - np.float32(1)).astype(np.float32)
    else:
        w = rng.random((T, G, Hi), dtype=np.float32)
    cu = np.zeros(len(doc_lens) + 1, np.int32)
    cu[1:] = np.cumsum(doc_lens)
    return qI, kI, w, cu


@pytest.mark.parametrize("T,G,Hi,Di,c,budget,doc_lens", [
    (1500, 4, 16, 128, 4, 128, [1500]),
    (1200, 2, 32, 64, 16, 128, [300, 7, 893]),
    (900, 8, 8, 128, 2, 64, [450, 450]),
])
def test_grouped_routes_and_scores(irs, T, G, Hi, Di, c, budget, doc_lens):
    qI, kI, w, cu = _grouped_inputs(T, G, Hi, Di, c, budget, doc_lens, seed=T + G)
    ld = max(doc_lens) // c
    t_qI = torch.from_numpy(qI).view(torch.bfloat16).to(DEV)
    t_kI = torch.from_numpy(kI).view(torch.bfloat16).to(DEV)
    t_w = torch.from_numpy(w).to(DEV)
    t_cu = torch.from_numpy(cu).to(DEV)
    scores = torch.full((T, G, ld), float("nan"), dtype=torch.float32, device=DEV)
    route = irs.sparse_index_score_topk_grouped(t_qI, t_kI, t_w, t_cu, c, budget, max_doc_len=max(doc_lens),
                                                scores_out=scores)
    irs.check_device_errors(DEV)
    g_route = route.cpu().numpy()
    g_scores = scores.cpu().numpy()
    wl_like = irs_synth.custom(T, 2, 1, 64, 128, Hi=Hi, Di=Di, c=c, budget=budget, doc_lens=doc_lens, seed=1)
    for g in range(G):
        # each group is the plain indexer on that group's queries and weights
        wl_like.arrays.update(qI=np.ascontiguousarray(qI[:, g]), kI=kI, w=np.ascontiguousarray(w[:, g]),
                              cu_seqlens=cu)
        ref_r, ref_s = O.index_routes(qI[:, g], kI, w[:, g], cu, c, budget, want_scores=True, ldS=ld)
        parity.check_scores(g_scores[:, g], ref_s, wl_like, np.arange(T))
        parity.check_routes_e2e(g_route[:, g], ref_r, ref_s, wl_like, np.arange(T))
        # and bit-identical to the single-group entry point on the same group
        single = irs.sparse_index_score_topk(torch.from_numpy(np.ascontiguousarray(qI[:, g])).view(torch.bfloat16).to(DEV),
                                             t_kI, torch.from_numpy(np.ascontiguousarray(w[:, g])).to(DEV), t_cu, c,
                                             budget, max_doc_len=max(doc_lens))
        assert torch.equal(single, route[:, g])
    # the oracle's grouped selection on a few rows, through its own entry point
    rows = np.asarray([0, T // 3, T - 1])
    ref_g = O.index_routes_grouped(qI, kI, w, cu, c, budget, rows=rows)
    for i, t in enumerate(rows):
        for g in range(G):
            ref_sc = O.index_routes(qI[:, g], kI, w[:, g], cu, c, budget, rows=[t], want_scores=True, ldS=ld)[1]
            wl_like.arrays.update(qI=np.ascontiguousarray(qI[:, g]), w=np.ascontiguousarray(w[:, g]))
            parity.check_routes_e2e(g_route[t:t + 1, g], ref_g[i:i + 1, g], ref_sc, wl_like, [t])


@pytest.mark.parametrize("Hq,Hkv,Dqk,Dv,W", [(16, 4, 128, 128, 300), (32, 2, 192, 128, 129), (6, 3, 64, 256, 64)])
def test_grouped_attention(irs, Hq, Hkv, Dqk, Dv, W):
    T = 400
    wl = irs_synth.custom(T, Hq, Hkv, Dqk, Dv, 2, 64, 4, 8, doc_lens=[150, 250], seed=Hq + W)
    a = wl.arrays
    rng = np.random.default_rng(W)
    routes = np.stack([irs_synth.random_routes(rng, T, T, W, wl.cu_seqlens, frac_invalid=0.2) for _ in range(Hkv)],
                      axis=1)
    routes[7, 1, 3] = 10 * T          # out of range: padding + device flag
    q, k, v = (torch.from_numpy(a[x]).view(torch.bfloat16).to(DEV) for x in ("q", "k", "v"))
    irs.read_device_errors(DEV)
    out, lse = irs.sparse_gqa_attn_fwd_grouped(q, k, v, torch.from_numpy(np.ascontiguousarray(routes)).to(DEV),
                                               wl.scale)
    assert irs.read_device_errors(DEV) & irs.DEVERR_ROUTE_ID
    ref_o, ref_l = O.attention_grouped(a["q"], a["k"], a["v"], routes, wl.scale)
    parity.check_attention(out, lse, ref_o, ref_l, np.arange(T))
