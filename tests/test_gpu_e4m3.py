"""Step-5 E4M3 scoring operands on the GPU (kind::f8f6f4 tensor cores, through the C ABI)
against the CPU oracle's `index_routes(operands="e4m3")` (Step-5 sparse page,
`indexer_score_tile`: queries and summaries rounded to FP8 E4M3)."""
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


@pytest.mark.parametrize("case", ["mid_small", "windowed_small", "multi_doc_signed", "hi256"])
def test_e4m3_scores_and_routes(irs, case):
    if case == "mid_small":
        wl = irs_synth.make("mid", small=True)
    elif case == "windowed_small":
        wl = irs_synth.make("windowed", small=True)
    elif case == "multi_doc_signed":
        wl = irs_synth.custom(1800, 2, 1, 64, 128, Hi=8, Di=128, c=4, budget=64, doc_lens=[600, 3, 1197], seed=21,
                              w_kind="signed")
    else:
        wl = irs_synth.custom(700, 2, 1, 64, 128, Hi=256, Di=128, c=4, budget=32, doc_lens=[700], seed=22)
    a = wl.arrays
    t = irs_synth.as_torch(wl, device=DEV)
    ld = max(1, wl.max_doc_len // wl.c)
    scores = torch.full((wl.T, ld), float("nan"), dtype=torch.float32, device=DEV)
    route = irs.sparse_index_score_topk(t["qI"], t["kI"], t["w"], t["cu_seqlens"], wl.c, wl.budget,
                                        max_doc_len=wl.max_doc_len, scores_out=scores, operands="e4m3")
    irs.check_device_errors(DEV)
    rows = np.arange(wl.T) if wl.T <= 2048 else parity.sample_rows(wl, 384, seed=6)
    ref_r, ref_s = O.index_routes(a["qI"], a["kI"], a["w"], wl.cu_seqlens, wl.c, wl.budget, rows=rows,
                                  want_scores=True, ldS=ld, operands="e4m3")
    idx = torch.as_tensor(rows, device=DEV)
    parity.check_scores(scores[idx].cpu().numpy(), ref_s, wl, rows)
    parity.check_routes_e2e(route[idx].cpu().numpy(), ref_r, ref_s, wl, rows)
    # the E4M3 scores are not the bf16 ones (the roundings are applied)
    if case == "mid_small":
        ref_bf = O.index_routes(a["qI"], a["kI"], a["w"], wl.cu_seqlens, wl.c, wl.budget, rows=rows[-4:],
                                want_scores=True, ldS=ld)[1]
        got = scores[idx[-4:]].cpu().numpy()
        fin = ~np.isnan(ref_bf)
        assert np.abs(got[fin] - ref_bf[fin]).max() > 1e-3 * np.abs(ref_bf[fin]).max()
