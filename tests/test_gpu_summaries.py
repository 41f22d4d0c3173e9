"""Step-5 learned-logit region summaries on the GPU (through the C ABI) against the CPU
oracle (Step-5 sparse page: `project_keys` compression logits, `_summarize_region_payload`
FP32 summaries with the bf16 and E4M3 roundings, `indexer_score_tile` scoring them,
`region_metadata` resetting regions at document boundaries)."""
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


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _to_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits)).view(torch.bfloat16).to(DEV)


SUMMARY_CASES = {
    # name: (T, Di, c, doc_lens, logit scale)
    "c4_one_doc": (2048, 128, 4, [2048], 2.0),
    "c64_ragged_docs": (4000, 128, 64, [1000, 63, 2937], 2.0),
    "di64_tiny_docs": (1203, 64, 4, [600, 3, 1, 599], 2.0),
    "equal_logits": (1024, 128, 8, [517, 507], 0.0),
    "sharp_logits_underflow": (1536, 64, 16, [1536], 60.0),
    "c1": (300, 128, 1, [100, 200], 2.0),
}


@pytest.mark.parametrize("case", sorted(SUMMARY_CASES))
def test_region_summaries_bit_exact(irs, case):
    T, Di, c, lens, scale = SUMMARY_CASES[case]
    wl = irs_synth.custom(T, 2, 1, 64, 128, Hi=4, Di=Di, c=c, budget=c, doc_lens=lens, seed=T + c)
    kI = wl.arrays["kI"]
    z = irs_synth.compression_logits(T, Di, seed=T + 7, scale=scale)
    cu = wl.arrays["cu_seqlens"]
    out = irs.region_summaries(_to_dev(kI), _to_dev(z), torch.from_numpy(cu).to(DEV), c, max_doc_len=max(lens))
    irs.check_device_errors(DEV)
    got = _bits(out)
    ref, offs = O.region_summaries_e4m3(kI, z, cu, c)
    n = int(offs[-1])
    want = irs_synth.f32_to_bf16_bits(ref.astype(np.float32))   # E4M3 values are exact in bf16
    np.testing.assert_array_equal(got[:n], want)
    assert not got[n:].any(), "rows past the last region must be zero"
    if scale == 0.0:
        # equal logits: the summaries are the E4M3 roundings of the bf16 means
        kbar, _ = O.pool_keys(kI, cu, c)
        np.testing.assert_array_equal(got[:n], irs_synth.f32_to_bf16_bits(
            O.round_to_e4m3(O.round_to_bf16(kbar).astype(np.float64)).astype(np.float32)))


INDEX_CASES = {
    # name: (T, G, Hi, Di, c, budget, doc_lens, operands, w_kind)
    "e4m3_one_group": (2048, 1, 16, 128, 4, 256, [2048], "e4m3", "uniform"),
    "e4m3_grouped_signed": (1500, 4, 8, 128, 4, 128, [700, 5, 795], "e4m3", "signed"),
    "bf16_queries_di64": (1200, 2, 32, 64, 16, 128, [300, 7, 893], "bf16", "signed"),
    "bf16_queries_c64": (4096, 1, 32, 128, 64, 1024, [4096], "bf16", "uniform"),
}


@pytest.mark.parametrize("case", sorted(INDEX_CASES))
def test_summary_indexer_scores_and_routes(irs, case):
    T, G, Hi, Di, c, budget, lens, operands, w_kind = INDEX_CASES[case]
    rng = np.random.default_rng(T + G + Hi)
    qI = irs_synth.f32_to_bf16_bits(rng.standard_normal((T, G, Hi, Di), dtype=np.float32))
    kI = irs_synth.f32_to_bf16_bits(rng.standard_normal((T, Di), dtype=np.float32))
    if w_kind == "signed":
        w = (rng.random((T, G, Hi), dtype=np.float32) * np.float32(2) - np.float32(1)).astype(np.float32)
    else:
        w = rng.random((T, G, Hi), dtype=np.float32)
    z = irs_synth.compression_logits(T, Di, seed=T + 3)
    cu = np.zeros(len(lens) + 1, np.int32)
    cu[1:] = np.cumsum(lens)
    ld = max(lens) // c
    scores = torch.full((T, G, ld), float("nan"), dtype=torch.float32, device=DEV)
    route = irs.sparse_index_score_topk_summaries(_to_dev(qI), _to_dev(kI), _to_dev(z), torch.from_numpy(w).to(DEV),
                                                  torch.from_numpy(cu).to(DEV), c, budget, operands=operands,
                                                  max_doc_len=max(lens), scores_out=scores)
    irs.check_device_errors(DEV)
    g_route, g_scores = route.cpu().numpy(), scores.cpu().numpy()
    ktilde, _ = O.region_summaries_e4m3(kI, z, cu, c)
    wl_like = irs_synth.custom(T, 2, 1, 64, 128, Hi=Hi, Di=Di, c=c, budget=budget, doc_lens=lens, seed=1)
    rows = np.arange(T) if T * G <= 3000 else parity.sample_rows(wl_like, 400, seed=9)
    for g in range(G):
        wl_like.arrays.update(qI=np.ascontiguousarray(qI[:, g]), kI=kI, w=np.ascontiguousarray(w[:, g]),
                              cu_seqlens=cu)
        ref_r, ref_s = O.index_routes(qI[:, g], kI, w[:, g], cu, c, budget, rows=rows, want_scores=True, ldS=ld,
                                      operands=operands, logits=z)
        parity.check_scores(g_scores[rows, g], ref_s, wl_like, rows, ktilde=ktilde)
        parity.check_routes_e2e(g_route[rows, g], ref_r, ref_s, wl_like, rows)
    # the summaries change the selection: the mean-pooled indexer picks other blocks somewhere
    if G == 1 and operands == "e4m3":
        plain = irs.sparse_index_score_topk(_to_dev(qI[:, 0]), _to_dev(kI), torch.from_numpy(w[:, 0]).to(DEV),
                                            torch.from_numpy(cu).to(DEV), c, budget, max_doc_len=max(lens),
                                            operands="e4m3")
        assert not torch.equal(plain, route)
