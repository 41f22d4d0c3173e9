"""The indexer entry point that allocates nothing (collected last on purpose).

irs_sparse_index_score_topk_noalloc serves callers that cannot give the library device
memory (e.g. runtime plugins without an allocator, or loops that must not risk the
synchronisation of a cudaMalloc): its scratch is a fixed 16 MiB array inside libirs.so.
These tests call it through the C ABI and compare it with the workspace entry point,
twice in a row, so results left in the shared array by one call cannot leak into the next.
"""

import numpy as np
import pytest
import torch

import irs_synth

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def _noalloc(L, t, wl, route, scores):
    ld = scores.stride(0) if scores is not None else 0
    return L.irs_sparse_index_score_topk_noalloc(
        t["qI"].data_ptr(), t["kI"].data_ptr(), t["w"].data_ptr(), t["cu_seqlens"].data_ptr(), wl.ndocs,
        wl.max_doc_len, wl.T, wl.Hi, wl.Di, wl.c, wl.budget, route.data_ptr(),
        scores.data_ptr() if scores is not None else None, ld, None,
        torch.cuda.current_stream(DEV).cuda_stream)


@pytest.mark.parametrize("name, with_scores", [("tiny", False), ("mid", True)])
def test_noalloc_matches_workspace_entry_point_twice(name, with_scores):
    import indexer_routed_sparse_gb300 as irs

    L = irs.lib()
    wl = irs_synth.make(name, small=(name != "tiny"))
    t = irs_synth.as_torch(wl, device=DEV)
    ld = max(1, wl.max_doc_len // wl.c)
    ref_scores = torch.full((wl.T, ld), float("nan"), dtype=torch.float32, device=DEV)
    ref = irs.sparse_index_score_topk(t["qI"], t["kI"], t["w"], t["cu_seqlens"], wl.c, wl.budget,
                                      max_doc_len=wl.max_doc_len, scores_out=ref_scores)
    irs.check_device_errors(DEV)
    sparse = ~torch.isnan(ref_scores)
    for call in range(2):
        route = torch.full_like(ref, -7)
        scores = torch.full((wl.T, ld), float("nan"), dtype=torch.float32, device=DEV) if with_scores else None
        st = _noalloc(L, t, wl, route, scores)
        assert st == 0, L.irs_last_error()
        torch.cuda.synchronize(DEV)
        assert torch.equal(route, ref), f"call {call}: routes differ from the workspace entry point"
        if scores is not None:
            got = scores[sparse].double()
            exp = ref_scores[sparse].double()
            rel = ((got - exp).abs() / exp.abs().clamp_min(1e-30)).max().item()
            assert rel <= 1e-4, f"call {call}: scores differ (max rel {rel:.2e})"


def test_noalloc_rejects_sizes_beyond_the_fixed_scratch():
    import indexer_routed_sparse_gb300 as irs

    L = irs.lib()
    wl = irs_synth.make("mid")          # 64 MB of score rows without a score buffer: over 16 MiB
    t = irs_synth.as_torch(wl, device=DEV)
    route = torch.empty((wl.T, wl.budget + wl.c - 1), dtype=torch.int32, device=DEV)
    st = _noalloc(L, t, wl, route, None)
    assert st == 2
    assert b"fixed array" in L.irs_last_error()
