"""Failure detection on the GPU without a fault: a bounded on-device wait that nothing
releases gives up, reports IRS_DEVERR_TIMEOUT through the caller's error word, and leaves
the context usable for the next call."""
import time

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


def test_wait_gives_up_reports_and_context_stays_usable(irs):
    t0 = time.perf_counter()
    err = irs.check_bounded_wait(limit_ms=20.0, device=DEV)
    torch.cuda.synchronize()
    assert int(err.item()) & irs.DEVERR_TIMEOUT
    assert time.perf_counter() - t0 < 10.0
    # an ordinary call afterwards runs and matches the oracle
    T = 64
    wl = irs_synth.custom(T, 4, 2, 128, 128, 2, 64, 4, 8, seed=5)
    a = wl.arrays
    routes = irs_synth.random_routes(np.random.default_rng(2), T, T, 40, wl.cu_seqlens)
    q, k, v = (torch.from_numpy(a[n]).view(torch.bfloat16).to(DEV) for n in ("q", "k", "v"))
    out, lse = irs.sparse_gqa_attn_fwd(q, k, v, torch.from_numpy(routes).to(DEV), wl.scale)
    irs.check_device_errors(DEV)
    ref_o, ref_l = O.attention(a["q"], a["k"], a["v"], routes, wl.scale)
    parity.check_attention(out, lse, ref_o, ref_l, np.arange(T))


def test_limits_are_checked(irs):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    with pytest.raises(ValueError):
        irs.check_bounded_wait(limit_ms=0.1, device=DEV, err=err)
