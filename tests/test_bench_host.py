"""Host-side pieces of bench.py: the oracle sample behind the CPU baseline and the
reference arm must work for every workload (no GPU)."""
import numpy as np

import bench
import irs_synth
from oracle import irs_oracle as O


def test_oracle_rows_every_workload_kind():
    for name in ("tiny", "latent", "windowed"):
        wl = irs_synth.make(name, small=True)
        bench._WL = wl
        rows = np.array([0, wl.T // 2, wl.T - 1])
        pairs = bench._oracle_rows(rows)
        if wl.latent:
            expect = int(np.count_nonzero(wl.arrays["route"][rows] >= 0))
        else:
            a = wl.arrays
            r = O.index_routes(a["qI"], a["kI"], a["w"], wl.cu_seqlens, wl.c, wl.budget, rows=rows)
            if wl.window:
                full = np.full((wl.T, r.shape[1]), -1, np.int32)
                full[rows] = r
                r = O.compose_window(full, wl.cu_seqlens, wl.T, wl.window, rows=rows)
            expect = int(np.count_nonzero(r >= 0))
        assert pairs == expect > 0, (name, pairs, expect)


def test_worker_init_builds_the_named_workload():
    bench._worker_init("latent", True)
    assert bench._WL.name == "latent" and bench._WL.T == irs_synth.make("latent", small=True).T
    bench._worker_init("tiny", False)
    assert bench._WL.name == "tiny"


def test_backward_kernel_named_by_the_dispatch_rule():
    """The kernel name the backward report carries follows the library's dispatch: the
    tensor-core kernel for 8 or more query heads per KV head (when its tiles fit), the
    CUDA-core warp-per-row kernel for smaller head groups, the general kernel for latent
    rows."""
    expect = {"tiny": "attn_bwd_fast_kernel", "mid": "attn_bwd_fast_kernel", "packed": "attn_bwd_tc_kernel",
              "windowed": "attn_bwd_tc_kernel", "latent": "attn_bwd_kernel"}
    for name, kernel in expect.items():
        assert bench.backward_kernel_name(irs_synth.make(name, small=True)) == kernel, name
    # a head shape the tensor-core tiles cannot hold (Dv 256 with Dqk 128 needs more than
    # 227 KB of stages and tiles) falls back to the CUDA-core kernel even with 32 heads
    wl = irs_synth.custom(64, 32, 1, 128, 256, 2, 64, 4, 8)
    assert bench.backward_kernel_name(wl) == "attn_bwd_fast_kernel"
