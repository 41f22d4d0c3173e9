"""Indexer front half on the GPU (through the C ABI) against the CPU oracle.

QSA page, `Qwen3_8_FlashNextQSAIndexer` (K RMSNorm and group-start RoPE on the FP32 group
means; RMSNorm and RoPE on the index queries) and `apply_qsa_rope` (rotate-half over the
first rope_dims dims). Both sides evaluate the transform in FP32 in the same order and
round once to bf16, so the transformed operands must agree bit for bit; scores and routes
then follow the indexer's own tolerances."""
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


def _front(wl, rope_dims, seed):
    f = irs_synth.front_half_inputs(wl.T, wl.Di, rope_dims, wl.cu_seqlens, seed=seed)
    dev = {"q_weight": torch.from_numpy(f["q_weight"]).to(DEV), "k_weight": torch.from_numpy(f["k_weight"]).to(DEV),
           "eps": f["eps"], "rope": torch.from_numpy(np.ascontiguousarray(f["rope"])).to(DEV) if rope_dims else None}
    host = dict(f)
    if not rope_dims:
        host["rope"] = np.zeros((wl.T, 0), np.float32)
    return host, dev


CASES = [
    ("mid_small", dict(), 128),
    ("multi_doc", dict(T=2000, Hi=4, Di=64, c=4, budget=64, doc_lens=[300, 1, 451, 1248]), 32),
    ("no_rope", dict(T=700, Hi=8, Di=128, c=2, budget=32, doc_lens=[700]), 0),
    ("windowed_small", dict(), 64),
]


def _workload(name, kw):
    if name == "mid_small":
        return irs_synth.make("mid", small=True)
    if name == "windowed_small":
        return irs_synth.make("windowed", small=True)
    lens = kw.pop("doc_lens")
    T = kw.pop("T")
    return irs_synth.custom(T, 2, 1, 64, 128, doc_lens=lens, seed=T + len(lens), **kw)


@pytest.mark.parametrize("name,kw,rope_dims", CASES)
def test_front_operands_bit_exact(irs, name, kw, rope_dims):
    wl = _workload(name, dict(kw))
    a = wl.arrays
    host, dev = _front(wl, rope_dims, seed=7)
    t = irs_synth.as_torch(wl, device=DEV)
    q_out, k_out = irs.index_front_operands(t["qI"], t["kI"], t["cu_seqlens"], wl.c, wl.budget, dev,
                                            max_doc_len=wl.max_doc_len)
    irs.check_device_errors(DEV)
    ref_k, blk_off = O.front_keys(a["kI"], wl.cu_seqlens, wl.c, host["k_weight"], host["eps"], host["rope"])
    nblk = ref_k.shape[0]
    got_k = k_out[:nblk].float().cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(got_k, ref_k)
    assert torch.all(k_out[nblk:] == 0)
    rows = np.arange(wl.T) if wl.T <= 2048 else parity.sample_rows(wl, 512, seed=3)
    got_q = q_out[torch.as_tensor(rows, device=DEV)].float().cpu().numpy().astype(np.float64)
    for i, tt in enumerate(rows):
        ref_q = O.front_query_row(a["qI"][tt], host["q_weight"], host["eps"], host["rope"][tt])
        np.testing.assert_array_equal(got_q[i], ref_q, err_msg=f"query row {tt}")


@pytest.mark.parametrize("name,kw,rope_dims", CASES)
def test_front_scores_and_routes(irs, name, kw, rope_dims):
    wl = _workload(name, dict(kw))
    a = wl.arrays
    host, dev = _front(wl, rope_dims, seed=8)
    t = irs_synth.as_torch(wl, device=DEV)
    ld = max(1, wl.max_doc_len // wl.c)
    scores = torch.full((wl.T, ld), float("nan"), dtype=torch.float32, device=DEV)
    route = irs.sparse_index_score_topk(t["qI"], t["kI"], t["w"], t["cu_seqlens"], wl.c, wl.budget,
                                        max_doc_len=wl.max_doc_len, scores_out=scores, front=dev)
    irs.check_device_errors(DEV)
    rows = np.arange(wl.T) if wl.T <= 2048 else parity.sample_rows(wl, 384, seed=4)
    ref_r, ref_s = O.index_routes(a["qI"], a["kI"], a["w"], wl.cu_seqlens, wl.c, wl.budget, rows=rows,
                                  want_scores=True, ldS=ld, front=host)
    idx = torch.as_tensor(rows, device=DEV)
    # the score tolerance's cancellation floor, with the transformed operands
    fk, _ = O.front_keys(a["kI"], wl.cu_seqlens, wl.c, host["k_weight"], host["eps"], host["rope"])
    fq = np.stack([O.front_query_row(a["qI"][tt], host["q_weight"], host["eps"], host["rope"][tt]) for tt in rows])
    _check_scores_front(scores[idx].cpu().numpy(), ref_s, fq, fk, wl, rows)
    parity.check_routes_e2e(route[idx].cpu().numpy(), ref_r, ref_s, wl, rows)


def _check_scores_front(got, ref, fq, fk, wl, rows):
    cu = np.asarray(wl.cu_seqlens, np.int64)
    _, blk_off = O.pool_keys(wl.arrays["kI"], wl.cu_seqlens, wl.c)
    kb = wl.budget // wl.c
    n = 0
    for i, t in enumerate(rows):
        d = int(np.searchsorted(cu, t, side="right") - 1)
        nv = (int(t) - int(cu[d]) + 1) // wl.c
        if nv <= kb:
            continue
        kt = np.abs(fk[blk_off[d]: blk_off[d] + nv])
        floor = 1e-3 * (np.abs(wl.arrays["w"][t].astype(np.float64)) @ (np.abs(fq[i]) @ kt.T))
        r = ref[i, :nv].astype(np.float64)
        rel = np.abs(got[i, :nv].astype(np.float64) - r) / np.maximum(np.abs(r), floor)
        assert rel.max() <= parity.SCORE_RTOL, f"row {t}: score rel err {rel.max():.3e}"
        n += nv
    assert n > 0
