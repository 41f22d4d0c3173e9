"""Comparison helpers for the GPU parity tests (CUDA path vs the CPU oracle).

Tolerances (from the acceptance criteria of the routed sparse-attention benchmark):
* block scores: |gpu - ref| <= 1e-4 * max(|ref|, floor), floor = 1e-3 * sum_h |w_h| (|q_h| . |k~_b|)
  (the floor keeps heavily cancelling dot products from blowing the relative error up);
* routes from identical FP32 scores: bit-exact;
* routes end to end: a slot may differ only where the oracle's scores of the blocks
  involved are within 1e-5 relative of the kb-th score (a near tie at the boundary);
* attention: max-abs <= 2e-2 and mean-abs <= 2e-3 against the FP32 oracle output,
  lse within 2e-3 absolute (reading: scores are FP32 sums of bf16 products, about 1e-6
  relative, and the bf16 probabilities only enter the output).
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import irs_oracle as O

SCORE_RTOL = 1e-4
TIE_RTOL = 1e-5
OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 2e-3
LSE_ABS = 2e-3


def doc_starts(cu, rows):
    cu = np.asarray(cu, np.int64)
    d = np.searchsorted(cu, np.asarray(rows), side="right") - 1
    return cu[d]


def check_scores(gpu_scores: np.ndarray, ref_scores: np.ndarray, wl, rows, ktilde=None) -> None:
    """gpu_scores / ref_scores: [len(rows), ld]; entries [0, nvis) of sparse rows compared.
    ktilde: the scored block keys (float64 values) when they are not the bf16 means."""
    a = wl.arrays
    kbar, blk_off = O.pool_keys(a["kI"], wl.cu_seqlens, wl.c)
    kt_abs = np.abs(O.round_to_bf16(kbar).astype(np.float64) if ktilde is None else np.asarray(ktilde, np.float64))
    cu = np.asarray(wl.cu_seqlens, np.int64)
    kb = wl.budget // wl.c
    worst = 0.0
    n_checked = 0
    for i, t in enumerate(rows):
        d = int(np.searchsorted(cu, t, side="right") - 1)
        tau = int(t) - int(cu[d])
        nv = (tau + 1) // wl.c
        if nv <= kb:
            continue
        q_abs = np.abs(O.bf16_to_f64(a["qI"][t]))
        w_abs = np.abs(a["w"][t].astype(np.float64))
        floor = 1e-3 * (w_abs @ (q_abs @ kt_abs[blk_off[d]: blk_off[d] + nv].T))
        ref = ref_scores[i, :nv].astype(np.float64)
        got = gpu_scores[i, :nv].astype(np.float64)
        rel = np.abs(got - ref) / np.maximum(np.abs(ref), floor)
        worst = max(worst, float(rel.max()))
        n_checked += nv
        assert rel.max() <= SCORE_RTOL, f"row {t}: score rel err {rel.max():.3e} at block {int(rel.argmax())}"
    assert n_checked > 0 or all(((int(t) - int(doc_starts(cu, [t])[0]) + 1) // wl.c) <= kb for t in rows)


def route_blocks(row: np.ndarray, budget: int, c: int) -> list[int]:
    blk = row[:budget]
    return blk[blk >= 0][::c].tolist()


def check_routes_e2e(gpu_routes: np.ndarray, ref_routes: np.ndarray, ref_scores: np.ndarray, wl, rows) -> int:
    """Rows must match except at oracle near-ties of the kb-th score. Returns #rows that differ."""
    c, budget = wl.c, wl.budget
    kb = budget // c
    cu = np.asarray(wl.cu_seqlens, np.int64)
    ndiff = 0
    for i, t in enumerate(rows):
        g, r = gpu_routes[i], ref_routes[i]
        if np.array_equal(g, r):
            continue
        ndiff += 1
        assert np.array_equal(g[budget:], r[budget:]), f"row {t}: tail differs"
        d = int(np.searchsorted(cu, t, side="right") - 1)
        s = int(cu[d])
        nv = (int(t) - s + 1) // c
        assert nv > kb, f"row {t}: dense row differs"
        sc = ref_scores[i, :nv].astype(np.float64)
        boundary = np.sort(sc)[::-1][kb - 1]
        gb = set(((np.asarray(route_blocks(g, budget, c)) - s) // c).tolist())
        rb = set(((np.asarray(route_blocks(r, budget, c)) - s) // c).tolist())
        assert len(gb) == kb, f"row {t}: gpu selected {len(gb)} blocks"
        for b in gb ^ rb:
            assert 0 <= b < nv, f"row {t}: block {b} not visible"
            gap = abs(sc[b] - boundary)
            assert gap <= TIE_RTOL * max(abs(boundary), 1e-30), \
                f"row {t}: block {b} differs but is not a near tie ({sc[b]} vs boundary {boundary})"
    return ndiff


def check_attention(out_gpu: torch.Tensor, lse_gpu: torch.Tensor, ref_o: np.ndarray, ref_l: np.ndarray,
                    rows) -> tuple[float, float]:
    idx = torch.as_tensor(np.asarray(rows), device=out_gpu.device)
    got = out_gpu[idx].float().cpu().numpy()
    err = np.abs(got - ref_o)
    assert np.isfinite(got).all(), "non-finite output"
    mx, mean = float(err.max()), float(err.mean())
    assert mx <= OUT_MAX_ABS, f"max-abs {mx:.3e}"
    assert mean <= OUT_MEAN_ABS, f"mean-abs {mean:.3e}"
    if lse_gpu is not None:
        gl = lse_gpu[idx].cpu().numpy()
        fin = np.isfinite(ref_l)
        assert np.array_equal(np.isneginf(gl), np.isneginf(ref_l)), "empty-row lse mismatch"
        if fin.any():
            assert np.abs(gl[fin] - ref_l[fin]).max() <= LSE_ABS, f"lse err {np.abs(gl[fin] - ref_l[fin]).max():.3e}"
    return mx, mean


def sample_rows(wl, n: int, seed: int = 0) -> np.ndarray:
    """Rows that exercise document starts/ends, tau in 0..c, the sparse boundary and random rows."""
    rng = np.random.default_rng(seed)
    cu = np.asarray(wl.arrays.get("cu_seqlens", np.asarray([0, wl.T])), np.int64)
    T = wl.T
    picks = set()
    kb_tau = (wl.budget // wl.c + 1) * wl.c - 1 if wl.c else 0
    for d in range(cu.shape[0] - 1):
        s, e = int(cu[d]), int(cu[d + 1])
        for off in list(range(0, min(e - s, wl.c + 1))) + [kb_tau - 1, kb_tau, kb_tau + 1]:
            if 0 <= off < e - s:
                picks.add(s + off)
        picks.add(e - 1)
        if len(picks) > n // 2:
            break
    while len(picks) < n:
        picks.add(int(rng.integers(0, T)))
    return np.asarray(sorted(picks)[:max(n, 1)])


def window_like_routes(T: int, Tk: int, W: int, cu) -> np.ndarray:
    """Cheap deterministic causal routes (the W most recent tokens of the document)."""
    cu = np.asarray(cu, np.int64)
    t = np.arange(T, dtype=np.int64)[:, None]
    s = cu[np.searchsorted(cu, np.arange(T), side="right") - 1][:, None]
    ids = t - np.arange(W, dtype=np.int64)[None, :]
    ids[ids < s] = -1
    return ids.astype(np.int32)
