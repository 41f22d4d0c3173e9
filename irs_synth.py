"""Seeded synthetic inputs for indexer-routed sparse attention.

This module only draws random numbers and lays them out. It holds none of the
method's arithmetic: no pooling, scoring, selection, routing or softmax. Both
the CPU oracle (through the tests) and the CUDA path (through the tests, the
smoke check and the benchmark) take their inputs from here, so the two sides
see identical bits.

bf16 tensors are returned as ``numpy.uint16`` bit patterns, rounded from
float32 draws with round-to-nearest-even. ``as_torch`` turns a bundle into
torch tensors (bf16 views of the same bits) on a chosen device.

Draw order within one workload is fixed: q, k, v, qI, kI, w, then the
document lengths (packed workload) or the route indices (latent workload).
Large arrays are drawn in row chunks so that peak host memory stays bounded;
the chunking is part of the recipe and is deterministic.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

# rows drawn per call when filling large arrays (part of the deterministic recipe)
_DRAW_ROWS = 4096


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round-to-nearest-even); return uint16 bits.

    Input generation only: the draws are finite normals or uniforms.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    r = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 values (exact)."""
    return (np.ascontiguousarray(u, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape: tuple[int, ...]) -> np.ndarray:
    rows = shape[0]
    inner = shape[1:]
    out = np.empty(shape, dtype=np.uint16)
    for r0 in range(0, rows, _DRAW_ROWS):
        r1 = min(rows, r0 + _DRAW_ROWS)
        out[r0:r1] = f32_to_bf16_bits(rng.standard_normal((r1 - r0,) + inner, dtype=np.float32))
    return out


def _uniform_f32(rng: np.random.Generator, shape: tuple[int, ...]) -> np.ndarray:
    return rng.random(shape, dtype=np.float32)


@dataclass
class Workload:
    """One seeded workload: shapes, parameters and host arrays."""

    name: str
    seed: int
    T: int                      # query tokens (flattened THD)
    Tk: int                     # key/value tokens
    Hq: int
    Hkv: int
    Dqk: int
    Dv: int
    scale: float
    # indexer (absent for the latent workload, whose routes are given)
    Hi: int = 0
    Di: int = 0
    c: int = 0
    budget: int = 0
    window: int = 0             # sliding window composed in front of the indexer route (0 = none)
    latent: bool = False        # k and v are one latent tensor; v is its first Dv dims
    arrays: dict = field(default_factory=dict)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def route_width(self) -> int:
        if self.latent:
            return int(self.arrays["route"].shape[1])
        w = self.budget + self.c - 1
        return w + self.window

    @property
    def cu_seqlens(self) -> np.ndarray:
        return self.arrays["cu_seqlens"]

    @property
    def ndocs(self) -> int:
        return int(self.arrays["cu_seqlens"].shape[0] - 1)

    @property
    def max_doc_len(self) -> int:
        cu = self.arrays["cu_seqlens"].astype(np.int64)
        return int(np.max(cu[1:] - cu[:-1]))


# --------------------------------------------------------------------------------------
# The five workloads. Sizes, distributions and seeds follow the workload list of the
# routed sparse-attention benchmark; `small=True` keeps structure but shrinks T so the
# CPU oracle covers every row (used by tests only).
# --------------------------------------------------------------------------------------

WORKLOADS = ("tiny", "mid", "packed", "windowed", "latent")


def packed_doc_lengths(rng: np.random.Generator, row_len: int, rows: int,
                       mean: float = 4096.0, sigma: float = 1.0,
                       lo: int = 256, hi: int = 32768) -> list[int]:
    """Document lengths for packed rows.

    Lengths are lognormal with arithmetic mean `mean` (so mu = ln(mean) - sigma^2/2),
    rounded, clipped to [lo, hi]. Each row is filled in order; a draw that would
    leave fewer than `lo` tokens in the row takes the whole remainder, so every
    document is at least `lo` long and each row boundary is a document boundary.
    """
    mu = math.log(mean) - 0.5 * sigma * sigma
    out: list[int] = []
    for _ in range(rows):
        remaining = row_len
        while remaining > 0:
            L = int(np.clip(np.rint(rng.lognormal(mu, sigma)), lo, hi))
            if remaining - L < lo:
                L = remaining
            out.append(L)
            remaining -= L
    return out


def latent_routes(rng: np.random.Generator, nq: int, Tk: int, width: int) -> np.ndarray:
    """Causal random routes for the latent workload.

    Query i sits at key position p_i = Tk - nq + i. Its valid prefix length is
    L_i ~ U{1..width}; the prefix holds L_i distinct key IDs drawn uniformly
    without replacement from [0, p_i], sorted ascending; the remaining slots are -1.
    """
    out = np.full((nq, width), -1, dtype=np.int32)
    lens = rng.integers(1, width + 1, size=nq)
    for i in range(nq):
        p = Tk - nq + i
        n = int(lens[i])
        ids = rng.choice(p + 1, size=n, replace=False)
        ids.sort()
        out[i, :n] = ids
    return out


def make(name: str, small: bool = False, seed: int | None = None) -> Workload:
    """Build one named workload with its seeded arrays."""
    if name == "tiny":
        wl = Workload("tiny", 0 if seed is None else seed, T=1024, Tk=1024, Hq=8, Hkv=2, Dqk=128, Dv=128,
                      scale=1.0 / math.sqrt(128), Hi=4, Di=64, c=4, budget=256)
        doc_lens = [wl.T]
    elif name == "mid":
        T = 2048 if small else 8192
        wl = Workload("mid", 1 if seed is None else seed, T=T, Tk=T, Hq=32, Hkv=8, Dqk=128, Dv=128,
                      scale=1.0 / math.sqrt(128), Hi=16, Di=128, c=4, budget=2048 if not small else 512)
        doc_lens = [T]
    elif name == "packed":
        row_len = 4096 if small else 32768
        T = 2 * row_len
        wl = Workload("packed", 2 if seed is None else seed, T=T, Tk=T, Hq=64, Hkv=8, Dqk=128, Dv=128,
                      scale=1.0 / math.sqrt(128), Hi=64, Di=128, c=4, budget=2048 if not small else 256)
        doc_lens = None  # drawn after the tensors
    elif name == "windowed":
        T = 8192 if small else 65536
        wl = Workload("windowed", 3 if seed is None else seed, T=T, Tk=T, Hq=64, Hkv=4, Dqk=192, Dv=128,
                      scale=1.0 / math.sqrt(192), Hi=32, Di=128, c=64, budget=16 * 64, window=512)
        doc_lens = [T]
    elif name == "latent":
        nq = 1024 if small else 16384
        Tk = 4096 if small else 65536
        wl = Workload("latent", 4 if seed is None else seed, T=nq, Tk=Tk, Hq=128, Hkv=1, Dqk=576, Dv=512,
                      scale=1.0 / math.sqrt(576), latent=True)
        doc_lens = None
    else:
        raise ValueError(f"unknown workload {name!r}; expected one of {WORKLOADS}")

    rng = np.random.default_rng(wl.seed)
    a = wl.arrays
    if wl.latent:
        a["q"] = _normal_bf16(rng, (wl.T, wl.Hq, wl.Dqk))
        a["kv"] = _normal_bf16(rng, (wl.Tk, 1, wl.Dqk))
        a["route"] = latent_routes(rng, wl.T, wl.Tk, 256 if small else 2048)
        return wl
    a["q"] = _normal_bf16(rng, (wl.T, wl.Hq, wl.Dqk))
    a["k"] = _normal_bf16(rng, (wl.Tk, wl.Hkv, wl.Dqk))
    a["v"] = _normal_bf16(rng, (wl.Tk, wl.Hkv, wl.Dv))
    a["qI"] = _normal_bf16(rng, (wl.T, wl.Hi, wl.Di))
    a["kI"] = _normal_bf16(rng, (wl.T, wl.Di))
    a["w"] = _uniform_f32(rng, (wl.T, wl.Hi))
    if doc_lens is None:
        doc_lens = packed_doc_lengths(rng, wl.T // 2, 2)
    cu = np.zeros(len(doc_lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(doc_lens, dtype=np.int64))
    assert int(cu[-1]) == wl.T
    a["cu_seqlens"] = cu
    return wl


def custom(T: int, Hq: int, Hkv: int, Dqk: int, Dv: int, Hi: int, Di: int, c: int, budget: int,
           doc_lens: list[int] | None = None, seed: int = 0, window: int = 0,
           w_kind: str = "uniform", name: str = "custom") -> Workload:
    """A small seeded workload of any shape (edge-case tests)."""
    wl = Workload(name, seed, T=T, Tk=T, Hq=Hq, Hkv=Hkv, Dqk=Dqk, Dv=Dv, scale=1.0 / math.sqrt(Dqk),
                  Hi=Hi, Di=Di, c=c, budget=budget, window=window)
    rng = np.random.default_rng(seed)
    a = wl.arrays
    a["q"] = _normal_bf16(rng, (T, Hq, Dqk))
    a["k"] = _normal_bf16(rng, (T, Hkv, Dqk))
    a["v"] = _normal_bf16(rng, (T, Hkv, Dv))
    a["qI"] = _normal_bf16(rng, (T, Hi, Di))
    a["kI"] = _normal_bf16(rng, (T, Di))
    if w_kind == "uniform":
        a["w"] = _uniform_f32(rng, (T, Hi))
    elif w_kind == "signed":
        a["w"] = (rng.random((T, Hi), dtype=np.float32) * np.float32(2.0) - np.float32(1.0)).astype(np.float32)
    elif w_kind == "ones":
        a["w"] = np.ones((T, Hi), dtype=np.float32)
    else:
        raise ValueError(w_kind)
    lens = [T] if doc_lens is None else list(doc_lens)
    assert sum(lens) == T and all(x > 0 for x in lens)
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    a["cu_seqlens"] = cu
    return wl


def front_half_inputs(T: int, Di: int, rope_dims: int, cu_seqlens: np.ndarray, seed: int = 0,
                      base: float = 10000.0, eps: float = 1e-6) -> dict:
    """Inputs of the indexer front half: RMSNorm weights for queries and keys (float32,
    U(0.5, 1.5)), eps, and a per-token rotary table [T, rope_dims] stored as
    cat(cos, sin). The table is what a model composes for document-local positions p
    (restarting at every document) with angles p * base^(-i / (rope_dims / 2)); here it
    is only a seeded input.
    """
    rng = np.random.default_rng(seed)
    q_weight = rng.uniform(0.5, 1.5, Di).astype(np.float32)
    k_weight = rng.uniform(0.5, 1.5, Di).astype(np.float32)
    cu = np.asarray(cu_seqlens, np.int64)
    t = np.arange(T, dtype=np.int64)
    pos = (t - cu[np.searchsorted(cu, t, side="right") - 1]).astype(np.float64)
    h = rope_dims // 2
    ang = pos[:, None] * base ** (-np.arange(h, dtype=np.float64) / h)[None, :]
    rope = np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)
    return dict(q_weight=q_weight, k_weight=k_weight, eps=eps, rope=rope)


def projection_inputs(T: int, H: int, Hi: int, Di: int, seed: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """Hidden states and the indexer's projection weights, bf16 bits: hidden [T, H] ~ N(0, 1)
    and weight [(Hi+1)*Di + Hi, H] ~ N(0, 1/H), so every projected value is about N(0, 1).
    Synthetic stand-ins for a model's activations and trained weights."""
    rng = np.random.default_rng(seed)
    hidden = np.empty((T, H), dtype=np.uint16)
    for r0 in range(0, T, _DRAW_ROWS):
        r1 = min(T, r0 + _DRAW_ROWS)
        hidden[r0:r1] = f32_to_bf16_bits(rng.standard_normal((r1 - r0, H), dtype=np.float32))
    N = (Hi + 1) * Di + Hi
    weight = f32_to_bf16_bits((rng.standard_normal((N, H), dtype=np.float32) * np.float32(1.0 / np.sqrt(H)))
                              .astype(np.float32))
    return hidden, weight


def compression_logits(T: int, Di: int, seed: int = 0, scale: float = 2.0) -> np.ndarray:
    """Step-5 compression logits shaped like the index keys: bf16 bits [T, Di] of
    scale * N(0, 1). scale 2 gives softmax weights that are neither flat nor one-hot over a
    region; 0 gives equal logits; a large scale gives near one-hot weights with underflow."""
    rng = np.random.default_rng(seed)
    out = np.empty((T, Di), dtype=np.uint16)
    for r0 in range(0, T, _DRAW_ROWS):
        r1 = min(T, r0 + _DRAW_ROWS)
        x = rng.standard_normal((r1 - r0, Di), dtype=np.float32) * np.float32(scale)
        out[r0:r1] = f32_to_bf16_bits(x.astype(np.float32))
    return out


def random_routes(rng: np.random.Generator, T: int, Tk: int, width: int, cu_seqlens: np.ndarray,
                  frac_invalid: float = 0.25) -> np.ndarray:
    """Arbitrary causal, document-confined routes with -1 holes at random slots.

    Row t holds distinct IDs from its own document prefix [s_d, t] in random
    order, with about `frac_invalid` of the slots set to -1 (attention tests that
    do not depend on the indexer).
    """
    out = np.full((T, width), -1, dtype=np.int32)
    cu = cu_seqlens.astype(np.int64)
    doc = np.searchsorted(cu, np.arange(T), side="right") - 1
    for t in range(T):
        s = int(cu[doc[t]])
        n_avail = t - s + 1
        n = min(width, n_avail)
        ids = s + rng.choice(n_avail, size=n, replace=False)
        slots = rng.permutation(width)[:n]
        keep = rng.random(n) >= frac_invalid
        if not keep.any():
            keep[0] = True
        out[t, slots[keep]] = ids[keep]
    return out


def as_torch(wl: Workload, device="cpu", pin: bool = False) -> dict:
    """Torch views of a workload's arrays (bf16 bits reinterpreted, no rounding)."""
    import torch

    out = {}
    for key, arr in wl.arrays.items():
        t = torch.from_numpy(np.ascontiguousarray(arr))
        if arr.dtype == np.uint16:
            t = t.view(torch.bfloat16)
        if pin:
            t = t.pin_memory()
        if device != "cpu":
            t = t.to(device, non_blocking=pin)
        out[key] = t
    return out
