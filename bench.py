"""Benchmark of the indexer-routed sparse attention hot path on GB300.

One step = one pass of the whole path over one batch of the windowed workload, the largest
single-GPU configuration that runs every stage (T=65536 single document, Hq=64, Hkv=4,
Dqk=192, Dv=128; indexer Hi=32, Di=128, c=64, top-16 regions; a 512-token causal window):
  sparse_index_score_topk (layout, pool, score, top-k + expansion) -> sparse_gqa_attn_fwd
  with the window (the window's keys are added inside the attention kernel).

Prints one JSON line (rank 0). `value` is the routed sparse-attention forward rate in
TFLOP/s over the whole step (algorithmic attention FLOPs / step time, inputs resident in
HBM, L2 flushed between timed steps); the indexer's queries/s, each kernel group's own rate,
cold- and warm-L2 times (mean and median) and the roofline of the dominant kernel, against
HBM and against an L2-aware bound, are reported beside it. `per_workload` repeats the
measurement for the other four workloads (tiny, mid, packed, latent). `--impl reference`
times the CPU oracle on a bounded row sample of the headline workload instead.

Multi-GPU: one process per GPU under torchrun; each rank runs its own replica of the
workload (weak scaling, no data-path collective); the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import irs_synth  # noqa: E402

METRIC = "routed sparse-attn fwd TFLOP/s & % roofline; indexer score+top-k queries/s"
WORKLOAD = "windowed"
L2_FLUSH_BYTES = 512 << 20    # > 129 MB L2


# --------------------------------------------------------------------------------------
# algorithmic counts (closed forms from the definitions; no GPU data involved)
# --------------------------------------------------------------------------------------
def valid_per_row(wl) -> np.ndarray:
    """Valid route entries of each row: min(nvis, kb)*c + (tau+1) % c."""
    cu = np.asarray(wl.cu_seqlens, np.int64)
    t = np.arange(wl.T, dtype=np.int64)
    s = cu[np.searchsorted(cu, t, side="right") - 1]
    tau = t - s
    nvis = (tau + 1) // wl.c
    kb = wl.budget // wl.c
    return np.minimum(nvis, kb) * wl.c + (tau + 1) % wl.c


def counts(wl, pairs: int | None = None) -> dict:
    """Algorithmic FLOPs and bytes of one step (closed forms from the definitions).

    The number of valid (query, key) pairs is the closed form min(nvis, kb)*c + (tau+1) % c per
    row, except where it depends on data: the latent workload's routes are an input (counted
    from them) and the windowed workload's window skips indexer IDs inside it (counted from
    the step's routes, passed in as `pairs`). The attention reads the indexer's route rows
    (budget + c - 1 wide); a window adds no reads.
    """
    if wl.latent:
        pairs = int(np.count_nonzero(np.asarray(wl.arrays["route"]) >= 0))
        attn_flops = 2.0 * (wl.Dqk + wl.Dv) * wl.Hq * pairs
        attn_bytes = (pairs * wl.Dqk * 2 + wl.T * wl.Hq * wl.Dqk * 2 + wl.T * wl.Hq * wl.Dv * 2 + wl.T * wl.Hq * 4
                      + wl.T * wl.route_width * 4)
        return dict(pairs=pairs, score_pairs=0, attn_flops=attn_flops, attn_bytes=attn_bytes, idx_flops=0.0,
                    idx_bytes=0, sparse_rows=0)
    if pairs is None:
        pairs = int(valid_per_row(wl).sum())
    cu = np.asarray(wl.cu_seqlens, np.int64)
    t = np.arange(wl.T, dtype=np.int64)
    s = cu[np.searchsorted(cu, t, side="right") - 1]
    nvis = (t - s + 1) // wl.c
    kb = wl.budget // wl.c
    sparse = nvis > kb
    score_pairs = int(nvis[sparse].sum())
    W = wl.budget + wl.c - 1
    attn_flops = 2.0 * (wl.Dqk + wl.Dv) * wl.Hq * pairs
    attn_bytes = (pairs * wl.Hkv * (wl.Dqk + wl.Dv) * 2          # gathered K and V rows
                  + wl.T * wl.Hq * wl.Dqk * 2                     # Q
                  + wl.T * wl.Hq * wl.Dv * 2                      # O
                  + wl.T * wl.Hq * 4                              # lse
                  + wl.T * W * 4)                                 # routes
    idx_flops = 2.0 * wl.Hi * wl.Di * score_pairs
    W_idx = wl.budget + wl.c - 1
    idx_bytes = (wl.T * wl.Hi * wl.Di * 2 + wl.T * wl.Di * 2 + wl.T * wl.Hi * 4 + wl.T * W_idx * 4)
    return dict(pairs=pairs, score_pairs=score_pairs, attn_flops=attn_flops, attn_bytes=attn_bytes,
                idx_flops=idx_flops, idx_bytes=idx_bytes, sparse_rows=int(sparse.sum()))


def describe(wl) -> str:
    if wl.latent:
        return (f"{wl.name}: {wl.T} queries x {wl.Hq} heads x {wl.Dqk}, latent {wl.Tk} x {wl.Dqk}, Dv {wl.Dv}, "
                f"route width {wl.route_width}, seed {wl.seed}")
    docs = f"{wl.ndocs} documents" if wl.ndocs > 1 else "single document"
    win = f", window {wl.window}" if wl.window else ""
    return (f"{wl.name} ({docs}): T={wl.T} Hq={wl.Hq} Hkv={wl.Hkv} Dqk={wl.Dqk} Dv={wl.Dv}, indexer Hi={wl.Hi} "
            f"Di={wl.Di} c={wl.c} budget={wl.budget}{win} (route width {wl.route_width}), scale 1/sqrt({wl.Dqk}), "
            f"seed {wl.seed}")


def profile_traffic(name: str, source: str) -> int | None:
    """DRAM bytes per launch recorded by the committed ncu summary, if it was taken on the
    kernel source as it is now (else None)."""
    import hashlib

    prof = os.path.join(ROOT, "profiles", name)
    src = os.path.join(ROOT, source)
    if not (os.path.exists(prof) and os.path.exists(src)):
        return None
    rec = {}
    with open(prof) as f:
        for line in f:
            if ":" in line and not line.startswith(("|", "#")):
                k, _, v = line.partition(":")
                rec[k.strip()] = v.strip()
    cur = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    if rec.get("source_sha256_16") != cur or "dram_bytes_per_launch" not in rec:
        return None
    return int(rec["dram_bytes_per_launch"])


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


# --------------------------------------------------------------------------------------
# clocks sampled during the timed region
# --------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.proc = None
        self.uuid = uuid

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(x: float, world: int, device) -> float:
    """Max of a host float over ranks (identity for one rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def measure_l2_gbs(dev, stream) -> tuple[float, str]:
    """L2 bandwidth measured live, the better of two L2-resident torch ops, each replayed 20
    times from a CUDA graph (no launch gaps), best of 5 replays:
    a 16 MiB -> 16 MiB copy (read + write bytes) and a column sum over a 48 MiB fp32
    matrix (read bytes)."""
    import torch

    best = (0.0, "none")
    a = torch.ones(8 << 20, dtype=torch.bfloat16, device=dev)
    b = torch.empty_like(a)
    x = torch.ones((3072, 4096), dtype=torch.float32, device=dev)
    col = torch.empty(4096, dtype=torch.float32, device=dev)
    probes = (("copy 16 MiB -> 16 MiB", lambda: b.copy_(a), 2.0 * a.numel() * a.element_size()),
              ("column sum of 48 MiB", lambda: torch.sum(x, dim=0, out=col), float(x.numel() * x.element_size())))
    for name, fn, nbytes in probes:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for _ in range(5):
                fn()
        stream.wait_stream(side)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(20):
                fn()
        g.replay()
        torch.cuda.synchronize(dev)
        t_best = float("inf")
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            e1.synchronize()
            t_best = min(t_best, e0.elapsed_time(e1) * 1e-3 / 20)
        gbs = nbytes / t_best / 1e9
        if gbs > best[0]:
            best = (gbs, name)
        del g
    return best


class Path:
    """Device buffers and the two halves of one step (indexer, attention) for a workload."""

    def __init__(self, irs, wl, dev, want_host: bool = False):
        import torch

        self.irs, self.wl, self.dev = irs, wl, dev
        host = irs_synth.as_torch(wl, device="cpu", pin=want_host)
        self.host = host if want_host else None
        self.d = {k: v.to(dev) for k, v in host.items()}
        T = wl.T
        self.out = torch.empty((T, wl.Hq, wl.Dv), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((T, wl.Hq), dtype=torch.float32, device=dev)
        self.err = irs.device_error_flag(dev)
        self.has_index = not wl.latent
        if self.has_index:
            W_idx = wl.budget + wl.c - 1
            self.route_idx = torch.empty((T, W_idx), dtype=torch.int32, device=dev)
            # the windowed workload's window is added by the attention kernel itself
            self.route = self.route_idx
            self.ws = torch.empty(irs.index_workspace_bytes(T, wl.Hi, wl.Di, wl.c, wl.budget, wl.ndocs,
                                                            wl.max_doc_len, True), dtype=torch.uint8, device=dev)
        else:
            self.route = self.d["route"]
        self.kv_v = self.d["kv"][:, :, :wl.Dv] if wl.latent else None
        self.kernels_per_step = path_kernels(wl)

    def index(self, d=None):
        wl = self.wl
        d = self.d if d is None else d
        if not self.has_index:
            return
        self.irs.sparse_index_score_topk(d["qI"], d["kI"], d["w"], d["cu_seqlens"], wl.c, wl.budget, ndocs=wl.ndocs,
                                         max_doc_len=wl.max_doc_len, out=self.route_idx, workspace=self.ws,
                                         err=self.err)

    def attend(self, d=None, out=None, lse=None):
        wl = self.wl
        d = self.d if d is None else d
        out = self.out if out is None else out
        lse = self.lse if lse is None else lse
        if wl.latent:
            route = d["route"]
            kv_v = d["kv"][:, :, :wl.Dv]
            self.irs.sparse_gqa_attn_fwd(d["q"], d["kv"], kv_v, route, wl.scale, out=out, lse=lse, err=self.err)
        elif wl.window:
            self.irs.sparse_gqa_attn_fwd(d["q"], d["k"], d["v"], self.route, wl.scale, window=wl.window,
                                         cu_seqlens=d["cu_seqlens"], ndocs=wl.ndocs, out=out, lse=lse, err=self.err)
        else:
            self.irs.sparse_gqa_attn_fwd(d["q"], d["k"], d["v"], self.route, wl.scale, out=out, lse=lse,
                                         err=self.err)

    def unique_kv_rows(self) -> int:
        """Distinct key rows the step's routes touch (outside any timed region)."""
        import torch

        r = self.route
        ids = r[(r >= 0) & (r < self.wl.Tk)].long()
        mask = torch.zeros(self.wl.Tk, dtype=torch.bool, device=self.dev)
        mask[ids] = True
        if self.has_index and self.wl.window:
            mask[:self.wl.T] = True   # every token is in its own query's window
        return int(mask.sum().item())

    def valid_pairs(self) -> int | None:
        """Valid pairs where they depend on data (the windowed workload: the window's tokens
        plus the route IDs before it); else None."""
        import torch

        wl = self.wl
        if not (self.has_index and wl.window):
            return None
        t = torch.arange(wl.T, device=self.dev, dtype=torch.int64)
        cu = self.d["cu_seqlens"].long()
        s = cu[torch.searchsorted(cu, t, right=True) - 1]
        lo_w = t - wl.window + 1
        nwin = t - torch.maximum(s, lo_w) + 1
        r = self.route
        routed = ((r >= 0) & (r.long() < lo_w[:, None])).sum()
        return int((nwin.sum() + routed).item())


def time_steps(path: Path, steps: int, flush, stream, cold: bool):
    """Per-step device times (ms) of the indexer half and the attention half, with CUDA
    events on the launching stream; `cold` writes a buffer larger than L2 before each step."""
    import torch

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    torch.cuda.synchronize(path.dev)
    for i in range(steps):
        if cold:
            flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        path.index()
        ev[i][1].record(stream)
        path.attend()
        ev[i][2].record(stream)
    torch.cuda.synchronize(path.dev)
    idx = np.asarray([e[0].elapsed_time(e[1]) for e in ev])
    att = np.asarray([e[1].elapsed_time(e[2]) for e in ev])
    return idx, att


def attention_report(wl, cnt, att_ms, att_warm_ms, peaks, l2_gbs, unique_rows) -> dict:
    """Attention rates and both rooflines for one workload (times in ms, per launch group).

    HBM roofline (the spec definition): every gathered K/V byte plus Q, O, lse and
    routes at the measured HBM copy bandwidth, or the FLOPs at the bf16 peak if slower.
    L2-aware roofline: the distinct K/V rows (plus Q, O, lse, routes) must come from HBM
    while every gathered byte passes through L2, at the L2 bandwidth measured live
    (measure_l2_gbs); the bound is the slowest of those two and the tensor time.
    """
    att_s = float(np.mean(att_ms)) * 1e-3
    rows_bytes = (wl.Dqk * 2) if wl.latent else wl.Hkv * (wl.Dqk + wl.Dv) * 2
    other_bytes = cnt["attn_bytes"] - cnt["pairs"] * rows_bytes
    t_hbm = cnt["attn_bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_tc = cnt["attn_flops"] / (peaks["bf16_tflops"] * 1e12)
    roof_s = max(t_hbm, t_tc)
    uniq_bytes = unique_rows * rows_bytes + other_bytes
    t_uniq = uniq_bytes / (peaks["hbm_gbs"] * 1e9)
    t_l2 = cnt["attn_bytes"] / (l2_gbs * 1e9)
    l2_roof_s = max(t_uniq, t_l2, t_tc)
    l2_bound = "hbm (distinct rows)" if l2_roof_s == t_uniq else ("l2" if l2_roof_s == t_l2 else "tensor")
    frac = roof_s / att_s
    rep = {"ms": round(att_s * 1e3, 4), "ms_median": round(float(np.median(att_ms)), 4),
           "ms_warm_l2": round(float(np.mean(att_warm_ms)), 4),
           "ms_warm_l2_median": round(float(np.median(att_warm_ms)), 4),
           "tflops": round(cnt["attn_flops"] / att_s / 1e12, 3),
           "routed_pairs_per_s": round(cnt["pairs"] * wl.Hq / att_s, 1),
           "valid_pairs": cnt["pairs"], "flops": cnt["attn_flops"], "algorithmic_bytes": int(cnt["attn_bytes"]),
           "roofline_bound": "hbm" if t_hbm >= t_tc else "tensor", "roofline_ms": round(roof_s * 1e3, 4),
           "roofline_frac": round(frac, 4),
           "l2_aware": {"bound": l2_bound, "roofline_ms": round(l2_roof_s * 1e3, 4),
                        "frac": round(l2_roof_s / att_s, 4), "distinct_kv_rows": int(unique_rows),
                        "distinct_bytes": int(uniq_bytes), "l2_gbs": round(l2_gbs, 1)}}
    if frac > 1.0:
        rep["note"] = ("bound not binding: the gathered K/V rows are re-read from L2, so the HBM roofline "
                       "understates what the kernel can reach; see l2_aware")
    return rep


def indexer_report(wl, cnt, idx_ms, idx_warm_ms, peaks) -> dict:
    idx_s = float(np.mean(idx_ms)) * 1e-3
    t_hbm = cnt["idx_bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_tc = cnt["idx_flops"] / (peaks["bf16_tflops"] * 1e12)
    roof_s = max(t_hbm, t_tc)
    return {"ms": round(idx_s * 1e3, 4), "ms_median": round(float(np.median(idx_ms)), 4),
            "ms_warm_l2": round(float(np.mean(idx_warm_ms)), 4),
            "queries_per_s": round(wl.T / idx_s, 1), "tflops": round(cnt["idx_flops"] / idx_s / 1e12, 3),
            "roofline_bound": "hbm" if t_hbm >= t_tc else "tensor",
            "roofline_frac": round(roof_s / idx_s, 4), "roofline_us": round(roof_s * 1e6, 2),
            "algorithmic_bytes": int(cnt["idx_bytes"]), "flops": cnt["idx_flops"],
            "window": "added inside the attention kernel" if wl.window else None}


def measure_other_workload(irs, name, args, dev, stream, flush, peaks, l2_gbs) -> dict:
    """One workload other than the headline one: cold and warm step times, attention and
    indexer rates and rooflines (no end-to-end leg, no CPU baseline)."""
    import torch

    wl = irs_synth.make(name)
    path = Path(irs, wl, dev)
    for _ in range(args.warmup):
        path.index()
        path.attend()
    torch.cuda.synchronize(dev)
    irs.check_device_errors(dev)
    cnt = counts(wl, path.valid_pairs())
    uniq = path.unique_kv_rows()
    steps = max(3, min(args.steps, 20))
    idx_ms, att_ms = time_steps(path, steps, flush, stream, cold=True)
    idx_w, att_w = time_steps(path, steps, flush, stream, cold=False)
    irs.check_device_errors(dev)
    rep = {"workload": describe(wl), "steps": steps,
           "ms_per_step": round(float(np.mean(idx_ms + att_ms)), 4),
           "kernels_per_step": path.kernels_per_step,
           "attention": attention_report(wl, cnt, att_ms, att_w, peaks, l2_gbs, uniq)}
    if path.has_index:
        rep["indexer"] = indexer_report(wl, cnt, idx_ms, idx_w, peaks)
    del path
    torch.cuda.empty_cache()
    return rep


def measure_indexer_variants(irs, wl, d, dev, stream, flush, peaks, steps: int) -> dict:
    """The indexer rows beyond the plain one, on the headline workload's indexer shape
    (T, Hi, Di, c, budget, documents), each timed cold (L2 flushed before every call):
    the projections from hidden states (one GEMM, synthetic hidden size 4096), the QSA front half (RMSNorm + RoPE, 64 rotary dims), FP8 E4M3 operands, per-KV-group
    selection (G = Hkv groups of Hi heads), and the Step-5 configuration (learned-logit
    summaries, E4M3 queries, per group). Grouped queries, weights and the compression logits
    come from a seeded device generator. Roofline: the score FLOPs at the tensor peak of the
    operand type (E4M3 at twice the measured bf16 rate, the nominal ratio) or the
    algorithmic bytes at the HBM rate, whichever is slower."""
    import torch

    T, Hi, Di, c, budget, G = wl.T, wl.Hi, wl.Di, wl.c, wl.budget, max(wl.Hkv, 1)
    W = budget + c - 1
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234)
    qg = torch.empty((T, G, Hi, Di), dtype=torch.bfloat16, device=dev)
    for r0 in range(0, T, 4096):
        r1 = min(T, r0 + 4096)
        qg[r0:r1] = torch.randn((r1 - r0, G, Hi, Di), generator=gen, device=dev, dtype=torch.float32)
    wg = torch.rand((T, G, Hi), generator=gen, device=dev, dtype=torch.float32)
    z = (2.0 * torch.randn((T, Di), generator=gen, device=dev, dtype=torch.float32)).to(torch.bfloat16)
    fr = irs_synth.front_half_inputs(T, Di, 64, wl.cu_seqlens, seed=5)
    front = {k: (torch.from_numpy(v).to(dev) if isinstance(v, np.ndarray) else v) for k, v in fr.items()}
    err = irs.device_error_flag(dev)
    kw = dict(ndocs=wl.ndocs, max_doc_len=wl.max_doc_len, err=err)
    score_pairs = counts(wl)["score_pairs"]
    base_bytes = T * Hi * Di * 2 + T * Di * 2 + T * Hi * 4 + T * W * 4
    variants = {
        "front_half": (lambda: irs.sparse_index_score_topk(d["qI"], d["kI"], d["w"], d["cu_seqlens"], c, budget,
                                                           front=front, **kw),
                       1, "bf16", base_bytes + T * 64 * 4 + 2 * Di * 4),
        "e4m3": (lambda: irs.sparse_index_score_topk(d["qI"], d["kI"], d["w"], d["cu_seqlens"], c, budget,
                                                     operands="e4m3", **kw), 1, "e4m3", base_bytes),
        f"grouped_g{G}": (lambda: irs.sparse_index_score_topk_grouped(qg, d["kI"], wg, d["cu_seqlens"], c, budget,
                                                                      **kw),
                          G, "bf16", G * (T * Hi * Di * 2 + T * Hi * 4 + T * W * 4) + T * Di * 2),
        f"step5_summaries_e4m3_g{G}": (lambda: irs.sparse_index_score_topk_summaries(
            qg, d["kI"], z, wg, d["cu_seqlens"], c, budget, operands="e4m3", **kw),
            G, "e4m3", G * (T * Hi * Di * 2 + T * Hi * 4 + T * W * 4) + 2 * T * Di * 2),
    }
    out = {}
    # the indexer's projections from hidden states (synthetic hidden size 4096): one GEMM
    H = 4096
    N = (Hi + 1) * Di + Hi
    hid = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    for r0 in range(0, T, 8192):
        r1 = min(T, r0 + 8192)
        hid[r0:r1] = torch.randn((r1 - r0, H), generator=gen, device=dev, dtype=torch.float32)
    wproj = (torch.randn((N, H), generator=gen, device=dev, dtype=torch.float32) / H ** 0.5).to(torch.bfloat16)
    proj_out = (torch.empty((T, Hi, Di), dtype=torch.bfloat16, device=dev),
                torch.empty((T, Di), dtype=torch.bfloat16, device=dev),
                torch.empty((T, Hi), dtype=torch.float32, device=dev))
    proj = lambda: irs.indexer_projection(hid, wproj, Hi, Di, out=proj_out, err=err)
    for _ in range(3):
        proj()
    torch.cuda.synchronize(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for i in range(steps):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        proj()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    irs.check_device_errors(dev)
    ms = np.asarray([e[0].elapsed_time(e[1]) for e in ev])
    sec = float(np.mean(ms)) * 1e-3
    flops = 2.0 * T * H * N
    pbytes = T * H * 2 + N * H * 2 + T * (Hi + 1) * Di * 2 + T * Hi * 4
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    t_hbm = pbytes / (peaks["hbm_gbs"] * 1e9)
    out["projection_h4096"] = {"ms": round(sec * 1e3, 4), "ms_median": round(float(np.median(ms)), 4),
                               "tflops": round(flops / sec / 1e12, 1), "hidden_size": H, "output_columns": N,
                               "roofline_bound": "tensor" if t_tc >= t_hbm else "hbm",
                               "roofline_frac": round(max(t_tc, t_hbm) / sec, 4),
                               "tensor_peak_tflops": round(peaks["bf16_tflops"], 1)}
    # projection then the front-half indexer: the queries' front half as its own pass, or
    # fused into the projection's epilogue
    def pipeline(fused: bool):
        if fused:
            q, k, wv = irs.indexer_projection(hid, wproj, Hi, Di, front=front, out=proj_out, err=err)
            return irs.sparse_index_score_topk(q, k, wv, d["cu_seqlens"], c, budget, front=front, queries_ready=True,
                                               **kw)
        q, k, wv = irs.indexer_projection(hid, wproj, Hi, Di, out=proj_out, err=err)
        return irs.sparse_index_score_topk(q, k, wv, d["cu_seqlens"], c, budget, front=front, **kw)
    for fused in (False, True):
        for _ in range(3):
            pipeline(fused)
        torch.cuda.synchronize(dev)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        for i in range(steps):
            flush.fill_(i & 0xFF)
            ev[i][0].record(stream)
            pipeline(fused)
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        irs.check_device_errors(dev)
        ms = np.asarray([e[0].elapsed_time(e[1]) for e in ev])
        key = "projection_front_fused_then_indexer_h4096" if fused else "projection_then_front_half_indexer_h4096"
        out[key] = {"ms": round(float(np.mean(ms)), 4), "ms_median": round(float(np.median(ms)), 4),
                    "queries_per_s": round(T / (float(np.mean(ms)) * 1e-3), 1)}
    del hid, wproj, proj_out
    for name, (fn, groups, dtype, nbytes) in variants.items():
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        for i in range(steps):
            flush.fill_(i & 0xFF)
            ev[i][0].record(stream)
            fn()
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        irs.check_device_errors(dev)
        ms = np.asarray([e[0].elapsed_time(e[1]) for e in ev])
        sec = float(np.mean(ms)) * 1e-3
        flops = 2.0 * Hi * Di * score_pairs * groups
        tc_peak = peaks["bf16_tflops"] * (2.0 if dtype == "e4m3" else 1.0)
        t_tc = flops / (tc_peak * 1e12)
        t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
        roof = max(t_tc, t_hbm)
        out[name] = {"ms": round(sec * 1e3, 4), "ms_median": round(float(np.median(ms)), 4),
                     "queries_per_s": round(T / sec, 1), "groups": groups, "operands": dtype,
                     "tflops": round(flops / sec / 1e12, 3), "roofline_bound": "tensor" if t_tc >= t_hbm else "hbm",
                     "roofline_frac": round(roof / sec, 4),
                     "tensor_peak_tflops": round(tc_peak, 1) if dtype == "bf16" else
                     f"{2 * peaks['bf16_tflops']:.1f} (2x measured bf16, nominal E4M3 ratio)"}
    del qg, wg, z
    return out


def e2e_pipelined(path, steps: int, flush, stream, dev, warmup: int = 2) -> float:
    """Mean ms per step end to end through the public API with host buffers, copies
    overlapped with compute: inputs and outputs are double-buffered on the device; step
    i+1's host-to-device copies (pinned memory, their own stream) and step i-1's
    device-to-host copies (another stream) run while step i computes. Every step copies
    all of its inputs in and its outputs (out, lse) back; L2 is flushed before each step's
    compute. The first `warmup` steps (which touch every buffer once) run untimed; the
    timed region runs from the first timed step's first copy to the last copy's end."""
    import torch

    host = path.host
    sets = [path.d, {k: torch.empty_like(v) for k, v in path.d.items()}]
    outs = [(path.out, path.lse), (torch.empty_like(path.out), torch.empty_like(path.lse))]
    outs_h = [(torch.empty(path.out.shape, dtype=path.out.dtype, pin_memory=True),
               torch.empty(path.lse.shape, dtype=path.lse.dtype, pin_memory=True)) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    in_ready, in_free, done, out_free = [ev(), ev()], [ev(), ev()], [ev(), ev()], [ev(), ev()]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    for i in range(warmup + steps):
        b = i & 1
        if i == warmup:
            s_in.wait_stream(s_out)                # the warm-up steps have left the device
            s_in.wait_stream(stream)
            start.record(s_in)
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(in_free[b])        # step i-2 no longer reads this input set
            for k_, v_ in host.items():
                sets[b][k_].copy_(v_, non_blocking=True)
            in_ready[b].record(s_in)
        stream.wait_event(in_ready[b])
        if i >= 2:
            stream.wait_event(out_free[b])         # step i-2's outputs have left this set
        flush.fill_(i & 0xFF)
        path.index(sets[b])
        path.attend(sets[b], *outs[b])
        in_free[b].record(stream)
        done[b].record(stream)
        s_out.wait_event(done[b])
        with torch.cuda.stream(s_out):
            outs_h[b][0].copy_(outs[b][0], non_blocking=True)
            outs_h[b][1].copy_(outs[b][1], non_blocking=True)
            out_free[b].record(s_out)
    s_out.wait_stream(s_in)
    end.record(s_out)
    end.synchronize()
    return start.elapsed_time(end) / steps


def run_variants_only(args) -> dict:
    """The indexer variants alone on the workload's indexer inputs (qI, kI, w, cu_seqlens)."""
    import torch

    import indexer_routed_sparse_gb300 as irs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    irs.lib()
    wl = irs_synth.make(args.workload, small=args.small)
    if wl.latent:
        raise SystemExit("the latent workload has no indexer")
    keys = ("qI", "kI", "w", "cu_seqlens")
    host = irs_synth.as_torch(wl, device="cpu")
    d = {k: host[k].to(dev) for k in keys}
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    variants = measure_indexer_variants(irs, wl, d, dev, torch.cuda.current_stream(dev), flush, load_peaks(),
                                        max(3, min(args.steps, 20)))
    return {"workload": describe(wl), "indexer_variants": variants}


def run_gpu(args) -> dict | None:
    import torch

    import indexer_routed_sparse_gb300 as irs

    world, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    irs.lib()
    wl = irs_synth.make(args.workload, small=args.small)
    peaks = load_peaks()
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    l2_gbs, l2_probe = measure_l2_gbs(dev, stream)

    path = Path(irs, wl, dev, want_host=True)
    for _ in range(args.warmup):
        path.index()
        path.attend()
    torch.cuda.synchronize(dev)
    irs.check_device_errors(dev)
    cnt = counts(wl, path.valid_pairs())
    uniq = path.unique_kv_rows()

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        if not uuid.startswith("GPU-"):
            uuid = "GPU-" + uuid
    except Exception:
        uuid = None
    clocks = ClockSampler(uuid if rank == 0 else None)
    if rank == 0:
        clocks.start()

    # ---- device-timed region: K steps, L2 flushed before each, per-kernel-group events ----
    barrier(world)
    wall0 = time.perf_counter()
    idx_ms, att_ms = time_steps(path, args.steps, flush, stream, cold=True)
    barrier(world)
    wall = time.perf_counter() - wall0
    step_ms = reduce_max(float(np.mean(idx_ms + att_ms)), world, dev)
    irs.check_device_errors(dev)
    # the same steps without the flush (L2 keeps what the previous step left)
    idx_w, att_w = time_steps(path, max(3, args.steps // 2), flush, stream, cold=False)

    # ---- end to end through the public API with host buffers ----
    host = path.host
    out_h = torch.empty(path.out.shape, dtype=path.out.dtype, pin_memory=True)
    lse_h = torch.empty(path.lse.shape, dtype=path.lse.dtype, pin_memory=True)
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()
    e2e_steps = max(3, args.steps // 2)
    ee = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(e2e_steps)]
    # untimed warm-up steps: the first copies into freshly pinned buffers pay for the
    # buffers' first use, which is not a per-step cost
    for _ in range(2):
        for k_, v_ in host.items():
            path.d[k_].copy_(v_, non_blocking=True)
        path.index()
        path.attend()
        out_h.copy_(path.out, non_blocking=True)
        lse_h.copy_(path.lse, non_blocking=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    for i in range(e2e_steps):
        flush.fill_(i & 0xFF)
        ee[i][0].record(stream)
        for k_, v_ in host.items():
            path.d[k_].copy_(v_, non_blocking=True)
        path.index()
        path.attend()
        out_h.copy_(path.out, non_blocking=True)
        lse_h.copy_(path.lse, non_blocking=True)
        ee[i][1].record(stream)
        ee[i][1].synchronize()
    barrier(world)
    e2e_serial_ms = reduce_max(float(np.mean([ee[i][0].elapsed_time(ee[i][1]) for i in range(e2e_steps)])), world,
                               dev)
    barrier(world)
    e2e_ms = reduce_max(e2e_pipelined(path, e2e_steps, flush, stream, dev), world, dev)
    barrier(world)
    variants = None
    if not args.no_per_workload and not args.small and args.workload == WORKLOAD and not wl.latent:
        variants = measure_indexer_variants(irs, wl, path.d, dev, stream, flush, peaks, max(3, min(args.steps, 20)))
    bwd = time_backward(args, wl, irs, path.d, path.route, path.kv_v, path.out, path.lse, flush, path.err, stream,
                        dev) if args.with_backward else None
    clk = clocks.stop() if rank == 0 else None
    irs.check_device_errors(dev)

    attn = attention_report(wl, cnt, att_ms, att_w, peaks, l2_gbs, uniq)
    att_avg_s = float(np.mean(att_ms)) * 1e-3
    value = world * cnt["attn_flops"] / (step_ms * 1e-3) / 1e12
    if attn["roofline_bound"] == "hbm":
        achieved = cnt["attn_bytes"] / att_avg_s / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4)}
    else:
        achieved = cnt["attn_flops"] / att_avg_s / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(achieved / peaks["bf16_tflops"], 4)}
    # the latent workload runs on the latent-attention kernel, the others on the GQA kernel
    kname, ksrc = (("mla_fwd_kernel", "irs_mla.cu") if wl.latent else ("attn_fwd_kernel", "irs_attn.cu"))
    kprof = f"{kname.replace('_kernel', '')}_{wl.name}{'_small' if args.small else ''}.md"
    roof.update({"traffic": profile_traffic(kprof, f"indexer_routed_sparse_gb300/csrc/{ksrc}"),
                 "kernel": kname, "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs, burst)",
                 "l2_aware_frac": attn["l2_aware"]["frac"], "l2_aware_bound": attn["l2_aware"]["bound"]})
    if roof["frac"] > 1.0:
        roof["note"] = "bound not binding (gathered rows re-read from L2): see l2_aware_frac"
    del path
    torch.cuda.empty_cache()
    per_workload = {}
    if not args.no_per_workload and not args.small and args.workload == WORKLOAD:
        for name in irs_synth.WORKLOADS:
            if name != WORKLOAD:
                per_workload[name] = measure_other_workload(irs, name, args, dev, stream, flush, peaks, l2_gbs)

    if rank != 0:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()
        return None
    res = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 4),
        "ms_per_step_median": round(float(np.median(idx_ms + att_ms)), 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 inputs, U(0,1) fp32 head weights)",
        "config": {"workload": describe(wl), "l2": "flushed (512 MiB write) before every timed step",
                   "l2_bandwidth_probe": f"{l2_probe}: {l2_gbs:.0f} GB/s",
                   "parallelism": f"replicas x{world}"},
        "roofline": roof,
        "attention": attn,
        "e2e": {"value": round(world * cnt["attn_flops"] / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "steps": e2e_steps,
                "overlap": "double-buffered: step i+1's host-to-device copies and step i-1's device-to-host "
                           "copies run on their own streams while step i computes",
                "serial_ms_per_step": round(e2e_serial_ms, 4),
                "serial_value": round(world * cnt["attn_flops"] / (e2e_serial_ms * 1e-3) / 1e12, 3)},
        "gpu_launches": path_kernels(wl) * args.steps,
        "clocks": clk,
        "wall_s_timed": round(wall, 3),
    }
    if not wl.latent:
        res["indexer"] = indexer_report(wl, cnt, idx_ms, idx_w, peaks)
    if variants is not None:
        res["indexer_variants"] = variants
    if bwd is not None:
        res["backward"] = backward_report(wl, cnt, bwd, peaks)
    if per_workload:
        res["per_workload"] = per_workload
    if not args.no_cpu_baseline and world == 1 and args.workload == WORKLOAD and not args.small:
        res["cpu_baseline"] = cpu_baseline(wl, cnt, budget_s=args.cpu_seconds, small=args.small)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return res


def path_kernels(wl) -> int:
    """Our kernels launched per step: layout, pool, score, top-k and one attention launch per
    8 KV heads (the window, where there is one, is added inside the attention kernel)."""
    return (0 if wl.latent else 4) + (wl.Hkv + 7) // 8


def time_backward(args, wl, irs, d, route, kv_v, out, lse, flush, err, stream, dev) -> float:
    """Mean device time (s) of one sparse_gqa_attn_bwd call (accumulators zeroed inside the
    call's timed region, L2 flushed before each), on the step's routes and forward outputs."""
    import torch

    gen = torch.Generator(device=dev)
    gen.manual_seed(wl.seed + 1000)
    dout = torch.randn(out.shape, generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
    if wl.window:
        # the forward attended the window in front of each route: its backward takes the
        # composed route (window + route), built once outside the timed region
        route = irs.compose_window_routes(route, d["cu_seqlens"], wl.window)
    k, v = (d["kv"], kv_v) if wl.latent else (d["k"], d["v"])
    dq = torch.empty((wl.T, wl.Hq, wl.Dqk), dtype=torch.float32, device=dev)
    dk = torch.empty((wl.Tk, wl.Hkv, wl.Dqk), dtype=torch.float32, device=dev)
    dv = None if wl.latent else torch.empty((wl.Tk, wl.Hkv, wl.Dv), dtype=torch.float32, device=dev)

    def backward():
        dk.zero_()
        if dv is not None:
            dv.zero_()
        irs.sparse_gqa_attn_bwd(d["q"], k, v, route, out, lse, dout, wl.scale, dq=dq, dk=dk, dv=dv, err=err)

    for _ in range(args.warmup):
        backward()
    torch.cuda.synchronize(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        backward()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    irs.check_device_errors(dev)
    return float(np.mean([e[0].elapsed_time(e[1]) for e in ev])) * 1e-3


def backward_kernel_name(wl) -> str:
    """The kernel sparse_gqa_attn_bwd launches for this shape: the tensor-core kernel for
    separate K and V whose tiles fit (dims multiples of 64 up to 256, TMEM and shared-memory
    budgets) with 8 or more query heads per KV head; else the CUDA-core warp-per-row kernel
    for the listed dims; else the tensor-core kernel if it fits, else the staged CUDA-core
    kernel (latent rows)."""
    if wl.latent:
        return "attn_bwd_kernel"
    W = wl.route_width
    smem = (512 * (wl.Dqk + wl.Dv) + 32 * (wl.Dqk + wl.Dv) + 2 * 128 * 128 + 2 * 16 * 128 + ((4 * W + 15) & ~15)
            + 4 * 16 * 36 * 4 + 1392)
    tc = (wl.Dqk % 64 == 0 and wl.Dv % 64 == 0 and max(wl.Dqk, wl.Dv) <= 256 and 96 + wl.Dqk + wl.Dv <= 512
          and smem <= 227 * 1024)
    if tc and min(wl.Hq // wl.Hkv, 16) >= 8:
        return "attn_bwd_tc_kernel"
    fast_dims = {(64, 64), (64, 128), (128, 128), (128, 256), (192, 128)}
    if (wl.Dqk, wl.Dv) in fast_dims:
        return "attn_bwd_fast_kernel"
    return "attn_bwd_tc_kernel" if tc else "attn_bwd_kernel"


def backward_report(wl, cnt, bwd_s: float, peaks: dict) -> dict:
    """Backward rate against the forward's roofline definition.

    FLOPs per (valid pair, query head): s and dp (2 Dqk + 2 Dv), dq and dk (4 Dqk) and dv
    (2 Dv). Bytes: the gathered K/V rows of every valid pair (as in the forward), q, dout,
    out, lse and dq per query head, the routes, and dk/dv written once.
    """
    rows = 1 if wl.latent else wl.Hkv
    kv_dims = wl.Dqk + (0 if wl.latent else wl.Dv)
    flops = cnt["pairs"] * wl.Hq * 2.0 * (3 * wl.Dqk + 2 * wl.Dv)
    nbytes = (cnt["pairs"] * rows * kv_dims * 2
              + wl.T * wl.Hq * (wl.Dqk * 2 + 2 * wl.Dv * 2 + 4 + wl.Dqk * 4)
              + wl.T * wl.route_width * 4
              + wl.Tk * rows * kv_dims * 4)
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    roof_s = max(t_hbm, t_tc)
    return {"ms": round(bwd_s * 1e3, 4), "tflops": round(flops / bwd_s / 1e12, 3),
            "gbs": round(nbytes / bwd_s / 1e9, 1), "bound": "hbm" if t_hbm >= t_tc else "tensor",
            "roofline_ms": round(roof_s * 1e3, 4), "roofline_frac": round(roof_s / bwd_s, 4),
            "algorithmic_bytes": int(nbytes), "flops": flops, "kernel": backward_kernel_name(wl),
            "launches_per_call": 1,
            "note": "timed separately, not part of the step or of value"}


# --------------------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)
# --------------------------------------------------------------------------------------
_WL = None


def _worker_init(name: str = WORKLOAD, small: bool = False, meta=None, shared_dir: str | None = None):
    """Worker set-up: the workload's arrays mapped read-only from `shared_dir` (written once
    by the parent), or drawn again from the seeded recipe when there is none."""
    global _WL
    if shared_dir is None:
        _WL = irs_synth.make(name, small=small)
        return
    arrays = {f[:-4]: np.load(os.path.join(shared_dir, f), mmap_mode="r")
              for f in os.listdir(shared_dir) if f.endswith(".npy")}
    _WL = dataclasses.replace(meta, arrays=arrays)


def share_arrays(wl) -> str | None:
    """Write the workload's arrays once to a temporary directory (in /dev/shm when it has
    room) so that the oracle's worker processes map them instead of drawing them again."""
    import shutil
    import tempfile

    need = sum(int(v.nbytes) for v in wl.arrays.values()) * 1.2 + (64 << 20)
    base = None
    if os.path.isdir("/dev/shm") and shutil.disk_usage("/dev/shm").free > need:
        base = "/dev/shm"
    elif shutil.disk_usage(tempfile.gettempdir()).free <= need:
        return None
    d = tempfile.mkdtemp(prefix="irs_oracle_", dir=base)
    for k, v in wl.arrays.items():
        np.save(os.path.join(d, k + ".npy"), np.ascontiguousarray(v))
    return d


def _oracle_rows(rows) -> int:
    """Indexer + attention of the oracle on some rows; returns their valid route entries."""
    from oracle import irs_oracle as O

    wl = _WL
    a = wl.arrays
    rows = np.asarray(rows, np.int64)
    if wl.latent:   # routes are given; attention over the latent rows only
        O.latent_attention(a["q"], a["kv"], a["route"], wl.scale, Dv=wl.Dv, rows=rows)
        return int(np.count_nonzero(a["route"][rows] >= 0))
    r = O.index_routes(a["qI"], a["kI"], a["w"], wl.cu_seqlens, wl.c, wl.budget, rows=rows)
    full = np.full((wl.T, r.shape[1]), -1, np.int32)
    full[rows] = r
    if wl.window:
        r = O.compose_window(full, wl.cu_seqlens, wl.T, wl.window, rows=rows)
        full = np.full((wl.T, r.shape[1]), -1, np.int32)
        full[rows] = r
    O.attention(a["q"], a["k"], a["v"], full, wl.scale, rows=rows)
    return int(np.count_nonzero(r >= 0))


def oracle_sample(n_rows: int, cores: int, pool) -> tuple[float, int, float]:
    """Time the oracle on n_rows rows spread over the workload; returns (seconds, pairs, flops)."""
    wl = _WL
    rows = np.linspace(0, wl.T - 1, n_rows).astype(np.int64)
    shards = [rows[i::cores] for i in range(cores) if rows[i::cores].size]
    t0 = time.perf_counter()
    pairs = sum(pool.map(_oracle_rows, shards))
    dt = time.perf_counter() - t0
    return dt, pairs, 2.0 * (wl.Dqk + wl.Dv) * wl.Hq * pairs


def make_pool(cores: int, wl, small: bool = False):
    """Spawned oracle workers (spawn: never forked from a process that has used the GPU) and
    the shared-array directory to remove afterwards (or None)."""
    import multiprocessing as mp

    os.environ.setdefault("OMP_NUM_THREADS", "1")
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    os.environ.setdefault("MKL_NUM_THREADS", "1")
    shared = share_arrays(wl)
    ctx = mp.get_context("spawn")
    meta = dataclasses.replace(wl, arrays={})
    pool = ctx.Pool(cores, initializer=_worker_init, initargs=(wl.name, small, meta, shared))
    pool.map(_worker_init_probe, range(cores))   # workers are up and hold the workload
    return pool, shared


def close_pool(pool, shared: str | None):
    import shutil

    pool.terminate()
    pool.join()
    if shared is not None:
        shutil.rmtree(shared, ignore_errors=True)


def _worker_init_probe(_):
    return 0


def cpu_baseline(wl, cnt, budget_s: float = 15.0, small: bool = False) -> dict:
    global _WL
    _WL = wl
    cores = os.cpu_count() or 1
    pool, shared = make_pool(cores, wl, small)
    try:
        oracle_sample(cores, cores, pool)                           # first calls per worker run slow
        dt1, _, _ = oracle_sample(cores, cores, pool)               # calibration: one row per core
        n = int(max(cores, min(wl.T, cores * max(1, int(budget_s / max(dt1, 1e-3))))))
        dt, pairs, flops = oracle_sample(n, cores, pool)
    finally:
        close_pool(pool, shared)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} of {wl.T} query rows spread evenly ({'attention' if wl.latent else 'indexer + attention'}, "
                      f"all {wl.Hq} heads), "
                      f"{dt:.1f} s wall on {cores} single-threaded worker processes",
            "seconds": round(dt, 3), "rows": n}


def run_reference(args) -> dict | None:
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    global _WL
    wl = irs_synth.make(WORKLOAD)
    _WL = wl
    cores = os.cpu_count() or 1
    pool, shared = make_pool(cores, wl)
    try:
        dt1, _, _ = oracle_sample(cores, cores, pool)
        per_step_s = max(0.5, args.reference_seconds / max(1, args.steps + args.warmup))
        n = int(max(cores, min(wl.T, cores * max(1, int(per_step_s / max(dt1, 1e-3))))))
        for _ in range(args.warmup):
            oracle_sample(n, cores, pool)
        times, fl = [], 0.0
        for _ in range(args.steps):
            dt, _, fl = oracle_sample(n, cores, pool)
            times.append(dt)
    finally:
        close_pool(pool, shared)
    ms = float(np.mean(times)) * 1e3
    value = fl / (ms * 1e-3) / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(wl), "sample_rows_per_step": n},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n} of {wl.T} query rows per step (indexer + attention)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("irs", "reference"), default="irs")
    ap.add_argument("--workload", choices=irs_synth.WORKLOADS, default=WORKLOAD,
                    help="workload of the step (the headline line uses the windowed workload, the "
                         "largest single-GPU configuration that runs the whole path)")
    ap.add_argument("--small", action="store_true",
                    help="the workload's reduced-size variant (test sizes; for profiler captures, not a bench line)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="time only the headline workload (skip the other four)")
    ap.add_argument("--with-backward", action="store_true",
                    help="also time sparse_gqa_attn_bwd on the step's routes (reported under 'backward')")
    ap.add_argument("--variants-only", action="store_true",
                    help="time only the indexer rows beyond the plain one (front half, E4M3, per-group, "
                         "Step-5 summaries) on the workload's indexer shape; a few GB on the device "
                         "(profiler captures), not a bench line")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--reference-seconds", type=float, default=150.0)
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "irs":
        args.warmup = 3
    if args.variants_only:
        res = run_variants_only(args)
    else:
        res = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
