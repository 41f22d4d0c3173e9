"""Benchmark of the indexer-routed sparse attention hot path on GB300.

One step = one pass of the whole path over one batch of the mid-size single-document
workload (B=1, S=8192, Hq=32, Hkv=8, D=128; indexer Hi=16, Di=128, c=4, budget=2048):
  sparse_index_score_topk (layout, pool, score, top-k + expansion)  ->  sparse_gqa_attn_fwd.

Prints one JSON line (rank 0). `value` is the routed sparse-attention forward rate in
TFLOP/s over the whole step (algorithmic attention FLOPs / step time, inputs resident in
HBM, L2 flushed between timed steps); the indexer's queries/s, each kernel's own rate and
the roofline of the dominant kernel are reported beside it. `--impl reference` times the
CPU oracle on a bounded row sample of the same workload instead.

Multi-GPU: one process per GPU under torchrun; each rank runs its own replica of the
workload (weak scaling, no data-path collective); the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
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
WORKLOAD = "mid"
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
    from them) and the windowed workload's composed routes drop indexer IDs inside the window
    (counted from the routes the step attends, passed in as `pairs`).
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
    W = wl.route_width
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

    host = irs_synth.as_torch(wl, device="cpu", pin=True)
    d = {k: v.to(dev) for k, v in host.items()}
    T = wl.T
    out = torch.empty((T, wl.Hq, wl.Dv), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, wl.Hq), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    err = irs.device_error_flag(dev)
    has_index = not wl.latent
    if has_index:
        W_idx = wl.budget + wl.c - 1
        route_idx = torch.empty((T, W_idx), dtype=torch.int32, device=dev)
        route = torch.empty((T, wl.route_width), dtype=torch.int32, device=dev) if wl.window else route_idx
        ws = torch.empty(irs.index_workspace_bytes(T, wl.Hi, wl.Di, wl.c, wl.budget, wl.ndocs, wl.max_doc_len, True),
                         dtype=torch.uint8, device=dev)
        max_doc_len, ndocs = wl.max_doc_len, wl.ndocs
    kv_v = d["kv"][:, :, :wl.Dv] if wl.latent else None

    def index(dd):
        if not has_index:
            return
        irs.sparse_index_score_topk(dd["qI"], dd["kI"], dd["w"], dd["cu_seqlens"], wl.c, wl.budget, ndocs=ndocs,
                                    max_doc_len=max_doc_len, out=route_idx, workspace=ws, err=err)
        if wl.window:
            irs.compose_window_routes(route_idx, dd["cu_seqlens"], wl.window, out=route, err=err)

    def attend(dd):
        if wl.latent:
            irs.sparse_gqa_attn_fwd(dd["q"], dd["kv"], kv_v, dd["route"], wl.scale, out=out, lse=lse, err=err)
        else:
            irs.sparse_gqa_attn_fwd(dd["q"], dd["k"], dd["v"], route, wl.scale, out=out, lse=lse, err=err)

    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        index(d)
        attend(d)
    torch.cuda.synchronize(dev)
    irs.check_device_errors(dev)
    # valid pairs: closed form, except for the window-composed routes (data dependent)
    pairs = int((route >= 0).sum().item()) if (has_index and wl.window) else None
    cnt = counts(wl, pairs)
    kernels_per_step = (4 if has_index else 0) + (1 if wl.window else 0) + (wl.Hkv + 7) // 8

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

    # ---- device-timed region: K steps, L2 flushed before each, per-kernel events ----
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        index(d)
        ev[i][1].record(stream)
        attend(d)
        ev[i][2].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    wall = time.perf_counter() - wall0
    idx_ms = np.asarray([ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps)])
    att_ms = np.asarray([ev[i][1].elapsed_time(ev[i][2]) for i in range(args.steps)])
    step_ms_local = float(np.mean(idx_ms + att_ms))
    step_ms = reduce_max(step_ms_local, world, dev)
    irs.check_device_errors(dev)

    # ---- end to end through the public API with host buffers ----
    out_h = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    lse_h = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()
    e2e_steps = max(3, args.steps // 2)
    ee = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(e2e_steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    for i in range(e2e_steps):
        flush.fill_(i & 0xFF)
        ee[i][0].record(stream)
        for k_, v_ in host.items():
            d[k_].copy_(v_, non_blocking=True)
        index(d)
        attend(d)
        out_h.copy_(out, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)
        ee[i][1].record(stream)
        ee[i][1].synchronize()
    barrier(world)
    e2e_ms = reduce_max(float(np.mean([ee[i][0].elapsed_time(ee[i][1]) for i in range(e2e_steps)])), world, dev)
    bwd = time_backward(args, wl, irs, d, route if has_index else d["route"], kv_v, out, lse, flush, err, stream,
                        dev) if args.with_backward else None
    clk = clocks.stop() if rank == 0 else None
    irs.check_device_errors(dev)

    if rank != 0:
        return None
    att_avg_s = float(np.mean(att_ms)) * 1e-3
    idx_avg_s = float(np.mean(idx_ms)) * 1e-3
    attn_gbs = cnt["attn_bytes"] / att_avg_s / 1e9
    attn_tflops = cnt["attn_flops"] / att_avg_s / 1e12
    attn_roof_s = max(cnt["attn_bytes"] / (peaks["hbm_gbs"] * 1e9), cnt["attn_flops"] / (peaks["bf16_tflops"] * 1e12))
    attn_bound = "hbm" if cnt["attn_bytes"] / peaks["hbm_gbs"] >= cnt["attn_flops"] / (peaks["bf16_tflops"] * 1e3) \
        else "tensor"
    value = world * cnt["attn_flops"] / (step_ms * 1e-3) / 1e12
    if attn_bound == "hbm":
        roof = {"bound": "hbm", "achieved": round(attn_gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(attn_gbs / peaks["hbm_gbs"], 4)}
    else:
        roof = {"bound": "tensor", "achieved": round(attn_tflops, 2), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(attn_tflops / peaks["bf16_tflops"], 4)}
    # the latent workload runs on the latent-attention kernel, the others on the GQA kernel
    kname, ksrc = (("mla_fwd_kernel", "irs_mla.cu") if wl.latent else ("attn_fwd_kernel", "irs_attn.cu"))
    kprof = f"{kname.replace('_kernel', '')}_{wl.name}{'_small' if args.small else ''}.md"
    roof.update({"traffic": profile_traffic(kprof, f"indexer_routed_sparse_gb300/csrc/{ksrc}"),
                 "kernel": kname, "peak_source": peaks["source"]})
    res = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 inputs, U(0,1) fp32 head weights)",
        "config": {"workload": describe(wl), "l2": "flushed (512 MiB write) before every timed step",
                   "parallelism": f"replicas x{world}"},
        "roofline": roof,
        "attention": {"ms": round(att_avg_s * 1e3, 4), "tflops": round(attn_tflops, 3),
                      "routed_pairs_per_s": round(cnt["pairs"] * wl.Hq / att_avg_s, 1),
                      "roofline_frac": round(attn_roof_s / att_avg_s, 4), "roofline_ms": round(attn_roof_s * 1e3, 4),
                      "algorithmic_bytes": cnt["attn_bytes"], "flops": cnt["attn_flops"], "valid_pairs": cnt["pairs"]},
        "e2e": {"value": round(world * cnt["attn_flops"] / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": kernels_per_step * args.steps,
        "clocks": clk,
        "wall_s_timed": round(wall, 3),
    }
    if has_index:
        idx_roof_s = max(cnt["idx_bytes"] / (peaks["hbm_gbs"] * 1e9), cnt["idx_flops"] / (peaks["bf16_tflops"] * 1e12))
        res["indexer"] = {"ms": round(idx_avg_s * 1e3, 4), "queries_per_s": round(wl.T / idx_avg_s, 1),
                          "tflops": round(cnt["idx_flops"] / idx_avg_s / 1e12, 3),
                          "roofline_frac": round(idx_roof_s / idx_avg_s, 4), "roofline_us": round(idx_roof_s * 1e6, 2),
                          "algorithmic_bytes": cnt["idx_bytes"], "flops": cnt["idx_flops"],
                          "includes_window_composition": bool(wl.window)}
    if bwd is not None:
        res["backward"] = backward_report(wl, cnt, bwd, peaks)
    if not args.no_cpu_baseline and world == 1 and args.workload == WORKLOAD:
        res["cpu_baseline"] = cpu_baseline(wl, cnt, budget_s=args.cpu_seconds, small=args.small)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return res


def time_backward(args, wl, irs, d, route, kv_v, out, lse, flush, err, stream, dev) -> float:
    """Mean device time (s) of one sparse_gqa_attn_bwd call (accumulators zeroed inside the
    call's timed region, L2 flushed before each), on the step's routes and forward outputs."""
    import torch

    gen = torch.Generator(device=dev)
    gen.manual_seed(wl.seed + 1000)
    dout = torch.randn(out.shape, generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
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
            "algorithmic_bytes": int(nbytes), "flops": flops, "kernel": "attn_bwd_kernel",
            "launches_per_call": 1,
            "note": "FP32 CUDA-core kernel; timed separately, not part of the step or of value"}


# --------------------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)
# --------------------------------------------------------------------------------------
_WL = None


def _worker_init(name: str = WORKLOAD, small: bool = False):
    global _WL
    _WL = irs_synth.make(name, small=small)


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


def make_pool(cores: int, name: str = WORKLOAD, small: bool = False):
    import multiprocessing as mp

    os.environ.setdefault("OMP_NUM_THREADS", "1")
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    os.environ.setdefault("MKL_NUM_THREADS", "1")
    ctx = mp.get_context("spawn")
    pool = ctx.Pool(cores, initializer=_worker_init, initargs=(name, small))
    pool.map(_worker_init_probe, range(cores))   # workers are up and have built the workload
    return pool


def _worker_init_probe(_):
    return 0


def cpu_baseline(wl, cnt, budget_s: float = 15.0, small: bool = False) -> dict:
    global _WL
    _WL = wl
    cores = os.cpu_count() or 1
    pool = make_pool(cores, wl.name, small)
    try:
        oracle_sample(cores, cores, pool)                           # first calls per worker run slow
        dt1, _, _ = oracle_sample(cores, cores, pool)               # calibration: one row per core
        n = int(max(cores, min(wl.T, cores * max(1, int(budget_s / max(dt1, 1e-3))))))
        dt, pairs, flops = oracle_sample(n, cores, pool)
    finally:
        pool.terminate()
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
    pool = make_pool(cores)
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
        pool.terminate()
    ms = float(np.mean(times)) * 1e3
    value = fl / (ms * 1e-3) / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "mid single-document: B=1 S=8192 Hq=32 Hkv=8 D=128, indexer Hi=16 Di=128 c=4 "
                               "budget=2048, seed 1", "sample_rows_per_step": n},
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
                    help="workload of the step (the headline line uses the mid workload)")
    ap.add_argument("--small", action="store_true",
                    help="the workload's reduced-size variant (test sizes; for profiler captures, not a bench line)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--with-backward", action="store_true",
                    help="also time sparse_gqa_attn_bwd on the step's routes (reported under 'backward')")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--reference-seconds", type=float, default=150.0)
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "irs":
        args.warmup = 3
    res = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
