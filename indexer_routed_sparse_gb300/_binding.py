"""ctypes binding of libirs.so (include/irs.h).

Argument marshalling only: tensors are checked, outputs and scratch are allocated
with torch on the tensors' device, and the C entry points are called with raw
device pointers and the current torch stream. There is no other code path: if the
library is missing or the device is not an sm_103 GPU, the calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libirs.so")

IRS_OK, IRS_ERR_TYPE, IRS_ERR_VALUE, IRS_ERR_RUNTIME = 0, 1, 2, 3
DEVERR_ROUTE_ID, DEVERR_CU_SEQLENS, DEVERR_TIMEOUT = 0x1, 0x2, 0x4

_lib = None
_lock = threading.Lock()
_err_flags: dict[int, torch.Tensor] = {}

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_F = ctypes.c_float

_SIGNATURES = {
    "irs_abi_version": (_I, []),
    "irs_last_error": (ctypes.c_char_p, []),
    "irs_index_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I, _I, _I]),
    "irs_sparse_index_score_topk": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _I64, _P, _SZ, _P, _P]),
    "irs_sparse_index_score_topk_noalloc": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _I64, _P, _P]),
    "irs_index_front_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I, _I, _I]),
    "irs_sparse_index_score_topk_front": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _F, _P, _I, _P, _P,
                                               _I64, _P, _SZ, _P, _P]),
    "irs_index_front_operands": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _F, _P, _I, _P, _P, _P, _SZ, _P,
                                      _P]),
    "irs_sparse_index_score_topk_grouped": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P, _I64, _P,
                                                 _SZ, _P, _P]),
    "irs_sparse_gqa_attn_fwd_grouped": (_I, [_P, _I64, _I64, _P, _I64, _I64, _P, _I64, _I64, _P, _I64, _I64, _I, _I,
                                             _I, _I, _I, _I, _I, _F, _P, _P, _P, _P]),
    "irs_index_e4m3_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I, _I, _I]),
    "irs_sparse_index_score_topk_e4m3": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _I64, _P, _SZ, _P,
                                              _P]),
    "irs_region_summaries_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "irs_region_summaries": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _SZ, _P, _P]),
    "irs_index_summaries_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I, _I, _I, _I, _I]),
    "irs_sparse_index_score_topk_summaries": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P,
                                                   _I64, _P, _SZ, _P, _P]),
    "irs_indexer_projection": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
    "irs_indexer_projection_front": (_I, [_P, _P, _I, _I, _I, _I, _P, _F, _P, _I, _P, _P, _P, _P, _P]),
    "irs_sparse_index_score_topk_front_keys": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _F, _P, _I, _P,
                                                    _P, _I64, _P, _SZ, _P, _P]),
    "irs_topk_from_scores": (_I, [_P, _I64, _P, _I, _I, _I, _I, _I, _P, _P, _P]),
    "irs_compose_window_routes": (_I, [_P, _I, _P, _I, _I, _I, _P, _P, _P]),
    "irs_sparse_gqa_attn_fwd": (_I, [_P, _I64, _I64, _P, _I64, _I64, _P, _I64, _I64, _P, _I64, _I, _I, _I, _I, _I, _I,
                                     _I, _F, _P, _P, _P, _P]),
    "irs_sparse_gqa_attn_fwd_windowed": (_I, [_P, _I64, _I64, _P, _I64, _I64, _P, _I64, _I64, _P, _I64, _P, _I, _I,
                                              _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P]),
    "irs_sparse_gqa_attn_bwd": (_I, [_P, _I64, _I64, _P, _I64, _I64, _P, _I64, _I64, _P, _I64, _P, _P, _P, _I, _I,
                                     _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P]),
    "irs_check_bounded_wait": (_I, [ctypes.c_uint64, _P, _P]),
}


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; "
                                   f"g.build()\"` (nvcc, sm_103a)")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def exported_symbols() -> list[str]:
    return list(_SIGNATURES)


def _check(status: int, what: str) -> None:
    if status == IRS_OK:
        return
    msg = f"{what}: {lib().irs_last_error().decode(errors='replace')}"
    if status == IRS_ERR_TYPE:
        raise TypeError(msg)
    if status == IRS_ERR_VALUE:
        raise ValueError(msg)
    raise RuntimeError(msg)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(dev: torch.device) -> int:
    return torch.cuda.current_stream(dev).cuda_stream


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, ndim: int | None = None) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")


def device_error_flag(device=None) -> torch.Tensor:
    """The per-device int32 word the kernels OR IRS_DEVERR_* bits into."""
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else torch.device(device).index)
    if dev.index not in _err_flags:
        _err_flags[dev.index] = torch.zeros(1, dtype=torch.int32, device=dev)
    return _err_flags[dev.index]


def read_device_errors(device=None, reset: bool = True) -> int:
    """Synchronise and return (then clear) the device error bits."""
    f = device_error_flag(device)
    torch.cuda.synchronize(f.device)
    v = int(f.item())
    if reset:
        f.zero_()
    return v


def check_device_errors(device=None) -> None:
    v = read_device_errors(device)
    if v:
        names = [n for b, n in ((DEVERR_ROUTE_ID, "route id out of range"),
                                (DEVERR_CU_SEQLENS, "malformed cu_seqlens"),
                                (DEVERR_TIMEOUT, "on-device wait timed out")) if v & b]
        raise RuntimeError("device reported: " + ", ".join(names))


def index_workspace_bytes(T, Hi, Di, c, budget, ndocs, max_doc_len, with_score_buffer=True) -> int:
    return int(lib().irs_index_workspace_bytes(T, Hi, Di, c, budget, ndocs, max_doc_len, int(bool(with_score_buffer))))


def _doc_stats(cu_seqlens: torch.Tensor, ndocs, max_doc_len, T: int):
    """Host sizes of the document layout without reading device data: ndocs from the
    tensor's shape and, unless the caller gives it, T as the bound on a document's length
    (a tighter max_doc_len shrinks the score scratch; the kernels check it on the device)."""
    if ndocs is None:
        ndocs = cu_seqlens.numel() - 1
    if max_doc_len is None:
        max_doc_len = T
    return int(ndocs), int(max_doc_len)


def _front_args(front: dict, Di: int):
    """(q_weight, k_weight, eps, rope, rope_dims) of a front-half dict, checked."""
    qw, kw, rope = front["q_weight"], front["k_weight"], front.get("rope")
    _need(qw, "q_weight", torch.float32, 1)
    _need(kw, "k_weight", torch.float32, 1)
    if qw.numel() != Di or kw.numel() != Di or not (qw.is_contiguous() and kw.is_contiguous()):
        raise ValueError("q_weight and k_weight must be contiguous fp32 [Di]")
    rope_dims = 0
    if rope is not None:
        _need(rope, "rope", torch.float32, 2)
        if not rope.is_contiguous():
            raise ValueError("rope must be contiguous [T, rope_dims]")
        rope_dims = rope.shape[1]
    return qw, kw, float(front["eps"]), rope, rope_dims


def sparse_index_score_topk(qI: torch.Tensor, kI: torch.Tensor, w: torch.Tensor, cu_seqlens: torch.Tensor,
                            c: int, budget: int, *, ndocs: int | None = None, max_doc_len: int | None = None,
                            scores_out: torch.Tensor | None = None, out: torch.Tensor | None = None,
                            workspace: torch.Tensor | None = None, err: torch.Tensor | None = None,
                            front: dict | None = None, operands: str = "bf16",
                            queries_ready: bool = False) -> torch.Tensor:
    """Route IDs int32 [T, budget + c - 1] from the compressed-block indexer.

    qI bf16 [T, Hi, Di], kI bf16 [T, Di] (or [T, 1, Di]), w fp32 [T, Hi], cu_seqlens int32
    [ndocs + 1] on the same device. `scores_out` (fp32 [T, ld >= max_doc_len // c]) receives
    the block scores of every row with more than budget // c visible blocks. `front` (a dict
    of fp32 device tensors q_weight [Di], k_weight [Di], rope [T, rope_dims] and a float eps)
    adds the indexer's front half: RMSNorm and RoPE of queries and pooled keys.
    operands="e4m3" scores with the Step-5 FP8 E4M3 roundings of queries and pooled keys.
    queries_ready (with `front`): qI already holds transformed queries (from
    indexer_projection(front=...)); only the pooled keys get the front half.
    """
    if operands not in ("bf16", "e4m3"):
        raise ValueError("operands must be 'bf16' or 'e4m3'")
    if operands == "e4m3" and front is not None:
        raise ValueError("E4M3 operands are not combined with the front half")
    if queries_ready and front is None:
        raise ValueError("queries_ready needs the front half's key weights (front=...)")
    _need(qI, "qI", torch.bfloat16, 3)
    _need(kI, "kI", torch.bfloat16)
    _need(w, "w", torch.float32, 2)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    T, Hi, Di = qI.shape
    if kI.dim() == 3:
        kI = kI.reshape(kI.shape[0], kI.shape[2])
    if tuple(kI.shape) != (T, Di) or tuple(w.shape) != (T, Hi):
        raise ValueError(f"shape mismatch: qI {tuple(qI.shape)}, kI {tuple(kI.shape)}, w {tuple(w.shape)}")
    if not (qI.is_contiguous() and kI.is_contiguous() and w.is_contiguous() and cu_seqlens.is_contiguous()):
        raise ValueError("qI, kI, w and cu_seqlens must be contiguous")
    ndocs, max_doc_len = _doc_stats(cu_seqlens, ndocs, max_doc_len, T)
    W = budget + c - 1
    dev = qI.device
    if out is None:
        out = torch.empty((T, W), dtype=torch.int32, device=dev)
    ld = 0
    if scores_out is not None:
        _need(scores_out, "scores_out", torch.float32, 2)
        if scores_out.shape[0] != T or scores_out.stride(1) != 1:
            raise ValueError("scores_out must be [T, ld] with unit inner stride")
        ld = scores_out.stride(0)
    if operands == "e4m3":
        nbytes = int(lib().irs_index_e4m3_workspace_bytes(T, Hi, Di, c, budget, ndocs, max_doc_len,
                                                          int(scores_out is None)))
    elif front is None:
        nbytes = index_workspace_bytes(T, Hi, Di, c, budget, ndocs, max_doc_len, scores_out is None)
    else:
        nbytes = int(lib().irs_index_front_workspace_bytes(T, Hi, Di, c, budget, ndocs, max_doc_len,
                                                           int(scores_out is None)))
    if nbytes == 0:
        _check(IRS_ERR_VALUE, "sparse_index_score_topk")
    if workspace is None or workspace.numel() < nbytes:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    if err is None:
        err = device_error_flag(dev)
    if operands == "e4m3":
        st = lib().irs_sparse_index_score_topk_e4m3(
            _ptr(qI), _ptr(kI), _ptr(w), _ptr(cu_seqlens), ndocs, max_doc_len, T, Hi, Di, c, budget, _ptr(out),
            _ptr(scores_out), ld, _ptr(workspace), workspace.numel(), _ptr(err), _stream(dev))
    elif front is None:
        st = lib().irs_sparse_index_score_topk(
            _ptr(qI), _ptr(kI), _ptr(w), _ptr(cu_seqlens), ndocs, max_doc_len, T, Hi, Di, c, budget, _ptr(out),
            _ptr(scores_out), ld, _ptr(workspace), workspace.numel(), _ptr(err), _stream(dev))
    elif queries_ready:
        _, kw, eps, rope, rope_dims = _front_args(dict(front, q_weight=front["k_weight"]), Di)
        st = lib().irs_sparse_index_score_topk_front_keys(
            _ptr(qI), _ptr(kI), _ptr(w), _ptr(cu_seqlens), ndocs, max_doc_len, T, Hi, Di, c, budget, _ptr(kw), eps,
            _ptr(rope), rope_dims, _ptr(out), _ptr(scores_out), ld, _ptr(workspace), workspace.numel(), _ptr(err),
            _stream(dev))
    else:
        qw, kw, eps, rope, rope_dims = _front_args(front, Di)
        st = lib().irs_sparse_index_score_topk_front(
            _ptr(qI), _ptr(kI), _ptr(w), _ptr(cu_seqlens), ndocs, max_doc_len, T, Hi, Di, c, budget, _ptr(qw),
            _ptr(kw), eps, _ptr(rope), rope_dims, _ptr(out), _ptr(scores_out), ld, _ptr(workspace),
            workspace.numel(), _ptr(err), _stream(dev))
    _check(st, "sparse_index_score_topk")
    return out


def index_front_operands(qI: torch.Tensor, kI: torch.Tensor, cu_seqlens: torch.Tensor, c: int, budget: int,
                         front: dict, *, ndocs: int | None = None, max_doc_len: int | None = None,
                         err: torch.Tensor | None = None) -> tuple[torch.Tensor, torch.Tensor]:
    """The indexer front half alone: (transformed queries bf16 [T, Hi, Di], transformed
    pooled keys bf16 [T // c, Di], pooled order; rows past the last complete block are 0)."""
    _need(qI, "qI", torch.bfloat16, 3)
    _need(kI, "kI", torch.bfloat16)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    T, Hi, Di = qI.shape
    if kI.dim() == 3:
        kI = kI.reshape(kI.shape[0], kI.shape[2])
    if not (qI.is_contiguous() and kI.is_contiguous() and cu_seqlens.is_contiguous()):
        raise ValueError("qI, kI and cu_seqlens must be contiguous")
    ndocs, max_doc_len = _doc_stats(cu_seqlens, ndocs, max_doc_len, T)
    dev = qI.device
    qw, kw, eps, rope, rope_dims = _front_args(front, Di)
    q_out = torch.empty_like(qI)
    k_out = torch.empty((max(1, T // c), Di), dtype=torch.bfloat16, device=dev)
    nbytes = int(lib().irs_index_front_workspace_bytes(T, Hi, Di, c, budget, ndocs, max_doc_len, 0))
    if nbytes == 0:
        _check(IRS_ERR_VALUE, "index_front_operands")
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    if err is None:
        err = device_error_flag(dev)
    st = lib().irs_index_front_operands(_ptr(qI), _ptr(kI), _ptr(cu_seqlens), ndocs, max_doc_len, T, Hi, Di, c,
                                        budget, _ptr(qw), _ptr(kw), eps, _ptr(rope), rope_dims, _ptr(q_out),
                                        _ptr(k_out), _ptr(ws), ws.numel(), _ptr(err), _stream(dev))
    _check(st, "index_front_operands")
    return q_out, k_out


def topk_from_scores(scores: torch.Tensor, cu_seqlens: torch.Tensor, c: int, budget: int, *,
                     ndocs: int | None = None, max_doc_len: int | None = None, out: torch.Tensor | None = None,
                     err: torch.Tensor | None = None) -> torch.Tensor:
    """Routes from given FP32 block scores [T, ld] (top-k, bitmap, expansion)."""
    _need(scores, "scores", torch.float32, 2)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    if scores.stride(1) != 1:
        raise ValueError("scores must have unit inner stride")
    T = scores.shape[0]
    if max_doc_len is None:   # the longest document whose block scores fit in a row of `scores`
        max_doc_len = min(T, (scores.shape[1] + 1) * c - 1)
    ndocs, max_doc_len = _doc_stats(cu_seqlens, ndocs, max_doc_len, T)
    dev = scores.device
    if out is None:
        out = torch.empty((T, budget + c - 1), dtype=torch.int32, device=dev)
    if err is None:
        err = device_error_flag(dev)
    st = lib().irs_topk_from_scores(_ptr(scores), scores.stride(0), _ptr(cu_seqlens), ndocs, max_doc_len, T, c,
                                    budget, _ptr(out), _ptr(err), _stream(dev))
    _check(st, "topk_from_scores")
    return out


def compose_window_routes(route_ids: torch.Tensor, cu_seqlens: torch.Tensor, window: int, *,
                          out: torch.Tensor | None = None, err: torch.Tensor | None = None) -> torch.Tensor:
    """[causal window of `window` tokens | route with in-window IDs set to -1], int32 [T, window + W]."""
    _need(route_ids, "route_ids", torch.int32, 2)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    if not route_ids.is_contiguous():
        raise ValueError("route_ids must be contiguous")
    T, W = route_ids.shape
    dev = route_ids.device
    if out is None:
        out = torch.empty((T, window + W), dtype=torch.int32, device=dev)
    if err is None:
        err = device_error_flag(dev)
    st = lib().irs_compose_window_routes(_ptr(route_ids), W, _ptr(cu_seqlens), cu_seqlens.numel() - 1, T, window,
                                         _ptr(out), _ptr(err), _stream(dev))
    _check(st, "compose_window_routes")
    return out


def sparse_gqa_attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, route_ids: torch.Tensor,
                        scale: float | None = None, *, window: int = 0, cu_seqlens: torch.Tensor | None = None,
                        ndocs: int | None = None, out: torch.Tensor | None = None,
                        lse: torch.Tensor | None = None, want_lse: bool = True,
                        err: torch.Tensor | None = None) -> tuple[torch.Tensor, torch.Tensor | None]:
    """Sparse attention over routed keys: (out bf16 [T, Hq, Dv], lse fp32 [T, Hq]).

    q bf16 [T, Hq, Dqk], k bf16 [Tk, Hkv, Dqk], v bf16 [Tk, Hkv, Dv] (innermost dim
    contiguous; v may be a view of k's leading Dv dims, as in latent attention),
    route_ids int32 [T, W] with -1 padding. With window > 0 (and cu_seqlens int32
    [ndocs + 1]) every query also attends the `window` most recent tokens of its document,
    in front of its route; route IDs inside the window are skipped.
    """
    _need(q, "q", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(route_ids, "route_ids", torch.int32, 2)
    T, Hq, Dqk = q.shape
    Tk, Hkv, Dk = k.shape
    Tv, Hv, Dv = v.shape
    if Dk != Dqk or Tv != Tk or Hv != Hkv or route_ids.shape[0] != T:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)} k {tuple(k.shape)} v {tuple(v.shape)} "
                         f"route {tuple(route_ids.shape)}")
    for name, t in (("q", q), ("k", k), ("v", v), ("route_ids", route_ids)):
        if t.stride(-1) != 1:
            raise ValueError(f"{name} must have unit inner stride")
    W = route_ids.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(Dqk)
    dev = q.device
    if out is None:
        out = torch.empty((T, Hq, Dv), dtype=torch.bfloat16, device=dev)
    elif tuple(out.shape) != (T, Hq, Dv) or not out.is_contiguous() or out.dtype != torch.bfloat16:
        raise ValueError("out must be a contiguous bf16 tensor [T, Hq, Dv]")
    if lse is not None and (tuple(lse.shape) != (T, Hq) or not lse.is_contiguous() or lse.dtype != torch.float32):
        raise ValueError("lse must be a contiguous fp32 tensor [T, Hq]")
    if lse is None and want_lse:
        lse = torch.empty((T, Hq), dtype=torch.float32, device=dev)
    if err is None:
        err = device_error_flag(dev)
    if window:
        if cu_seqlens is None:
            raise ValueError("a window needs cu_seqlens")
        _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
        if not cu_seqlens.is_contiguous():
            raise ValueError("cu_seqlens must be contiguous")
        nd = cu_seqlens.numel() - 1 if ndocs is None else int(ndocs)
        st = lib().irs_sparse_gqa_attn_fwd_windowed(
            _ptr(q), q.stride(0), q.stride(1), _ptr(k), k.stride(0), k.stride(1), _ptr(v), v.stride(0), v.stride(1),
            _ptr(route_ids), route_ids.stride(0), _ptr(cu_seqlens), nd, int(window), T, Tk, Hq, Hkv, Dqk, Dv, W,
            float(scale), _ptr(out), _ptr(lse), _ptr(err), _stream(dev))
        _check(st, "sparse_gqa_attn_fwd (windowed)")
        return out, lse
    st = lib().irs_sparse_gqa_attn_fwd(
        _ptr(q), q.stride(0), q.stride(1), _ptr(k), k.stride(0), k.stride(1), _ptr(v), v.stride(0), v.stride(1),
        _ptr(route_ids), route_ids.stride(0), T, Tk, Hq, Hkv, Dqk, Dv, W, float(scale), _ptr(out), _ptr(lse),
        _ptr(err), _stream(dev))
    _check(st, "sparse_gqa_attn_fwd")
    return out, lse


def _values_alias_keys(k: torch.Tensor, v: torch.Tensor) -> bool:
    return v.data_ptr() == k.data_ptr() and v.stride(0) == k.stride(0) and v.stride(1) == k.stride(1)


def sparse_gqa_attn_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, route_ids: torch.Tensor,
                        out: torch.Tensor, lse: torch.Tensor, dout: torch.Tensor, scale: float | None = None, *,
                        dq: torch.Tensor | None = None, dk: torch.Tensor | None = None,
                        dv: torch.Tensor | None = None,
                        err: torch.Tensor | None = None) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor | None]:
    """Backward of `sparse_gqa_attn_fwd` for the loss sum(out * dout): (dq, dk, dv), fp32.

    out and lse are the forward's outputs, dout bf16 [T, Hq, Dv]. When v is a view of k's
    leading Dv dims (latent attention), the rows are one tensor: its gradient is returned
    as dk [Tk, Hkv, Dqk] (key plus value gradient) and dv is None. dk and dv, if given,
    are added to; by default they are allocated zeroed.
    """
    _need(q, "q", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(route_ids, "route_ids", torch.int32, 2)
    _need(out, "out", torch.bfloat16, 3)
    _need(lse, "lse", torch.float32, 2)
    _need(dout, "dout", torch.bfloat16, 3)
    T, Hq, Dqk = q.shape
    Tk, Hkv, Dk = k.shape
    Tv, Hv, Dv = v.shape
    if Dk != Dqk or Tv != Tk or Hv != Hkv or route_ids.shape[0] != T:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)} k {tuple(k.shape)} v {tuple(v.shape)} "
                         f"route {tuple(route_ids.shape)}")
    for name, t in (("q", q), ("k", k), ("v", v), ("route_ids", route_ids)):
        if t.stride(-1) != 1:
            raise ValueError(f"{name} must have unit inner stride")
    for name, t, shape in (("out", out, (T, Hq, Dv)), ("dout", dout, (T, Hq, Dv)), ("lse", lse, (T, Hq))):
        if tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous with shape {shape}")
    W = route_ids.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(Dqk)
    dev = q.device
    shared = _values_alias_keys(k, v) and Dv <= Dqk
    if shared and dv is not None:
        raise ValueError("v is a view of k: the shared row gradient is returned as dk, so dv must be None")
    if dq is None:
        dq = torch.empty((T, Hq, Dqk), dtype=torch.float32, device=dev)
    if dk is None:
        dk = torch.zeros((Tk, Hkv, Dqk), dtype=torch.float32, device=dev)
    if not shared and dv is None:
        dv = torch.zeros((Tk, Hkv, Dv), dtype=torch.float32, device=dev)
    for name, t, shape in (("dq", dq, (T, Hq, Dqk)), ("dk", dk, (Tk, Hkv, Dqk))) + (
            () if shared else (("dv", dv, (Tk, Hkv, Dv)),)):
        if t.dtype != torch.float32 or tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous fp32 tensor {shape}")
    if err is None:
        err = device_error_flag(dev)
    st = lib().irs_sparse_gqa_attn_bwd(
        _ptr(q), q.stride(0), q.stride(1), _ptr(k), k.stride(0), k.stride(1), _ptr(v), v.stride(0), v.stride(1),
        _ptr(route_ids), route_ids.stride(0), _ptr(out), _ptr(lse), _ptr(dout), T, Tk, Hq, Hkv, Dqk, Dv, W,
        float(scale), _ptr(dq), _ptr(dk), _ptr(dk if shared else dv), _ptr(err), _stream(dev))
    _check(st, "sparse_gqa_attn_bwd")
    return dq, dk, (None if shared else dv)


def check_bounded_wait(limit_ms: float = 20.0, device=None, err: torch.Tensor | None = None) -> torch.Tensor:
    """Run one on-device wait that nothing releases; it gives up after `limit_ms` and sets
    DEVERR_TIMEOUT in the returned error word (asynchronous on the current stream)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    st = lib().irs_check_bounded_wait(int(limit_ms * 1e6), _ptr(err), _stream(dev))
    _check(st, "check_bounded_wait")
    return err


def sparse_index_score_topk_grouped(qI: torch.Tensor, kI: torch.Tensor, w: torch.Tensor, cu_seqlens: torch.Tensor,
                                    c: int, budget: int, *, ndocs: int | None = None, max_doc_len: int | None = None,
                                    scores_out: torch.Tensor | None = None, out: torch.Tensor | None = None,
                                    err: torch.Tensor | None = None) -> torch.Tensor:
    """Per-KV-group routes int32 [T, G, budget + c - 1] (Step-5 selection per group).

    qI bf16 [T, G, Hi, Di], kI bf16 [T, Di], w fp32 [T, G, Hi]; scores_out fp32 [T, G, ld].
    """
    _need(qI, "qI", torch.bfloat16, 4)
    _need(kI, "kI", torch.bfloat16)
    _need(w, "w", torch.float32, 3)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    T, G, Hi, Di = qI.shape
    if kI.dim() == 3:
        kI = kI.reshape(kI.shape[0], kI.shape[2])
    if tuple(kI.shape) != (T, Di) or tuple(w.shape) != (T, G, Hi):
        raise ValueError(f"shape mismatch: qI {tuple(qI.shape)}, kI {tuple(kI.shape)}, w {tuple(w.shape)}")
    if not (qI.is_contiguous() and kI.is_contiguous() and w.is_contiguous() and cu_seqlens.is_contiguous()):
        raise ValueError("qI, kI, w and cu_seqlens must be contiguous")
    ndocs, max_doc_len = _doc_stats(cu_seqlens, ndocs, max_doc_len, T)
    dev = qI.device
    W = budget + c - 1
    if out is None:
        out = torch.empty((T, G, W), dtype=torch.int32, device=dev)
    ld = 0
    if scores_out is not None:
        _need(scores_out, "scores_out", torch.float32, 3)
        if tuple(scores_out.shape[:2]) != (T, G) or not scores_out.is_contiguous():
            raise ValueError("scores_out must be a contiguous fp32 [T, G, ld]")
        ld = scores_out.shape[2]
    nbytes = index_workspace_bytes(T, Hi, Di, c, budget, ndocs, max_doc_len, scores_out is None)
    if nbytes == 0:
        _check(IRS_ERR_VALUE, "sparse_index_score_topk_grouped")
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    if err is None:
        err = device_error_flag(dev)
    st = lib().irs_sparse_index_score_topk_grouped(
        _ptr(qI), _ptr(kI), _ptr(w), _ptr(cu_seqlens), ndocs, max_doc_len, T, G, Hi, Di, c, budget, _ptr(out),
        _ptr(scores_out), ld, _ptr(ws), ws.numel(), _ptr(err), _stream(dev))
    _check(st, "sparse_index_score_topk_grouped")
    return out


def indexer_projection(hidden: torch.Tensor, weight: torch.Tensor, Hi: int, Di: int, *,
                       front: dict | None = None, out: tuple | None = None, err: torch.Tensor | None = None):
    """The indexer's queries, raw keys and signed head weights from hidden states:
    (qI bf16 [T, Hi, Di], kI bf16 [T, Di], w fp32 [T, Hi]).

    hidden bf16 [T, H]; weight bf16 [(Hi+1)*Di + Hi, H] (row n gives output column n:
    queries head-major, then keys, then head weights). `front` (q_weight, eps, rope as for
    sparse_index_score_topk) fuses the queries' RMSNorm and RoPE into the projection: qI
    then holds the transformed queries, for sparse_index_score_topk(queries_ready=True).
    """
    _need(hidden, "hidden", torch.bfloat16, 2)
    _need(weight, "weight", torch.bfloat16, 2)
    T, H = hidden.shape
    N = (Hi + 1) * Di + Hi
    if tuple(weight.shape) != (N, H):
        raise ValueError(f"weight must be [(Hi+1)*Di + Hi, H] = [{N}, {H}], got {tuple(weight.shape)}")
    if not (hidden.is_contiguous() and weight.is_contiguous()):
        raise ValueError("hidden and weight must be contiguous")
    dev = hidden.device
    if out is None:
        out = (torch.empty((T, Hi, Di), dtype=torch.bfloat16, device=dev),
               torch.empty((T, Di), dtype=torch.bfloat16, device=dev),
               torch.empty((T, Hi), dtype=torch.float32, device=dev))
    qI, kI, w = out
    if err is None:
        err = device_error_flag(dev)
    if front is None:
        st = lib().irs_indexer_projection(_ptr(hidden), _ptr(weight), T, H, Hi, Di, _ptr(qI), _ptr(kI), _ptr(w),
                                          _ptr(err), _stream(dev))
    else:
        qw, _, eps, rope, rope_dims = _front_args(dict(front, k_weight=front["q_weight"]), Di)
        st = lib().irs_indexer_projection_front(_ptr(hidden), _ptr(weight), T, H, Hi, Di, _ptr(qw), eps, _ptr(rope),
                                                rope_dims, _ptr(qI), _ptr(kI), _ptr(w), _ptr(err), _stream(dev))
    _check(st, "indexer_projection")
    return qI, kI, w


def region_summaries(kI: torch.Tensor, z: torch.Tensor, cu_seqlens: torch.Tensor, c: int, *,
                     ndocs: int | None = None, max_doc_len: int | None = None, out: torch.Tensor | None = None,
                     err: torch.Tensor | None = None) -> torch.Tensor:
    """Step-5 learned-logit region summaries, bf16 [T // c, Di] holding E4M3 values.

    kI and z (the compression logits) bf16 [T, Di]. Row blk_off[d] + b is region b of
    document d; rows past the last region are zero.
    """
    _need(kI, "kI", torch.bfloat16, 2)
    _need(z, "z", torch.bfloat16, 2)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    T, Di = kI.shape
    if tuple(z.shape) != (T, Di) or not (kI.is_contiguous() and z.is_contiguous() and cu_seqlens.is_contiguous()):
        raise ValueError("kI and z must be contiguous bf16 [T, Di] of one shape")
    ndocs, max_doc_len = _doc_stats(cu_seqlens, ndocs, max_doc_len, T)
    dev = kI.device
    rows = max(T // c, 1)
    if out is None:
        out = torch.empty((rows, Di), dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, 2)
    if tuple(out.shape) != (rows, Di) or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous bf16 [{rows}, {Di}]")
    nbytes = int(lib().irs_region_summaries_workspace_bytes(T, Di, c, ndocs, max_doc_len))
    if nbytes == 0:
        _check(IRS_ERR_VALUE, "region_summaries")
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    if err is None:
        err = device_error_flag(dev)
    st = lib().irs_region_summaries(_ptr(kI), _ptr(z), _ptr(cu_seqlens), ndocs, max_doc_len, T, Di, c, _ptr(out),
                                    _ptr(ws), ws.numel(), _ptr(err), _stream(dev))
    _check(st, "region_summaries")
    return out


def sparse_index_score_topk_summaries(qI: torch.Tensor, kI: torch.Tensor, z: torch.Tensor, w: torch.Tensor,
                                      cu_seqlens: torch.Tensor, c: int, budget: int, *, operands: str = "e4m3",
                                      ndocs: int | None = None, max_doc_len: int | None = None,
                                      scores_out: torch.Tensor | None = None, out: torch.Tensor | None = None,
                                      workspace: torch.Tensor | None = None,
                                      err: torch.Tensor | None = None) -> torch.Tensor:
    """Step-5 indexer: routes scored against the learned-logit region summaries of kI under
    the compression logits z, per KV group.

    qI bf16 [T, G, Hi, Di] (or [T, Hi, Di] for one group), kI and z bf16 [T, Di], w fp32
    [T, G, Hi] (or [T, Hi]). operands "e4m3" rounds the queries to E4M3 too (Di 128),
    "bf16" keeps them. Returns int32 [T, G, budget + c - 1] ([T, budget + c - 1] for 3-D qI);
    scores_out fp32 [T, G, ld] (or [T, ld]).
    """
    if operands not in ("bf16", "e4m3"):
        raise ValueError("operands must be 'bf16' or 'e4m3'")
    _need(qI, "qI", torch.bfloat16)
    _need(kI, "kI", torch.bfloat16)
    _need(z, "z", torch.bfloat16)
    _need(w, "w", torch.float32)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    flat = qI.dim() == 3
    q4 = qI.unsqueeze(1) if flat else qI
    w3 = w.unsqueeze(1) if flat else w
    if q4.dim() != 4:
        raise ValueError("qI must be [T, Hi, Di] or [T, G, Hi, Di]")
    T, G, Hi, Di = q4.shape
    if kI.dim() == 3:
        kI = kI.reshape(kI.shape[0], kI.shape[2])
    if z.dim() == 3:
        z = z.reshape(z.shape[0], z.shape[2])
    if tuple(kI.shape) != (T, Di) or tuple(z.shape) != (T, Di) or tuple(w3.shape) != (T, G, Hi):
        raise ValueError(f"shape mismatch: qI {tuple(qI.shape)}, kI {tuple(kI.shape)}, z {tuple(z.shape)}, "
                         f"w {tuple(w.shape)}")
    if not all(t.is_contiguous() for t in (q4, kI, z, w3, cu_seqlens)):
        raise ValueError("qI, kI, z, w and cu_seqlens must be contiguous")
    ndocs, max_doc_len = _doc_stats(cu_seqlens, ndocs, max_doc_len, T)
    dev = qI.device
    W = budget + c - 1
    if out is None:
        out = torch.empty((T, W) if flat else (T, G, W), dtype=torch.int32, device=dev)
    ld = 0
    if scores_out is not None:
        _need(scores_out, "scores_out", torch.float32)
        s3 = scores_out.unsqueeze(1) if flat else scores_out
        if s3.dim() != 3 or tuple(s3.shape[:2]) != (T, G) or not s3.is_contiguous():
            raise ValueError("scores_out must be a contiguous fp32 [T, G, ld] ([T, ld] for one group)")
        ld = s3.shape[2]
    e4 = int(operands == "e4m3")
    nbytes = int(lib().irs_index_summaries_workspace_bytes(T, G, Hi, Di, c, budget, ndocs, max_doc_len, e4,
                                                            int(scores_out is None)))
    if nbytes == 0:
        _check(IRS_ERR_VALUE, "sparse_index_score_topk_summaries")
    if workspace is None or workspace.numel() < nbytes:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    if err is None:
        err = device_error_flag(dev)
    st = lib().irs_sparse_index_score_topk_summaries(
        _ptr(q4), _ptr(kI), _ptr(z), _ptr(w3), _ptr(cu_seqlens), ndocs, max_doc_len, T, G, Hi, Di, c, budget, e4,
        _ptr(out), _ptr(scores_out), ld, _ptr(workspace), workspace.numel(), _ptr(err), _stream(dev))
    _check(st, "sparse_index_score_topk_summaries")
    return out


def sparse_gqa_attn_fwd_grouped(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, route_ids: torch.Tensor,
                                scale: float | None = None, *, err: torch.Tensor | None = None):
    """Attention with a route per KV group: route_ids int32 [T, Hkv, W]; the query heads of
    KV head g attend route_ids[t, g]. Returns (out bf16 [T, Hq, Dv], lse fp32 [T, Hq])."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(route_ids, "route_ids", torch.int32, 3)
    T, Hq, Dqk = q.shape
    Tk, Hkv, _ = k.shape
    Dv = v.shape[2]
    if route_ids.shape[0] != T or route_ids.shape[1] != Hkv or route_ids.stride(2) != 1:
        raise ValueError("route_ids must be [T, Hkv, W] with unit inner stride")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.stride(-1) != 1:
            raise ValueError(f"{name} must have unit inner stride")
    W = route_ids.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(Dqk)
    dev = q.device
    out = torch.empty((T, Hq, Dv), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, Hq), dtype=torch.float32, device=dev)
    if err is None:
        err = device_error_flag(dev)
    st = lib().irs_sparse_gqa_attn_fwd_grouped(
        _ptr(q), q.stride(0), q.stride(1), _ptr(k), k.stride(0), k.stride(1), _ptr(v), v.stride(0), v.stride(1),
        _ptr(route_ids), route_ids.stride(0), route_ids.stride(1), T, Tk, Hq, Hkv, Dqk, Dv, W, float(scale),
        _ptr(out), _ptr(lse), _ptr(err), _stream(dev))
    _check(st, "sparse_gqa_attn_fwd_grouped")
    return out, lse
