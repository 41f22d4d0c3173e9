"""The C ABI library: loads, exports what include/irs.h declares, validates on the host.

No compute call is made here: every call below fails host-side validation before the
library touches a GPU.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import indexer_routed_sparse_gb300 as irs

    if not os.path.exists(irs.LIB_PATH):
        from indexer_routed_sparse_gb300 import build

        build.build()
    return irs.lib()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "irs.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(irs_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ("irs_sparse_index_score_topk", "irs_sparse_gqa_attn_fwd", "irs_topk_from_scores",
                 "irs_compose_window_routes", "irs_index_workspace_bytes", "irs_last_error", "irs_abi_version"):
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    import indexer_routed_sparse_gb300 as irs

    for name in declared_symbols():
        assert hasattr(lib, name), f"{name} declared in include/irs.h but not exported"
        assert name in irs.exported_symbols(), f"{name} has no binding"
    assert lib.irs_abi_version() == 1


def test_workspace_size_rules(lib):
    import indexer_routed_sparse_gb300 as irs

    n = irs.index_workspace_bytes(8192, 16, 128, 4, 2048, 1, 8192, True)
    # pooled keys (8192/4 x 128 bf16) + score rows (8192 x 2048 fp32) at least
    assert n >= 2048 * 128 * 2 + 8192 * 2048 * 4
    n0 = irs.index_workspace_bytes(8192, 16, 128, 4, 2048, 1, 8192, False)
    assert 2048 * 128 * 2 <= n0 < n
    assert irs.index_workspace_bytes(8192, 12, 128, 4, 2048, 1, 8192, True) == 0     # Hi not a power of two
    assert irs.index_workspace_bytes(8192, 16, 96, 4, 2048, 1, 8192, True) == 0      # unsupported Di
    assert irs.index_workspace_bytes(8192, 16, 128, 4, 2047, 1, 8192, True) == 0     # budget % c
    assert n % 256 == 0


@pytest.mark.parametrize("case, field", [
    (dict(Hi=3), "Hi"), (dict(Di=32), "Di"), (dict(c=0), "c"), (dict(budget=6, c=4), "budget"),
    (dict(ndocs=0), "ndocs"), (dict(max_doc_len=0), "max_doc_len"),
])
def test_index_validation_is_value_error(lib, case, field):
    args = dict(T=64, Hi=4, Di=64, c=4, budget=16, ndocs=1, max_doc_len=64)
    args.update(case)
    st = lib.irs_sparse_index_score_topk(None, None, None, None, args["ndocs"], args["max_doc_len"], args["T"],
                                         args["Hi"], args["Di"], args["c"], args["budget"], None, None, 0, None, 0,
                                         None, None)
    assert st == 2, field
    assert lib.irs_last_error()


def test_index_null_pointers_are_value_error(lib):
    st = lib.irs_sparse_index_score_topk(None, None, None, None, 1, 64, 64, 4, 64, 4, 16, None, None, 0, None, 0,
                                         None, None)
    assert st == 2 and b"NULL" in lib.irs_last_error()


@pytest.mark.parametrize("case", [
    dict(Hq=6, Hkv=4), dict(Dqk=100), dict(Dqk=640), dict(Dv=64), dict(Dv=640), dict(W=0), dict(W=5000),
    dict(scale=0.0), dict(scale=-1.0), dict(scale=float("inf")), dict(route_stride=3, W=4),
])
def test_attention_validation_is_value_error(lib, case):
    a = dict(T=4, Tk=16, Hq=4, Hkv=2, Dqk=128, Dv=128, W=8, scale=0.1, route_stride=8)
    a.update(case)
    st = lib.irs_sparse_gqa_attn_fwd(None, 0, 0, None, 0, 0, None, 0, 0, None, a["route_stride"], a["T"], a["Tk"],
                                     a["Hq"], a["Hkv"], a["Dqk"], a["Dv"], a["W"], a["scale"], None, None, None, None)
    assert st == 2, case


def test_attention_misaligned_strides_are_value_error(lib):
    # strides must be multiples of 8 elements; checked before any device access
    buf = ctypes.create_string_buffer(64)
    p = ctypes.addressof(buf) + (16 - ctypes.addressof(buf) % 16) % 16
    st = lib.irs_sparse_gqa_attn_fwd(p, 12, 128, p, 128, 128, p, 128, 128, p, 8, 4, 16, 4, 2, 128, 128, 8, 0.1, p,
                                     None, None, None)
    assert st == 2 and b"multiples of 8" in lib.irs_last_error()


def test_binding_rejects_wrong_dtypes_on_cpu():
    import torch

    import indexer_routed_sparse_gb300 as irs

    q = torch.zeros(4, 2, 64, dtype=torch.float32)
    with pytest.raises(TypeError):
        irs.sparse_gqa_attn_fwd(q, q, q, torch.zeros(4, 4, dtype=torch.int32))
    qb = torch.zeros(4, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):   # not a CUDA tensor
        irs.sparse_gqa_attn_fwd(qb, qb, qb, torch.zeros(4, 4, dtype=torch.int32))


def _bwd_call(lib, p=None, **kw):
    a = dict(T=4, Tk=16, Hq=4, Hkv=2, Dqk=128, Dv=128, W=8, scale=0.1, route_stride=8, q_st=512, dk=p, dv=p)
    a.update(kw)
    return lib.irs_sparse_gqa_attn_bwd(p, a["q_st"], 128, p, 256, 128, p, 256, 128, p, a["route_stride"], p, p, p,
                                       a["T"], a["Tk"], a["Hq"], a["Hkv"], a["Dqk"], a["Dv"], a["W"], a["scale"],
                                       p, a["dk"], a["dv"], None, None)


@pytest.mark.parametrize("case", [
    dict(Hq=6, Hkv=4), dict(Dqk=100), dict(Dqk=640), dict(Dv=64), dict(Dv=640), dict(W=0), dict(W=5000),
    dict(scale=0.0), dict(scale=float("nan")), dict(route_stride=3, W=4),
])
def test_backward_validation_is_value_error(lib, case):
    assert _bwd_call(lib, None, **case) == 2, case


def test_backward_host_checks(lib):
    buf = ctypes.create_string_buffer(64)
    p = ctypes.addressof(buf) + (16 - ctypes.addressof(buf) % 16) % 16
    assert _bwd_call(lib, None) == 2 and b"NULL" in lib.irs_last_error()
    assert _bwd_call(lib, p, q_st=12) == 2 and b"multiples of 8" in lib.irs_last_error()
    assert _bwd_call(lib, p, dk=p + 4) == 2 and b"16-byte aligned" in lib.irs_last_error()
    # a shared dk/dv buffer needs the value rows to fit in the key rows
    assert _bwd_call(lib, p, Dqk=128, Dv=256) == 2 and b"Dv <= Dqk" in lib.irs_last_error()
    assert _bwd_call(lib, p, T=0) == 0          # nothing to do
    # separate value rows with a shared gradient buffer would mix the two gradients
    st = lib.irs_sparse_gqa_attn_bwd(p, 512, 128, p, 256, 128, p + 16, 256, 128, p, 8, p, p, p, 4, 16, 4, 2, 128, 128,
                                     8, 0.1, p, p, p, None, None)
    assert st == 2 and b"view of k" in lib.irs_last_error()


def test_backward_binding_rejects_wrong_inputs_on_cpu():
    import torch

    import indexer_routed_sparse_gb300 as irs

    qb = torch.zeros(4, 2, 128, dtype=torch.bfloat16)
    r = torch.zeros(4, 4, dtype=torch.int32)
    lse = torch.zeros(4, 2)
    with pytest.raises(TypeError):      # q must be bf16
        irs.sparse_gqa_attn_bwd(qb.float(), qb, qb, r, qb, lse, qb)
    with pytest.raises(ValueError):     # not CUDA tensors
        irs.sparse_gqa_attn_bwd(qb, qb, qb, r, qb, lse, qb)


def test_front_half_validation_is_value_error(lib):
    import ctypes as C
    buf = C.create_string_buffer(256)
    p = C.addressof(buf) + (16 - C.addressof(buf) % 16) % 16
    def call(rope_dims=32, qw=p, kw=p, eps=1e-6, rope=p):
        return lib.irs_sparse_index_score_topk_front(p, p, p, p, 1, 64, 64, 4, 64, 4, 16, qw, kw, eps, rope, rope_dims,
                                                     p, None, 0, p, 1 << 20, None, None)
    assert call(rope_dims=24) == 2 and b"rope_dims" in lib.irs_last_error()
    assert call(rope_dims=80) == 2
    assert call(qw=None) == 2 and b"RMSNorm" in lib.irs_last_error()
    assert call(eps=-1.0) == 2 and b"eps" in lib.irs_last_error()
    assert call(rope=None) == 2 and b"rotary" in lib.irs_last_error()
    assert call(qw=p + 4) == 2 and b"16-byte aligned" in lib.irs_last_error()
    assert call(rope=p + 8) == 2 and b"16-byte aligned" in lib.irs_last_error()
    assert lib.irs_index_front_workspace_bytes(64, 4, 64, 4, 16, 1, 64, 1) > lib.irs_index_workspace_bytes(
        64, 4, 64, 4, 16, 1, 64, 1)


def test_summaries_validation_is_value_error(lib):
    import ctypes as C
    buf = C.create_string_buffer(512)
    p = C.addressof(buf) + (256 - C.addressof(buf) % 256) % 256

    def call(z=p, Di=128, e4=1, G=1):
        return lib.irs_sparse_index_score_topk_summaries(p, p, z, p, p, 1, 64, 64, G, 4, Di, 4, 16, e4, p, None, 0,
                                                         p, 1 << 30, None, None)
    assert call(z=None) == 2 and b"compression logits" in lib.irs_last_error()
    assert call(Di=64, e4=1) == 2 and b"Di = 128" in lib.irs_last_error()
    assert call(z=p + 2) == 2 and b"16-byte" in lib.irs_last_error()
    assert call(G=0) == 2
    one = lib.irs_index_summaries_workspace_bytes(64, 1, 4, 128, 4, 16, 1, 64, 1, 1)
    two = lib.irs_index_summaries_workspace_bytes(64, 2, 4, 128, 4, 16, 1, 64, 1, 1)
    assert 0 < one < two                       # the E4M3 query copy holds every group
    assert lib.irs_index_summaries_workspace_bytes(64, 1, 4, 64, 4, 16, 1, 64, 1, 1) == 0
    assert lib.irs_index_summaries_workspace_bytes(64, 1, 4, 64, 4, 16, 1, 64, 0, 1) > 0
    # the summaries alone
    assert lib.irs_region_summaries_workspace_bytes(64, 96, 4, 1, 64) == 0
    assert lib.irs_region_summaries_workspace_bytes(64, 128, 4, 1, 64) > 0
    st = lib.irs_region_summaries(p, None, p, 1, 64, 64, 128, 4, p, p, 1 << 20, None, None)
    assert st == 2 and b"NULL" in lib.irs_last_error()
    st = lib.irs_region_summaries(p, p + 8, p, 1, 64, 64, 128, 4, p, p, 1 << 20, None, None)
    assert st == 2 and b"aligned" in lib.irs_last_error()
    st = lib.irs_region_summaries(p, p, p, 1, 64, 64, 128, 4, p, p, 16, None, None)
    assert st == 2 and b"workspace too small" in lib.irs_last_error()


def test_projection_validation_is_value_error(lib):
    import ctypes as C
    buf = C.create_string_buffer(512)
    p = C.addressof(buf) + (256 - C.addressof(buf) % 256) % 256

    def call(T=64, H=128, Hi=4, Di=64, hid=p, wt=p, q=p, k=p, w=p):
        return lib.irs_indexer_projection(hid, wt, T, H, Hi, Di, q, k, w, None, None)
    assert call(H=100) == 2 and b"multiple of 8" in lib.irs_last_error()
    assert call(Di=12) == 2 and b"multiple of 8" in lib.irs_last_error()
    assert call(T=0) == 2
    assert call(Hi=0) == 2
    assert call(wt=None) == 2 and b"NULL" in lib.irs_last_error()
    assert call(q=p + 8) == 2 and b"16-byte aligned" in lib.irs_last_error()
    assert call(w=p + 2) == 2 and b"4-byte aligned" in lib.irs_last_error()


def test_fused_projection_and_keys_only_validation(lib):
    import ctypes as C
    buf = C.create_string_buffer(512)
    p = C.addressof(buf) + (256 - C.addressof(buf) % 256) % 256
    st = lib.irs_indexer_projection_front(p, p, 64, 128, 4, 96, p, 1e-6, p, 32, p, p, p, None, None)
    assert st == 2 and b"Di = 64 or 128" in lib.irs_last_error()
    st = lib.irs_indexer_projection_front(p, p, 64, 128, 4, 64, None, 1e-6, p, 32, p, p, p, None, None)
    assert st == 2 and b"RMSNorm" in lib.irs_last_error()
    st = lib.irs_sparse_index_score_topk_front_keys(p, p, p, p, 1, 64, 64, 4, 64, 4, 16, p, 1e-6, p, 24, p, None, 0,
                                                    p, 1 << 20, None, None)
    assert st == 2 and b"rope_dims" in lib.irs_last_error()
