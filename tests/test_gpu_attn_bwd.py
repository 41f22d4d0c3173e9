"""Sparse attention backward on the GPU (through the C ABI) against the CPU oracle.

The kernel gets the oracle's forward outputs (out rounded to bf16, as a forward saves
it, and the FP32 lse) and an arbitrary bf16 output gradient; its dq, dk and dv are
compared with the oracle's backward element by element, against bounds derived from the
arithmetic (`grad_bounds`), and per tensor:
    dq, dk:  max |gpu - ref| <= 2e-2 max |ref| + 1e-4,  mean |gpu - ref| <= 5e-3 mean |ref| + 1e-5
    dv:      max |gpu - ref| <= 1e-4 max |ref| + 1e-6,  mean |gpu - ref| <= 2e-5 mean |ref| + 1e-7
Reading: the kernel takes D = dO . out from the bf16 output, while the oracle sums
p_r dO.v_r exactly. An FP32 emulation of the kernel's arithmetic on these shapes puts
that effect at up to 3e-3 of the largest dq/dk entry and 1e-3 of the mean, about a
sixth of the bound. dv does not involve D (FP32 sums, about 2e-6), so its tight bound
checks every probability, key and route. The absolute floors cover gradients that are
exactly zero in the oracle (one key per row).
GQA shapes with 8 or more query heads per KV head run on the tensor cores, where P and dS
are bf16 operands (each rounded once, at most 2^-9 relative, as the forward rounds P):
every GQA case carries c = 2^-9 + 1e-4 per term magnitude in its element-wise bounds
instead of 1e-4, and dv the loose per-tensor bound (the FP32 CUDA-core kernel, which takes
the smaller head groups, meets these too).
"""
import math

import numpy as np
import pytest
import torch

import irs_synth
from oracle import irs_oracle as O

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
TOL = {"loose": (2e-2, 1e-4, 5e-3, 1e-5), "tight": (1e-4, 1e-6, 2e-5, 1e-7)}
C_TC = 2.0 ** -9 + 1e-4   # per-term bound with bf16 P and dS operands (one rounding each)


@pytest.fixture(scope="module")
def irs():
    import indexer_routed_sparse_gb300 as m

    m.lib()
    return m


def bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits)).view(torch.bfloat16).to(DEV)


def check_grad(name, got, ref, tc=False):
    """dv gets the tight bound (the loose one on the tensor-core path, tc), every gradient
    that involves D the loose one."""
    max_rel, max_abs, mean_rel, mean_abs = TOL["tight" if name == "dv" and not tc else "loose"]
    got = got.double().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, name
    assert np.all(np.isfinite(got)), name
    err = np.abs(got - ref)
    assert err.max() <= max_rel * np.abs(ref).max() + max_abs, (name, err.max(), np.abs(ref).max())
    assert err.mean() <= mean_rel * np.abs(ref).mean() + mean_abs, (name, err.mean(), np.abs(ref).mean())


def grad_bounds(q, k, v, routes, scale, dout, out_bf16, rows=None, c=1e-4):
    """Element-wise bounds on |kernel - oracle| for dq (the given rows), dk and dv, from the
    arithmetic (reading R13). The kernel takes D = dO . out from the bf16 output, so a row's
    ds_r = p_r (dp_r - D) is off by p_r dD with dD = dO . (out - bf16(out)): dq[h, d] moves by
    scale dD sum_r p_r |K[r, d]| and dk[r, d] by scale p_r dD |q[h, d]|, both computed exactly
    here. Everything else is FP32 rounding (probabilities from the FP32 lse and FP32 scores,
    sums over at most a few thousand terms): c times the sums of the terms' magnitudes,
    c = 1e-4, 10 to 100 times the FP32 worst case at these lengths. Empty rows bound to 0."""
    T, Hq, Dqk = q.shape
    Tk, Hkv, _ = k.shape
    Dv = v.shape[2]
    G = Hq // Hkv
    rows = np.arange(T) if rows is None else np.asarray(rows)
    qf, kf, vf, dO = O.bf16_to_f64(q), O.bf16_to_f64(k), O.bf16_to_f64(v), O.bf16_to_f64(dout)
    ob = np.asarray(out_bf16, np.float64)
    dq_b = np.zeros((rows.shape[0], Hq, Dqk))
    dk_b = np.zeros((Tk, Hkv, Dqk))
    dv_b = np.zeros((Tk, Hkv, Dv))
    for i, t in enumerate(rows):
        ids = np.asarray(routes[t], np.int64)
        ids = ids[(ids >= 0) & (ids < Tk)]
        if ids.shape[0] == 0:
            continue
        for h in range(Hq):
            g = h // G
            K, V = kf[ids, g], vf[ids, g]
            sc = scale * (K @ qf[t, h])
            p = np.exp(sc - sc.max())
            p /= p.sum()
            dp = V @ dO[t, h]
            D = p @ dp
            dD = abs(dO[t, h] @ (p @ V - ob[t, h]))
            wgt = p * (np.abs(dp) + abs(D))
            dq_b[i, h] = scale * (dD * (p @ np.abs(K)) + c * (wgt @ np.abs(K)))
            np.add.at(dk_b[:, g], ids, scale * np.outer(p * dD + c * wgt, np.abs(qf[t, h])))
            np.add.at(dv_b[:, g], ids, c * np.outer(p, np.abs(dO[t, h])))
    return dq_b, dk_b, dv_b


def check_grad_elementwise(name, got, ref, bound):
    """|got - ref| <= 2 bound + 1e-7 in every element (bound from grad_bounds)."""
    got = got.double().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    err = np.abs(got - np.asarray(ref, np.float64))
    lim = 2.0 * bound + 1e-7
    bad = err > lim
    assert not bad.any(), (name, int(bad.sum()), float((err / lim).max()), np.unravel_index(int(np.argmax(err / lim)), err.shape))


def forward_outputs(q, k, v, routes, scale):
    out, lse = O.attention(q, k, v, routes, scale)
    return torch.from_numpy(out).to(torch.bfloat16).to(DEV), torch.from_numpy(lse).to(DEV)


def run_gqa(irs, q, k, v, routes, scale, dout, dk0=None):
    out_d, lse_d = forward_outputs(q, k, v, routes, scale)
    kd = bf16_dev(k)
    dk = None if dk0 is None else torch.from_numpy(dk0).to(DEV)
    dq, dk, dv = irs.sparse_gqa_attn_bwd(bf16_dev(q), kd, bf16_dev(v), torch.from_numpy(routes).to(DEV), out_d,
                                         lse_d, bf16_dev(dout), scale, dk=dk)
    return dq, dk, dv


GQA_CASES = [
    # (T, Hq, Hkv, Dqk, Dv, W, doc_lens, seed)
    (300, 8, 2, 128, 128, 64, [120, 180], 21),      # several staged chunks, two documents
    (200, 4, 4, 64, 128, 33, [200], 22),            # one head per KV head, Dv > Dqk
    (150, 6, 2, 192, 128, 100, [50, 60, 40], 23),   # three heads per KV head
    (64, 32, 1, 128, 256, 80, [64], 24),            # two head blocks per KV head
    (512, 32, 8, 128, 128, 512, [512], 25),         # mid-workload head shape
    # tensor-core kernel (8 or more heads per KV head)
    (256, 16, 2, 128, 128, 150, [100, 156], 32),    # 8 heads, several chunks, two documents
    (160, 32, 2, 192, 128, 300, [60, 100], 33),     # the windowed workload's head shape
    (140, 16, 1, 64, 128, 130, [1, 139], 34),       # Dqk = 64, one KV head, a one-token document
    (96, 24, 2, 128, 128, 70, [96], 35),            # 12 heads per KV head: a partial head block
]


@pytest.mark.parametrize("T, Hq, Hkv, Dqk, Dv, W, lens, seed", GQA_CASES)
def test_gqa_backward_matches_oracle(irs, T, Hq, Hkv, Dqk, Dv, W, lens, seed):
    wl = irs_synth.custom(T, Hq, Hkv, Dqk, Dv, 2, 64, 4, 8, doc_lens=lens, seed=seed)
    rng = np.random.default_rng(seed)
    routes = irs_synth.random_routes(rng, T, T, W, wl.cu_seqlens)
    dout = irs_synth.f32_to_bf16_bits(rng.standard_normal((T, Hq, Dv)).astype(np.float32))
    scale = 1.0 / math.sqrt(Dqk)
    q, k, v = wl.arrays["q"], wl.arrays["k"], wl.arrays["v"]
    dq, dk, dv = run_gqa(irs, q, k, v, routes, scale, dout)
    irs.check_device_errors(DEV)
    ref_dq, ref_dk, ref_dv = O.attention_bwd(q, k, v, routes, scale, dout)
    check_grad("dq", dq, ref_dq, tc=True)
    check_grad("dk", dk, ref_dk, tc=True)
    check_grad("dv", dv, ref_dv, tc=True)
    # element by element, against bounds derived from the arithmetic
    out_bf16 = torch.from_numpy(O.attention(q, k, v, routes, scale)[0]).to(torch.bfloat16).double().numpy()
    bq, bk, bv = grad_bounds(q, k, v, routes, scale, dout, out_bf16, c=C_TC)
    check_grad_elementwise("dq", dq, ref_dq, bq)
    check_grad_elementwise("dk", dk, ref_dk, bk)
    check_grad_elementwise("dv", dv, ref_dv, bv)


def test_gradients_are_added_to_the_given_buffers(irs):
    T, Hq, Hkv, D = 96, 4, 2, 128
    wl = irs_synth.custom(T, Hq, Hkv, D, D, 2, 64, 4, 8, seed=26)
    rng = np.random.default_rng(26)
    routes = irs_synth.random_routes(rng, T, T, 40, wl.cu_seqlens)
    dout = irs_synth.f32_to_bf16_bits(rng.standard_normal((T, Hq, D)).astype(np.float32))
    base = rng.standard_normal((T, Hkv, D)).astype(np.float32)
    q, k, v = wl.arrays["q"], wl.arrays["k"], wl.arrays["v"]
    _, dk, _ = run_gqa(irs, q, k, v, routes, 0.1, dout, dk0=base)
    irs.check_device_errors(DEV)
    _, ref_dk, _ = O.attention_bwd(q, k, v, routes, 0.1, dout)
    check_grad("dk", dk.cpu().numpy() - base, ref_dk, tc=True)


def test_latent_backward_matches_oracle(irs):
    rng = np.random.default_rng(27)
    Tq, H, D, Dv, Tk, W = 24, 128, 576, 512, 700, 128
    q = irs_synth.f32_to_bf16_bits(rng.standard_normal((Tq, H, D)).astype(np.float32))
    kv = irs_synth.f32_to_bf16_bits(rng.standard_normal((Tk, 1, D)).astype(np.float32))
    routes = irs_synth.latent_routes(rng, Tq, Tk, W)
    dout = irs_synth.f32_to_bf16_bits(rng.standard_normal((Tq, H, Dv)).astype(np.float32))
    scale = 1.0 / math.sqrt(D)
    out, lse = O.latent_attention(q, kv, routes, scale, Dv=Dv)
    kvd = bf16_dev(kv)
    dq, dkv, dv = irs.sparse_gqa_attn_bwd(bf16_dev(q), kvd, kvd[:, :, :Dv], torch.from_numpy(routes).to(DEV),
                                          torch.from_numpy(out).to(torch.bfloat16).to(DEV),
                                          torch.from_numpy(lse).to(DEV), bf16_dev(dout), scale)
    irs.check_device_errors(DEV)
    assert dv is None
    ref_dq, ref_dkv = O.latent_attention_bwd(q, kv, routes, scale, dout, Dv=Dv)
    check_grad("dq", dq, ref_dq)
    check_grad("dkv", dkv, ref_dkv)
    out_bf16 = torch.from_numpy(out).to(torch.bfloat16).double().numpy()
    bq, bk, bv = grad_bounds(q, kv, kv[:, :, :Dv], routes, scale, dout, out_bf16)
    bk[:, :, :Dv] += bv
    check_grad_elementwise("dq", dq, ref_dq, bq)
    check_grad_elementwise("dkv", dkv, ref_dkv, bk)


def test_single_key_empty_rows_and_bad_ids(irs):
    T, Hq, Hkv, D, Tk = 64, 8, 2, 128, 64
    wl = irs_synth.custom(T, Hq, Hkv, D, D, 2, 64, 4, 8, seed=28)
    rng = np.random.default_rng(28)
    q, k, v = wl.arrays["q"], wl.arrays["k"], wl.arrays["v"]
    dout = irs_synth.f32_to_bf16_bits(rng.standard_normal((T, Hq, D)).astype(np.float32))
    # W = 1: every row attends one key, so dq and dk vanish and dv collects dO
    r1 = (np.arange(T, dtype=np.int32) // 2).reshape(T, 1)
    dq, dk, dv = run_gqa(irs, q, k, v, r1, 0.2, dout)
    irs.check_device_errors(DEV)
    ref = O.attention_bwd(q, k, v, r1, 0.2, dout)
    for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        check_grad(name, got, want, tc=True)
    ob = torch.from_numpy(O.attention(q, k, v, r1, 0.2)[0]).to(torch.bfloat16).double().numpy()
    for name, got, want, b in zip(("dq", "dk", "dv"), (dq, dk, dv), ref,
                                  grad_bounds(q, k, v, r1, 0.2, dout, ob, c=C_TC)):
        check_grad_elementwise(name, got, want, b)
    # rows without keys give no gradient; an ID outside [-1, Tk) is padding and is reported
    r2 = irs_synth.random_routes(rng, T, Tk, 12, wl.cu_seqlens)
    r2[::3] = -1
    r2[1, 0] = Tk + 5
    dq, dk, dv = run_gqa(irs, q, k, v, r2, 0.2, dout)
    flags = irs.read_device_errors(DEV)
    assert flags & irs.DEVERR_ROUTE_ID
    ref = O.attention_bwd(q, k, v, r2, 0.2, dout)
    assert torch.all(dq[::3] == 0)
    for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        check_grad(name, got, want, tc=True)
    ob = torch.from_numpy(O.attention(q, k, v, r2, 0.2)[0]).to(torch.bfloat16).double().numpy()
    for name, got, want, b in zip(("dq", "dk", "dv"), (dq, dk, dv), ref,
                                  grad_bounds(q, k, v, r2, 0.2, dout, ob, c=C_TC)):
        check_grad_elementwise(name, got, want, b)


@pytest.mark.parametrize("name", ["mid", "windowed_small"])
def test_mid_backward_full_size(irs, name):
    """Large cases in the launch configuration the backward timing uses: the mid workload at
    full size (T 8192, Hq 32, Hkv 8, D 128, routes of 2051 IDs from the GPU indexer; the
    CUDA-core kernel) and the windowed workload's shape at T 8192 (Hq 64, Hkv 4, Dqk 192,
    Dv 128; the 512-token window composed with the indexer's routes, 2111 slots; the
    tensor-core kernel), forward outputs from the GPU forward. Checked against the oracle on
    sampled outputs it can compute one by one: dq of 24 query rows, and the complete dk / dv
    rows of 6 key rows, each summed by the oracle over every query row that routes that key.
    Every dk / dv row is also checked by two invariants: per KV group the value gradients sum
    to the group's sum of dO (the weights of each row sum to one), and the key gradients sum
    to zero (the softmax is invariant to a shift of the logits)."""
    wl = irs_synth.make("windowed", small=True) if name == "windowed_small" else irs_synth.make("mid")
    a = wl.arrays
    t = irs_synth.as_torch(wl, device=DEV)
    route = irs.sparse_index_score_topk(t["qI"], t["kI"], t["w"], t["cu_seqlens"], wl.c, wl.budget,
                                        max_doc_len=wl.max_doc_len)
    if wl.window:
        route = irs.compose_window_routes(route, t["cu_seqlens"], wl.window)
    out, lse = irs.sparse_gqa_attn_fwd(t["q"], t["k"], t["v"], route, wl.scale)
    rng = np.random.default_rng(31)
    dout = irs_synth.f32_to_bf16_bits(rng.standard_normal((wl.T, wl.Hq, wl.Dv)).astype(np.float32))
    dq, dk, dv = irs.sparse_gqa_attn_bwd(t["q"], t["k"], t["v"], route, out, lse, bf16_dev(dout), wl.scale)
    irs.check_device_errors(DEV)
    routes = route.cpu().numpy()
    q, k, v = a["q"], a["k"], a["v"]
    # sampled query rows: dq against the oracle
    rows = np.unique(np.concatenate([[0, 1, 3, 2047, 2048, wl.T - 1], rng.integers(0, wl.T, 18)]))
    ref_dq, _, _ = O.attention_bwd(q, k, v, routes, wl.scale, dout, rows=rows)
    check_grad("dq", dq[torch.as_tensor(rows, device=DEV)], ref_dq, tc=True)
    out_np = out.double().cpu().numpy()
    bq, _, _ = grad_bounds(q, k, v, routes, wl.scale, dout, out_np, rows=rows, c=C_TC)
    check_grad_elementwise("dq", dq[torch.as_tensor(rows, device=DEV)], ref_dq, bq)
    # sampled key rows: all of their query rows, so the oracle's dk / dv rows are complete
    ids = routes[routes >= 0]
    fan_in = np.bincount(ids, minlength=wl.T)
    cand = np.flatnonzero((fan_in >= 2) & (fan_in <= 12))
    keys = np.unique(cand[np.linspace(0, cand.shape[0] - 1, 6).astype(np.int64)])
    users = np.flatnonzero(np.isin(routes, keys).any(axis=1))
    _, ref_dk, ref_dv = O.attention_bwd(q, k, v, routes, wl.scale, dout, rows=users)
    kidx = torch.as_tensor(keys, device=DEV)
    check_grad("dk", dk[kidx], ref_dk[keys], tc=True)
    check_grad("dv", dv[kidx], ref_dv[keys], tc=True)
    _, bk, bv = grad_bounds(q, k, v, routes, wl.scale, dout, out_np, rows=users, c=C_TC)
    check_grad_elementwise("dk", dk[kidx], ref_dk[keys], bk[keys])
    check_grad_elementwise("dv", dv[kidx], ref_dv[keys], bv[keys])
    # invariants over every key row (float64 sums of the FP32 gradients)
    G = wl.Hq // wl.Hkv
    dO = O.bf16_to_f64(dout).reshape(wl.T, wl.Hkv, G, wl.Dv).sum(axis=(0, 2))       # [Hkv, Dv]
    dv_sum = dv.double().sum(dim=0).cpu().numpy()
    # with bf16 weights each row's weights sum to 1 only within their unbiased roundings
    # (at most 2^-9 relative each): the deviation of a column sum is a sum of independent
    # terms with standard deviation at most 2^-9 sqrt(sum dO^2); allow twice that
    dO2 = (O.bf16_to_f64(dout) ** 2).reshape(wl.T, wl.Hkv, G, wl.Dv).sum(axis=(0, 2))
    assert np.all(np.abs(dv_sum - dO) <= 2 * 2.0 ** -9 * np.sqrt(dO2) + 1e-2), np.abs(dv_sum - dO).max()
    dk_abs = dk.double().abs().sum(dim=0).cpu().numpy()
    dk_sum = dk.double().sum(dim=0).cpu().numpy()
    # the kernel's D = dO . out uses the bf16 output, so each row's ds sums to about 2^-9 |out||dO|
    # instead of 0; over 32768 (row, head) pairs that leaves about 4e-4 of sum |dk|
    assert np.all(np.abs(dk_sum) <= 2e-3 * dk_abs + 1e-3), float(np.max(np.abs(dk_sum) / (dk_abs + 1e-30)))
