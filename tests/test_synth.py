"""Seeded input generator: determinism and the workload recipes."""
import numpy as np

import irs_synth


def test_tiny_is_deterministic_and_shaped():
    a = irs_synth.make("tiny")
    b = irs_synth.make("tiny")
    for k in a.arrays:
        np.testing.assert_array_equal(a.arrays[k], b.arrays[k])
    assert a.arrays["q"].shape == (1024, 8, 128) and a.arrays["q"].dtype == np.uint16
    assert a.arrays["qI"].shape == (1024, 4, 64)
    assert a.arrays["kI"].shape == (1024, 64)
    assert a.arrays["w"].dtype == np.float32 and a.arrays["w"].min() >= 0 and a.arrays["w"].max() < 1
    assert a.route_width == 259
    assert a.cu_seqlens.tolist() == [0, 1024]


def test_bf16_rounding_of_draws_is_round_to_nearest_even():
    import torch

    x = np.random.default_rng(0).standard_normal(10000).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(irs_synth.f32_to_bf16_bits(x), ref)


def test_packed_document_lengths():
    rng = np.random.default_rng(2)
    lens = irs_synth.packed_doc_lengths(rng, 32768, 2)
    assert sum(lens) == 65536
    assert min(lens) >= 256 and max(lens) <= 32768
    cs = np.cumsum(lens)
    assert 32768 in cs.tolist(), "row boundary must be a document boundary"


def test_latent_routes_are_causal_sorted_prefixes():
    rng = np.random.default_rng(4)
    r = irs_synth.latent_routes(rng, 64, 1000, 32)
    for i in range(64):
        p = 1000 - 64 + i
        v = r[i][r[i] >= 0]
        n = v.shape[0]
        assert 1 <= n <= 32
        assert np.all(r[i][n:] == -1)
        assert np.all(np.diff(v) > 0) and v.max() <= p and v.min() >= 0


def test_random_routes_are_document_confined():
    rng = np.random.default_rng(1)
    cu = np.asarray([0, 10, 30], np.int32)
    r = irs_synth.random_routes(rng, 30, 30, 8, cu)
    for t in range(30):
        s = 0 if t < 10 else 10
        v = r[t][r[t] >= 0]
        assert v.shape[0] >= 1 and np.all((v >= s) & (v <= t)) and len(set(v.tolist())) == v.shape[0]


def test_front_half_inputs():
    cu = np.asarray([0, 5, 12], np.int32)
    a = irs_synth.front_half_inputs(12, 16, 8, cu, seed=3)
    b = irs_synth.front_half_inputs(12, 16, 8, cu, seed=3)
    for k in ("q_weight", "k_weight", "rope"):
        np.testing.assert_array_equal(a[k], b[k])
    assert a["rope"].shape == (12, 8) and a["rope"].dtype == np.float32
    cos, sin = a["rope"][:, :4].astype(np.float64), a["rope"][:, 4:].astype(np.float64)
    np.testing.assert_allclose(cos * cos + sin * sin, 1.0, atol=1e-6)
    # document-local positions: position 0 at every document start (angle 0), then growing
    for t in (0, 5):
        np.testing.assert_array_equal(a["rope"][t], [1, 1, 1, 1, 0, 0, 0, 0])
    np.testing.assert_array_equal(a["rope"][6], a["rope"][1])
    assert 0.5 <= a["q_weight"].min() and a["k_weight"].max() <= 1.5
