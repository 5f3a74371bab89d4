"""The seeded input module: determinism, bf16 rounding, quantiser layout."""

import numpy as np
import torch

import moe_inputs as mi


def test_bf16_rounding_matches_torch_cast():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(10000).astype(np.float32) * 3,
                        np.float32([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3.4e38])])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(mi.f32_to_bf16_bits(x), ref)


def test_draws_are_deterministic_and_seed_dependent():
    wl = mi.get_workload("tiny")
    a = mi.make_layer_inputs(wl)
    b = mi.make_layer_inputs(wl)
    for k in ("router", "gate_up", "down", "dense_gate", "dense_up", "dense_down"):
        np.testing.assert_array_equal(a[k], b[k])
    np.testing.assert_array_equal(mi.make_tokens(wl), mi.make_tokens(wl))
    c = mi.make_layer_inputs(mi.get_workload("tiny", seed=5))
    assert not np.array_equal(a["gate_up"], c["gate_up"])


def test_shapes_and_distribution_of_tiny_workload():
    wl = mi.get_workload("tiny")
    p = mi.make_layer_inputs(wl)
    assert p["router"].shape == (16, 256)
    assert p["gate_up"].shape == (16, 128, 256)
    assert p["down"].shape == (16, 256, 64)
    assert p["dense_gate"].shape == (128, 256) and p["dense_down"].shape == (256, 128)
    f = lambda b: (b.astype(np.uint32) << 16).view(np.float32)
    assert abs(f(p["gate_up"]).std() - 0.02) < 0.001
    assert abs(f(p["router"]).std() - 1 / 16) < 0.003
    assert abs(f(mi.make_tokens(wl)).std() - 1.0) < 0.02
    assert np.all(p["w_post_ff"] == 0x3F80) and p["layer_scalar"] == 1.0


def test_quantised_workload_reuses_bf16_draws():
    wl = mi.get_workload("tiny")
    wq = mi.get_workload("tiny", quant=(4, 4, 8), draw_seed=0)
    p = mi.make_layer_inputs(wl)
    pq = mi.make_layer_inputs(wq)
    ref = mi.quantize_affine(p["gate_up"], 4)
    for k in ("q", "scales", "biases"):
        np.testing.assert_array_equal(pq["gate_up"][k], ref[k])
    assert pq["router"]["q"].dtype == np.uint8 and pq["router"]["q"].shape == (16, 256)
    assert pq["gate_up"]["q"].dtype == np.uint32 and pq["gate_up"]["q"].shape == (16, 128, 32)
    assert pq["gate_up"]["scales"].shape == (16, 128, 4)


def test_zipf_bias_is_a_permuted_zipf_profile():
    rng = np.random.default_rng(3)
    b = mi.zipf_router_bias(rng, 128, 1.0)
    p = np.sort(np.exp(b))[::-1]
    k = np.arange(1, 129)
    ref = k ** -1.2 / (k ** -1.2).sum()
    np.testing.assert_allclose(p, ref, rtol=1e-5)
