"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test checks one function of ``oracle.moe_oracle`` against brute force on
tiny inputs, a closed form, an identity of the mathematics, a special case
that reduces to a library routine, or a value printed on the pages, so that a
plausible slip in the oracle (a dropped term, a swapped operand, a wrong axis
or index, the erf GELU, eps outside the root) fails at least one of them.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle as o

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed=0):
    return np.random.default_rng(seed)


def _small_params(rng, H=32, E=6, I=8, D=12, std=0.3):
    f = lambda *s: rng.standard_normal(s) * std
    return {
        "router": f(E, H), "gate_up": f(E, 2 * I, H), "down": f(E, H, I),
        "dense_gate": f(D, H), "dense_up": f(D, H), "dense_down": f(H, D),
        "router_scale": rng.uniform(0.5, 1.5, H),
        "per_expert_scale": np.ones(E),
        "w_pre_ff": rng.uniform(0.5, 1.5, H), "w_pre_ff2": rng.uniform(0.5, 1.5, H),
        "w_post_ff1": rng.uniform(0.5, 1.5, H), "w_post_ff2": rng.uniform(0.5, 1.5, H),
        "w_post_ff": rng.uniform(0.5, 1.5, H), "router_bias": None,
        "layer_scalar": 0.75,
    }


# ---------------------------------------------------------------- constants

def test_workload_shapes_match_printed_constants():
    g = json.load(open(os.path.join(GOLDEN, "model_constants.json")))
    for name in ("canvas256", "canvas256_q4", "batch2048_zipf", "stack30_q4"):
        wl = mi.get_workload(name)
        assert (wl.hidden, wl.n_experts, wl.top_k, wl.expert_inter, wl.dense_inter) == (
            g["hidden"], g["n_experts"], g["top_k"], g["expert_inter"], g["dense_inter"])
    assert 2 * g["expert_inter"] == g["gate_up_rows"]
    assert o.EPS == g["rms_eps"]
    wl = mi.get_workload("canvas256_q4")
    assert wl.quant == (g["expert_bits"], g["expert_bits"], g["router_bits"])


# ---------------------------------------------------------------- RMSNorm

def test_rms_norm_matches_torch_library_routine():
    rng = _rng(1)
    x = rng.standard_normal((5, 40)) * 3.0
    w = rng.uniform(0.5, 1.5, 40)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (40,),
                                       torch.from_numpy(w), eps=1e-6).numpy()
    np.testing.assert_allclose(o.rms_norm(x, w), ref, rtol=1e-13, atol=0)


def test_rms_norm_eps_inside_root_closed_form():
    # x = c * ones: rms_norm(x) = c / sqrt(c^2 + eps), which separates eps
    # inside the root from eps added to the norm
    for c in (1e-3, 0.5, 3.0):
        x = np.full((1, 7), c)
        np.testing.assert_allclose(o.rms_norm(x), c / math.sqrt(c * c + 1e-6), rtol=1e-14)


# ---------------------------------------------------------------- GELU

def test_gelu_tanh_identity_and_library_value():
    x = np.linspace(-6, 6, 241)
    np.testing.assert_allclose(o.gelu_tanh(x) - o.gelu_tanh(-x), x, atol=1e-14)
    ref = torch.nn.functional.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    np.testing.assert_allclose(o.gelu_tanh(x), ref, rtol=1e-12, atol=1e-15)
    # the tanh form, not the erf form: they differ visibly at x = 1
    erf1 = 0.5 * (1 + math.erf(1 / math.sqrt(2)))
    assert abs(o.gelu_tanh(np.array([1.0]))[0] - erf1) > 1e-4


# ---------------------------------------------------------------- router

def test_router_norm_closed_form_with_identity_projection():
    # Wr = I makes the logits the router input itself; with unit scale its
    # norm is |h| / sqrt(|h|^2 + H eps)
    rng = _rng(2)
    H = 16
    for mag in (1e-4, 1e-2, 1.0, 10.0):
        h = rng.standard_normal((3, H)) * mag
        z = o.router_logits(h, np.eye(H), np.ones(H))
        nh = np.linalg.norm(h, axis=1)
        np.testing.assert_allclose(np.linalg.norm(z, axis=1),
                                   nh / np.sqrt(nh ** 2 + H * 1e-6), rtol=1e-12)
    # router_scale multiplies per channel and H^-0.5 is applied once
    h = rng.standard_normal((2, H))
    sc = rng.uniform(0.5, 1.5, H)
    r = 1 / np.sqrt((h ** 2).mean(1, keepdims=True) + 1e-6)
    np.testing.assert_allclose(o.router_logits(h, np.eye(H), sc), h * r * sc / 4.0,
                               rtol=1e-13)


def _brute_topk(zrow, k):
    order = sorted(range(len(zrow)), key=lambda e: (-zrow[e], e))
    return sorted(order[:k])


def test_topk_equals_full_sort_with_and_without_ties():
    rng = _rng(3)
    z = rng.standard_normal((50, 20))
    zt = rng.integers(-3, 3, (50, 20)).astype(np.float64)   # many exact ties
    for zz in (z, zt):
        for k in (1, 3, 8, 20):
            idx = o.select_topk(zz, k)
            for t in range(zz.shape[0]):
                assert list(idx[t]) == _brute_topk(list(zz[t]), k)


def test_routing_weights_two_forms_agree_and_sum_to_one():
    rng = _rng(4)
    z = rng.standard_normal((30, 16)) * 2
    k = 4
    idx = o.select_topk(z, k)
    w = o.routing_weights(z, idx, np.ones(16))
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-14)
    # softmax taken over the k selected logits only (the MLX form)
    for t in range(30):
        sel = [z[t, e] for e in idx[t]]
        m = max(sel)
        ex = [math.exp(v - m) for v in sel]
        ref = [v / sum(ex) for v in ex]
        np.testing.assert_allclose(w[t], ref, rtol=1e-12)
    pes = rng.uniform(0.5, 1.5, 16)
    np.testing.assert_allclose(o.routing_weights(z, idx, pes), w * pes[idx], rtol=1e-14)


def test_zero_token_routes_to_first_k_with_equal_weights():
    p = _small_params(_rng(5))
    h = np.zeros((2, 32))
    h[1] = _rng(6).standard_normal(32)
    r = o.moe_block_forward(h, p, top_k=3, inter=8)
    assert list(r["idx"][0]) == [0, 1, 2]
    np.testing.assert_allclose(r["w"][0], 1 / 3, rtol=1e-15)
    assert np.all(r["out"][0] == 0.0)   # every branch maps 0 to 0


def test_duplicate_router_rows_lower_index_wins():
    rng = _rng(7)
    H, E, k = 32, 6, 3
    h = rng.standard_normal((1, H))
    Wr = rng.standard_normal((E, H)) * 0.01
    # experts 0 and 4 clearly first; 2 and 5 identical and next: only 2 fits
    Wr[0] = h[0] * 3.0
    Wr[4] = h[0] * 2.0
    Wr[2] = Wr[5] = h[0] * 1.0
    _, idx, _ = o.route(h, Wr, np.ones(H), np.ones(E), k)
    assert list(idx[0]) == [0, 2, 4]


def test_routing_invariant_under_scaling_of_h():
    wl = mi.get_workload("tiny")
    p = mi.make_layer_inputs(wl)
    h = o.bf16_to_f64(mi.make_tokens(wl))
    Wr, sc = o.to_f64(p["router"]), o.to_f64(p["router_scale"])
    _, i1, _ = o.route(h, Wr, sc, np.ones(wl.n_experts), wl.top_k)
    _, i2, _ = o.route(2.0 * h, Wr, sc, np.ones(wl.n_experts), wl.top_k)
    assert np.array_equal(i1, i2)


# ---------------------------------------------------------------- experts

def test_single_feature_expert_closed_form_pins_gate_up_down_orientation():
    # one expert, inter 1: gate row a*e_0, up row b*e_1, down column c*e_2
    # -> y = c * gelu(a x0) * (b x1) on channel 2 only
    H, a, b, c = 6, 0.7, -1.3, 2.0
    gate_up = np.zeros((1, 2, H))
    gate_up[0, 0, 0] = a
    gate_up[0, 1, 1] = b
    down = np.zeros((1, H, 1))
    down[0, 2, 0] = c
    x = np.array([[0.9, -0.4, 5.0, 1.0, 1.0, 1.0]])
    y = o.experts_forward(x, np.array([[0]]), np.array([[1.0]]), gate_up, down, 1)
    g = a * 0.9
    expect = c * 0.5 * g * (1 + math.tanh(math.sqrt(2 / math.pi) * (g + 0.044715 * g ** 3))) * (b * -0.4)
    ref = np.zeros((1, H))
    ref[0, 2] = expect
    np.testing.assert_allclose(y, ref, rtol=1e-14, atol=1e-300)


def test_grouped_experts_equal_per_token_loop():
    rng = _rng(8)
    T, H, E, I, k = 9, 16, 5, 4, 2
    x = rng.standard_normal((T, H))
    gu = rng.standard_normal((E, 2 * I, H)) * 0.3
    dn = rng.standard_normal((E, H, I)) * 0.3
    idx = np.array([sorted(rng.choice(E, k, replace=False)) for _ in range(T)], np.int32)
    w = rng.uniform(0, 1, (T, k))
    y = o.experts_forward(x, idx, w, gu, dn, I)
    for t in range(T):
        acc = [0.0] * H
        for j in range(k):
            e = idx[t, j]
            act = []
            for f in range(I):
                gs = sum(gu[e, f, i] * x[t, i] for i in range(H))
                us = sum(gu[e, I + f, i] * x[t, i] for i in range(H))
                gl = 0.5 * gs * (1 + math.tanh(math.sqrt(2 / math.pi) * (gs + 0.044715 * gs ** 3)))
                act.append(gl * us)
            for hh in range(H):
                acc[hh] += w[t, j] * sum(dn[e, hh, f] * act[f] for f in range(I))
        np.testing.assert_allclose(y[t], acc, rtol=1e-10, atol=1e-13)


def test_identical_experts_collapse_to_one_mlp():
    rng = _rng(9)
    p = _small_params(rng)
    for n in ("gate_up", "down"):
        p[n] = np.repeat(p[n][:1], p[n].shape[0], axis=0)
    h = rng.standard_normal((7, 32))
    r = o.moe_block_forward(h, p, top_k=3, inter=8)
    single = o.geglu_mlp(r["xe"], p["gate_up"][0, :8], p["gate_up"][0, 8:], p["down"][0])
    np.testing.assert_allclose(r["y_moe"], single, rtol=1e-12, atol=1e-14)


def test_topk_equal_to_all_experts_is_dense_mixture():
    rng = _rng(10)
    p = _small_params(rng)
    E = p["router"].shape[0]
    h = rng.standard_normal((5, 32))
    r = o.moe_block_forward(h, p, top_k=E, inter=8)
    for t in range(5):
        zt = list(r["z"][t])
        m = max(zt)
        ex = [math.exp(v - m) for v in zt]
        pr = [v / sum(ex) for v in ex]
        mix = sum(pr[e] * o.geglu_mlp(r["xe"][t:t + 1], p["gate_up"][e, :8],
                                     p["gate_up"][e, 8:], p["down"][e])[0] for e in range(E))
        np.testing.assert_allclose(r["y_moe"][t], mix, rtol=1e-11, atol=1e-14)


def test_mlp_of_zero_is_zero():
    p = _small_params(_rng(11))
    y = o.geglu_mlp(np.zeros((1, 32)), p["dense_gate"], p["dense_up"], p["dense_down"])
    assert np.all(y == 0)


# ---------------------------------------------------------------- combine

def test_combine_closed_form_rms_of_branch_sum():
    rng = _rng(12)
    H = 24
    h = rng.standard_normal((4, H))
    yd = rng.standard_normal((4, H)) * 0.1
    ym = rng.standard_normal((4, H)) * 5.0
    s = 0.6
    out = o.combine(h, yd, ym, np.ones(H), np.ones(H), np.ones(H), s)
    ob = out / s - h
    # post_ff output is RMS-normalised: its RMS is sqrt(m / (m + eps))
    m = np.mean((o.rms_norm(yd) + o.rms_norm(ym)) ** 2, axis=1)
    np.testing.assert_allclose(np.sqrt(np.mean(ob ** 2, axis=1)), np.sqrt(m / (m + 1e-6)),
                               rtol=1e-12)
    # each branch is normalised before the sum: scaling a branch whose mean
    # square is far above eps changes the output only by O(eps) terms
    yd1 = rng.standard_normal((4, H))
    base = o.combine(h, yd1, ym, np.ones(H), np.ones(H), np.ones(H), s)
    out2 = o.combine(h, yd1 * 7.0, ym * 0.5, np.ones(H), np.ones(H), np.ones(H), s)
    np.testing.assert_allclose(out2, base, rtol=1e-5, atol=1e-5)


def test_block_output_with_zero_mlps_is_scaled_residual():
    rng = _rng(13)
    p = _small_params(rng)
    for n in ("gate_up", "down", "dense_gate", "dense_up", "dense_down"):
        p[n] = np.zeros_like(p[n])
    h = rng.standard_normal((3, 32))
    r = o.moe_block_forward(h, p, top_k=2, inter=8)
    np.testing.assert_array_equal(r["out"], h * p["layer_scalar"])


# ---------------------------------------------------------------- permutation

def _brute_perm(idx, E):
    T, k = idx.shape
    perm, counts = [], [0] * E
    for e in range(E):
        for t in range(T):
            for j in range(k):
                if idx[t, j] == e:
                    perm.append(t * k + j)
                    counts[e] += 1
    return counts, perm


def test_permutation_matches_brute_force_and_is_a_bijection():
    rng = _rng(14)
    for (T, E, k) in [(1, 4, 2), (13, 8, 3), (40, 16, 4), (7, 5, 5)]:
        idx = np.array([sorted(rng.choice(E, k, replace=False)) for _ in range(T)], np.int32)
        off, perm = o.permutation(idx, E)
        counts, bperm = _brute_perm(idx, E)
        assert list(perm) == bperm
        assert off[0] == 0 and off[-1] == T * k and np.all(np.diff(off) == counts)
        assert sorted(perm) == list(range(T * k))
        for e in range(E):
            seg = perm[off[e]:off[e + 1]]
            assert all(idx.reshape(-1)[a] == e for a in seg)


# ---------------------------------------------------------------- quantised path

def _dequant_by_hand(qt):
    """Bit-by-bit decode, written independently of the oracle's vectorised one."""
    q = np.asarray(qt["q"])
    bits, g = qt["bits"], qt["group"]
    lead = q.shape[:-1]
    K = q.shape[-1] * (8 if bits == 4 else 1)
    out = np.empty(lead + (K,))
    sc = qt["scales"].astype(np.uint32)
    bi = qt["biases"].astype(np.uint32)
    for pos in itertools.product(*[range(n) for n in lead]):
        for kk in range(K):
            if bits == 4:
                code = (int(q[pos + (kk // 8,)]) >> (4 * (kk % 8))) & 15
            else:
                code = int(q[pos + (kk,)])
            s = float(np.array([sc[pos + (kk // g,)] << 16], np.uint32).view(np.float32)[0])
            b = float(np.array([bi[pos + (kk // g,)] << 16], np.uint32).view(np.float32)[0])
            out[pos + (kk,)] = s * code + b
    return out


@pytest.mark.parametrize("bits", [4, 8])
def test_dequant_matches_hand_decode_and_nearest_level(bits):
    rng = _rng(20 + bits)
    w = mi.f32_to_bf16_bits(rng.standard_normal((3, 128)).astype(np.float32) * 0.02)
    qt = mi.quantize_affine(w, bits)
    deq = o.dequant_affine(qt)
    np.testing.assert_array_equal(deq, _dequant_by_hand(qt))
    wf = o.bf16_to_f64(w)
    # every decoded weight is the level nearest to the original one
    s = np.repeat(o.bf16_to_f64(qt["scales"]), 64, axis=-1)
    b = np.repeat(o.bf16_to_f64(qt["biases"]), 64, axis=-1)
    levels = b[..., None] + s[..., None] * np.arange(2 ** bits)
    best = np.abs(levels - wf[..., None]).min(axis=-1)
    assert np.all(np.abs(deq - wf) <= best + 1e-12)


def test_dequant_constant_group_is_exact():
    w = np.full((2, 64), mi.f32_to_bf16_bits(np.float32([0.0123]))[0], np.uint16)
    for bits in (4, 8):
        deq = o.dequant_affine(mi.quantize_affine(w, bits))
        np.testing.assert_array_equal(deq, o.bf16_to_f64(w))


def test_quantised_block_equals_dequant_then_bf16_block():
    wl = mi.get_workload("tiny", quant=(4, 4, 8))
    pq = mi.make_layer_inputs(wl, randvec=True)
    h = mi.make_tokens(wl)[:6]
    pd = dict(pq)
    for n in ("router", "gate_up", "down", "dense_gate", "dense_up", "dense_down"):
        if n in ("gate_up", "down"):
            pd[n] = np.stack([_dequant_by_hand({**pq[n], "q": pq[n]["q"][e],
                                                "scales": pq[n]["scales"][e],
                                                "biases": pq[n]["biases"][e]})
                              for e in range(wl.n_experts)])
        else:
            pd[n] = _dequant_by_hand(pq[n])
    rq = o.moe_block_forward(h, pq, wl.top_k, wl.expert_inter)
    rd = o.moe_block_forward(h, pd, wl.top_k, wl.expert_inter)
    assert np.array_equal(rq["idx"], rd["idx"])
    np.testing.assert_allclose(rq["out"], rd["out"], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("bits", [4, 8])
def test_quantised_sc_mlp_equals_the_mlp_on_hand_decoded_weights(bits):
    # the self-conditioning MLP on 4- and 8-bit (q8) affine weights is the
    # same MLP on the weights decoded by hand
    wl = mi.get_workload("sc_tiny", quant=(bits, bits, 8))
    pq = mi.make_sc_inputs(wl, randvec=True, quantise=True)
    assert all(pq[n]["bits"] == bits for n in ("gate", "up", "down"))
    pd = dict(pq)
    for n in ("gate", "up", "down"):
        pd[n] = _dequant_by_hand(pq[n])
    e, sg = pq["embeds"][:5], pq["signal"][:5]
    np.testing.assert_allclose(o.sc_mlp_forward(e, sg, pq), o.sc_mlp_forward(e, sg, pd),
                               rtol=1e-12, atol=1e-12)


def test_bf16_decoded_weights_are_the_rounded_exact_decode():
    # the bf16_weights variant: exact decode by hand, then round to nearest
    # even bf16 through the input module's independent rounding (the decode
    # s*q + b of bf16 s, b and a 4-bit q is exact in float32)
    rng = _rng(31)
    w = mi.f32_to_bf16_bits(rng.standard_normal((4, 256)).astype(np.float32) * 0.02)
    qt = mi.quantize_affine(w, 4)
    exact = _dequant_by_hand(qt)
    want = o.bf16_to_f64(mi.f32_to_bf16_bits(exact.astype(np.float32)))
    assert np.array_equal(exact.astype(np.float32).astype(np.float64), exact)
    got = o.decoded(qt, bf16_weights=True)
    np.testing.assert_array_equal(got, want)
    # within half a bf16 ulp of the exact decode, and not all equal to it
    ulp = np.ldexp(1.0, np.floor(np.log2(np.abs(np.where(exact == 0, 1, exact)))).astype(int) - 7)
    assert np.all(np.abs(got - exact) <= ulp / 2)
    assert np.any(got != exact)
    # bf16 weights and float64 weights pass through unchanged
    assert np.array_equal(o.decoded(w, True), o.bf16_to_f64(w))


def test_bf16_weights_variant_leaves_bf16_block_unchanged_and_changes_q4_block():
    wl = mi.get_workload("tiny")
    h = mi.make_tokens(wl)[:8]
    pb = mi.make_layer_inputs(wl, randvec=True)
    r0 = o.moe_block_forward(h, pb, wl.top_k, wl.expert_inter)
    r1 = o.moe_block_forward(h, pb, wl.top_k, wl.expert_inter, bf16_weights=True)
    assert np.array_equal(r0["out"], r1["out"])
    pq = mi.make_layer_inputs(wl, randvec=True, quantise=True)
    q0 = o.moe_block_forward(h, pq, wl.top_k, wl.expert_inter)
    q1 = o.moe_block_forward(h, pq, wl.top_k, wl.expert_inter, bf16_weights=True)
    assert np.array_equal(q0["idx"], q1["idx"])         # the router stays exact
    d = np.abs(q1["out"] - q0["out"]).max()
    assert 0 < d < 0.05 * np.sqrt(np.mean(q0["out"] ** 2))


# ---------------------------------------------------------------- whole block

def test_canvas_permutation_permutes_outputs():
    wl = mi.get_workload("tiny")
    p = mi.make_layer_inputs(wl, randvec=True)
    h = mi.make_tokens(wl)
    r = o.moe_block_forward(h, p, wl.top_k, wl.expert_inter)
    pi = _rng(15).permutation(wl.tokens)
    rp = o.moe_block_forward(h[pi], p, wl.top_k, wl.expert_inter)
    assert np.array_equal(rp["idx"], r["idx"][pi])
    np.testing.assert_allclose(rp["out"], r["out"][pi], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(rp["w"], r["w"][pi], rtol=1e-12)


def test_block_against_direct_formula_on_tiny_workload():
    """The whole block written out per token with python loops over experts,
    against moe_block_forward (2 tokens of the tiny workload)."""
    wl = mi.get_workload("tiny")
    p = mi.make_layer_inputs(wl, randvec=True)
    h = o.bf16_to_f64(mi.make_tokens(wl)[:2])
    r = o.moe_block_forward(h, p, wl.top_k, wl.expert_inter)
    H, E, K, I = wl.hidden, wl.n_experts, wl.top_k, wl.expert_inter
    f = lambda n: o.to_f64(p[n])
    for t in range(2):
        x = h[t]
        rr = 1 / math.sqrt(sum(v * v for v in x) / H + 1e-6)
        xr = x * rr * f("router_scale") / math.sqrt(H)
        z = [float(np.dot(f("router")[e], xr)) for e in range(E)]
        sel = _brute_topk(z, K)
        m = max(z)
        pr = [math.exp(v - m) for v in z]
        tot = sum(pr[e] for e in sel)
        ww = [pr[e] / tot * f("per_expert_scale")[e] for e in sel]
        xe = x * rr * f("w_pre_ff2")
        xd = x * rr * f("w_pre_ff")
        ym = np.zeros(H)
        for e, we in zip(sel, ww):
            gu = f("gate_up")[e]
            ym += we * o.geglu_mlp(xe[None], gu[:I], gu[I:], f("down")[e])[0]
        yd = o.geglu_mlp(xd[None], f("dense_gate"), f("dense_up"), f("dense_down"))[0]
        n = lambda v, w: v / math.sqrt(float(np.mean(v * v)) + 1e-6) * w
        out = (x + n(n(yd, f("w_post_ff1")) + n(ym, f("w_post_ff2")), f("w_post_ff"))) * p["layer_scalar"]
        assert list(r["idx"][t]) == sel
        np.testing.assert_allclose(r["w"][t], ww, rtol=1e-12)
        np.testing.assert_allclose(r["out"][t], out, rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- bf16 rounding

def test_round_bf16_ties_to_even_and_nearest():
    ulp = 2.0 ** -7
    cases = {1.0 + ulp / 2: 1.0, 1.0 + 3 * ulp / 2: 1.0 + 2 * ulp, -(1.0 + ulp / 2): -1.0,
             1.0 + ulp / 2 + 1e-12: 1.0 + ulp, 3.0: 3.0, 0.0: 0.0}
    for x, want in cases.items():
        assert o.round_bf16(np.array([x]))[0] == want, x
    # brute force: the nearest of all bf16 values of the same binade
    rng = _rng(30)
    x = rng.standard_normal(2000) * 10.0 ** rng.integers(-3, 3, 2000)
    got = o.round_bf16(x)
    for xi, gi in zip(x, got):
        e = math.floor(math.log2(abs(xi)))
        grid = np.sign(xi) * (1 + np.arange(0, 129) / 128.0) * 2.0 ** e
        d = np.abs(grid - xi)
        assert abs(gi - xi) <= d.min() + 1e-300
        assert abs(gi) >= 2.0 ** e or gi == 0


def test_bf16_activation_variant_rounds_only_the_activations():
    rng = _rng(31)
    T, H, E, I, k = 6, 16, 4, 8, 2
    x = rng.standard_normal((T, H))
    gu = rng.standard_normal((E, 2 * I, H)) * 0.3
    dn = rng.standard_normal((E, H, I)) * 0.3
    idx = np.array([sorted(rng.choice(E, k, replace=False)) for _ in range(T)], np.int32)
    w = rng.uniform(0, 1, (T, k))
    y = o.experts_forward(x, idx, w, gu, dn, I, bf16_activations=True)
    xb = o.round_bf16(x)
    ref = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            a = o.round_bf16(o.gelu_tanh(gu[e, :I] @ xb[t]) * (gu[e, I:] @ xb[t]))
            ref[t] += w[t, j] * (dn[e] @ a)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-14)
    y0 = o.experts_forward(x, idx, w, gu, dn, I)
    assert 1e-4 < np.abs(y - y0).max() / np.abs(y0).max() < 2e-2


# ---------------------------------------------------------------- self-conditioning MLP

def test_sc_zero_signal_is_the_weightless_norm_of_the_embeddings():
    # the MLP maps 0 to 0 ("DiffusionGemma Explained": relevant for the
    # self-conditioning MLP on the first decode step), so only the post-norm
    # of the embeddings remains; checked against torch's RMSNorm routine
    import torch
    wl = mi.get_workload("sc_tiny")
    p = mi.make_sc_inputs(wl, randvec=True)
    zero = np.zeros_like(p["signal"])
    got = o.sc_mlp_forward(p["embeds"], zero, p)
    x = torch.from_numpy(o.bf16_to_f64(p["embeds"]))
    want = torch.nn.functional.rms_norm(x, (x.shape[-1],), eps=1e-6).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_sc_composition_prenorm_signal_residual_then_weightless_postnorm():
    # structure of the pages' listing: RMSNorm_w on the signal, GEGLU MLP,
    # add to the embeddings, RMSNorm without weight; torch ops as the reference
    import torch
    wl = mi.get_workload("sc_tiny")
    p = mi.make_sc_inputs(wl, randvec=True)
    got = o.sc_mlp_forward(p["embeds"], p["signal"], p)
    t = lambda a: torch.from_numpy(o.bf16_to_f64(a))
    H = wl.hidden
    n = torch.nn.functional.rms_norm(t(p["signal"]), (H,), weight=t(p["pre_norm"]), eps=1e-6)
    g = torch.nn.functional.gelu(n @ t(p["gate"]).T, approximate="tanh")
    s = (g * (n @ t(p["up"]).T)) @ t(p["down"]).T
    want = torch.nn.functional.rms_norm(t(p["embeds"]) + s, (H,), eps=1e-6).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-10)
    # every output row has unit RMS up to eps
    assert np.all(np.abs(np.sqrt((got ** 2).mean(1)) - 1) < 1e-5)


def test_sc_permuting_tokens_permutes_outputs():
    wl = mi.get_workload("sc_tiny")
    p = mi.make_sc_inputs(wl)
    pi = np.random.default_rng(9).permutation(wl.tokens)
    a = o.sc_mlp_forward(p["embeds"], p["signal"], p)
    b = o.sc_mlp_forward(p["embeds"][pi], p["signal"][pi], p)
    np.testing.assert_array_equal(a[pi], b)


# ---------------------------------------------------------------- decoder-layer neighbours

def _planes(T=16, H=256, seed=3):
    r = np.random.default_rng(seed)
    bits = lambda a: mi.f32_to_bf16_bits(a.astype(np.float32))
    return (bits(r.standard_normal((T, H))), bits(r.standard_normal((T, H)) * 3.0),
            bits(r.uniform(0.5, 1.5, H)))


def test_attn_residual_with_zero_attention_is_the_residual():
    x, a, w = _planes()
    got = o.attn_residual(x, np.zeros_like(a), w)
    np.testing.assert_array_equal(got, o.bf16_to_f64(x))


def test_attn_residual_constant_attention_rows_add_plus_minus_one():
    # rows of a constant c normalise to sign(c) (1 - O(eps / c^2), which
    # rounds to 1 in bf16), so with a unit weight h = bf16(x + sign(c))
    x, _, _ = _planes()
    T, H = x.shape
    c = np.where(np.arange(T) % 2 == 0, 0.75, -2.5)
    a = mi.f32_to_bf16_bits(np.repeat(c[:, None], H, 1).astype(np.float32))
    ones = np.full(H, mi.BF16_ONE, dtype=np.uint16)
    got = o.attn_residual(x, a, ones)
    want = o.round_bf16(o.bf16_to_f64(x) + np.sign(c)[:, None])
    np.testing.assert_array_equal(got, want)


def test_attn_residual_against_torch_rms_norm():
    import torch
    x, a, w = _planes()
    t = lambda b: torch.from_numpy(o.bf16_to_f64(b))
    n = torch.nn.functional.rms_norm(t(a), (a.shape[1],), weight=t(w), eps=1e-6)
    n = n.to(torch.bfloat16).to(torch.float64)          # torch's own rounding
    want = (t(x) + n).to(torch.bfloat16).to(torch.float64).numpy()
    got = o.attn_residual(x, a, w)
    # torch rounds through fp32: identical except on the rare double-rounding case
    diff = np.abs(got - want) / np.maximum(np.abs(want), 1e-30)
    assert (got == want).mean() > 0.999 and diff.max() <= 2.0 ** -7


def test_next_input_norm_constant_rows_give_the_weight():
    _, _, w = _planes()
    H = w.shape[0]
    out = mi.f32_to_bf16_bits(np.array([[1.5] * H, [-0.25] * H], np.float32))
    got = o.next_input_norm(out, w)
    np.testing.assert_array_equal(got[0], o.bf16_to_f64(w))
    np.testing.assert_array_equal(got[1], -o.bf16_to_f64(w))


def test_next_input_norm_against_torch_rms_norm():
    import torch
    x, _, w = _planes()
    t = lambda b: torch.from_numpy(o.bf16_to_f64(b))
    want = torch.nn.functional.rms_norm(t(x), (x.shape[1],), weight=t(w), eps=1e-6)
    want = want.to(torch.bfloat16).to(torch.float64).numpy()
    got = o.next_input_norm(x, w)
    diff = np.abs(got - want) / np.maximum(np.abs(want), 1e-30)
    assert (got == want).mean() > 0.999 and diff.max() <= 2.0 ** -7


# ---------------------------------------------------------------- NVFP4 weights

def test_e4m3_decode_matches_torch_float8():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)   # no NaN
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(o.e4m3_value(codes), want)


def test_e2m1_decode_values():
    # the sixteen fp4 e2m1 values (sign, exponent bias 1, one mantissa bit)
    want = [0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.0, -0.5, -1, -1.5, -2, -3, -4, -6]
    np.testing.assert_array_equal(o.e2m1_value(np.arange(16)), want)


def test_nvfp4_decode_bit_by_bit():
    w = mi._normal_bf16(np.random.default_rng(5), (3, 8, 48), 0.02)
    qt = mi.quantize_nvfp4(w)
    got = o.dequant_nvfp4(qt)
    ref = np.zeros((3, 8, 48))
    e2m1 = {0: 0.0, 1: 0.5, 2: 1.0, 3: 1.5, 4: 2.0, 5: 3.0, 6: 4.0, 7: 6.0}
    for e in range(3):
        for r in range(8):
            for k in range(48):
                byte = int(qt["q"][e, r, k // 2])
                c = (byte >> 4) if k % 2 else (byte & 15)
                v = e2m1[c & 7] * (-1 if c & 8 else 1)
                sc = int(qt["scales"][e, r, k // 16])
                ex, m = sc >> 3, sc & 7
                s = m * 2.0 ** -9 if ex == 0 else (1 + m / 8) * 2.0 ** (ex - 7)
                ref[e, r, k] = v * s * float(qt["globals"][e])
    np.testing.assert_array_equal(got, ref)


def test_nvfp4_round_trip_error_bound():
    # within one e2m1 step of the block scale (the widest step, 4 -> 6, is 2),
    # beyond saturation at 6 when the e4m3 scale rounded down
    w = mi._normal_bf16(np.random.default_rng(6), (4, 32, 256), 0.02)
    qt = mi.quantize_nvfp4(w)
    wf = o.bf16_to_f64(w)
    deq = o.dequant_nvfp4(qt)
    sg = (o.e4m3_value(qt["scales"]) * qt["globals"].astype(np.float64)[:, None, None])
    sg = np.repeat(sg, 16, axis=-1)
    err = np.abs(wf - deq)
    assert np.all(err <= 1.0 * sg + np.maximum(np.abs(wf) - 6 * sg, 0) + 1e-12)
    # the decode of the block maximum is its nearest level: relative error small
    assert np.abs(deq - wf).mean() < 0.1 * np.abs(wf).mean()


def test_nvfp4_block_times_scale_is_bf16_exact():
    # an e2m1 value times an e4m3 scale has at most 6 significant bits, so the
    # GPU's bf16 decode of it is exact; the matrix scale comes after the sum
    w = mi._normal_bf16(np.random.default_rng(7), (2, 16, 64), 0.02)
    qt = mi.quantize_nvfp4(w)
    q = qt["q"]
    codes = np.stack([q & 0xF, q >> 4], -1).reshape(*q.shape[:-1], q.shape[-1] * 2)
    v = o.e2m1_value(codes).reshape(2, 16, 4, 16) * o.e4m3_value(qt["scales"])[..., None]
    np.testing.assert_array_equal(o.round_bf16(v), v)
