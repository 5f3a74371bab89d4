"""Seeded synthetic inputs for the routed-MoE feed-forward block.

This module is the only code shared by the CPU oracle and the CUDA path.  It
draws the tensors of a layer (activations, router, expert and dense weights,
norm vectors) from numpy's PCG64 generator, rounds them to bf16 and, for the
quantised workloads, encodes them in the group-64 affine format.  It holds none
of the block's forward arithmetic: no normalisation, routing, GEMM, activation
or dequantisation.

Workloads (the shapes are the DiffusionGemma MoE layer: hidden 2816, 128
experts, top-8, expert FFN 704, dense FFN 2112; "diffgemma — architecture &
implemented contract", Part II §1 model constants; "DiffusionGemma port —
plan & parity strategy", Reference dossier §1 top-level config):

* ``tiny``      32 tokens, hidden 256, 16 experts top-4, expert 64, dense 128;
                weights N(0, 0.02), router N(0, 1/16), activations N(0, 1).
* ``canvas256`` one full-shape layer over a 256-token canvas, bf16 weights
                N(0, 0.02) (router included), activations N(0, 1).
* ``canvas256_q4`` the same draws as ``canvas256``, expert and dense weights
                4-bit group-64 affine, router 8-bit group-64 affine.
* ``batch2048_zipf`` 8 canvases (2048 tokens), bf16, and a per-expert router
                logit bias beta*ln(p) with p Zipf(1.2) over a seeded expert
                permutation, so that expert loads are skewed.
* ``batch2048_zipf_b1`` the same with beta 1 (the literal bias): routing
                collapses onto about eight experts (stress case).
* ``stack30_q4``  30 stacked layers, 64 canvases (16384 tokens), 4-bit
                weights, 8-bit router, layer scalars U(0.5, 1.5).

Seeding: ``SeedSequence(seed).spawn(1 + n_layers)``; child 0 draws the
activations, child 1 + l draws layer l (router, then per expert gate_up and
down, then dense gate, up, down, then the layer's extra vectors).  With
``randvec=True`` the norm weights, router scale, per-expert scale and the
layer scalar are drawn U(0.5, 1.5) from ``default_rng(seed + 100)`` instead of
being ones, so that no multiply by them is dead code.
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

__all__ = [
    "Workload",
    "WORKLOADS",
    "get_workload",
    "f32_to_bf16_bits",
    "quantize_affine",
    "make_layer_inputs",
    "make_tokens",
    "zipf_router_bias",
    "SC_WORKLOADS",
    "make_sc_inputs",
    "quantize_nvfp4",
]

BF16_ONE = np.uint16(0x3F80)
NVFP4 = 16   # weight "bits" code of the NVFP4 format in a workload's quant tuple


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    tokens: int
    hidden: int
    n_experts: int
    top_k: int
    expert_inter: int
    dense_inter: int
    seed: int
    weight_std: float
    router_std: float
    n_layers: int = 1
    # None for bf16 weights; otherwise bits for (experts, dense, router)
    quant: Optional[tuple] = None
    # seed whose bf16 draws are quantised (the 4-bit canvas reuses canvas256's)
    draw_seed: Optional[int] = None
    zipf_beta: Optional[float] = None
    layer_scalar_range: Optional[tuple] = None

    @property
    def quantised(self) -> bool:
        return self.quant is not None


WORKLOADS = {
    "tiny": Workload("tiny", 32, 256, 16, 4, 64, 128, seed=0,
                     weight_std=0.02, router_std=1.0 / 16.0),
    "canvas256": Workload("canvas256", 256, 2816, 128, 8, 704, 2112, seed=1,
                          weight_std=0.02, router_std=0.02),
    "canvas256_q4": Workload("canvas256_q4", 256, 2816, 128, 8, 704, 2112,
                             seed=1, weight_std=0.02, router_std=0.02,
                             quant=(4, 4, 8), draw_seed=1),
    # the dense branch at 8 bits (the pages' quantisation predicate for the
    # dense MLP), experts at 4, router at 8
    "canvas256_q4d8": Workload("canvas256_q4d8", 256, 2816, 128, 8, 704, 2112,
                               seed=1, weight_std=0.02, router_std=0.02,
                               quant=(4, 8, 8), draw_seed=1),
    # NVFP4 experts and dense (the pages' nvfp4 profile), 8-bit router
    "canvas256_fp4": Workload("canvas256_fp4", 256, 2816, 128, 8, 704, 2112,
                              seed=1, weight_std=0.02, router_std=0.02,
                              quant=(16, 16, 8), draw_seed=1),
    "batch2048_zipf": Workload("batch2048_zipf", 2048, 2816, 128, 8, 704,
                               2112, seed=2, weight_std=0.02, router_std=0.02,
                               zipf_beta=0.02),
    # the literal reading of the Zipf bias (beta 1): routing collapses onto
    # a handful of experts; a stress case of the same draws
    "batch2048_zipf_b1": Workload("batch2048_zipf_b1", 2048, 2816, 128, 8, 704,
                                  2112, seed=2, weight_std=0.02, router_std=0.02,
                                  zipf_beta=1.0),
    "stack30_q4": Workload("stack30_q4", 16384, 2816, 128, 8, 704, 2112,
                           seed=4, weight_std=0.02, router_std=0.02,
                           n_layers=30, quant=(4, 4, 8),
                           layer_scalar_range=(0.5, 1.5)),
}


# The self-conditioning MLP (dense-FFN shapes, before layer 0) over one
# canvas: the soft signal and the token embeddings drawn N(0, 1).
SC_WORKLOADS = {
    # weight std 0.1 so that the MLP's share of the output (about the
    # embeddings' RMS, as on the full shape) is not hidden by the embeddings
    "sc_tiny": Workload("sc_tiny", 32, 256, 1, 1, 64, 128, seed=6,
                        weight_std=0.1, router_std=0.02),
    "sc_canvas256": Workload("sc_canvas256", 256, 2816, 1, 1, 704, 2112, seed=5,
                             weight_std=0.02, router_std=0.02),
    "sc_canvas256_q4": Workload("sc_canvas256_q4", 256, 2816, 1, 1, 704, 2112, seed=5,
                                weight_std=0.02, router_std=0.02, quant=(4, 4, 8)),
    "sc_canvas256_q8": Workload("sc_canvas256_q8", 256, 2816, 1, 1, 704, 2112, seed=5,
                                weight_std=0.02, router_std=0.02, quant=(8, 8, 8)),
}


def get_workload(name: str, **overrides) -> Workload:
    w = WORKLOADS[name] if name in WORKLOADS else SC_WORKLOADS[name]
    return dataclasses.replace(w, **overrides) if overrides else w


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest even); returns the
    16-bit patterns as uint16.  Inputs are finite draws, so no NaN care."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def _bits_to_f32(b: np.ndarray) -> np.ndarray:
    # widening a bf16 pattern to float32 is exact; used only by the quantiser
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def quantize_affine(w_bits: np.ndarray, bits: int, group: int = 64) -> dict:
    """Encode bf16 weights [..., K] in the group-wise affine format.

    Per group of ``group`` consecutive elements along K: ``lo = min``,
    ``hi = max``; ``scale = bf16((hi - lo) / (2**bits - 1))``;
    ``bias = bf16(lo)``; ``q = clamp(rint((w - bias) / scale), 0, 2**bits-1)``
    using the stored scale and bias (scale 0 gives q 0).  The decoded weight
    is ``scale * q + bias`` ("DiffusionGemma port — plan & parity strategy",
    Reference dossier §1: OptiQ affine quant, group_size 64, 4-bit experts,
    8-bit router).

    Storage (the MLX affine layout): 4-bit codes packed 8 per uint32 word,
    element k at bits 4*(k % 8) of word k // 8, shape [..., K/8]; 8-bit codes
    as uint8 [..., K]; scales and biases as bf16 bits [..., K/group].
    """
    if bits not in (4, 8):
        raise ValueError("bits must be 4 or 8")
    if w_bits.ndim == 3:   # stacked experts: one expert at a time (memory)
        parts = [quantize_affine(w_bits[e], bits, group) for e in range(w_bits.shape[0])]
        return {"bits": bits, "group": group,
                **{k: np.stack([q[k] for q in parts]) for k in ("q", "scales", "biases")}}
    K = w_bits.shape[-1]
    if K % group:
        raise ValueError("K must be a multiple of the group size")
    lead = w_bits.shape[:-1]
    w = _bits_to_f32(w_bits).reshape(*lead, K // group, group)
    lo = w.min(axis=-1)
    hi = w.max(axis=-1)
    levels = np.float32(2 ** bits - 1)
    s_bits = f32_to_bf16_bits((hi - lo) / levels)
    b_bits = f32_to_bf16_bits(lo)
    s = _bits_to_f32(s_bits)[..., None]
    b = _bits_to_f32(b_bits)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(s > 0, np.rint((w - b) / np.where(s > 0, s, 1)), 0)
    q = np.clip(q, 0, levels).astype(np.uint32).reshape(*lead, K)
    if bits == 8:
        packed = q.astype(np.uint8)
    else:
        q8 = q.reshape(*lead, K // 8, 8)
        shifts = (np.arange(8, dtype=np.uint32) * np.uint32(4))
        packed = np.bitwise_or.reduce(q8 << shifts, axis=-1).astype(np.uint32)
    return {"bits": bits, "group": group, "q": packed,
            "scales": s_bits, "biases": b_bits}


# e2m1 magnitudes by code (bits e1 e0 m): 0, 0.5, 1, 1.5, 2, 3, 4, 6
_E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _e4m3_encode(v: np.ndarray) -> np.ndarray:
    """Non-negative float64 -> fp8 e4m3 (bias 7, no infinity, max 448) codes,
    rounded to nearest, ties to even; values above 448 saturate."""
    v = np.minimum(np.asarray(v, np.float64), 448.0)
    code = np.zeros(v.shape, np.uint8)
    pos = v > 0
    e = np.floor(np.log2(np.where(pos, v, 1.0)))
    sub = pos & (e < -6)
    m_sub = np.rint(np.where(sub, v, 0.0) / 2.0 ** -9)          # ties to even
    code = np.where(sub, m_sub.astype(np.uint8), code)            # 8 -> 2^-6, code 8
    nrm = pos & ~sub
    en = np.where(nrm, e, 0.0)
    m = np.rint((np.where(nrm, v, 1.0) / 2.0 ** en - 1.0) * 8.0)
    carry = m >= 8
    en = np.where(carry, en + 1, en)
    m = np.where(carry, 0, m)
    c = ((en + 7).astype(np.int64) << 3) | m.astype(np.int64)
    code = np.where(nrm, np.minimum(c, 0x7E).astype(np.uint8), code)
    return code


def _e4m3_value(code: np.ndarray) -> np.ndarray:
    c = np.asarray(code, np.int64)
    e, m = (c >> 3) & 15, c & 7
    return np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * 2.0 ** (e - 7))


def _e2m1_encode(x: np.ndarray) -> np.ndarray:
    """float64 -> e2m1 codes (sign bit 3), nearest magnitude with ties to the
    even code, saturating at 6."""
    a = np.abs(x)
    d = np.abs(a[..., None] - _E2M1_MAG)
    best = np.argmin(d + 1e-9 * (np.arange(8) & 1), axis=-1)   # ties: even code
    return (best | np.where(x < 0, 8, 0)).astype(np.uint8)


def quantize_nvfp4(w_bits: np.ndarray) -> dict:
    """Encode bf16 weights [..., K] in NVFP4 ("diffgemma — architecture &
    implemented contract", §8 quantisation profiles: nvfp4 experts, K a
    multiple of 16): e2m1 codes, two a byte (element k in the low nibble of
    byte k // 2 when k is even), one fp8 e4m3 scale per 16 consecutive
    elements along K, and one fp32 scale per matrix (per expert for a stack).
    global = amax / (6 * 448); block scale = e4m3(block amax / 6 / global);
    code = e2m1(w / (block scale * global)).  The decoded weight is
    e2m1 * block scale * global."""
    w = _bits_to_f32(w_bits).astype(np.float64)
    K = w.shape[-1]
    if K % 16:
        raise ValueError("K must be a multiple of 16")
    lead = w.shape[:-1]
    mats = w.reshape(-1, *w.shape[-2:]) if w.ndim >= 2 else w.reshape(1, 1, K)
    amax = np.abs(mats).reshape(mats.shape[0], -1).max(axis=1)
    g = np.where(amax > 0, amax / (6.0 * 448.0), 1.0).astype(np.float32)
    gf = g.astype(np.float64)[:, None, None]
    blocks = mats.reshape(mats.shape[0], mats.shape[1], K // 16, 16)
    bamax = np.abs(blocks).max(axis=-1)
    sc = _e4m3_encode(bamax / 6.0 / gf)
    codes = np.empty(blocks.shape, np.uint8)
    for m in range(blocks.shape[0]):   # one matrix at a time bounds the memory
        sv = _e4m3_value(sc[m])[..., None] * gf[m, ..., None]
        with np.errstate(divide="ignore", invalid="ignore"):
            codes[m] = _e2m1_encode(np.where(sv > 0, blocks[m] / np.where(sv > 0, sv, 1.0), 0.0))
    codes = codes.reshape(*lead, K)
    packed = (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)
    return {"fmt": "nvfp4", "q": packed, "scales": sc.reshape(*lead, K // 16),
            "globals": g if w.ndim == 3 else g[:1]}


def _normal_bf16(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    x = rng.standard_normal(shape, dtype=np.float32)
    x *= np.float32(std)
    return f32_to_bf16_bits(x)


def zipf_router_bias(rng: np.random.Generator, n_experts: int, beta: float,
                     s: float = 1.2) -> np.ndarray:
    """Per-expert additive router-logit bias beta*ln(p[pi(e)]), with
    p_k proportional to k^-s over k = 1..E and pi a seeded permutation."""
    k = np.arange(1, n_experts + 1, dtype=np.float64)
    p = k ** (-s)
    p /= p.sum()
    pi = rng.permutation(n_experts)
    return (beta * np.log(p[pi])).astype(np.float32)


def make_tokens(wl: Workload, tokens: Optional[int] = None) -> np.ndarray:
    """Activations h [T, H] as bf16 bits, N(0, 1)."""
    T = wl.tokens if tokens is None else tokens
    child = np.random.SeedSequence(wl.seed).spawn(1 + wl.n_layers)[0]
    rng = np.random.default_rng(child)
    return _normal_bf16(rng, (T, wl.hidden), 1.0)


def _vectors(wl: Workload, randvec: bool, layer: int) -> dict:
    H, E = wl.hidden, wl.n_experts
    names = ["router_scale", "w_pre_ff", "w_pre_ff2", "w_post_ff1",
             "w_post_ff2", "w_post_ff"]
    out = {}
    if randvec:
        rng = np.random.default_rng(wl.seed + 100 + 1000 * layer)
        for n in names:
            out[n] = f32_to_bf16_bits(rng.uniform(0.5, 1.5, H).astype(np.float32))
        out["per_expert_scale"] = f32_to_bf16_bits(
            rng.uniform(0.5, 1.5, E).astype(np.float32))
        ls = float(_bits_to_f32(f32_to_bf16_bits(
            np.float32([rng.uniform(0.5, 1.5)])))[0])
    else:
        for n in names:
            out[n] = np.full(H, BF16_ONE, dtype=np.uint16)
        out["per_expert_scale"] = np.full(E, BF16_ONE, dtype=np.uint16)
        ls = 1.0
    out["layer_scalar"] = ls
    return out


def make_layer_inputs(wl: Workload, layer: int = 0, randvec: bool = False,
                      quantise: Optional[bool] = None) -> dict:
    """Draw one layer's parameters.

    Returns a dict of numpy arrays: bf16 tensors as uint16 bit patterns,
    quantised tensors as the dicts of :func:`quantize_affine`.  Keys:
    router [E, H], gate_up [E, 2I, H] (rows 0..I-1 gate, I..2I-1 up),
    down [E, H, I], dense_gate [D, H], dense_up [D, H], dense_down [H, D],
    router_scale [H], per_expert_scale [E], w_pre_ff, w_pre_ff2, w_post_ff1,
    w_post_ff2, w_post_ff [H], router_bias [E] float32 or None, and the
    python float layer_scalar.
    """
    H, E, I, D = wl.hidden, wl.n_experts, wl.expert_inter, wl.dense_inter
    seed = wl.draw_seed if wl.draw_seed is not None else wl.seed
    child = np.random.SeedSequence(seed).spawn(1 + wl.n_layers)[1 + layer]
    rng = np.random.default_rng(child)
    p = {}
    p["router"] = _normal_bf16(rng, (E, H), wl.router_std)
    gate_up = np.empty((E, 2 * I, H), dtype=np.uint16)
    down = np.empty((E, H, I), dtype=np.uint16)
    for e in range(E):
        gate_up[e] = _normal_bf16(rng, (2 * I, H), wl.weight_std)
        down[e] = _normal_bf16(rng, (H, I), wl.weight_std)
    p["gate_up"], p["down"] = gate_up, down
    p["dense_gate"] = _normal_bf16(rng, (D, H), wl.weight_std)
    p["dense_up"] = _normal_bf16(rng, (D, H), wl.weight_std)
    p["dense_down"] = _normal_bf16(rng, (H, D), wl.weight_std)
    p["router_bias"] = (zipf_router_bias(rng, E, wl.zipf_beta)
                        if wl.zipf_beta is not None else None)
    p.update(_vectors(wl, randvec, layer))
    if wl.layer_scalar_range is not None and not randvec:
        lo, hi = wl.layer_scalar_range
        v = np.float32([rng.uniform(lo, hi)])
        p["layer_scalar"] = float(_bits_to_f32(f32_to_bf16_bits(v))[0])
    do_q = wl.quantised if quantise is None else quantise
    if do_q:
        # bits 4 / 8: group-64 affine; NVFP4 (code 16): e2m1 with e4m3 scales
        eb, db, rb = wl.quant if wl.quant is not None else (4, 4, 8)
        quant = lambda w, b: quantize_nvfp4(w) if b == NVFP4 else quantize_affine(w, b)
        p["router"] = quantize_affine(p["router"], rb)
        p["gate_up"] = quant(p["gate_up"], eb)
        p["down"] = quant(p["down"], eb)
        for n in ("dense_gate", "dense_up", "dense_down"):
            p[n] = quant(p[n], db)
    return p


def make_sc_inputs(wl: Workload, randvec: bool = False, quantise: Optional[bool] = None,
                   tokens: Optional[int] = None) -> dict:
    """Draws of the self-conditioning MLP: token embeddings and soft signal
    [T, H] (N(0, 1), bf16 bits), gate and up [D, H], down [H, D] (N(0, std)),
    and the pre_norm vector (ones, or U(0.5, 1.5) with randvec).  Seeding:
    SeedSequence(seed).spawn(2): child 0 the activations (embeddings, then
    signal), child 1 the weights (gate, up, down).  With quantise (default: the
    workload's own), gate/up/down in the group-64 affine format at the
    workload's dense bits."""
    T = wl.tokens if tokens is None else tokens
    H, D = wl.hidden, wl.dense_inter
    ca, cw = np.random.SeedSequence(wl.seed).spawn(2)
    ra, rw = np.random.default_rng(ca), np.random.default_rng(cw)
    out = {"embeds": _normal_bf16(ra, (T, H), 1.0), "signal": _normal_bf16(ra, (T, H), 1.0)}
    out["gate"] = _normal_bf16(rw, (D, H), wl.weight_std)
    out["up"] = _normal_bf16(rw, (D, H), wl.weight_std)
    out["down"] = _normal_bf16(rw, (H, D), wl.weight_std)
    if randvec:
        r = np.random.default_rng(wl.seed + 100)
        out["pre_norm"] = f32_to_bf16_bits(r.uniform(0.5, 1.5, H).astype(np.float32))
    else:
        out["pre_norm"] = np.full(H, BF16_ONE, dtype=np.uint16)
    do_q = wl.quantised if quantise is None else quantise
    if do_q:
        bits = wl.quant[1] if wl.quant is not None else 4
        for n in ("gate", "up", "down"):
            out[n] = quantize_affine(out[n], bits)
    return out
