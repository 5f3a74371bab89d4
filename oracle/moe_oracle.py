"""Plain fp64 CPU oracle of the routed-MoE feed-forward block.

TEST INFRASTRUCTURE.  Only the tests, the smoke check of ``__graft_entry__``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
this module.  The product (the CUDA library and its Python binding) never
calls it, and it shares no code with the product: its only input is the raw
bit patterns produced by :mod:`moe_inputs`.

Every step is written the plain way, in float64, in the order the pages give:

* RMSNorm ``x / sqrt(mean(x^2) + eps) * w`` with eps 1e-6, the weight
  multiplied directly ("diffgemma — architecture & implemented contract",
  Part II §2.1 Norms and §1 RMS eps; "DiffusionGemma port — plan & parity
  strategy", Reference dossier §1 rms_norm_eps; "Independent GGUF Forward
  Pass ...", §4 fact 9).
* Router: weightless RMSNorm of the raw residual stream, times router.scale
  and hidden^-0.5, as two literal steps (not folded into one weighted norm),
  then a linear map to E logits, softmax over all E, top-k, renormalise the
  k selected to sum 1, multiply by per_expert_scale ("diffgemma ...", Part II
  §2.1 MoE order; "DiffusionGemma Explained", MOEBlock.forward; "DiffusionGemma
  port ...", Reference dossier §2 Router and the D1 router-norm finding).
  Ties: the higher logit wins, equal logits go to the lower expert index
  ("diffgemma ...", §2.1 tie-break).  The selection is taken on the logits,
  which order the experts exactly as the probabilities do.
* Experts: ``down(gelu_tanh(gate(x)) * up(x))`` with gate_up stored fused,
  gate rows first ("diffgemma ...", §2.1; "DiffusionGemma Explained", MLP;
  "DiffusionGemma port ...", Reference dossier §2 MLP and Experts), input
  ``pre_feedforward_layernorm_2(h)``; combined as the routing-weighted sum.
* Dense always-on GEGLU MLP on ``pre_feedforward_layernorm(h)``.
* FFN sandwich: ``h1 = post_ff_1(dense)``, ``h2 = post_ff_2(moe)``,
  ``out = (h + post_ff(h1 + h2)) * layer_scalar`` ("DiffusionGemma port ...",
  Reference dossier §2 DecoderLayer; "DiffusionGemma Explained",
  MOEBlock.forward and the layer-scalar discussion).
* Group-wise affine weights decode as ``scale * q + bias`` per group of 64
  along K ("DiffusionGemma port ...", Reference dossier §1).

Readings where the pages are silent or disagree are listed in the design
notes; the ones that touch this file: eps inside the square root; the tanh
form of GELU; selection on exact logits with ties to the lower index; the k
selected experts reported in ascending expert order; the canonical
permutation sorted by (expert, token); no rounding of intermediates.

Two variants serve the intermediate checks of the tensor-core path, not the
block's definition: ``bf16_activations`` rounds the activation planes to bf16,
and ``bf16_weights`` rounds each group-wise affine weight, once decoded
exactly, to bf16 (the operand type of the bf16 tensor-core product).
"""

from __future__ import annotations

import numpy as np

EPS = 1e-6

__all__ = [
    "EPS", "bf16_to_f64", "round_bf16", "dequant_affine", "to_f64", "decoded", "rms_norm",
    "gelu_tanh",
    "router_logits", "select_topk", "routing_weights", "route",
    "geglu_mlp", "experts_forward", "dense_forward", "combine",
    "permutation", "moe_block_forward", "sc_mlp_forward", "attn_residual", "next_input_norm",
    "e4m3_value", "e2m1_value", "dequant_nvfp4",
]


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Decode bf16 bit patterns (uint16) to float64 exactly."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (8 significant bits,
    ties to even), returned as float64.  Used by the bf16-activation and
    bf16-weight variants and for the bf16 planes around the block
    (:func:`attn_residual`, :func:`next_input_norm`); finite normal-range
    inputs."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                       # x = m 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


def dequant_affine(qt: dict) -> np.ndarray:
    """Decode a group-wise affine tensor to float64: W = scale * q + bias.

    ``qt`` holds ``bits`` (4 or 8), ``group``, ``q`` (4-bit: uint32 words with
    element k at bits 4*(k % 8) of word k // 8; 8-bit: uint8), ``scales`` and
    ``biases`` (bf16 bits, one per group along the last axis)."""
    bits, group = qt["bits"], qt["group"]
    q = np.asarray(qt["q"])
    if bits == 4:
        shifts = np.arange(8, dtype=np.uint32) * np.uint32(4)
        codes = (q[..., None].astype(np.uint32) >> shifts) & np.uint32(0xF)
        codes = codes.reshape(*q.shape[:-1], q.shape[-1] * 8)
    elif bits == 8:
        codes = q.astype(np.uint32)
    else:
        raise ValueError("bits must be 4 or 8")
    s = bf16_to_f64(qt["scales"])
    b = bf16_to_f64(qt["biases"])
    K = codes.shape[-1]
    c = codes.astype(np.float64).reshape(*codes.shape[:-1], K // group, group)
    w = s[..., None] * c + b[..., None]
    return w.reshape(*codes.shape[:-1], K)


def e2m1_value(codes) -> np.ndarray:
    """fp4 e2m1 (sign, 2 exponent bits with bias 1, 1 mantissa bit): e = 0
    gives m / 2, else 2^(e-1) (1 + m/2); the values 0, 0.5, 1, 1.5, 2, 3, 4, 6."""
    c = np.asarray(codes, np.int64)
    e, m = (c >> 1) & 3, c & 1
    mag = np.where(e == 0, 0.5 * m, 2.0 ** (e - 1) * (1.0 + 0.5 * m))
    return np.where(c & 8, -mag, mag)


def e4m3_value(codes) -> np.ndarray:
    """fp8 e4m3 (bias 7, no infinity): e = 0 gives m 2^-9, else
    (1 + m/8) 2^(e-7); sign bit 7 (the block scales are non-negative)."""
    c = np.asarray(codes, np.int64)
    e, m = (c >> 3) & 15, c & 7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * 2.0 ** (e - 7))
    return np.where(c & 0x80, -mag, mag)


def dequant_nvfp4(qt: dict) -> np.ndarray:
    """Decode an NVFP4 tensor to float64: e2m1 code * e4m3 scale of its block
    of 16 along K * the matrix's fp32 scale ("diffgemma — architecture &
    implemented contract", §8: nvfp4 expert profile, K a multiple of 16).
    ``q``: two codes a byte, element k in the low nibble of byte k // 2 for
    even k; ``scales``: e4m3 bytes [..., K/16]; ``globals``: one float32 per
    matrix (per expert of a stack)."""
    q = np.asarray(qt["q"])
    codes = np.stack([q & 0xF, q >> 4], axis=-1).reshape(*q.shape[:-1], q.shape[-1] * 2)
    K = codes.shape[-1]
    v = e2m1_value(codes).reshape(*codes.shape[:-1], K // 16, 16)
    v = v * e4m3_value(qt["scales"])[..., None]
    g = np.asarray(qt["globals"], np.float64)
    v = v.reshape(*codes.shape[:-1], K)
    if v.ndim == 3:
        v = v * g[:, None, None]
    else:
        v = v * g[0]
    return v


def to_f64(t) -> np.ndarray:
    """A weight given as bf16 bits (uint16), as a group-wise affine or NVFP4
    dict, or already as float64 -> float64."""
    if isinstance(t, dict):
        return dequant_nvfp4(t) if t.get("fmt") == "nvfp4" else dequant_affine(t)
    t = np.asarray(t)
    if t.dtype == np.float64:
        return t
    return bf16_to_f64(t)


def _slice(t, e):
    """Expert e of a stacked weight (bf16 bits, affine or NVFP4 dict)."""
    if isinstance(t, dict) and t.get("fmt") == "nvfp4":
        return {"fmt": "nvfp4", "q": t["q"][e], "scales": t["scales"][e],
                "globals": t["globals"][e:e + 1]}
    if isinstance(t, dict):
        return {"bits": t["bits"], "group": t["group"], "q": t["q"][e],
                "scales": t["scales"][e], "biases": t["biases"][e]}
    return t[e]


def rms_norm(x: np.ndarray, w=None, eps: float = EPS) -> np.ndarray:
    """x / sqrt(mean(x^2, last axis) + eps), times w when given."""
    y = x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return y if w is None else y * w


def gelu_tanh(x: np.ndarray) -> np.ndarray:
    """GELU, tanh form: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))."""
    return 0.5 * x * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (x + 0.044715 * x ** 3)))


def router_logits(h: np.ndarray, Wr: np.ndarray, router_scale: np.ndarray,
                  bias=None) -> np.ndarray:
    """z = (rms_norm(h) * router_scale * H^-0.5) @ Wr^T (+ per-expert bias).

    The normalisation is applied to the raw residual stream, before the
    projection, as two literal steps."""
    H = h.shape[-1]
    xr = rms_norm(h)
    xr = xr * router_scale * (H ** -0.5)
    z = xr @ Wr.T
    if bias is not None:
        z = z + np.asarray(bias, dtype=np.float64)
    return z


def select_topk(z: np.ndarray, k: int) -> np.ndarray:
    """Per token, the k experts with the largest logits; equal logits go to
    the lower expert index.  Returned in ascending expert order, int32."""
    T, E = z.shape
    idx = np.empty((T, k), dtype=np.int32)
    experts = np.arange(E)
    for t in range(T):
        order = np.lexsort((experts, -z[t]))   # by -z, then by expert id
        idx[t] = np.sort(order[:k])
    return idx


def routing_weights(z: np.ndarray, idx: np.ndarray, pes: np.ndarray) -> np.ndarray:
    """Softmax over all E logits, keep the selected, renormalise them to sum
    1, multiply by per_expert_scale of the selected expert."""
    zmax = z.max(axis=-1, keepdims=True)
    p = np.exp(z - zmax)
    p = p / p.sum(axis=-1, keepdims=True)
    sel = np.take_along_axis(p, idx.astype(np.int64), axis=-1)
    sel = sel / sel.sum(axis=-1, keepdims=True)
    return sel * pes[idx]


def route(h, Wr, router_scale, pes, k, bias=None):
    """Router of the block: (logits [T, E], idx [T, k] int32, weights [T, k])."""
    z = router_logits(h, Wr, router_scale, bias)
    idx = select_topk(z, k)
    w = routing_weights(z, idx, pes)
    return z, idx, w


def decoded(t, bf16_weights: bool = False) -> np.ndarray:
    """A weight as float64; with bf16_weights, a group-wise affine weight is
    rounded to bf16 after its exact decode (bf16 weights are unchanged, and so
    are NVFP4 weights: a code times its e4m3 block scale is a bf16 number,
    the matrix scale is applied to the fp32 product)."""
    w = to_f64(t)
    affine = isinstance(t, dict) and t.get("fmt") != "nvfp4"
    return round_bf16(w) if (bf16_weights and affine) else w


def geglu_mlp(x: np.ndarray, W_gate: np.ndarray, W_up: np.ndarray,
              W_down: np.ndarray) -> np.ndarray:
    """down(gelu_tanh(x W_gate^T) * (x W_up^T)); weights stored [out, in]."""
    return (gelu_tanh(x @ W_gate.T) * (x @ W_up.T)) @ W_down.T


def experts_forward(xe: np.ndarray, idx: np.ndarray, w: np.ndarray,
                    gate_up, down, inter: int, bf16_activations: bool = False,
                    bf16_weights: bool = False) -> np.ndarray:
    """y[t] = sum_k w[t, k] * MLP_{idx[t, k]}(xe[t]); one expert at a time,
    over the tokens routed to it.  gate_up[e] rows 0..inter-1 are the gate,
    rows inter..2*inter-1 the up projection.

    bf16_activations: round the expert input and the GEGLU activation to bf16
    before they are multiplied, as the activation planes are bf16 in the
    precision policy ("diffgemma — architecture & implemented contract",
    Part III, precision policy); everything else stays float64.
    bf16_weights: decode affine weights exactly, then round them to bf16."""
    T, H = xe.shape
    E = (gate_up["q"] if isinstance(gate_up, dict) else gate_up).shape[0]
    if bf16_activations:
        xe = round_bf16(xe)
    y = np.zeros((T, H), dtype=np.float64)
    for e in range(E):
        tok, slot = np.nonzero(idx == e)
        if tok.size == 0:
            continue
        gu = decoded(_slice(gate_up, e), bf16_weights)
        dn = decoded(_slice(down, e), bf16_weights)
        x = xe[tok]
        act = gelu_tanh(x @ gu[:inter].T) * (x @ gu[inter:].T)
        if bf16_activations:
            act = round_bf16(act)
        y[tok] += w[tok, slot][:, None] * (act @ dn.T)
    return y


def dense_forward(xd, dense_gate, dense_up, dense_down,
                  bf16_activations: bool = False, bf16_weights: bool = False) -> np.ndarray:
    """The always-on dense GEGLU MLP (bf16_activations, bf16_weights as in
    experts_forward)."""
    Wg, Wu, Wd = (decoded(t, bf16_weights) for t in (dense_gate, dense_up, dense_down))
    if not bf16_activations:
        return geglu_mlp(xd, Wg, Wu, Wd)
    x = round_bf16(xd)
    act = round_bf16(gelu_tanh(x @ Wg.T) * (x @ Wu.T))
    return act @ Wd.T


def combine(h, y_dense, y_moe, w_post1, w_post2, w_post, layer_scalar):
    """out = (h + rms(rms(y_dense) w_post1 + rms(y_moe) w_post2) w_post) * s."""
    h1 = rms_norm(y_dense, w_post1)
    h2 = rms_norm(y_moe, w_post2)
    o = rms_norm(h1 + h2, w_post)
    return (h + o) * layer_scalar


def permutation(idx: np.ndarray, n_experts: int):
    """Canonical grouping of the T*k assignments by expert.

    Assignment (t, j) has id t*k + j.  Returns ``offsets`` [E+1] (exclusive
    prefix sum of the per-expert counts) and ``perm`` [T*k]: the assignment
    ids sorted by (expert ascending, token ascending)."""
    T, k = idx.shape
    expert = idx.reshape(-1).astype(np.int64)
    token = np.repeat(np.arange(T, dtype=np.int64), k)
    perm = np.lexsort((token, expert)).astype(np.int32)   # by expert, then token
    counts = np.bincount(expert, minlength=n_experts)
    offsets = np.zeros(n_experts + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    return offsets, perm


def moe_block_forward(h_bits, p: dict, top_k: int, inter: int,
                      layer_scalar=None, with_perm: bool = True,
                      bf16_weights: bool = False) -> dict:
    """The whole block on one [T, H] activation, with its intermediates.

    ``h_bits`` is bf16 bits (uint16) or float64; ``p`` a parameter dict as
    produced by :func:`moe_inputs.make_layer_inputs`.  bf16_weights: the
    expert and dense affine weights rounded to bf16 after their exact decode
    (the block on bf16-decoded weights; the router is left exact)."""
    h = bf16_to_f64(h_bits) if np.asarray(h_bits).dtype == np.uint16 else np.asarray(h_bits, np.float64)
    s = p["layer_scalar"] if layer_scalar is None else layer_scalar
    vec = {n: to_f64(p[n]) for n in ("router_scale", "per_expert_scale",
                                          "w_pre_ff", "w_pre_ff2", "w_post_ff1",
                                          "w_post_ff2", "w_post_ff")}
    Wr = to_f64(p["router"])
    z, idx, w = route(h, Wr, vec["router_scale"], vec["per_expert_scale"],
                      top_k, p.get("router_bias"))
    xd = rms_norm(h, vec["w_pre_ff"])
    xe = rms_norm(h, vec["w_pre_ff2"])
    y_moe = experts_forward(xe, idx, w, p["gate_up"], p["down"], inter,
                            bf16_weights=bf16_weights)
    y_dense = dense_forward(xd, p["dense_gate"], p["dense_up"], p["dense_down"],
                            bf16_weights=bf16_weights)
    out = combine(h, y_dense, y_moe, vec["w_post_ff1"], vec["w_post_ff2"],
                  vec["w_post_ff"], s)
    res = {"z": z, "idx": idx, "w": w, "xd": xd, "xe": xe, "y_moe": y_moe,
           "y_dense": y_dense, "out": out}
    if with_perm:
        E = Wr.shape[0]
        res["offsets"], res["perm"] = permutation(idx, E)
    return res


def sc_mlp_forward(embeds_bits, signal_bits, p: dict, bf16_weights: bool = False) -> np.ndarray:
    """The self-conditioning MLP on a canvas: the soft signal (previous-step
    probabilities times the embedding table) through a pre-normed GEGLU MLP of
    the dense FFN's shape, added to the token embeddings, then RMS-normalised
    without a weight ("DiffusionGemma port — plan & parity strategy",
    Reference dossier §3 Self-conditioning; "diffgemma — architecture &
    implemented contract", Part II §2.1 SC injection; "DiffusionGemma
    Explained", MLP with conditioning_mlp).  p: gate, up, down weights and the
    pre_norm vector; inputs bf16 bits [T, H]."""
    x = bf16_to_f64(embeds_bits)
    sig = bf16_to_f64(signal_bits)
    normed = rms_norm(sig, to_f64(p["pre_norm"]))
    sc = geglu_mlp(normed, decoded(p["gate"], bf16_weights), decoded(p["up"], bf16_weights),
                   decoded(p["down"], bf16_weights))
    return rms_norm(x + sc)


def attn_residual(x_bits, attn_bits, w_post_attn) -> np.ndarray:
    """The block's input from the attention half of the decoder layer:
    ``h = residual + post_attention_layernorm(attn)`` ("DiffusionGemma port —
    plan & parity strategy", Reference dossier §2 DecoderLayer), with the
    normed attention output and the sum each a bf16 activation plane
    ("diffgemma — architecture & implemented contract", Part III precision
    policy), so each is rounded once.  Inputs bf16 bits [T, H] and the norm
    weight; returns float64 values that are bf16 numbers."""
    n = round_bf16(rms_norm(bf16_to_f64(attn_bits), to_f64(w_post_attn)))
    return round_bf16(bf16_to_f64(x_bits) + n)


def next_input_norm(out_bits, w_in_next) -> np.ndarray:
    """The next decoder layer's input_layernorm of this layer's bf16 output
    plane ("DiffusionGemma port ...", Reference dossier §2 DecoderLayer: the
    layer opens with ``h = input_layernorm(x)``), rounded to bf16."""
    return round_bf16(rms_norm(bf16_to_f64(out_bits), to_f64(w_in_next)))
