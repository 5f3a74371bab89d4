"""PyTorch-side holder of one MoE FFN layer on the GPU.

PyTorch only allocates device memory (weights, workspace, outputs) and
supplies the CUDA stream; every step of the forward runs in the CUDA library
through the C ABI (:mod:`.binding`).
"""

from __future__ import annotations

import numpy as np
import torch

from . import binding as B

WEIGHTS = ("router", "gate_up", "down", "dense_gate", "dense_up", "dense_down")
VECTORS = ("router_scale", "per_expert_scale", "w_pre_ff", "w_pre_ff2", "w_post_ff1",
           "w_post_ff2", "w_post_ff")


def _to_device(a: np.ndarray, device) -> torch.Tensor:
    """numpy array -> device tensor with the same bytes (bf16 bits stay bits)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    if a.dtype == np.uint32:
        return torch.from_numpy(a.view(np.int32)).to(device)
    if a.dtype in (np.uint8, np.float32, np.int32):
        return torch.from_numpy(a).to(device)
    raise TypeError(f"unsupported dtype {a.dtype}")


def _quant_to_device(v: dict, device) -> dict:
    if v.get("fmt") == "nvfp4":
        return {"fmt": "nvfp4", "q": _to_device(v["q"], device),
                "scales": _to_device(v["scales"], device),
                "globals": _to_device(np.asarray(v["globals"], np.float32), device)}
    return {"bits": v["bits"], "group": v["group"], "q": _to_device(v["q"], device),
            "scales": _to_device(v["scales"], device), "biases": _to_device(v["biases"], device)}


def params_to_device(p: dict, device) -> dict:
    """Copy a layer's parameters (bf16 bit patterns as uint16 arrays,
    group-wise affine dicts {bits, group, q, scales, biases} or NVFP4 dicts
    {fmt, q, scales, globals}) to the device."""
    out = {}
    for k in WEIGHTS:
        v = p[k]
        if isinstance(v, dict) and v.get("fmt") == "nvfp4":
            out[k] = _quant_to_device(v, device)
        elif isinstance(v, dict):
            out[k] = {"bits": v["bits"], "group": v["group"],
                      "q": _to_device(v["q"], device),
                      "scales": _to_device(v["scales"], device),
                      "biases": _to_device(v["biases"], device)}
        else:
            out[k] = _to_device(v, device)
    for k in VECTORS:
        out[k] = _to_device(p[k], device)
    rb = p.get("router_bias")
    out["router_bias"] = None if rb is None else _to_device(np.asarray(rb, np.float32), device)
    return out


def _fmt(w) -> int:
    if not isinstance(w, dict):
        return B.DG_FMT_BF16
    if w.get("fmt") == "nvfp4":
        return B.DG_FMT_NVFP4_G16
    return {4: B.DG_FMT_AFFINE_U4_G64, 8: B.DG_FMT_AFFINE_U8_G64}[w["bits"]]


def _qt(w) -> B.dg_qtensor_t:
    if isinstance(w, dict) and w.get("fmt") == "nvfp4":
        return B.dg_qtensor_t(w["q"].data_ptr(), w["scales"].data_ptr(), w["globals"].data_ptr())
    if isinstance(w, dict):
        return B.dg_qtensor_t(w["q"].data_ptr(), w["scales"].data_ptr(), w["biases"].data_ptr())
    return B.dg_qtensor_t(w.data_ptr(), None, None)


class MoEBlock:
    """One layer: device weights (borrowed by the C handle), a workspace and
    the handle.  ``forward`` runs the block on a bf16 [T, H] device tensor."""

    def __init__(self, weights: dict, *, hidden: int, n_experts: int, top_k: int,
                 expert_inter: int, dense_inter: int, max_tokens: int, rms_eps: float = 1e-6,
                 workspace: torch.Tensor = None):
        """workspace: optional uint8 device tensor to use instead of a private
        one (at least workspace_bytes(...) + 1024 bytes).  Layers that run
        one after another on one stream may share a workspace; the handle
        keeps only its device status word there between forwards."""
        self.weights = weights  # keeps the device tensors alive
        self.hidden, self.n_experts, self.top_k = hidden, n_experts, top_k
        self.expert_inter, self.dense_inter, self.max_tokens = expert_inter, dense_inter, max_tokens
        self.cfg = B.dg_moe_config_t(hidden, n_experts, top_k, expert_inter, dense_inter,
                                     max_tokens, _fmt(weights["gate_up"]),
                                     _fmt(weights["dense_gate"]), _fmt(weights["router"]),
                                     rms_eps, 0)
        self.device = weights["router_scale"].device
        ws_bytes = B.dg_moe_workspace_size(self.cfg)
        if workspace is None:
            workspace = torch.empty(ws_bytes + 1024, dtype=torch.uint8, device=self.device)
        elif workspace.numel() < ws_bytes + 1024 or workspace.device != self.device:
            raise ValueError("shared workspace too small or on another device")
        self.workspace = workspace
        base = self.workspace.data_ptr()
        self._ws_ptr = (base + 1023) // 1024 * 1024
        self._ws_bytes = ws_bytes
        w = weights
        self.cw = B.dg_moe_weights_t(
            _qt(w["router"]), _qt(w["gate_up"]), _qt(w["down"]), _qt(w["dense_gate"]),
            _qt(w["dense_up"]), _qt(w["dense_down"]),
            w["router_scale"].data_ptr(), w["per_expert_scale"].data_ptr(),
            w["w_pre_ff"].data_ptr(), w["w_pre_ff2"].data_ptr(), w["w_post_ff1"].data_ptr(),
            w["w_post_ff2"].data_ptr(), w["w_post_ff"].data_ptr(),
            w["router_bias"].data_ptr() if w.get("router_bias") is not None else None)
        self.handle = B.dg_moe_create(self.cfg, self.cw, self._ws_ptr, ws_bytes)

    @classmethod
    def from_params(cls, p: dict, *, hidden, n_experts, top_k, expert_inter, dense_inter,
                    max_tokens, device="cuda", workspace=None):
        return cls(params_to_device(p, device), hidden=hidden, n_experts=n_experts, top_k=top_k,
                   expert_inter=expert_inter, dense_inter=dense_inter, max_tokens=max_tokens,
                   workspace=workspace)

    @staticmethod
    def workspace_bytes(*, hidden, n_experts, top_k, expert_inter, dense_inter, max_tokens,
                        expert_fmt=B.DG_FMT_BF16, dense_fmt=B.DG_FMT_BF16,
                        router_fmt=B.DG_FMT_BF16, rms_eps=1e-6) -> int:
        """Bytes to allocate for a workspace shared by layers of this shape
        (the C library's requirement plus 1024 bytes of alignment slack)."""
        cfg = B.dg_moe_config_t(hidden, n_experts, top_k, expert_inter, dense_inter, max_tokens,
                                expert_fmt, dense_fmt, router_fmt, rms_eps, 0)
        return B.dg_moe_workspace_size(cfg) + 1024

    def _stream(self, stream=None) -> int:
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        return s.cuda_stream

    def forward(self, h: torch.Tensor, layer_scalar: float = 1.0, out: torch.Tensor = None,
                debug: bool = False, stream=None):
        """h: bf16 [T, H] on the device.  Returns out (bf16 [T, H]) and, with
        debug=True, a dict of the routing and intermediate tensors."""
        assert h.dtype == torch.bfloat16 and h.is_contiguous() and h.shape[1] == self.hidden
        T = h.shape[0]
        if out is None:
            out = torch.empty_like(h)
        dbg = None
        tensors = None
        if debug:
            dev, K, H, E = self.device, self.top_k, self.hidden, self.n_experts
            tensors = {
                "idx": torch.empty(T, K, dtype=torch.int32, device=dev),
                "w": torch.empty(T, K, dtype=torch.float32, device=dev),
                "logits": torch.empty(T, E, dtype=torch.float32, device=dev),
                "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
                "perm": torch.empty(T * K, dtype=torch.int32, device=dev),
                "xd": torch.empty(T, H, dtype=torch.bfloat16, device=dev),
                "xe_perm": torch.empty(T * K, H, dtype=torch.bfloat16, device=dev),
                "y_moe": torch.empty(T, H, dtype=torch.float32, device=dev),
                "y_dense": torch.empty(T, H, dtype=torch.float32, device=dev),
                "n_refined": torch.zeros(1, dtype=torch.int32, device=dev),
            }
            dbg = B.dg_moe_debug_t(*[tensors[k].data_ptr() for k in (
                "idx", "w", "logits", "offsets", "perm", "xd", "xe_perm", "y_moe", "y_dense",
                "n_refined")])
        B.dg_moe_forward(self.handle, h.data_ptr(), out.data_ptr(), T, float(layer_scalar),
                         self._stream(stream), dbg)
        return (out, tensors) if debug else out

    def forward_neighbours(self, x: torch.Tensor, attn_out: torch.Tensor, w_post_attn: torch.Tensor,
                           w_next_in: torch.Tensor = None, layer_scalar: float = 1.0,
                           out: torch.Tensor = None, next_in: torch.Tensor = None,
                           h_mid: torch.Tensor = None, stream=None):
        """The block fused with the decoder layer's neighbours: x is the layer
        input (attention residual), attn_out the attention output before its
        post-norm; returns (out, next_in) where next_in is the next layer's
        input norm of out (None without w_next_in).  h_mid, if given,
        receives the block input x + post_attention_layernorm(attn_out)."""
        for t in (x, attn_out):
            assert t.dtype == torch.bfloat16 and t.is_contiguous() and t.shape[1] == self.hidden
        assert x.shape == attn_out.shape
        T = x.shape[0]
        if out is None:
            out = torch.empty_like(x)
        if w_next_in is not None and next_in is None:
            next_in = torch.empty_like(x)
        nb = B.dg_moe_neighbours_t(attn_out.data_ptr(), w_post_attn.data_ptr(),
                                   w_next_in.data_ptr() if w_next_in is not None else None,
                                   next_in.data_ptr() if w_next_in is not None else None,
                                   h_mid.data_ptr() if h_mid is not None else None)
        B.dg_moe_forward_neighbours(self.handle, x.data_ptr(), nb, out.data_ptr(), T,
                                    float(layer_scalar), self._stream(stream))
        return out, (next_in if w_next_in is not None else None)

    def forward_host(self, h_host: torch.Tensor, out_host: torch.Tensor, layer_scalar: float = 1.0,
                     stream=None) -> torch.Tensor:
        """End to end from host memory: copy in, forward, copy out, synchronise."""
        assert h_host.device.type == "cpu" and out_host.device.type == "cpu"
        B.dg_moe_forward_host(self.handle, h_host.data_ptr(), out_host.data_ptr(), h_host.shape[0],
                              float(layer_scalar), self._stream(stream))
        return out_host

    def device_status(self, stream=None):
        return B.dg_moe_last_device_status(self.handle, self._stream(stream))

    def close(self):
        if getattr(self, "handle", None):
            B.dg_moe_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class ScMlp:
    """The self-conditioning MLP (before layer 0 of a decode step): device
    weights (borrowed by the C handle), a workspace and the handle.
    ``forward(embeds, signal)`` returns the bf16 [T, H] result."""

    def __init__(self, weights: dict, *, hidden: int, inter: int, max_tokens: int,
                 rms_eps: float = 1e-6):
        self.weights = weights
        self.hidden, self.inter, self.max_tokens = hidden, inter, max_tokens
        self.cfg = B.dg_sc_mlp_config_t(hidden, inter, max_tokens, _fmt(weights["gate"]),
                                        rms_eps, 0)
        self.device = weights["pre_norm"].device
        ws_bytes = B.dg_sc_mlp_workspace_size(self.cfg)
        self.workspace = torch.empty(ws_bytes + 1024, dtype=torch.uint8, device=self.device)
        ptr = (self.workspace.data_ptr() + 1023) // 1024 * 1024
        self.cw = B.dg_sc_mlp_weights_t(_qt(weights["gate"]), _qt(weights["up"]),
                                        _qt(weights["down"]), weights["pre_norm"].data_ptr())
        self.handle = B.dg_sc_mlp_create(self.cfg, self.cw, ptr, ws_bytes)

    @classmethod
    def from_params(cls, p: dict, *, hidden, inter, max_tokens, device="cuda"):
        w = {}
        for k in ("gate", "up", "down"):
            v = p[k]
            if isinstance(v, dict):
                w[k] = {"bits": v["bits"], "group": v["group"],
                        "q": _to_device(v["q"], device),
                        "scales": _to_device(v["scales"], device),
                        "biases": _to_device(v["biases"], device)}
            else:
                w[k] = _to_device(v, device)
        w["pre_norm"] = _to_device(p["pre_norm"], device)
        return cls(w, hidden=hidden, inter=inter, max_tokens=max_tokens)

    def forward(self, embeds: torch.Tensor, signal: torch.Tensor, out: torch.Tensor = None,
                stream=None) -> torch.Tensor:
        for t in (embeds, signal):
            assert t.dtype == torch.bfloat16 and t.is_contiguous() and t.shape[1] == self.hidden
        assert embeds.shape == signal.shape
        if out is None:
            out = torch.empty_like(embeds)
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        B.dg_sc_mlp_forward(self.handle, embeds.data_ptr(), signal.data_ptr(), out.data_ptr(),
                            embeds.shape[0], s.cuda_stream)
        return out

    def device_status(self, stream=None) -> int:
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        return B.dg_sc_mlp_last_device_status(self.handle, s.cuda_stream)

    def close(self):
        if getattr(self, "handle", None):
            B.dg_sc_mlp_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
