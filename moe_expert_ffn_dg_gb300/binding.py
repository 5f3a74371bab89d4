"""ctypes binding of the C ABI in ``include/dg_moe.h``.

The functions below carry the C names and only marshal arguments; every step
of the block runs in the CUDA library ``lib/libdgmoe.so``.  There is no other
code path: if the library is missing, :func:`load_library` raises.
"""

from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int, c_size_t, c_uint, c_void_p

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libdgmoe.so")

DG_OK = 0
DG_ERR_INVALID_ARG = 1
DG_ERR_ALIGNMENT = 2
DG_ERR_UNSUPPORTED = 3
DG_ERR_CUDA = 4
DG_ERR_TIMEOUT = 5
DG_ERR_DEVICE_CHECK = 6
DG_ERR_WORKSPACE = 7

DG_FMT_BF16 = 0
DG_FMT_AFFINE_U4_G64 = 1
DG_FMT_AFFINE_U8_G64 = 2
DG_FMT_NVFP4_G16 = 3

EXPORTED = (
    "dg_moe_workspace_size", "dg_moe_create", "dg_moe_forward", "dg_moe_forward_host",
    "dg_moe_destroy", "dg_moe_last_device_status", "dg_moe_kernel_names",
    "dg_moe_set_profile_events", "dg_moe_status_string", "dg_moe_last_error",
    "dg_moe_route_noalloc", "dg_moe_forward_neighbours", "dg_moe_arm_wait_timeout_test",
    "dg_sc_mlp_workspace_size", "dg_sc_mlp_create", "dg_sc_mlp_forward",
    "dg_sc_mlp_last_device_status", "dg_sc_mlp_destroy", "dg_sc_mlp_kernel_names",
    "dg_sc_mlp_set_profile_events",
)


class dg_moe_config_t(ctypes.Structure):
    _fields_ = [("hidden", c_int), ("n_experts", c_int), ("top_k", c_int),
                ("expert_inter", c_int), ("dense_inter", c_int), ("max_tokens", c_int),
                ("expert_fmt", c_int), ("dense_fmt", c_int), ("router_fmt", c_int),
                ("rms_eps", c_float), ("flags", c_uint)]


class dg_qtensor_t(ctypes.Structure):
    _fields_ = [("q", c_void_p), ("scales", c_void_p), ("biases", c_void_p)]


class dg_moe_weights_t(ctypes.Structure):
    _fields_ = [("router", dg_qtensor_t), ("gate_up", dg_qtensor_t), ("down", dg_qtensor_t),
                ("dense_gate", dg_qtensor_t), ("dense_up", dg_qtensor_t),
                ("dense_down", dg_qtensor_t),
                ("router_scale", c_void_p), ("per_expert_scale", c_void_p),
                ("w_pre_ff", c_void_p), ("w_pre_ff2", c_void_p), ("w_post_ff1", c_void_p),
                ("w_post_ff2", c_void_p), ("w_post_ff", c_void_p), ("router_bias", c_void_p)]


class dg_moe_neighbours_t(ctypes.Structure):
    _fields_ = [("attn_out", c_void_p), ("w_post_attn", c_void_p), ("w_next_in", c_void_p),
                ("next_in", c_void_p), ("h_mid", c_void_p)]


class dg_moe_debug_t(ctypes.Structure):
    _fields_ = [("idx", c_void_p), ("w", c_void_p), ("logits", c_void_p),
                ("offsets", c_void_p), ("perm", c_void_p), ("xd", c_void_p),
                ("xe_perm", c_void_p), ("y_moe", c_void_p), ("y_dense", c_void_p),
                ("n_refined", c_void_p)]


class dg_sc_mlp_config_t(ctypes.Structure):
    _fields_ = [("hidden", c_int), ("inter", c_int), ("max_tokens", c_int), ("fmt", c_int),
                ("rms_eps", c_float), ("flags", c_uint)]


class dg_sc_mlp_weights_t(ctypes.Structure):
    _fields_ = [("gate", dg_qtensor_t), ("up", dg_qtensor_t), ("down", dg_qtensor_t),
                ("pre_norm", c_void_p)]


class DgError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {dg_moe_status_string(status)} (status {status})")


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} not found: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    lib.dg_moe_workspace_size.argtypes = [POINTER(dg_moe_config_t), POINTER(c_size_t)]
    lib.dg_moe_create.argtypes = [POINTER(dg_moe_config_t), POINTER(dg_moe_weights_t), c_void_p,
                                  c_size_t, POINTER(c_void_p)]
    lib.dg_moe_forward.argtypes = [c_void_p, c_void_p, c_void_p, c_int, c_float, c_void_p,
                                   POINTER(dg_moe_debug_t)]
    lib.dg_moe_forward_host.argtypes = [c_void_p, c_void_p, c_void_p, c_int, c_float, c_void_p]
    lib.dg_moe_forward_neighbours.argtypes = [c_void_p, c_void_p, POINTER(dg_moe_neighbours_t),
                                              c_void_p, c_int, c_float, c_void_p,
                                              POINTER(dg_moe_debug_t)]
    lib.dg_moe_destroy.argtypes = [c_void_p]
    lib.dg_moe_last_device_status.argtypes = [c_void_p, c_void_p, POINTER(c_uint), POINTER(c_uint)]
    lib.dg_moe_kernel_names.argtypes = [c_void_p, POINTER(c_char_p), POINTER(c_int)]
    lib.dg_moe_set_profile_events.argtypes = [c_void_p, POINTER(c_void_p), c_int]
    lib.dg_moe_arm_wait_timeout_test.argtypes = [c_void_p]
    lib.dg_moe_route_noalloc.argtypes = [POINTER(dg_moe_config_t), POINTER(dg_moe_weights_t),
                                         c_void_p, c_int, c_void_p, c_void_p, c_void_p]
    lib.dg_sc_mlp_workspace_size.argtypes = [POINTER(dg_sc_mlp_config_t), POINTER(c_size_t)]
    lib.dg_sc_mlp_create.argtypes = [POINTER(dg_sc_mlp_config_t), POINTER(dg_sc_mlp_weights_t),
                                     c_void_p, c_size_t, POINTER(c_void_p)]
    lib.dg_sc_mlp_forward.argtypes = [c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_void_p]
    lib.dg_sc_mlp_last_device_status.argtypes = [c_void_p, c_void_p]
    lib.dg_sc_mlp_destroy.argtypes = [c_void_p]
    lib.dg_sc_mlp_kernel_names.argtypes = [c_void_p, POINTER(c_char_p), POINTER(c_int)]
    lib.dg_sc_mlp_set_profile_events.argtypes = [c_void_p, POINTER(c_void_p), c_int]
    lib.dg_moe_status_string.argtypes = [c_int]
    lib.dg_moe_status_string.restype = c_char_p
    lib.dg_moe_last_error.argtypes = [c_void_p]
    lib.dg_moe_last_error.restype = c_char_p
    for name in EXPORTED:
        if name not in ("dg_moe_status_string", "dg_moe_last_error"):
            getattr(lib, name).restype = c_int
    _lib = lib
    return lib


def dg_moe_status_string(status: int) -> str:
    return load_library().dg_moe_status_string(status).decode()


def _check(status: int, what: str, handle: int = None) -> None:
    if status != DG_OK:
        detail = ""
        if handle and status == DG_ERR_CUDA:
            detail = " [" + dg_moe_last_error(handle) + "]"
        raise DgError(status, what + detail)


def dg_moe_last_error(handle: int) -> str:
    return load_library().dg_moe_last_error(c_void_p(handle)).decode()


def dg_moe_workspace_size(cfg: dg_moe_config_t) -> int:
    n = c_size_t(0)
    _check(load_library().dg_moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)),
           "dg_moe_workspace_size")
    return n.value


def dg_moe_create(cfg: dg_moe_config_t, weights: dg_moe_weights_t, workspace: int,
                  workspace_bytes: int) -> int:
    h = c_void_p(0)
    _check(load_library().dg_moe_create(ctypes.byref(cfg), ctypes.byref(weights),
                                        c_void_p(workspace), workspace_bytes, ctypes.byref(h)),
           "dg_moe_create")
    return h.value


def dg_moe_forward(handle: int, h_in: int, h_out: int, n_tokens: int, layer_scalar: float,
                   stream: int, dbg: dg_moe_debug_t | None = None) -> None:
    _check(load_library().dg_moe_forward(c_void_p(handle), c_void_p(h_in), c_void_p(h_out),
                                         n_tokens, layer_scalar, c_void_p(stream),
                                         ctypes.byref(dbg) if dbg is not None else None),
           "dg_moe_forward", handle)


def dg_moe_forward_neighbours(handle: int, x: int, nb: dg_moe_neighbours_t, out: int,
                              n_tokens: int, layer_scalar: float, stream: int,
                              dbg: dg_moe_debug_t | None = None) -> None:
    _check(load_library().dg_moe_forward_neighbours(
        c_void_p(handle), c_void_p(x), ctypes.byref(nb) if nb is not None else None,
        c_void_p(out), n_tokens, layer_scalar, c_void_p(stream),
        ctypes.byref(dbg) if dbg is not None else None), "dg_moe_forward_neighbours", handle)


def dg_moe_forward_host(handle: int, h_in_host: int, h_out_host: int, n_tokens: int,
                        layer_scalar: float, stream: int) -> None:
    _check(load_library().dg_moe_forward_host(c_void_p(handle), c_void_p(h_in_host),
                                              c_void_p(h_out_host), n_tokens, layer_scalar,
                                              c_void_p(stream)),
           "dg_moe_forward_host", handle)


def dg_moe_destroy(handle: int) -> None:
    _check(load_library().dg_moe_destroy(c_void_p(handle)), "dg_moe_destroy")


def dg_moe_last_device_status(handle: int, stream: int):
    """(status, where, info) of the device status word; clears it."""
    where, info = c_uint(0), c_uint(0)
    s = load_library().dg_moe_last_device_status(c_void_p(handle), c_void_p(stream),
                                                 ctypes.byref(where), ctypes.byref(info))
    return s, where.value, info.value


def _kernel_names(fn, handle: int) -> list:
    n = c_int(0)
    _check(fn(c_void_p(handle), None, ctypes.byref(n)), fn.__name__)
    arr = (c_char_p * n.value)()
    _check(fn(c_void_p(handle), arr, ctypes.byref(n)), fn.__name__)
    return [a.decode() for a in arr]


def _set_profile_events(fn, handle: int, events) -> None:
    if events is None:
        _check(fn(c_void_p(handle), None, 0), fn.__name__)
        _EVENT_ARRAYS.pop(handle, None)
        return
    arr = (c_void_p * len(events))(*events)
    _check(fn(c_void_p(handle), arr, len(events)), fn.__name__)
    # keep the array alive as long as the handle may use it
    _EVENT_ARRAYS[handle] = arr


def dg_moe_kernel_names(handle: int) -> list:
    return _kernel_names(load_library().dg_moe_kernel_names, handle)


def dg_moe_set_profile_events(handle: int, events) -> None:
    """events: list of cudaEvent_t handles (ints), or None to switch off."""
    _set_profile_events(load_library().dg_moe_set_profile_events, handle, events)


def dg_moe_arm_wait_timeout_test(handle: int) -> None:
    """Arm the bounded-wait test for the handle's next forward (see
    include/dg_moe.h): one device wait runs out after 10 ms and reports
    DG_ERR_TIMEOUT through dg_moe_last_device_status."""
    _check(load_library().dg_moe_arm_wait_timeout_test(c_void_p(handle)),
           "dg_moe_arm_wait_timeout_test")


def dg_sc_mlp_kernel_names(handle: int) -> list:
    return _kernel_names(load_library().dg_sc_mlp_kernel_names, handle)


def dg_sc_mlp_set_profile_events(handle: int, events) -> None:
    _set_profile_events(load_library().dg_sc_mlp_set_profile_events, handle, events)


_EVENT_ARRAYS: dict = {}


def dg_moe_route_noalloc(cfg: dg_moe_config_t, weights: dg_moe_weights_t, h_in: int,
                         n_tokens: int, idx_out: int, w_out: int, stream: int) -> None:
    """Routing only, with the library's fixed device scratch (no allocation);
    see include/dg_moe.h."""
    _check(load_library().dg_moe_route_noalloc(ctypes.byref(cfg), ctypes.byref(weights),
                                               c_void_p(h_in), n_tokens, c_void_p(idx_out),
                                               c_void_p(w_out), c_void_p(stream)),
           "dg_moe_route_noalloc")


def dg_sc_mlp_workspace_size(cfg: dg_sc_mlp_config_t) -> int:
    n = c_size_t(0)
    _check(load_library().dg_sc_mlp_workspace_size(ctypes.byref(cfg), ctypes.byref(n)),
           "dg_sc_mlp_workspace_size")
    return n.value


def dg_sc_mlp_create(cfg: dg_sc_mlp_config_t, weights: dg_sc_mlp_weights_t, workspace: int,
                     workspace_bytes: int) -> int:
    h = c_void_p(0)
    _check(load_library().dg_sc_mlp_create(ctypes.byref(cfg), ctypes.byref(weights),
                                           c_void_p(workspace), workspace_bytes, ctypes.byref(h)),
           "dg_sc_mlp_create")
    return h.value


def dg_sc_mlp_forward(handle: int, embeds: int, signal: int, out: int, n_tokens: int,
                      stream: int) -> None:
    _check(load_library().dg_sc_mlp_forward(c_void_p(handle), c_void_p(embeds), c_void_p(signal),
                                            c_void_p(out), n_tokens, c_void_p(stream)),
           "dg_sc_mlp_forward")


def dg_sc_mlp_last_device_status(handle: int, stream: int) -> int:
    return load_library().dg_sc_mlp_last_device_status(c_void_p(handle), c_void_p(stream))


def dg_sc_mlp_destroy(handle: int) -> None:
    _check(load_library().dg_sc_mlp_destroy(c_void_p(handle)), "dg_sc_mlp_destroy")
