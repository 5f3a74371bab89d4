"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function the header declares, and rejects bad arguments before any
CUDA call."""

import ctypes
import os
import re

import pytest

import moe_expert_ffn_dg_gb300 as pkg
from moe_expert_ffn_dg_gb300 import binding as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "dg_moe.h")


@pytest.fixture(scope="module")
def lib():
    pkg.build()
    return B.load_library()


def _cfg(**kw):
    c = dict(hidden=2816, n_experts=128, top_k=8, expert_inter=704, dense_inter=2112,
             max_tokens=256, expert_fmt=0, dense_fmt=0, router_fmt=0, rms_eps=1e-6, flags=0)
    c.update(kw)
    return B.dg_moe_config_t(**c)


def test_library_exports_every_declared_function(lib):
    decl = set(re.findall(r"\b(dg_(?:moe|sc_mlp)_\w+)\s*\(", open(HEADER).read()))
    assert decl == set(B.EXPORTED)
    for name in decl:
        assert hasattr(lib, name)


def test_status_strings(lib):
    for s in range(8):
        assert B.dg_moe_status_string(s) not in ("", "unknown status")
    assert B.dg_moe_status_string(99) == "unknown status"


def test_workspace_size_validation(lib):
    n = ctypes.c_size_t(0)
    assert lib.dg_moe_workspace_size(None, ctypes.byref(n)) == B.DG_ERR_INVALID_ARG
    assert lib.dg_moe_workspace_size(ctypes.byref(_cfg()), None) == B.DG_ERR_INVALID_ARG
    for bad, code in [(dict(top_k=129), B.DG_ERR_INVALID_ARG),
                      (dict(top_k=0), B.DG_ERR_INVALID_ARG),
                      (dict(max_tokens=0), B.DG_ERR_INVALID_ARG),
                      (dict(flags=1), B.DG_ERR_INVALID_ARG),
                      (dict(hidden=2880), B.DG_ERR_UNSUPPORTED),
                      (dict(expert_inter=700), B.DG_ERR_UNSUPPORTED),
                      (dict(n_experts=512, top_k=8), B.DG_ERR_UNSUPPORTED),
                      (dict(top_k=17, n_experts=32), B.DG_ERR_UNSUPPORTED),
                      (dict(router_fmt=1), B.DG_ERR_UNSUPPORTED)]:
        assert lib.dg_moe_workspace_size(ctypes.byref(_cfg(**bad)), ctypes.byref(n)) == code, bad
    size = B.dg_moe_workspace_size(_cfg())
    # dominated by the grouped expert rows (T*K*H bf16) and two f32 [T, H] planes
    assert 256 * 8 * 2816 * 2 < size < 64 * 2 ** 20
    big = B.dg_moe_workspace_size(_cfg(max_tokens=16384))
    assert big > 60 * size


def _weights(ptr=0x10000):
    q = lambda: B.dg_qtensor_t(ptr, None, None)
    return B.dg_moe_weights_t(q(), q(), q(), q(), q(), q(), ptr, ptr, ptr, ptr, ptr, ptr, ptr, None)


def test_create_rejects_bad_arguments_before_touching_the_gpu(lib):
    h = ctypes.c_void_p(0)
    cfg = _cfg()
    ws = 1 << 20
    size = B.dg_moe_workspace_size(cfg)
    assert lib.dg_moe_create(ctypes.byref(cfg), None, ws, size, ctypes.byref(h)) == B.DG_ERR_INVALID_ARG
    w = _weights()
    w.gate_up.q = None
    assert lib.dg_moe_create(ctypes.byref(cfg), ctypes.byref(w), ws, size, ctypes.byref(h)) == B.DG_ERR_INVALID_ARG
    w = _weights()
    w.down.q = 0x10008  # not 16-byte aligned
    assert lib.dg_moe_create(ctypes.byref(cfg), ctypes.byref(w), ws, size, ctypes.byref(h)) == B.DG_ERR_ALIGNMENT
    w = _weights()
    w.w_post_ff = None
    assert lib.dg_moe_create(ctypes.byref(cfg), ctypes.byref(w), ws, size, ctypes.byref(h)) == B.DG_ERR_INVALID_ARG
    w = _weights()
    assert lib.dg_moe_create(ctypes.byref(cfg), ctypes.byref(w), None, size, ctypes.byref(h)) == B.DG_ERR_WORKSPACE
    assert lib.dg_moe_create(ctypes.byref(cfg), ctypes.byref(w), ws, size - 1, ctypes.byref(h)) == B.DG_ERR_WORKSPACE
    assert lib.dg_moe_create(ctypes.byref(cfg), ctypes.byref(w), ws + 512, size, ctypes.byref(h)) == B.DG_ERR_WORKSPACE
    assert h.value is None
    bad = _cfg(top_k=200)
    assert lib.dg_moe_create(ctypes.byref(bad), ctypes.byref(w), ws, size, ctypes.byref(h)) == B.DG_ERR_INVALID_ARG


def test_null_handle_is_rejected_and_destroy_accepts_null(lib):
    assert lib.dg_moe_forward(None, 16, 16, 4, 1.0, None, None) == B.DG_ERR_INVALID_ARG
    assert lib.dg_moe_forward_host(None, 16, 16, 4, 1.0, None) == B.DG_ERR_INVALID_ARG
    nb = B.dg_moe_neighbours_t(16, 16, None, None, None)
    assert lib.dg_moe_forward_neighbours(None, 16, ctypes.byref(nb), 16, 4, 1.0, None,
                                         None) == B.DG_ERR_INVALID_ARG
    assert lib.dg_moe_destroy(None) == B.DG_OK
    n = ctypes.c_int(0)
    assert lib.dg_moe_kernel_names(None, None, ctypes.byref(n)) == B.DG_ERR_INVALID_ARG
    assert lib.dg_moe_set_profile_events(None, None, 0) == B.DG_ERR_INVALID_ARG


def _sc_cfg(**kw):
    c = dict(hidden=2816, inter=2112, max_tokens=256, fmt=0, rms_eps=1e-6, flags=0)
    c.update(kw)
    return B.dg_sc_mlp_config_t(**c)


def test_sc_mlp_workspace_and_create_validation(lib):
    assert B.dg_sc_mlp_workspace_size(_sc_cfg()) > 256 * 2816 * 4
    # bf16, 4-bit and 8-bit (q8) group-64 affine weights; NVFP4 is not an SC format
    for fmt in (B.DG_FMT_AFFINE_U4_G64, B.DG_FMT_AFFINE_U8_G64):
        assert B.dg_sc_mlp_workspace_size(_sc_cfg(fmt=fmt)) > 256 * 2816 * 4
    for bad in (dict(hidden=100), dict(inter=100), dict(fmt=B.DG_FMT_NVFP4_G16), dict(flags=1),
                dict(fmt=B.DG_FMT_AFFINE_U8_G64, hidden=3072)):
        with pytest.raises(B.DgError):
            B.dg_sc_mlp_workspace_size(_sc_cfg(**bad))
    w = B.dg_sc_mlp_weights_t()
    h = ctypes.c_void_p(0)
    # null weights and a null workspace are refused before any CUDA call
    assert lib.dg_sc_mlp_create(ctypes.byref(_sc_cfg()), ctypes.byref(w), None, 0,
                                ctypes.byref(h)) == B.DG_ERR_INVALID_ARG
    assert lib.dg_sc_mlp_forward(None, None, None, None, 1, None) == B.DG_ERR_INVALID_ARG
    assert lib.dg_sc_mlp_destroy(None) == B.DG_OK


def test_nvfp4_format_pairs(lib):
    n = ctypes.c_size_t(0)
    ok = _cfg(expert_fmt=B.DG_FMT_NVFP4_G16, dense_fmt=B.DG_FMT_NVFP4_G16, router_fmt=2)
    assert lib.dg_moe_workspace_size(ctypes.byref(ok), ctypes.byref(n)) == B.DG_OK
    mixed = _cfg(expert_fmt=B.DG_FMT_NVFP4_G16, dense_fmt=B.DG_FMT_AFFINE_U4_G64)
    assert lib.dg_moe_workspace_size(ctypes.byref(mixed), ctypes.byref(n)) == B.DG_ERR_UNSUPPORTED


def _route_noalloc(lib, cfg, w, h=0x10000, T=4, idx=0x20000, wo=0x30000):
    return lib.dg_moe_route_noalloc(None if cfg is None else ctypes.byref(cfg),
                                    None if w is None else ctypes.byref(w), h, T, idx, wo, None)


def test_route_noalloc_rejects_bad_arguments_before_any_cuda_call(lib):
    """Every rejection below returns before the scratch array is looked up or
    any kernel launched, so it runs without a GPU."""
    ok_cfg, ok_w = _cfg(), _weights()
    assert _route_noalloc(lib, None, ok_w) == B.DG_ERR_INVALID_ARG
    assert _route_noalloc(lib, ok_cfg, None) == B.DG_ERR_INVALID_ARG
    for bad, code in [(dict(top_k=129), B.DG_ERR_INVALID_ARG),        # K > E
                      (dict(top_k=0), B.DG_ERR_INVALID_ARG),
                      (dict(hidden=0), B.DG_ERR_INVALID_ARG),
                      (dict(rms_eps=-1.0), B.DG_ERR_INVALID_ARG),
                      (dict(flags=2), B.DG_ERR_INVALID_ARG),
                      (dict(hidden=2880), B.DG_ERR_UNSUPPORTED),      # H % 128
                      (dict(n_experts=512), B.DG_ERR_UNSUPPORTED),
                      (dict(router_fmt=B.DG_FMT_AFFINE_U4_G64), B.DG_ERR_UNSUPPORTED)]:
        assert _route_noalloc(lib, _cfg(**bad), ok_w) == code, bad
    # weights the routing kernels read
    w = _weights()
    w.router.q = None
    assert _route_noalloc(lib, ok_cfg, w) == B.DG_ERR_INVALID_ARG
    w = _weights()
    w.router.q = 0x10008
    assert _route_noalloc(lib, ok_cfg, w) == B.DG_ERR_ALIGNMENT
    w = _weights()
    w.router_scale = 0x10004
    assert _route_noalloc(lib, ok_cfg, w) == B.DG_ERR_ALIGNMENT
    w = _weights()
    w.w_pre_ff = None
    assert _route_noalloc(lib, ok_cfg, w) == B.DG_ERR_INVALID_ARG
    w = _weights()
    w.per_expert_scale = 0x10001
    assert _route_noalloc(lib, ok_cfg, w) == B.DG_ERR_ALIGNMENT
    w = _weights()
    w.router_bias = 0x10002          # f32 loads need 4-byte alignment
    assert _route_noalloc(lib, ok_cfg, w) == B.DG_ERR_ALIGNMENT
    # the 8-bit router needs its scales and biases (2-byte aligned)
    u8 = _cfg(router_fmt=B.DG_FMT_AFFINE_U8_G64)
    assert _route_noalloc(lib, u8, _weights()) == B.DG_ERR_INVALID_ARG
    w = _weights()
    w.router.scales, w.router.biases = 0x10001, 0x10000
    assert _route_noalloc(lib, u8, w) == B.DG_ERR_ALIGNMENT
    # token count and the per-call buffers
    assert _route_noalloc(lib, ok_cfg, ok_w, T=-1) == B.DG_ERR_INVALID_ARG
    assert _route_noalloc(lib, ok_cfg, ok_w, T=0) == B.DG_OK    # nothing to do
    assert _route_noalloc(lib, ok_cfg, ok_w, h=None) == B.DG_ERR_INVALID_ARG
    assert _route_noalloc(lib, ok_cfg, ok_w, idx=None) == B.DG_ERR_INVALID_ARG
    assert _route_noalloc(lib, ok_cfg, ok_w, h=0x10008) == B.DG_ERR_ALIGNMENT
    assert _route_noalloc(lib, ok_cfg, ok_w, idx=0x20002) == B.DG_ERR_ALIGNMENT
    assert _route_noalloc(lib, ok_cfg, ok_w, wo=0x30001) == B.DG_ERR_ALIGNMENT
    # beyond the fixed scratch: refused on the host
    assert _route_noalloc(lib, ok_cfg, ok_w, T=4096) == B.DG_ERR_UNSUPPORTED
