"""GPU parity of the block fused with its decoder-layer neighbours: the
attention half's residual + post_attention_layernorm built inside the router
kernels, and the next layer's input_layernorm written by the combine.

The block input h the GPU builds is compared with the oracle's
(``oracle.attn_residual``) within one bf16 ulp (fp32 products before the
rounding can land on the other side of a bf16 boundary); the block output is
held to the oracle block on the GPU's own h at the block's tolerance, and the
plain (unfused) forward on that h is checked by the usual parity helper; the
next layer's input is compared with ``oracle.next_input_norm`` of the GPU's
output within one ulp."""

import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
from gpu_util import assert_close, bf16_bits, bf16_ulp_distance, make_block, run_and_check, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import moe_expert_ffn_dg_gb300 as pkg
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkg.build()
    pkg.load_library()


def _neighbours(T, H, seed):
    r = np.random.default_rng(seed)
    bits = lambda a: mi.f32_to_bf16_bits(a.astype(np.float32))
    return {"x": bits(r.standard_normal((T, H))), "attn": bits(r.standard_normal((T, H)) * 4.0),
            "w_pa": bits(r.uniform(0.5, 1.5, H)), "w_next": bits(r.uniform(0.5, 1.5, H))}


def _f64_to_bits(v):
    return (np.asarray(v, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _check(wl, p, T, seed, alias=False, full_check=True, sample=None):
    nbr = _neighbours(T, wl.hidden, seed)
    blk = make_block(wl, p, max_tokens=max(T, 1))
    x = to_dev_bf16(nbr["x"])
    a = to_dev_bf16(nbr["attn"])
    w_pa, w_next = to_dev_bf16(nbr["w_pa"]), to_dev_bf16(nbr["w_next"])
    h_mid = torch.empty_like(x)
    out, nxt = blk.forward_neighbours(x, a, w_pa, w_next, layer_scalar=p["layer_scalar"],
                                      out=x if alias else None, h_mid=h_mid)
    torch.cuda.synchronize()
    assert blk.device_status()[0] == 0
    h_bits = bf16_bits(h_mid)
    # the block input against the oracle's attention residual.  The normed
    # attention n is a bf16 plane formed from fp32 products, so it may sit one
    # ulp from the exact value's rounding (as xd, xe); h = bf16(x + n) is then
    # exact given n, which a cancellation can turn into many ulps of h.  So h
    # must be the rounded sum for n or one of its bf16 neighbours, and equal
    # to the oracle's almost everywhere.
    h_ref = _f64_to_bits(oracle.attn_residual(nbr["x"], nbr["attn"], nbr["w_pa"]))
    n_ref = oracle.round_bf16(oracle.rms_norm(oracle.bf16_to_f64(nbr["attn"]),
                                              oracle.bf16_to_f64(nbr["w_pa"])))
    n_bits = _f64_to_bits(n_ref).astype(np.int32)
    xf = oracle.bf16_to_f64(nbr["x"])
    ok = h_bits == h_ref
    for step in (-1, 1):  # the neighbouring bf16 values of n (same sign)
        nb_bits = np.clip(n_bits + step, 0, 0xFFFF).astype(np.uint16)
        ok |= h_bits == _f64_to_bits(oracle.round_bf16(xf + oracle.bf16_to_f64(nb_bits)))
    assert ok.all() and (h_bits == h_ref).mean() > 0.999, (ok.mean(), (h_bits == h_ref).mean())
    # the block on the GPU's own h (on sampled tokens for large batches:
    # tokens are independent)
    out_bits = bf16_bits(out)
    rows = np.arange(T) if sample is None else np.sort(
        np.random.default_rng(seed).choice(T, sample, replace=False))
    ref = oracle.moe_block_forward(h_bits[rows], p, wl.top_k, wl.expert_inter,
                                   layer_scalar=p["layer_scalar"], with_perm=False)
    res = assert_close(out.float().cpu().numpy()[rows], ref["out"], "out", bf16_output=True)
    # the next layer's input norm of the GPU's output
    nx_ref = _f64_to_bits(oracle.next_input_norm(out_bits, nbr["w_next"]))
    dn = bf16_ulp_distance(bf16_bits(nxt), nx_ref)
    assert dn.max() <= 1 and (dn == 0).mean() > 0.999, (dn.max(), (dn == 0).mean())
    if full_check:
        # the plain forward on the same h: routing and permutation bit-exact,
        # the output (the branch checks, calibrated on the workloads' own
        # inputs, run in the plain parity tests)
        run_and_check(wl, p, h_bits, layer_scalar=p["layer_scalar"], blk=blk,
                      check_intermediates=False)
    blk.close()
    return res


@pytest.mark.parametrize("T", [32, 1, 17, 300, 4100])
def test_tiny_neighbours(T):
    wl = mi.get_workload("tiny")
    p = mi.make_layer_inputs(wl, randvec=True)
    _check(wl, p, T, seed=10 + T, sample=None if T <= 300 else 512)


def test_tiny_neighbours_out_aliases_x():
    wl = mi.get_workload("tiny")
    p = mi.make_layer_inputs(wl, randvec=True)
    _check(wl, p, 64, seed=3, alias=True, full_check=False)


def test_canvas256_neighbours():
    wl = mi.get_workload("canvas256")
    p = mi.make_layer_inputs(wl, randvec=True)
    print("canvas256 neighbours", _check(wl, p, wl.tokens, seed=7))


def test_canvas256_q4_neighbours_large_batch():
    # 4100 tokens: the register-tiled router (and its fused prologue) and the
    # 256-token 4-bit tiles
    wl = mi.get_workload("canvas256_q4")
    p = mi.make_layer_inputs(wl)
    _check(wl, p, 4100, seed=8, full_check=False, sample=256)


def test_neighbours_argument_checks():
    import moe_expert_ffn_dg_gb300.binding as B
    wl = mi.get_workload("tiny")
    p = mi.make_layer_inputs(wl)
    blk = make_block(wl, p)
    x = torch.zeros(wl.tokens, wl.hidden, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(wl.hidden, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    cases = [
        (B.dg_moe_neighbours_t(None, w.data_ptr(), None, None, None), B.DG_ERR_INVALID_ARG),
        (B.dg_moe_neighbours_t(x.data_ptr(), w.data_ptr(), w.data_ptr(), None, None),
         B.DG_ERR_INVALID_ARG),  # next-layer weight without an output
        (B.dg_moe_neighbours_t(x.data_ptr() + 2, w.data_ptr(), None, None, None),
         B.DG_ERR_ALIGNMENT),
    ]
    for nb, status in cases:
        with pytest.raises(B.DgError) as e:
            B.dg_moe_forward_neighbours(blk.handle, x.data_ptr(), nb, x.data_ptr(), wl.tokens,
                                        1.0, s)
        assert e.value.status == status
    blk.close()
