"""GPU parity of the self-conditioning MLP against the CPU oracle: the whole
output (bf16, unit RMS per token) within 2e-2 RMS beyond the bf16 half-ulp
and cosine 0.9999, and the MLP's own contribution out - rms(embeds) within
3e-2 of its RMS, so a wrong projection cannot hide behind the embeddings."""

import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
from gpu_util import assert_close, bf16_half_ulp, close_stats, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import moe_expert_ffn_dg_gb300 as pkg
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkg.build()
    pkg.load_library()


def _run(wl, p, ref_bf16_weights=False, T=None, alias=False):
    import moe_expert_ffn_dg_gb300 as pkg
    T = wl.tokens if T is None else T
    e, s = p["embeds"][:T], p["signal"][:T]
    sc = pkg.ScMlp.from_params(p, hidden=wl.hidden, inter=wl.dense_inter,
                               max_tokens=max(T, 1), device="cuda")
    ed = to_dev_bf16(e)
    out = sc.forward(ed, to_dev_bf16(s), out=ed if alias else None)
    torch.cuda.synchronize()
    assert sc.device_status() == 0
    got = out.float().cpu().numpy()
    ref = oracle.sc_mlp_forward(e, s, p, bf16_weights=ref_bf16_weights)
    res = assert_close(got, ref, "sc out", bf16_output=True)
    # the MLP's own share: the same error (beyond the output's half-ulp)
    # against the RMS of out - rms(embeds) instead of the RMS of out
    base = oracle.rms_norm(oracle.bf16_to_f64(e))
    excess = np.maximum(np.abs(got - ref) - bf16_half_ulp(ref), 0.0)
    _, c_rms, c_cos = close_stats(got - base, ref - base)
    assert float(excess.max()) <= 3e-2 * c_rms, (float(excess.max()), c_rms)
    assert c_cos >= 0.999, c_cos
    sc.close()
    return res, (c_rms, c_cos)


@pytest.mark.parametrize("randvec", [False, True])
def test_sc_tiny_bf16(randvec):
    wl = mi.get_workload("sc_tiny")
    print(_run(wl, mi.make_sc_inputs(wl, randvec=randvec)))


@pytest.mark.parametrize("T", [1, 17, 300])
def test_sc_tiny_ragged(T):
    wl = mi.get_workload("sc_tiny", tokens=T)
    _run(wl, mi.make_sc_inputs(wl, randvec=True))


def test_sc_tiny_q4():
    wl = mi.get_workload("sc_tiny")
    _run(wl, mi.make_sc_inputs(wl, randvec=True, quantise=True), ref_bf16_weights=True)


@pytest.mark.parametrize("T", [32, 1, 300])
def test_sc_tiny_q8(T):
    """8-bit group-64 affine gate/up/down (the q8 format the pages give the
    self-conditioning MLP beside 4-bit)."""
    wl = mi.get_workload("sc_tiny", quant=(8, 8, 8), tokens=T)
    _run(wl, mi.make_sc_inputs(wl, randvec=True, quantise=True), ref_bf16_weights=True)


def test_sc_zero_signal_gives_the_normed_embeddings():
    import moe_expert_ffn_dg_gb300 as pkg
    wl = mi.get_workload("sc_tiny")
    p = mi.make_sc_inputs(wl, randvec=True)
    sc = pkg.ScMlp.from_params(p, hidden=wl.hidden, inter=wl.dense_inter, max_tokens=wl.tokens,
                               device="cuda")
    zero = torch.zeros(wl.tokens, wl.hidden, dtype=torch.bfloat16, device="cuda")
    out = sc.forward(to_dev_bf16(p["embeds"]), zero)
    torch.cuda.synchronize()
    want = oracle.rms_norm(oracle.bf16_to_f64(p["embeds"]))
    got = out.float().cpu().numpy()
    # the only rounding left is the bf16 output itself (and fp32 1/rms)
    assert np.all(np.abs(got - want) <= bf16_half_ulp(want) + 1e-6 * np.abs(want) + 1e-30)
    sc.close()


def test_sc_output_may_alias_embeds():
    wl = mi.get_workload("sc_tiny")
    _run(wl, mi.make_sc_inputs(wl, randvec=True), alias=True)


def test_sc_canvas256_bf16():
    wl = mi.get_workload("sc_canvas256")
    print("sc_canvas256", _run(wl, mi.make_sc_inputs(wl, randvec=True)))


def test_sc_canvas256_q4_exact_decode():
    wl = mi.get_workload("sc_canvas256_q4")
    print("sc_canvas256_q4", _run(wl, mi.make_sc_inputs(wl, randvec=True)))


def test_sc_canvas256_q8_exact_decode():
    wl = mi.get_workload("sc_canvas256_q8")
    print("sc_canvas256_q8", _run(wl, mi.make_sc_inputs(wl, randvec=True)))
