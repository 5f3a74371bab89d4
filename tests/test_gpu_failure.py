"""Failure detection on the GPU without a fault: a bounded device wait that
runs out.

Every wait inside the kernels has a limit; when it runs out the kernel
records a timeout in the workspace status word, stops, drains the copies
and tensor-core operations it has in flight, releases its tensor memory and
returns.  dg_moe_arm_wait_timeout_test makes one such wait (block 0 of the
next forward's gate_up GEMM, on a barrier nothing arrives on, 10 ms limit)
run out.  The test checks that the host sees DG_ERR_TIMEOUT with the
reported site, that the status word is cleared by reading it, and that the
same handle's next forward is clean and matches the oracle.  Nothing
faults, traps or hangs.
"""

import pytest
import torch

import moe_inputs as mi
from gpu_util import make_block, run_and_check, to_dev_bf16

pytestmark = pytest.mark.gpu

SITE_GEMM_EPILOGUE = 3
STALL_INFO = 0x57A11


@pytest.fixture(scope="module", autouse=True)
def _built():
    import moe_expert_ffn_dg_gb300 as pkg
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkg.build()
    pkg.load_library()


@pytest.mark.parametrize("name,quantise", [("tiny", False), ("tiny", True),
                                           ("canvas256", False)])
def test_bounded_wait_runs_out_and_the_handle_recovers(name, quantise):
    from moe_expert_ffn_dg_gb300 import binding as B
    wl = mi.get_workload(name)
    p = mi.make_layer_inputs(wl, randvec=True, quantise=quantise)
    h = mi.make_tokens(wl)
    blk = make_block(wl, p)
    hd = to_dev_bf16(h)
    B.dg_moe_arm_wait_timeout_test(blk.handle)
    blk.forward(hd, p["layer_scalar"])
    torch.cuda.synchronize()
    assert blk.device_status() == (B.DG_ERR_TIMEOUT, SITE_GEMM_EPILOGUE, STALL_INFO)
    # reading the status cleared it, and the test was armed for one forward
    assert blk.device_status()[0] == B.DG_OK
    for _ in range(2):
        run_and_check(wl, p, h, blk=blk, ref_bf16_weights=quantise)
        assert blk.device_status()[0] == B.DG_OK
    blk.close()
