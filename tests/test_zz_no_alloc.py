"""The allocation-free routing entry point against the regular forward.

dg_moe_route_noalloc serves callers that may not allocate device memory (an
allocator hook or an arena that owns the device, a host framework that
forbids allocation on its hot path): it routes with a fixed scratch array
inside the library instead of a caller workspace.  Its routing must equal the
one dg_moe_forward computes, call after call, since every call reuses the
same scratch.  This file is collected last on purpose.
"""

import numpy as np
import pytest
import torch

import moe_inputs as mi
from gpu_util import W_ABS, make_block, to_dev_bf16
from moe_expert_ffn_dg_gb300 import binding as B

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import moe_expert_ffn_dg_gb300 as pkg
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkg.build()
    pkg.load_library()


@pytest.mark.parametrize("name,tokens", [
    ("tiny", 0), ("canvas256", 0),
    # 8-bit router (the 4-bit canvas workload quantises its router to 8 bits)
    ("canvas256_q4", 0),
    # from 4096 tokens the logits come from the register-tiled kernel; at
    # hidden 256 that still fits the fixed scratch
    ("tiny", 4100)])
def test_noalloc_routing_equals_forward_routing_twice(name, tokens):
    wl = mi.get_workload(name, **({"tokens": tokens} if tokens else {}))
    p = mi.make_layer_inputs(wl, randvec=True)
    h = to_dev_bf16(mi.make_tokens(wl))
    blk = make_block(wl, p)
    _, dbg = blk.forward(h, p["layer_scalar"], debug=True)
    torch.cuda.synchronize()
    idx_ref = dbg["idx"].cpu().numpy()
    w_ref = dbg["w"].cpu().numpy()
    T, K = wl.tokens, wl.top_k
    idx = torch.empty(T, K, dtype=torch.int32, device="cuda")
    w = torch.empty(T, K, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        idx.fill_(-1)
        w.fill_(float("nan"))
        B.dg_moe_route_noalloc(blk.cfg, blk.cw, h.data_ptr(), T, idx.data_ptr(), w.data_ptr(),
                               stream)
        torch.cuda.synchronize()
        assert np.array_equal(idx.cpu().numpy(), idx_ref)
        assert np.abs(w.cpu().numpy() - w_ref).max() <= W_ABS
    blk.close()


def test_noalloc_routing_rejects_calls_beyond_its_scratch():
    wl = mi.get_workload("canvas256")
    p = mi.make_layer_inputs(wl)
    blk = make_block(wl, p)
    h = to_dev_bf16(mi.make_tokens(wl))
    out = torch.empty(1, dtype=torch.int32, device="cuda")
    with pytest.raises(B.DgError) as e:
        # 4096 tokens of hidden 2816 need far more than the fixed scratch;
        # rejected on the host before anything is read or written
        B.dg_moe_route_noalloc(blk.cfg, blk.cw, h.data_ptr(), 4096, out.data_ptr(),
                               out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert e.value.status == B.DG_ERR_UNSUPPORTED
    blk.close()
