"""The multi-GPU path is replicas only: each rank runs the whole block on its
own canvases and nothing crosses ranks on the data path.  These CPU tests run
two ranks over gloo (127.0.0.1) and check the host-side logic the benchmark
uses: distinct canvases per rank, the slowest-rank time, the aggregate
throughput, and that splitting a batch by canvases reproduces the block on
the whole batch (tokens are independent, checked with the CPU oracle)."""

import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from moe_expert_ffn_dg_gb300 import replicas


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_dir):
    import torch
    import torch.distributed as dist

    import moe_inputs as mi
    import oracle

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    base = mi.get_workload("tiny")
    wl = mi.get_workload("tiny", seed=replicas.replica_seed(base.seed, rank))
    h = mi.make_tokens(wl)
    p = mi.make_layer_inputs(base, randvec=True)  # every replica holds the same weights
    out = oracle.moe_block_forward(h, p, base.top_k, base.expert_inter, with_perm=False)["out"]
    # the slowest rank's time
    slowest = replicas.max_over_ranks(1.0 + 0.5 * rank, dist)
    # canvases of all ranks, for the whole-batch comparison on rank 0
    hs = [torch.zeros(h.shape, dtype=torch.int32) for _ in range(world)]
    dist.all_gather(hs, torch.from_numpy(h.astype(np.int32)))
    outs = [torch.zeros(out.shape, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(outs, torch.from_numpy(out))
    if rank == 0:
        h_all = np.concatenate([t.numpy().astype(np.uint16) for t in hs])
        out_all = oracle.moe_block_forward(h_all, p, base.top_k, base.expert_inter,
                                           with_perm=False)["out"]
        np.savez(os.path.join(out_dir, "r0.npz"), h_all=h_all, out_all=out_all,
                 outs=np.stack([t.numpy() for t in outs]), slowest=slowest)
    else:
        np.savez(os.path.join(out_dir, f"r{rank}.npz"), slowest=slowest)
    dist.barrier()
    dist.destroy_process_group()


@pytest.fixture(scope="module")
def two_ranks(tmp_path_factory):
    d = str(tmp_path_factory.mktemp("replicas"))
    mp.start_processes(_rank_main, args=(2, _free_port(), d), nprocs=2, join=True,
                       start_method="spawn")
    return d


def test_ranks_draw_distinct_canvases(two_ranks):
    r0 = np.load(os.path.join(two_ranks, "r0.npz"))
    h_all = r0["h_all"]
    n = h_all.shape[0] // 2
    assert not np.array_equal(h_all[:n], h_all[n:])
    assert replicas.replica_seed(7, 0) == 7 and replicas.replica_seed(7, 1) != 7


def test_slowest_rank_time_on_every_rank(two_ranks):
    for r in (0, 1):
        assert float(np.load(os.path.join(two_ranks, f"r{r}.npz"))["slowest"]) == 1.5


def test_split_by_canvas_reproduces_the_whole_batch(two_ranks):
    r0 = np.load(os.path.join(two_ranks, "r0.npz"))
    n = r0["out_all"].shape[0] // 2
    for r in (0, 1):
        np.testing.assert_allclose(r0["outs"][r], r0["out_all"][r * n:(r + 1) * n],
                                   rtol=1e-12, atol=1e-12)


def test_aggregate_throughput_counts_every_replica():
    assert replicas.aggregate_throughput(4, 256, 0.001) == pytest.approx(1.024e6)
    assert replicas.max_over_ranks(3.0) == 3.0
