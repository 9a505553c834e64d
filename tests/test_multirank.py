"""The multi-rank host logic of bench.py on CPU: two gloo ranks, each with its own
vector sets, the step time taken as the maximum over ranks, and the whole-job rate."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import bench
    from bit_exact_emulation_gb300 import workloads as W
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank                       # rank 1 is the slow one
        slowest = bench.max_over_ranks(ms, dist, "cpu")
        a, b, c = W.gen_block_fma_set("bf16", 64, 4, seed=bench.rank_seed(4, rank))
        digest = torch.tensor([int(a.astype(np.int64).sum()), int(c.astype(np.int64).sum())])
        gathered = [torch.zeros_like(digest) for _ in range(world)]
        dist.all_gather(gathered, digest)
        out[rank] = (slowest, bench.whole_job_rate(1000, world, slowest),
                     [g.tolist() for g in gathered])
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        slowest, rate, digests = res[rank]
        assert slowest == 15.0
        assert rate == pytest.approx(2 * 1000 / 0.015)
        assert digests[0] != digests[1]              # each rank streams its own vector sets
    assert res[0][2] == res[1][2]
