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


def _shard_rank(rank, world, port, out):
    """Each rank evaluates its share with the CPU evaluator (the oracle) and rank 0
    assembles the whole: vector ranges, row bands of a GEMM, and word-pair products of
    a multi-word GEMM combined in the fixed order on the owner."""
    import oracle
    from oracle.presets import PRESETS, block_models
    from bit_exact_emulation_gb300 import shard, workloads as W
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        # block FMAs by index range
        spec = block_models("bf16", 4)["ga_rne"]
        a, b, c = W.gen_block_fma_set("bf16", 1001, 4, seed=9)
        lo, hi = shard.vector_range(1001, rank, world)
        part = torch.from_numpy(oracle.block_fma(spec, a[lo:hi], b[lo:hi], c[lo:hi]).astype(np.int64))
        parts = [None] * world
        dist.all_gather_object(parts, part.tolist())
        vec = np.array(sum(parts, []), dtype=np.uint32)
        # GEMM rows by whole 64-row tiles
        M, N, K = 150, 20, 48
        A, Bt, C = W.gen_dense_bf16(M, N, K, seed=3)
        r0, r1 = shard.row_band(M, rank, world)
        ii, jj = np.meshgrid(np.arange(r0, r1), np.arange(N), indexing="ij")
        band = oracle.gemm_entries(PRESETS["cdna3_bf16"], K, 8, A, Bt, C, ii.ravel(), jj.ravel())
        bands = [None] * world
        dist.all_gather_object(bands, band.tolist())
        gemm = np.array(sum(bands, []), dtype=np.uint32).reshape(M, N)
        # multi-word: each rank the fp32 products of its word pairs, the owner adds them
        Mw, Nw, Kw = 6, 5, 32
        Af, Bf = W.gen_multiword_fp64(Mw, Nw, Kw, seed=5)
        wa, wb = oracle.split_bf16(Af, 3).reshape(3, Mw, Kw), oracle.split_bf16(Bf, 3).reshape(3, Nw, Kw)
        zero = np.zeros((Mw, Nw), np.uint32)
        iw, jw = np.meshgrid(np.arange(Mw), np.arange(Nw), indexing="ij")
        mine = {}
        for (i, j) in shard.word_pairs(3, False, rank, world):
            mine[f"{i},{j}"] = oracle.gemm_entries(PRESETS["cdna3_bf16"], Kw, 8, wa[i - 1], wb[j - 1], zero,
                                                   iw.ravel(), jw.ravel()).tolist()
        prods = [None] * world
        dist.all_gather_object(prods, mine)
        allp = {k: v for d in prods for k, v in d.items()}
        D = np.zeros(Mw * Nw)
        for (i, j) in shard.combine_order(3, False):
            D = D + np.array(allp[f"{i},{j}"], np.uint32).view(np.float32).astype(np.float64)
        if rank == 0:
            out["vec"] = bool(np.array_equal(vec, oracle.block_fma(spec, a, b, c)))
            ii, jj = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
            whole = oracle.gemm_entries(PRESETS["cdna3_bf16"], K, 8, A, Bt, C, ii.ravel(), jj.ravel()).reshape(M, N)
            out["gemm"] = bool(np.array_equal(gemm, whole))
            want = oracle.multiword_entries(PRESETS["cdna3_bf16"], 8, 3, False, Af, Bf, iw.ravel(), jw.ravel())
            out["mw"] = bool(np.array_equal(D.view(np.uint64), want.view(np.uint64)))
    finally:
        dist.destroy_process_group()


def test_sharded_work_concatenates_to_the_single_rank_result():
    from bit_exact_emulation_gb300 import shard
    for n in (0, 1, 7, 1000):
        for world in (1, 2, 3, 8):
            ranges = [shard.vector_range(n, r, world) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == n
            assert all(ranges[r][1] == ranges[r + 1][0] for r in range(world - 1))
    assert len(shard.combine_order(3, False)) == 9 and len(shard.combine_order(3, True)) == 6
    assert shard.combine_order(3, False)[:3] == [(3, 3), (2, 3), (3, 2)]
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_shard_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res == {"vec": True, "gemm": True, "mw": True}
