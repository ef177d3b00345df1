"""The step on several processes: the work-balanced partition of a bank
(muon_partition, host only) and the way bench.py splits a world-sized bank
and aggregates its timing.  CPU only: the multi-rank test runs two `gloo`
ranks as child processes, each computing its own matrices with the oracle
(standing in for the GPU step, which the ranks never exchange data for).

The page "深入解析KellerJordan/modded-nanogpt中的训练架构与优化技术"
(reposource.net), section "Muon优化器：动量正交化技术", shards the step by
giving each rank its own parameters; what a rank computes for a matrix must
not depend on which rank computes it, and every matrix must have exactly one
owner.
"""

import ctypes
import os
import socket
import tempfile

import numpy as np
import pytest

import bench
from newton_schulz_08_gb300 import muon

WORKERS = 2


def work(shape):
    m, n = min(shape), max(shape)
    return m * (m + 1) * n + m * m * (m + 1) + 2 * m * m * n


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(muon.LIB_PATH):
        from newton_schulz_08_gb300 import build
        build.build()
    return muon.lib()


def test_partition_covers_and_balances(L):
    rng = np.random.default_rng(7)
    for trial in range(40):
        n = int(rng.integers(1, 60))
        world = int(rng.integers(1, 9))
        shapes = [(int(rng.integers(1, 3000)), int(rng.integers(1, 3000))) for _ in range(n)]
        owner = muon.partition(shapes, world)
        assert len(owner) == n and all(0 <= o < world for o in owner)
        assert muon.partition(shapes, world) == owner  # a pure function of its arguments
        load = np.zeros(world)
        for s, o in zip(shapes, owner):
            load[o] += work(s)
        # greedy longest-first: the last matrix placed on the busiest rank
        # went to the least-loaded rank, so the excess is at most one matrix
        assert load.max() <= load.sum() / world + max(work(s) for s in shapes) + 1e-6


def test_partition_special_cases(L):
    assert muon.partition([(64, 64)] * 5, 1) == [0] * 5
    # more ranks than matrices: each matrix on a rank of its own
    owner = muon.partition([(8, 8), (16, 16), (32, 32)], 6)
    assert len(set(owner)) == 3
    # heaviest first, ties to the lowest rank
    assert muon.partition([(8, 8), (32, 32), (16, 16)], 2) == [1, 0, 1]
    # identical banks repeated per rank: every rank gets one bank's mix
    gpt2 = bench.workload_shapes("gpt2")
    for world in (2, 3, 8):
        for rank in range(world):
            ids, shapes = bench.rank_bank(gpt2, world, rank)
            assert sorted(shapes) == sorted(gpt2)
    assert muon.partition([], 4) == []


def test_partition_rejects_bad_arguments(L):
    i64 = ctypes.c_int64 * 2
    owner = (ctypes.c_int * 2)(-5, -5)
    assert L.muon_partition(i64(4, 4), i64(4, 4), 2, 0, owner) == muon.MUON_ERR_INVALID_ARG
    assert L.muon_partition(i64(4, 0), i64(4, 4), 2, 2, owner) == muon.MUON_ERR_INVALID_ARG
    assert L.muon_partition(None, i64(4, 4), 2, 2, owner) == muon.MUON_ERR_INVALID_ARG
    assert L.muon_partition(i64(4, 4), i64(4, 4), -1, 2, owner) == muon.MUON_ERR_INVALID_ARG
    assert list(owner) == [-5, -5]  # untouched on error
    assert L.muon_partition(None, None, 0, 2, None) == muon.MUON_OK


# a small bank of mixed shapes (tall, wide, square, ragged)
SMALL_BANK = [(24, 40), (40, 24), (32, 32), (16, 48), (48, 16), (20, 20), (8, 56)]


def _oracle_step(gid, shape):
    from newton_schulz_08_gb300 import inputs
    from oracle import muon_step
    p = inputs.param(shape, gid).astype(np.float64)
    g = inputs.grad(shape, gid).astype(np.float64)
    b = inputs.buffer(shape, gid).astype(np.float64)
    new_p, new_b, _ = muon_step(p, g, b, 0.02, 0.95, True, 5, "fp64")
    return new_p, new_b


def _worker(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ids, shapes = bench.rank_bank(SMALL_BANK, world, rank)
        mine = {gid: _oracle_step(gid, s) for gid, s in zip(ids, shapes)}
        # timing aggregation: every rank sees the slowest rank's time
        got = bench.max_over_ranks(1.5 * (rank + 1), world)
        assert got == 1.5 * world, got
        gathered = [None] * world
        dist.all_gather_object(gathered, (ids, mine))
        if rank == 0:
            np.save(os.path.join(out_dir, "ids.npy"), np.array([g for ids_r, _ in gathered for g in ids_r]))
            results = {}
            for _, m in gathered:
                results.update(m)
            np.save(os.path.join(out_dir, "p.npy"),
                    np.concatenate([results[g][0].ravel() for g in sorted(results)]))
            np.save(os.path.join(out_dir, "buf.npy"),
                    np.concatenate([results[g][1].ravel() for g in sorted(results)]))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_share_a_world_sized_bank(L):
    import torch.multiprocessing as mp
    with tempfile.TemporaryDirectory() as d:
        mp.spawn(_worker, args=(WORKERS, _free_port(), d), nprocs=WORKERS, join=True)
        ids = np.load(os.path.join(d, "ids.npy"))
        p = np.load(os.path.join(d, "p.npy"))
        buf = np.load(os.path.join(d, "buf.npy"))
    total = len(SMALL_BANK) * WORKERS
    # every matrix of the world-sized bank has exactly one owner
    assert sorted(ids.tolist()) == list(range(total))
    # and the sharded result equals one process doing the whole bank
    full = [SMALL_BANK[g % len(SMALL_BANK)] for g in range(total)]
    ref = [_oracle_step(g, full[g]) for g in range(total)]
    np.testing.assert_array_equal(p, np.concatenate([r[0].ravel() for r in ref]))
    np.testing.assert_array_equal(buf, np.concatenate([r[1].ravel() for r in ref]))
