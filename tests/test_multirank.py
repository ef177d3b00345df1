"""The step on several processes: the work-balanced partition of a bank
(muon_partition, host only), the way bench.py splits a world-sized bank and
aggregates its timing, and the exchange of the sharded data-parallel step
(gradients averaged onto owners, parameters broadcast from owners).  The
multi-rank tests run two `gloo` ranks on CPU as child processes, each
computing its own matrices with the oracle standing in for the GPU step; one
GPU test runs sharded_muon_step itself over a one-rank NCCL group.

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


# ------------------------------------------------ sharded data-parallel step
def _sharded_worker(rank, world, port, out_dir):
    """The exchange of sharded_muon_step around the local step, on CPU
    tensors: gradients averaged onto owners, the owner's step (the oracle
    stands in for the CUDA step here), parameters broadcast from owners."""
    import torch
    import torch.distributed as dist

    from newton_schulz_08_gb300 import inputs, sharded
    from oracle import muon_step
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        params = [torch.from_numpy(inputs.param(s, i)) for i, s in enumerate(SMALL_BANK)]
        grads = [torch.from_numpy(inputs.grad(s, i, step=rank)) for i, s in enumerate(SMALL_BANK)]
        bufs = [torch.from_numpy(inputs.buffer(s, i)) for i, s in enumerate(SMALL_BANK)]
        owner = sharded.owners([p.shape for p in params], world)
        mine = sharded.reduce_grads_to_owners(grads, owner, rank, world)
        assert sorted(mine) == [i for i, o in enumerate(owner) if o == rank]
        for i, g in mine.items():
            new_p, _, _ = muon_step(params[i].numpy(), g.numpy(), bufs[i].numpy(), 0.02, 0.95, True, 5, "fp64")
            params[i].copy_(torch.from_numpy(new_p.astype(np.float32)))
        sharded.broadcast_params_from_owners(params, owner, world)
        np.save(os.path.join(out_dir, f"p{rank}.npy"), np.concatenate([p.numpy().ravel() for p in params]))
    finally:
        dist.destroy_process_group()


def test_sharded_step_exchange_on_two_gloo_ranks(L):
    import torch.multiprocessing as mp

    from newton_schulz_08_gb300 import inputs
    from oracle import muon_step
    with tempfile.TemporaryDirectory() as d:
        mp.spawn(_sharded_worker, args=(WORKERS, _free_port(), d), nprocs=WORKERS, join=True)
        got = [np.load(os.path.join(d, f"p{r}.npy")) for r in range(WORKERS)]
    # every rank ends with the same parameters ...
    np.testing.assert_array_equal(got[0], got[1])
    # ... equal to one process stepping every matrix with the averaged gradient
    ref = []
    for i, s in enumerate(SMALL_BANK):
        g = (inputs.grad(s, i, step=0) + inputs.grad(s, i, step=1)) / np.float32(WORKERS)
        new_p, _, _ = muon_step(inputs.param(s, i), g, inputs.buffer(s, i), 0.02, 0.95, True, 5, "fp64")
        ref.append(new_p.astype(np.float32).ravel())
    np.testing.assert_array_equal(got[0], np.concatenate(ref))


@pytest.mark.gpu
def test_sharded_step_on_one_nccl_rank_equals_muon_step():
    """sharded_muon_step with world size 1: the fp32-averaged gradient has the
    bf16 gradient's values, so the result equals muon_step bit for bit."""
    import torch
    import torch.distributed as dist

    from newton_schulz_08_gb300 import inputs, sharded
    shapes = [(256, 256), (300, 100), (100, 300), (768, 768)]
    dev = torch.device("cuda")
    mk = lambda f: [torch.from_numpy(f(s, i)).to(dev) for i, s in enumerate(shapes)]
    P1, B1 = mk(inputs.param), mk(inputs.buffer)
    P2, B2 = [p.clone() for p in P1], [b.clone() for b in B1]
    G = [g.to(torch.bfloat16) for g in mk(inputs.grad)]
    store = dist.TCPStore("127.0.0.1", _free_port(), 1, True)
    dist.init_process_group("nccl", store=store, rank=0, world_size=1)
    try:
        ws = sharded.sharded_muon_step(P1, G, B1)
        torch.cuda.synchronize()
        assert muon.muon_device_status(ws) == muon.MUON_OK
    finally:
        dist.destroy_process_group()
    muon.muon_step(P2, G, B2)
    torch.cuda.synchronize()
    for a, b in zip(P1 + B1, P2 + B2):
        assert torch.equal(a, b)
