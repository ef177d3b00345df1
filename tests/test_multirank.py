"""The step on several processes: the work-balanced partition of a bank
(muon_partition, host only), the way bench.py splits a world-sized bank and
aggregates its timing, and the exchange of the sharded data-parallel step
(ShardedBank: reduce-scatter of the gradients by size group, the owners'
steps, all-gather of the parameters).  The multi-rank tests run two `gloo`
ranks on CPU as child processes, each computing its own matrices with the
oracle standing in for the GPU step; one GPU test runs ShardedBank itself
over a one-rank NCCL group.

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
# several size groups (the 960-element group mixes a tall and a wide shape),
# uneven ownership within groups, tall, wide and square matrices
SHARD_BANK = [(24, 40), (24, 40), (40, 24), (24, 40), (32, 32), (32, 32), (16, 48), (20, 20), (20, 20), (20, 20),
              (8, 56)]
SHARD_STEPS = 2
HP = dict(lr=0.02, momentum=0.95, nesterov=True, ns_steps=5)


def _grad(shape, i, step, rank):
    from newton_schulz_08_gb300 import inputs
    return inputs.grad(shape, i, step=2 * step + rank)


def _oracle_local_step(params, grads, bufs, lr, momentum, nesterov, ns_steps, stream):
    """The owner's step with the oracle standing in for the CUDA path: fp32
    state in and out, the step in fp64."""
    import torch

    from oracle import muon_step
    for p, g, b in zip(params, grads, bufs):
        new_p, new_b, _ = muon_step(p.numpy().astype(np.float64), g.float().numpy().astype(np.float64),
                                    b.numpy().astype(np.float64), lr, momentum, nesterov, ns_steps, "fp64")
        p.copy_(torch.from_numpy(new_p.astype(np.float32)))
        b.copy_(torch.from_numpy(new_b.astype(np.float32)))


def _sharded_worker(rank, world, port, out_dir):
    """ShardedBank.step on CPU tensors over gloo: reduce-scatter of the bf16
    gradients, the owners' steps (the oracle stands in for the CUDA step),
    asynchronous all-gather of the parameters."""
    import torch
    import torch.distributed as dist

    from newton_schulz_08_gb300 import inputs, sharded
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bank = sharded.ShardedBank(SHARD_BANK, "cpu")
        for i, s in enumerate(SHARD_BANK):
            bank.params[i].copy_(torch.from_numpy(inputs.param(s, i)))
        for step in range(SHARD_STEPS):
            for i, s in enumerate(SHARD_BANK):
                bank.grads[i].copy_(torch.from_numpy(_grad(s, i, step, rank)))
            bank.step(local_step=_oracle_local_step, **HP)
        np.save(os.path.join(out_dir, f"p{rank}.npy"), np.concatenate([p.numpy().ravel() for p in bank.params]))
        np.save(os.path.join(out_dir, f"owned{rank}.npy"), np.array(bank.owned()))
        for i in bank.owned():
            np.save(os.path.join(out_dir, f"buf{i}.npy"), bank.bufs[i].numpy())
        assert all(bank.bufs[i] is None for i in range(len(SHARD_BANK)) if i not in bank.owned())
    finally:
        dist.destroy_process_group()


def test_sharded_step_exchange_on_two_gloo_ranks(L):
    import torch.multiprocessing as mp

    import oracle
    from newton_schulz_08_gb300 import inputs, sharded
    with tempfile.TemporaryDirectory() as d:
        mp.spawn(_sharded_worker, args=(WORKERS, _free_port(), d), nprocs=WORKERS, join=True)
        got = [np.load(os.path.join(d, f"p{r}.npy")) for r in range(WORKERS)]
        owned = [np.load(os.path.join(d, f"owned{r}.npy")).tolist() for r in range(WORKERS)]
        bufs = {i: np.load(os.path.join(d, f"buf{i}.npy")) for r in owned for i in r}
    # every matrix has exactly one owner, and the groups are uneven
    assert sorted(owned[0] + owned[1]) == list(range(len(SHARD_BANK)))
    own = sharded.owners(SHARD_BANK, WORKERS)
    groups = [sharded._Group(idx, SHARD_BANK, own, WORKERS) for idx in sharded.size_groups(SHARD_BANK)]
    assert any(len(g.members[0]) != len(g.members[1]) for g in groups)
    # every rank ends with the same parameters ...
    np.testing.assert_array_equal(got[0], got[1])
    # ... equal, bit for bit, to one process stepping every matrix with the
    # average of the ranks' bf16 gradients: their bf16 sum (one rounding for
    # two terms) halved (exact)
    ref_p, ref_b = [], {}
    for i, s in enumerate(SHARD_BANK):
        p, b = inputs.param(s, i), np.zeros(s, np.float32)
        for step in range(SHARD_STEPS):
            gs = [oracle.round_to_bf16(_grad(s, i, step, r)) for r in range(WORKERS)]
            g = oracle.round_to_bf16(gs[0] + gs[1]) / WORKERS
            new_p, new_b, _ = oracle.muon_step(p.astype(np.float64), g, b.astype(np.float64), HP["lr"],
                                               HP["momentum"], HP["nesterov"], HP["ns_steps"], "fp64")
            p, b = new_p.astype(np.float32), new_b.astype(np.float32)
        ref_p.append(p.ravel())
        ref_b[i] = b
    np.testing.assert_array_equal(got[0], np.concatenate(ref_p))
    for i, b in bufs.items():
        np.testing.assert_array_equal(b, ref_b[i])


def test_sharded_layout_is_owner_ordered_and_padded(L):
    """The flat buffers hold each rank's matrices in one segment per group,
    every segment padded to the group's longest."""
    from newton_schulz_08_gb300 import sharded
    groups = sharded.size_groups(SHARD_BANK)
    assert [SHARD_BANK[g[0]][0] * SHARD_BANK[g[0]][1] for g in groups] == [1024, 960, 768, 448, 400]
    owner = sharded.owners(SHARD_BANK, 3)
    for idx in groups:
        g = sharded._Group(idx, SHARD_BANK, owner, 3)
        assert g.seg == g.numel * max(len(m) for m in g.members)
        seen = set()
        for r, mem in enumerate(g.members):
            for k, i in enumerate(mem):
                assert owner[i] == r and g.offset[i] == r * g.seg + k * g.numel
                seen.add(i)
        assert seen == set(idx)


@pytest.mark.gpu
def test_sharded_step_on_one_nccl_rank_equals_muon_step():
    """ShardedBank.step with world size 1 (the reduce-scatter and the
    all-gather are copies): equal to muon_step bit for bit over two steps."""
    import torch
    import torch.distributed as dist

    from newton_schulz_08_gb300 import inputs, sharded
    shapes = [(256, 256), (300, 100), (100, 300), (768, 768), (768, 768)]
    dev = torch.device("cuda")
    P2 = [torch.from_numpy(inputs.param(s, i)).to(dev) for i, s in enumerate(shapes)]
    B2 = [torch.zeros(s, device=dev) for s in shapes]
    store = dist.TCPStore("127.0.0.1", _free_port(), 1, True)
    dist.init_process_group("nccl", store=store, rank=0, world_size=1)
    try:
        bank = sharded.ShardedBank(shapes, dev)
        for i, p in enumerate(P2):
            bank.params[i].copy_(p)
        for step in range(2):
            G = [torch.from_numpy(inputs.grad(s, i, step=step)).to(dev).to(torch.bfloat16)
                 for i, s in enumerate(shapes)]
            for i, g in enumerate(G):
                bank.grads[i].copy_(g)
            bank.step()
            muon.muon_step(P2, G, B2)
        torch.cuda.synchronize()
        assert muon.muon_device_status(bank.workspace) == muon.MUON_OK
    finally:
        dist.destroy_process_group()
    for i in range(len(shapes)):
        assert torch.equal(bank.params[i], P2[i]) and torch.equal(bank.bufs[i], B2[i])
