"""Multi-process (gloo, world_size 2, CPU) checks of the N>1 path: the N-shard
plan covers the weight exactly, sharded results equal the unsharded layer with
no exchange (CPU oracle on each rank), and the benchmark's max-over-ranks
aggregation."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from semi_structured_sparse_gb300 import shard


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_shard_plan_partitions_rows():
    for N in (128, 256, 4096, 14336, 28672):
        for world in (1, 2, 3, 4, 8):
            plan = shard.shard_plan(N, world)
            assert plan[0][0] == 0 and plan[-1][1] == N
            for (a, b), (c, d) in zip(plan, plan[1:]):
                assert b == c
            sizes = [b - a for a, b in plan]
            assert all(s % 128 == 0 for s in sizes)
            assert max(sizes) - min(sizes) <= 128
    with pytest.raises(ValueError):
        shard.shard_rows(200, 2, 0)


def _bench_worker(rank, world, port, result_path):
    """What bench.py --gpus N builds on each rank: its rows of the one layer's
    weight (split) or the whole layer on a batch of its own (replicas)."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import inputs
    assert bench.dist_env()[:2] == (rank, world)
    w0 = inputs.WORKLOADS["groupwise"]
    w, rows = bench.rank_workload(w0, world, rank, "split")
    r, _ = bench.rank_workload(w0, world, rank, "replicas")
    mine = torch.tensor([rows[0], rows[1], w.M, w.N, w.K, r.N, r.seed], dtype=torch.int64)
    got = [torch.zeros(7, dtype=torch.int64) for _ in range(world)]
    dist.all_gather(got, mine)
    if rank == 0:
        np.save(result_path, torch.stack(got).numpy())
    dist.destroy_process_group()


def test_bench_rank_shapes_two_ranks(tmp_path):
    world, port = 2, _free_port()
    path = str(tmp_path / "shapes.npy")
    mp.start_processes(_bench_worker, args=(world, port, path), nprocs=world, start_method="spawn")
    t = np.load(path)
    w0 = __import__("inputs").WORKLOADS["groupwise"]
    # split: contiguous whole-tile blocks of W's rows covering N once, full M and K on every rank
    assert t[0, 0] == 0 and t[0, 1] == t[1, 0] and t[1, 1] == w0.N
    assert all(t[i, 3] == t[i, 1] - t[i, 0] and t[i, 3] % 256 == 0 for i in range(world))
    assert all(t[i, 2] == w0.M and t[i, 4] == w0.K for i in range(world))
    # replicas: the whole layer, a batch of its own per rank
    assert all(t[i, 5] == w0.N for i in range(world)) and t[0, 6] != t[1, 6]


def _worker(rank, world, port, result_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import inputs
    import oracle
    w = inputs.Workload("mr", 24, 512, 256, gN=128, gK=128, seed=5)
    X, W, _, _ = inputs.generate(w)
    xq, sx = oracle.quantize_act(X.numpy(), 128)
    a, b = shard.shard_rows(w.N, world, rank)
    Wb = inputs.bf16_bits(W)[a:b]
    values, meta, sw = oracle.compress(Wb, 128, 128)
    y_local = oracle.gemm(xq, sx, values, meta, sw, 1, 128, 128)
    # gather only to check; the layer itself needs no exchange
    gathered = [torch.zeros((w.M, hi - lo), dtype=torch.float64) for lo, hi in shard.shard_plan(w.N, world)]
    dist.all_gather(gathered, torch.from_numpy(y_local))
    t = torch.tensor([0.010 * (rank + 1)])
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    if rank == 0:
        full = np.concatenate([g.numpy() for g in gathered], axis=1)
        v, m, s = oracle.compress(inputs.bf16_bits(W), 128, 128)
        ref = oracle.gemm(xq, sx, v, m, s, 1, 128, 128)
        np.save(result_path, np.stack([full, ref]))
        with open(result_path + ".t", "w") as f:
            f.write(repr(float(t.item())))
    dist.destroy_process_group()


def test_two_rank_sharded_layer_equals_unsharded(tmp_path):
    world, port = 2, _free_port()
    path = str(tmp_path / "res.npy")
    mp.start_processes(_worker, args=(world, port, path), nprocs=world, start_method="spawn")
    full, ref = np.load(path)
    assert np.array_equal(full, ref)  # bit-identical: shards see exactly the same arithmetic
    assert float(open(path + ".t").read()) == pytest.approx(0.020)
    assert shard.aggregate_throughput(10.0, [0.01, 0.02]) == pytest.approx(1000.0)
