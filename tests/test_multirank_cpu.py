"""The N > 1 path of bench.py on CPU: two gloo ranks, no GPU.

Each rank permutes its own batch (weak scaling, no collective on the data
path); the only cross-rank steps are the barrier and the max over ranks of the
timed region, from which rank 0 computes the whole-job throughput.  These tests
run those steps with world_size 2 on the gloo backend, and check that rank-local
oracle work on disjoint batch shards reassembles the single-rank result.
"""
import os
import socket
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import oracle
    from movement_tl_permute_gb300 import workloads

    assert bench.dist_env() == (rank, rank, world)
    # max over ranks of a per-rank time
    got = bench.reduce_max(10.0 + 5.0 * rank)
    bench.barrier()
    # each rank permutes its own leading shard of the tile batch
    w = workloads.get("tile_transpose")
    per_rank = 6
    lead = workloads.scaled(w, per_rank * world)
    src = workloads.make_input(lead)
    shard_elems = per_rank * 8192
    mine = src.view(np.uint16)[rank * shard_elems:(rank + 1) * shard_elems].copy().view(np.uint8)
    out = np.zeros_like(mine)
    oracle.permute(mine, out, (per_rank,) + w.shape[1:], w.src_strides, w.dst_strides, 2)
    np.save(os.path.join(out_dir, "shard%d.npy" % rank), out)
    np.save(os.path.join(out_dir, "max%d.npy" % rank), np.array([got]))
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_and_shard(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    for r in range(world):
        assert float(np.load(tmp_path / ("max%d.npy" % r))[0]) == 15.0
    # the shards, concatenated, are the single-process permute of the whole batch
    sys.path.insert(0, ROOT)
    import oracle
    from movement_tl_permute_gb300 import workloads

    w = workloads.get("tile_transpose")
    lead = workloads.scaled(w, 12)
    src = workloads.make_input(lead)
    want = np.zeros_like(src)
    oracle.permute(src, want, lead.shape, w.src_strides, w.dst_strides, 2)
    got = np.concatenate([np.load(tmp_path / ("shard%d.npy" % r)) for r in range(world)])
    assert np.array_equal(got, want)


def test_whole_job_throughput_is_weak_scaling():
    sys.path.insert(0, ROOT)
    import bench

    # 2 ranks, each 1 GB per step, 10 steps, slowest rank 10 ms -> 2 TB/s aggregate
    assert bench.whole_job_gbps(10**9, 10, 2, 10.0) == pytest.approx(2000.0)
    assert bench.whole_job_gbps(10**9, 10, 1, 10.0) == pytest.approx(1000.0)
    assert bench.reduce_max(3.5) == 3.5          # no process group: identity
