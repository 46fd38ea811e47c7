"""The benchmark's multi-process path on CPU: two gloo ranks rendezvous on 127.0.0.1 the
way torchrun launches bench.py, take the max of their step times over ranks, draw
different seeded batches (token-parallel replicas), and only rank 0 produces a line."""

import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    from moe_workloads import PARITY_WORKLOADS, make_inputs
    import torch.distributed as dist

    w_, r_, l_ = bench.dist_env()
    assert (w_, r_, l_) == (world, rank, rank)
    bench.dist_init(world, rank, backend="gloo")
    bench.barrier(world)
    my_ms = 1.0 + rank          # rank 1 is the slower one
    slowest = bench.allreduce_max(my_ms, world, device="cpu")
    w = PARITY_WORKLOADS["tiny_f32"]
    x = make_inputs(w, seed=rank)["x"]                 # each replica its own batch
    others = [torch.zeros_like(x) for _ in range(world)]
    dist.all_gather(others, x)
    ref_line = bench.run_reference(None, world, rank, rank) if rank != 0 else "rank0"
    results[rank] = dict(slowest=slowest, distinct=not torch.equal(others[0], others[1]),
                         ref_none=ref_line is None,
                         value=bench.replica_throughput(world, w.T, slowest))
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_distinct_batches():
    world = 2
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), results), nprocs=world, join=True)
        res = dict(results)
    assert res[0]["slowest"] == res[1]["slowest"] == 2.0
    assert res[0]["distinct"] and res[1]["distinct"]
    assert res[1]["ref_none"]                        # the reference arm runs on rank 0 only
    assert res[0]["value"] == pytest.approx(2 * 256 / 2e-3)
