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


def test_bench_gpus_flag_starts_that_many_ranks():
    """`bench.py --gpus 2` without a launcher starts two ranks itself (torch.distributed.run
    on 127.0.0.1); on CPU the reference arm joins a gloo group, rank 0 alone prints the
    line, and it reports both ranks."""
    import json
    import subprocess

    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(k, None)
    p = subprocess.run([sys.executable, "bench.py", "--gpus", "2", "--impl", "reference",
                        "--workload", "tiny_f32", "--steps", "3", "--warmup", "3"], cwd=ROOT,
                       env=env, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    r = json.loads(lines[0])
    assert r["n_gpus"] == 2 and r["impl"] == "reference" and r["steps"] == 3


def test_bench_gpus_flag_must_match_the_launcher():
    import subprocess

    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    p = subprocess.run([sys.executable, "bench.py", "--gpus", "2", "--impl", "reference"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode != 0 and "WORLD_SIZE" in p.stderr
