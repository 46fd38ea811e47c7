"""The reference arm of bench.py (the CPU oracle) prints one well-formed JSON line."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload",
                          "tiny_f32", "--steps", "3", "--warmup", "3"], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=300, check=True).stdout
    lines = [ln for ln in out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    r = json.loads(lines[0])
    assert r["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in r, key
    assert r["steps"] == 3 and r["warmup"] == 3 and r["n_gpus"] == 1
    assert r["value"] > 0 and r["higher_is_better"] is True
    assert r["config"]["workload"] == "tiny_f32"
    assert r["cpu_baseline"]["kind"] == "oracle" and r["cpu_baseline"]["value"] == r["value"]
    assert r["e2e"]["value"] == r["value"] and r["e2e"]["h2d_bytes_per_step"] == 0


def test_bench_rejects_short_warmup():
    p = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--warmup", "2"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert p.returncode != 0 and "warmup" in p.stderr


def test_roofline_bound_and_fraction():
    """The roofline object picks the bound from the algorithmic flops and bytes and
    divides by the right peak."""
    sys.path.insert(0, ROOT)
    import bench
    from moe_workloads import WORKLOADS

    peaks = dict(hbm_gbs=6500.0, bf16_tflops=1800.0, bf16_tflops_sustained=1400.0,
                 source="test")
    w = WORKLOADS["mixtral_prefill"]
    M = w.T * w.k
    flops, byts = bench.ffn_algorithmic(w, M, w.E)
    assert flops == 4.0 * M * w.d * w.h
    r = bench.roofline(w, M, w.E, 1e-3, peaks)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["achieved"] - flops / 1e-3 / 1e12) < 0.1
    assert abs(r["frac"] - r["achieved"] / 1800.0) < 1e-4
    d = WORKLOADS["decode"]
    r = bench.roofline(d, d.T * d.k, 24, 1e-3, peaks)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 6500.0
    assert r["algorithmic_bytes"] >= 24 * 2 * d.d * d.h * 2


def test_traffic_figure_is_dropped_when_the_gemm_sources_change(monkeypatch):
    """roofline.traffic comes from a capture of specific GEMM sources: with any other
    sources (a different hash) the figure is reported as null, not carried over."""
    sys.path.insert(0, ROOT)
    import bench

    name = next(iter(bench.NCU_TRAFFIC_BYTES))
    recorded = bench.NCU_TRAFFIC_BYTES[name][0]
    monkeypatch.setattr(bench, "gemm_source_hash", lambda: recorded)
    assert bench.ncu_traffic(name)[0] == bench.NCU_TRAFFIC_BYTES[name][1]
    monkeypatch.setattr(bench, "gemm_source_hash", lambda: "0" * 16)
    assert bench.ncu_traffic(name) == (None, None)


def test_forward_launch_count():
    """gpu_launches counts the forward's own kernels: eight, one fewer on a bf16 top-1 layer
    whose groups fit the weights-as-M GEMMs (the combine is folded into them), and one fewer
    again with fused_gather (no row copy)."""
    sys.path.insert(0, ROOT)
    import bench
    from moe_workloads import WORKLOADS, Workload

    assert bench.forward_launches(WORKLOADS["mixtral_prefill"]) == 8
    assert bench.forward_launches(WORKLOADS["decode"]) == 8
    assert bench.forward_launches(WORKLOADS["switch_capacity"]) == 7  # C = 80 rows
    assert bench.forward_launches(WORKLOADS["switch_capacity"], fused_gather=True) == 6
    assert bench.forward_launches(WORKLOADS["mixtral_prefill"], fused_gather=True) == 7
    # top-1 with groups above 128 rows, and top-1 in fp32 (groups of at most 64 rows), keep
    # the combine pass
    big = Workload("top1_big", T=4096, d=256, h=512, E=8, k=1, dtype="bf16", gate=1,
                   capacity_factor=0.0)
    assert bench.forward_launches(big) == 8
    f32 = Workload("top1_f32", T=64, d=64, h=128, E=8, k=1, dtype="f32", gate=1,
                   capacity_factor=0.0)
    assert bench.forward_launches(f32) == 8
