#!/usr/bin/env python3
"""Benchmark of the top-k MoE FFN forward (moe_forward through the C ABI) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one moe_forward (router, softmax/top-k, balance loss, dispatch, grouped
expert GEMMs, combine) over one batch of seeded synthetic tokens already resident in
HBM.  Default workload: the 8-expert top-2 prefill layer (T=4096, d=4096, h=14336,
bf16).  L2 is flushed (a 256 MB write) before every timed step, outside the step's
CUDA-event pair.  Under torchrun each rank runs an independent replica on its own
batch (token-parallel, no data-path collective): value = tokens of all ranks / the
slowest rank's time.  Rank 0 prints one JSON line.

The line carries: the device-timed tokens/s (`value`, T over the median step), the
end-to-end tokens/s with host-resident x and y copied in and out inside the timed region
(`e2e`: moe_forward_host over `steps` pinned batches, copies overlapped with the layer;
`e2e.serial_value` one step at a time), the grouped
expert GEMM pair timed alone against the measured roofline (`roofline`), the CPU
oracle timed on a bounded sample of the same workload (`cpu_baseline`), SM clocks
sampled during the timed region (`clocks`) and the number of our kernel launches in
the timed region (`gpu_launches`).

With the default workload the line also carries `workloads`: every configuration of
the layer family (tiny fp32, 8-expert prefill, 128-expert Switch with capacity,
256-expert top-8, 64-token decode) timed the same way (CUDA events, median step, L2
flushed before each step), each with its expert-GEMM pair against the measured roofline,
its routing stage's share of the forward and its own clock record.

--gpus N without a launcher starts N ranks of this script itself (torch.distributed.run
on 127.0.0.1); under a launcher --gpus must equal WORLD_SIZE.

--impl reference times the CPU oracle itself (the plain fp64 implementation the
parity tests use) on the host cores, each step a bounded sample of the workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import socket
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from moe_workloads import WORKLOADS, capacity_factor_or_none, input_recipe, make_inputs  # noqa: E402

METRIC = "MoE-layer fwd tokens/s at 1 B300; grouped-GEMM % BF16 peak; decode % HBM BW"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "mixtral_prefill"
L2_FLUSH_BYTES = 256 << 20
# A GPU-side wait (torch.cuda._sleep, in SM clock cycles: ~0.1 ms) enqueued after the L2
# flush and before each device-timed call's start event, so that the host has finished
# enqueueing the call before the event fires: device times exclude the host's enqueue
# work, which on the small layers is longer than the layer itself (e2e includes it).
HEAD_START_CYCLES = 200_000
KERNELS_PER_FORWARD = 8   # router GEMM, softmax/top-k, finalize/scan, place, row copy, GEMM1, GEMM2, combine
KERNELS_PER_EC_FORWARD = 7  # router GEMM, softmax, per-expert select, gather, GEMM1, GEMM2, combine


def forward_launches(w, fused_gather=False) -> int:
    """Our kernel launches in one top-k moe_forward of workload w: a bf16 top-1 layer whose
    expert groups fit the weights-as-M GEMMs (at most 128 rows) has no combine pass (the
    expert GEMMs write y); with fused_gather there is no row copy."""
    cap = math.ceil(w.T * w.capacity_factor / w.E) if w.capacity_factor > 0 else w.T
    fused_combine = w.k == 1 and w.dtype == "bf16" and min(cap, w.T) <= 128
    return KERNELS_PER_FORWARD - int(fused_combine) - int(bool(fused_gather))
# moe_backward: combine and gate backward, dA / dXp / router-dx GEMMs, the dx sum, dW2 / dW1 /
# dW_g GEMMs with two tail-packing kernels before each expert one, three two-kernel column sums
KERNELS_PER_BACKWARD = 19
TRAIN_METRIC = "MoE-layer fwd+bwd (training step) tokens/s at 1 B300; backward GEMMs % BF16 peak"
D_AUX = 0.01

# dram__bytes_read.sum + dram__bytes_write.sum of one moe_expert_ffn (the grouped GEMM
# pair G1 + G2) from an ncu capture: (hash of the GEMM sources that capture ran, bytes,
# how).  The 15 GB layers are captured on their reduced twins (same per-expert shapes,
# 32 or 8 experts) and scaled by the algorithmic bytes.  A figure whose hash differs from
# the current sources' (gemm_source_hash) is stale and reported as null.
NCU_TRAFFIC_BYTES = {
    "mixtral_prefill": ("cbf75181ceb343bf", 2965290752, "captured at full size"),
    "switch_capacity": ("cbf75181ceb343bf", 159500288,
                        "captured at full size (the forward's GEMMs, combine folded in)"),
    "deepseek_fine": ("cbf75181ceb343bf", 17516703744,
                      "deepseek_fine_e32 capture (1.0036 x its algorithmic bytes), scaled"),
    "decode": ("cbf75181ceb343bf", 4500414010,
               "decode_e8 capture (1.0062 x its algorithmic bytes), scaled"),
}
GEMM_SOURCES = ("sparse_mixture_experts_61_b300/csrc/gemm_tc.cu",
                "sparse_mixture_experts_61_b300/csrc/tc_pipe.cuh",
                "sparse_mixture_experts_61_b300/csrc/common.cuh")
# Configurations of the layer family reported in the default run's `workloads` map.
FAMILY = ("tiny_f32", "mixtral_prefill", "switch_capacity", "deepseek_fine", "decode")


def gemm_source_hash() -> str:
    h = hashlib.sha256()
    for rel in GEMM_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(name: str):
    """(bytes, how) of the current GEMM sources' capture for a workload, or (None, None)."""
    entry = NCU_TRAFFIC_BYTES.get(name)
    if entry is None or entry[0] != gemm_source_hash():
        return None, None
    return entry[1], entry[2]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return dict(hbm_gbs=p["hbm_gbs"], bf16_tflops=p["bf16_tflops"],
                    bf16_tflops_sustained=p.get("bf16_tflops_sustained"), source="measured")
    return dict(hbm_gbs=6400.0, bf16_tflops=1800.0, bf16_tflops_sustained=1400.0, source="fallback")


# ------------------------------------------------------------------ distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, local, backend="nccl"):
    """One process per GPU (NCCL); the gloo backend runs the same rendezvous on CPU."""
    if world > 1:
        import torch.distributed as dist
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(v: float, world: int, device: str = "cuda") -> float:
    """The slowest rank's value (timings are taken as the max over ranks)."""
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world: int, tokens_per_rank: int, slowest_ms: float) -> float:
    """Weak scaling: every rank runs its own batch; tokens of all ranks / slowest rank's time."""
    return world * tokens_per_rank / (slowest_ms / 1e3)


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampler of SM clocks and throttle reasons; keeps timestamped rows."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                    rows.append((ts, float(parts[1]), float(parts[2]), parts[4:]))
                except (ValueError, IndexError):
                    continue
            os.unlink(self.path)
        if not rows:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=[], samples=0)
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3][1:5])
                          if v.strip().lower() == "active"})
        return dict(sm_mhz=statistics.median(r[1] for r in inside),
                    sm_max_mhz=max(r[2] for r in inside), reasons=reasons, samples=len(inside))


# ------------------------------------------------------------------ oracle (CPU) timing
def oracle_tokens_step(w, host, fetch, tokens):
    """Runs the oracle's whole layer on the given tokens (a batch of its own).  Returns
    the seconds spent inside oracle calls (host copies of weights are not timed)."""
    import oracle

    cf = capacity_factor_or_none(w)
    xs = host["x"][torch.as_tensor(tokens)]
    spent = 0.0
    t = time.perf_counter()
    lg = oracle.logits(xs, host["w_gate"], host["logit_bias"])
    p = oracle.softmax(lg)
    idx = oracle.topk(lg, w.k)
    wts = oracle.gate_weights(lg, idx, w.gate)
    oracle.aux_loss(p, idx)
    disp = oracle.dispatch(idx, w.E, oracle.capacity(len(tokens), w.E, cf))
    spent += time.perf_counter() - t
    z = np.zeros((len(tokens), w.k, w.d))
    by_e = {}
    for a in range(len(tokens)):
        for j in range(w.k):
            if disp["slot_row"][a, j] >= 0:
                by_e.setdefault(int(idx[a, j]), []).append((a, j))
    for e, items in sorted(by_e.items()):
        w1, b1, w2, b2 = fetch(e)
        rows = xs[[a for a, _ in items]]
        t = time.perf_counter()
        ze = oracle.expert_rows(rows, w1, b1, w2, b2)
        spent += time.perf_counter() - t
        for q, (a, j) in enumerate(items):
            z[a, j] = ze[q]
    t = time.perf_counter()
    oracle.combine(disp["slot_row"], wts, z)
    spent += time.perf_counter() - t
    return spent


def oracle_ec_tokens_step(w, host, fetch, tokens):
    """The oracle's expert-choice layer on the given tokens as a batch of their own
    (C from the batch size).  Returns the seconds spent inside oracle calls."""
    import oracle

    xs = host["x"][torch.as_tensor(tokens)]
    spent = 0.0
    t = time.perf_counter()
    lg = oracle.logits(xs, host["w_gate"], host["logit_bias"])
    p = oracle.softmax(lg)
    C = min(len(tokens), oracle.capacity(len(tokens), w.E, w.capacity_factor))
    sel, sel_w = oracle.expert_choice(p, C)
    spent += time.perf_counter() - t
    z = np.zeros((w.E * C, w.d))
    for e in range(w.E):
        if C == 0:
            break
        w1, b1, w2, b2 = fetch(e)
        rows = xs[sel[e].tolist()]
        t = time.perf_counter()
        z[e * C:(e + 1) * C] = oracle.expert_rows(rows, w1, b1, w2, b2)
        spent += time.perf_counter() - t
    t = time.perf_counter()
    oracle.combine_expert_choice(len(tokens), sel, sel_w, z)
    spent += time.perf_counter() - t
    return spent


def tokens_step(w, host, fetch, tokens):
    if w.routing == "expert_choice":
        return oracle_ec_tokens_step(w, host, fetch, tokens)
    return oracle_tokens_step(w, host, fetch, tokens)


def host_view(inp):
    host = {"x": inp["x"].cpu(), "w_gate": inp["w_gate"].cpu(),
            "logit_bias": inp["logit_bias"].cpu() if inp["logit_bias"] is not None else None}
    cache = {}

    def fetch(e):
        if e not in cache:
            if len(cache) >= 16:
                cache.pop(next(iter(cache)))
            cache[e] = tuple(inp[n][e].cpu() for n in ("w1", "b1", "w2", "b2"))
        return cache[e]

    return host, fetch


def _oracle_rate(w, host, fetch, budget_s):
    """Tokens/s of the oracle over consecutive tokens from token 0, in growing batches,
    until about budget_s seconds of oracle work; returns (rate, tokens, seconds)."""
    done, spent, batch = 0, 0.0, 1
    while spent < budget_s and done < w.T:
        toks = list(range(done, min(w.T, done + batch)))
        spent += tokens_step(w, host, fetch, toks)
        done += len(toks)
        batch = min(batch * 2, 256)
    return done / spent, done, spent


def cpu_baseline(w, inp, budget_s=10.0, single_budget_s=6.0):
    """Oracle throughput on a bounded sample, on all host cores (the reported value)
    and on one thread."""
    import oracle

    host, fetch = host_view(inp)
    cores = oracle.num_threads()
    rate, done, spent = _oracle_rate(w, host, fetch, budget_s)
    oracle.set_num_threads(1)
    try:
        rate1, done1, spent1 = _oracle_rate(w, host, fetch, single_budget_s)
    finally:
        oracle.set_num_threads(cores)
    return dict(value=rate, unit=UNIT, cores=cores, kind="oracle",
                single_thread_value=rate1,
                sample=f"first {done} of {w.T} tokens of the workload, whole layer in fp64 "
                       f"({spent:.1f} s of oracle time on {cores} threads); single-thread "
                       f"figure over the first {done1} tokens ({spent1:.1f} s)")


# ------------------------------------------------------------------ roofline
def ffn_algorithmic(w, M, nonempty):
    s = 2 if w.dtype == "bf16" else 4
    flops = 4.0 * M * w.d * w.h
    byts = s * (2.0 * M * w.d + 2.0 * M * w.h + nonempty * (2.0 * w.d * w.h + w.h + w.d))
    return flops, byts


def roofline(w, M, nonempty, t_ffn_s, peaks):
    flops, byts = ffn_algorithmic(w, M, nonempty)
    t_tensor = flops / (peaks["bf16_tflops"] * 1e12)
    t_hbm = byts / (peaks["hbm_gbs"] * 1e9)
    traffic, traffic_how = ncu_traffic(w.name)
    if t_tensor >= t_hbm:
        achieved = flops / t_ffn_s / 1e12
        r = dict(bound="tensor", achieved=round(achieved, 1), peak=peaks["bf16_tflops"],
                 unit="TFLOP/s", frac=round(achieved / peaks["bf16_tflops"], 4))
        if peaks.get("bf16_tflops_sustained"):
            r["frac_of_sustained"] = round(achieved / peaks["bf16_tflops_sustained"], 4)
    else:
        achieved = byts / t_ffn_s / 1e9
        r = dict(bound="hbm", achieved=round(achieved, 1), peak=peaks["hbm_gbs"], unit="GB/s",
                 frac=round(achieved / peaks["hbm_gbs"], 4))
    r.update(traffic=traffic, traffic_source=traffic_how,
             kernel="grouped expert GEMM pair G1+G2 (moe_expert_ffn)",
             algorithmic_flops=flops, algorithmic_bytes=byts, peak_source=peaks["source"],
             ms=round(t_ffn_s * 1e3, 4))
    return r


# ------------------------------------------------------------------ our arm
def _median_event_ms(fn, steps, warmup, flush, stream):
    """Median CUDA-event time of fn() over `steps` calls after `warmup` calls, with L2
    flushed (a 256 MB write) and the host given a head start before every call, both
    outside the event pair."""
    ev = []
    for i in range(steps + warmup):
        flush.zero_()
        torch.cuda._sleep(HEAD_START_CYCLES)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        if i >= warmup:
            ev.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ev)


def ffn_alone(moe, w, cfg, inp, outs, C, dev):
    """Callable of the grouped expert GEMM pair alone (moe_expert_ffn) on the rows the
    layer's routing produces, plus its stage workspace.  Expert choice: the same call on
    its E groups of C rows, through a top-k configuration with capacity C (identical
    tile height and row count)."""
    i32 = dict(dtype=torch.int32, device=dev)
    ec = w.routing == "expert_choice"
    ffn_cfg = cfg
    if ec:
        ffn_cfg = moe.config(w.T, w.d, w.h, w.E, w.k, w.dtype, w.gate, w.capacity_factor)
        assert moe.moe_capacity(ffn_cfg) == C
    sws = torch.empty(moe.moe_stage_workspace_size(ffn_cfg), dtype=torch.uint8, device=dev)
    rows = w.T * w.k
    x_perm = torch.empty((rows, w.d), dtype=w.torch_dtype, device=dev)
    h_buf = torch.empty((rows, w.h), dtype=w.torch_dtype, device=dev)
    y_perm = torch.empty((rows, w.d), dtype=w.torch_dtype, device=dev)
    offsets = torch.empty((w.E + 1,), **i32)
    if ec:
        M = w.E * C
        torch.index_select(inp["x"], 0, outs["sel_token"].flatten().long(), out=x_perm[:M])
        offsets.copy_(torch.arange(w.E + 1, dtype=torch.int32, device=dev) * C)
    else:
        idx = torch.empty((w.T, w.k), **i32)
        wts = torch.empty((w.T, w.k), dtype=torch.float32, device=dev)
        slot_row = torch.empty((w.T, w.k), **i32)
        row_token = torch.empty((rows,), **i32)
        moe.moe_route(cfg, inp["x"], inp["w_gate"], inp["logit_bias"], None, idx, wts, None, None,
                      sws)
        moe.moe_dispatch(cfg, inp["x"], idx, offsets, None, slot_row, row_token, None, x_perm, sws)

    def call():
        moe.moe_expert_ffn(ffn_cfg, x_perm, offsets, inp["w1"], inp["b1"], inp["w2"], inp["b2"],
                           h_buf, y_perm, sws)
    return call, sws


def family_entry(moe, w, steps, warmup, flush, stream, dev, rank, world, peaks):
    """One configuration of the layer family: the forward's tokens/s (median of `steps`
    steps), the expert-GEMM pair alone against the roofline, the routing stage
    (moe_route with counts and balance loss) and its share of the forward, and the SM
    clocks sampled while they ran."""
    inp = make_inputs(w, seed=rank, device=str(dev))
    cfg = moe.config_from_workload(w)
    i32 = dict(dtype=torch.int32, device=dev)
    outs = dict(y=torch.empty((w.T, w.d), dtype=w.torch_dtype, device=dev),
                offsets=torch.empty((w.E + 1,), **i32), kept_counts=torch.empty((w.E,), **i32))
    ws = torch.empty(moe.moe_workspace_size(cfg), dtype=torch.uint8, device=dev)
    fwd_args = moe.forward_args(inp, outs)

    def fwd():
        moe.moe_forward(cfg, inp, outs, ws, stream, args=fwd_args)

    sws = torch.empty(moe.moe_stage_workspace_size(cfg), dtype=torch.uint8, device=dev)
    idx = torch.empty((w.T, w.k), **i32)
    wts = torch.empty((w.T, w.k), dtype=torch.float32, device=dev)
    counts = torch.empty((w.E,), **i32)
    aux = torch.empty((1,), dtype=torch.float32, device=dev)

    def route():
        moe.moe_route(cfg, inp["x"], inp["w_gate"], inp["logit_bias"], None, idx, wts, counts, aux,
                      sws)

    for _ in range(warmup):
        fwd()
    assert moe.moe_device_error(ws) == 0
    M = int(outs["offsets"][-1])
    nonempty = int((outs["kept_counts"] > 0).sum())
    ffn, fws = ffn_alone(moe, w, cfg, inp, outs, None, dev)
    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if clocks:
        clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    fwd_ms = _median_event_ms(fwd, steps, 0, flush, stream)
    ffn_ms = _median_event_ms(ffn, steps, warmup, flush, stream)
    route_ms = _median_event_ms(route, steps, warmup, flush, stream)
    t1 = time.time()
    if clocks:
        clocks.stop()
    assert moe.moe_device_error(ws) == 0 and moe.moe_device_error(fws) == 0
    assert moe.moe_device_error(sws) == 0
    fwd_ms = allreduce_max(fwd_ms, world)
    ffn_ms = allreduce_max(ffn_ms, world)
    route_ms = allreduce_max(route_ms, world)
    entry = {
        "tokens_per_s": round(replica_throughput(world, w.T, fwd_ms), 1),
        "ms_per_step": round(fwd_ms, 4),
        "kept_rows": M, "nonempty_experts": nonempty,
        "routing_ms": round(route_ms, 4), "routing_share": round(route_ms / fwd_ms, 4),
        "inputs": input_recipe(w),
        "clocks": clocks.summary(t0, t1) if clocks else None,
    }
    if w.dtype == "bf16":
        r = roofline(w, M, nonempty, ffn_ms / 1e3, peaks)
        flops, byts = r["algorithmic_flops"], r["algorithmic_bytes"]
        r["frac_of_hbm"] = round(byts / (ffn_ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4)
        r["frac_of_bf16_burst"] = round(flops / (ffn_ms / 1e3) / 1e12 / peaks["bf16_tflops"], 4)
        if peaks.get("bf16_tflops_sustained"):
            r["frac_of_bf16_sustained"] = round(
                flops / (ffn_ms / 1e3) / 1e12 / peaks["bf16_tflops_sustained"], 4)
        entry["roofline"] = r
    else:
        entry["gemm_pair_ms"] = round(ffn_ms, 4)
        entry["roofline"] = {"bound": "latency (fp32 SIMT GEMMs)", "ms": round(ffn_ms, 4)}
    return entry


def run_ours(args, world, rank, local):
    import sparse_mixture_experts_61_b300 as moe

    moe.lib()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = WORKLOADS[args.workload]
    inp = make_inputs(w, seed=rank, device=str(dev))
    cfg = moe.config_from_workload(w, fused_gather=int(args.fused_gather))
    i32 = dict(dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    ec = w.routing == "expert_choice"
    if ec:
        C = moe.moe_expert_choice_capacity(cfg)
        outs = dict(y=torch.empty((w.T, w.d), dtype=w.torch_dtype, device=dev),
                    sel_token=torch.empty((w.E, C), **i32))
        ws = torch.empty(moe.moe_expert_choice_workspace_size(cfg), dtype=torch.uint8, device=dev)
        ec_args = moe.expert_choice_args(inp, outs)

        def step():
            moe.moe_expert_choice_forward(cfg, inp, outs, ws, stream, args=ec_args)
    else:
        outs = dict(y=torch.empty((w.T, w.d), dtype=w.torch_dtype, device=dev),
                    offsets=torch.empty((w.E + 1,), **i32), kept_counts=torch.empty((w.E,), **i32))
        ws = torch.empty(moe.moe_workspace_size(cfg), dtype=torch.uint8, device=dev)
        fwd_args = moe.forward_args(inp, outs)

        def step():
            moe.moe_forward(cfg, inp, outs, ws, stream, args=fwd_args)

    for _ in range(args.warmup):
        step()
    assert moe.moe_device_error(ws) == 0
    if ec:
        M, nonempty = w.E * C, (w.E if C > 0 else 0)
    else:
        M = int(outs["offsets"][-1])
        nonempty = int((outs["kept_counts"] > 0).sum())

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if clocks:
        clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(args.steps):
        flush.zero_()
        torch.cuda._sleep(HEAD_START_CYCLES)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t1 = time.time()
    if clocks:
        clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    # tokens/s is T over the median step time; the mean is reported beside it.
    med_ms = allreduce_max(statistics.median(step_ms), world)
    mean_ms = allreduce_max(statistics.fmean(step_ms), world)
    assert moe.moe_device_error(ws) == 0

    # The grouped expert GEMM pair alone (same rows, same stream), for the roofline.
    ffn, sws = ffn_alone(moe, w, cfg, inp, outs, C if ec else None, dev)
    if ec:
        assert M <= w.T * w.k
    t_ffn = _median_event_ms(ffn, args.steps, args.warmup, flush, stream) / 1e3
    assert moe.moe_device_error(sws) == 0
    del ffn, sws

    # End to end with x and y in (pinned) host memory.  Headline: moe_forward_host, the
    # C call that takes host batches and overlaps their copies with the layer, over
    # `steps` batches after a `warmup`-batch call.  Beside it: one step at a time
    # (copy in, the layer, copy out, no overlap).
    routing = "expert_choice" if ec else "topk"
    n_bufs = min(args.steps, 4)
    xs = [inp["x"].cpu().pin_memory() for _ in range(n_bufs)]
    ys = [torch.empty((w.T, w.d), dtype=w.torch_dtype).pin_memory() for _ in range(n_bufs)]
    hws = torch.empty(moe.moe_forward_host_workspace_size(cfg, routing), dtype=torch.uint8,
                      device=dev)
    weights = {n: inp[n] for n in moe.WEIGHTS}

    def host_call(n):
        moe.moe_forward_host(cfg, weights, [xs[i % n_bufs] for i in range(n)],
                             [ys[i % n_bufs] for i in range(n)], hws, stream, routing=routing)

    host_call(args.warmup)
    e2e_a, e2e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e2e_a.record(stream)
    host_call(args.steps)
    e2e_b.record(stream)
    torch.cuda.synchronize()
    assert moe.moe_device_error(hws) == 0
    if not torch.equal(ys[(args.steps - 1) % n_bufs].to(dev), outs["y"]):
        raise RuntimeError("moe_forward_host returned a y that differs from moe_forward's")
    e2e_ms = allreduce_max(e2e_a.elapsed_time(e2e_b) / args.steps, world)
    del hws

    x_host, y_host, x_dev = xs[0], ys[0], inp["x"]
    ser_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    for i in range(args.steps + args.warmup):
        flush.zero_()
        if i >= args.warmup:
            ser_ev[i - args.warmup][0].record(stream)
        x_dev.copy_(x_host, non_blocking=True)
        step()
        y_host.copy_(outs["y"], non_blocking=True)
        if i >= args.warmup:
            ser_ev[i - args.warmup][1].record(stream)
    torch.cuda.synchronize()
    ser_ms = allreduce_max(statistics.median(a.elapsed_time(b) for a, b in ser_ev), world)

    if rank != 0:
        return None
    peaks = load_peaks()
    line = {
        "metric": METRIC,
        "value": round(replica_throughput(world, w.T, med_ms), 1),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(med_ms, 4),
        "ms_per_step_mean": round(mean_ms, 4),
        "timing": "median of the timed steps (CUDA events on the launching stream)",
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "d": w.d, "h": w.h, "E": w.E, "k": w.k,
                   "routing": w.routing,
                   "gate": ["topk_softmax", "softmax_topk_renorm"][w.gate],
                   "capacity_factor": w.capacity_factor, "kept_rows": M,
                   "nonempty_experts": nonempty, "inputs": input_recipe(w),
                   "l2": "flushed before every timed step (256 MB write outside the event pair)",
                   "fused_gather": bool(args.fused_gather),
                   "parallelism": f"replicas x{world} (token-parallel, no collective)"},
        "roofline": roofline(w, M, nonempty, t_ffn, peaks),
        "e2e": {"value": round(replica_throughput(world, w.T, e2e_ms), 1), "unit": UNIT,
                "h2d_bytes_per_step": x_host.numel() * x_host.element_size(),
                "d2h_bytes_per_step": y_host.numel() * y_host.element_size(),
                "ms_per_step": round(e2e_ms, 4),
                "call": f"moe_forward_host over {args.steps} pinned host batches (routing "
                        f"{routing}): each batch's x copied in and y copied out, overlapped "
                        "with the neighbouring batches' layers; no L2 flush between batches",
                "serial_value": round(replica_throughput(world, w.T, ser_ms), 1),
                "serial": "per step: x copied in, moe_forward, y copied out, no overlap "
                          "(L2 flushed before each step)"},
        "gpu_launches": (KERNELS_PER_EC_FORWARD if ec else
                         forward_launches(w, args.fused_gather)) * args.steps,
        "clocks": clocks.summary(t0, t1) if clocks else None,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, inp)
    return line


def run_family(args, world, rank, local, line):
    """Adds the `workloads` map (every configuration of the layer family) to the line."""
    import sparse_mixture_experts_61_b300 as moe

    dev = torch.device("cuda", local)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    peaks = load_peaks()
    fam = {}
    for name in FAMILY:
        torch.cuda.empty_cache()
        fam[name] = family_entry(moe, WORKLOADS[name], args.steps, args.warmup, flush, stream, dev,
                                 rank, world, peaks)
    if line is not None:
        line["workloads"] = fam
    return line


# ------------------------------------------------------------------ training step
def run_train(args, world, rank, local):
    """Forward (keeping its activations) + backward of the layer per step."""
    import sparse_mixture_experts_61_b300 as moe

    moe.lib()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = WORKLOADS[args.workload]
    if w.routing != "topk" or w.dtype != "bf16":
        raise SystemExit("--pass train needs a bf16 top-k workload")
    inp = make_inputs(w, seed=rank, device=str(dev))
    cfg = moe.config_from_workload(w)
    T, d, h, E, k = w.T, w.d, w.h, w.E, w.k
    rows = T * k
    i32 = dict(dtype=torch.int32, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    bf = dict(dtype=torch.bfloat16, device=dev)
    outs = dict(y=torch.empty((T, d), **bf), logits=torch.empty((T, E), **f32),
                topk_idx=torch.empty((T, k), **i32), topk_w=torch.empty((T, k), **f32),
                counts=torch.empty((E,), **i32), aux_loss=torch.empty((1,), **f32),
                offsets=torch.empty((E + 1,), **i32), kept_counts=torch.empty((E,), **i32),
                slot_row=torch.empty((T, k), **i32), x_perm=torch.empty((rows, d), **bf),
                h_act=torch.empty((rows, h), **bf), y_perm=torch.empty((rows, d), **bf),
                h_pre=torch.empty((rows, h), **bf))
    grads = dict(dx=torch.empty((T, d), **bf), dw_gate=torch.empty((E, d), **f32),
                 dlogit_bias=torch.empty((E,), **f32), dw1=torch.empty((E, h, d), **bf),
                 db1=torch.empty((E, h), **f32), dw2=torch.empty((E, d, h), **bf),
                 db2=torch.empty((E, d), **f32))
    gen = torch.Generator(device=dev)
    gen.manual_seed(1000 + rank)
    dy = torch.randn((T, d), generator=gen, device=dev).to(torch.bfloat16)
    ws = torch.empty(moe.moe_workspace_size(cfg), dtype=torch.uint8, device=dev)
    bws = torch.empty(moe.moe_backward_workspace_size(cfg), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    fwd_args = moe.forward_args(inp, outs)
    bin_ = dict(dy=dy, x=inp["x"], w_gate=inp["w_gate"], w1=inp["w1"], w2=inp["w2"])
    for n in ("logits", "topk_idx", "topk_w", "counts", "offsets", "slot_row", "x_perm", "h_pre",
              "h_act", "y_perm"):
        bin_[n] = outs[n]
    bwd_args = moe.backward_args(bin_, grads, D_AUX)

    def fwd():
        moe.moe_forward(cfg, inp, outs, ws, stream, args=fwd_args)

    def bwd():
        moe.moe_backward(cfg, bin_, grads, D_AUX, bws, stream, args=bwd_args)

    for _ in range(args.warmup):
        fwd()
        bwd()
    assert moe.moe_device_error(ws) == 0 and moe.moe_device_error(bws) == 0
    M = int(outs["offsets"][-1])
    nonempty = int((outs["kept_counts"] > 0).sum())
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if clocks:
        clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(args.steps):
        flush.zero_()
        torch.cuda._sleep(HEAD_START_CYCLES)
        ev[i][0].record(stream)
        fwd()
        ev[i][1].record(stream)
        bwd()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t1 = time.time()
    if clocks:
        clocks.stop()
    step_ms = allreduce_max(statistics.median(e[0].elapsed_time(e[2]) for e in ev), world)
    bwd_ms = statistics.median(e[1].elapsed_time(e[2]) for e in ev)
    assert moe.moe_device_error(bws) == 0
    if rank != 0:
        return None
    peaks = load_peaks()
    # Backward tensor-core work: four expert GEMMs of 2*M*d*h flops each, plus the router's
    # data and weight gradients (2 * 2*T*E*d).
    flops = 4 * 2.0 * M * d * h + 2 * 2.0 * T * E * d
    achieved = flops / (bwd_ms / 1e3) / 1e12
    return {
        "metric": TRAIN_METRIC,
        "value": round(replica_throughput(world, T, step_ms), 1),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic",
        "config": {"workload": w.name, "T": T, "d": d, "h": h, "E": E, "k": k,
                   "gate": ["topk_softmax", "softmax_topk_renorm"][w.gate],
                   "capacity_factor": w.capacity_factor, "kept_rows": M,
                   "nonempty_experts": nonempty, "d_aux": D_AUX, "inputs": input_recipe(w),
                   "l2": "flushed before every timed step (256 MB write outside the event pair)",
                   "parallelism": f"replicas x{world} (token-parallel, no collective)"},
        "backward_ms": round(bwd_ms, 4),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1),
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(achieved / peaks["bf16_tflops"], 4), "traffic": None,
                     "kernel": "moe_backward (all backward kernels; GEMM flops only)",
                     "algorithmic_flops": flops, "peak_source": peaks["source"],
                     "ms": round(bwd_ms, 4)},
        "gpu_launches": (KERNELS_PER_FORWARD + KERNELS_PER_BACKWARD) * args.steps,
        "clocks": clocks.summary(t0, t1) if clocks else None,
    }


# ------------------------------------------------------------------ reference arm
def run_reference(args, world, rank, local):
    """The CPU oracle on rank 0; under N ranks the others join a gloo group, wait for
    rank 0 at a barrier and return without work."""
    if world > 1 and args is not None:
        import torch.distributed as dist
        dist_init(world, local, backend="gloo")
        try:
            return _reference_line(args, world) if rank == 0 else None
        finally:
            dist.barrier()
            dist.destroy_process_group()
    if rank != 0:
        return None
    return _reference_line(args, world)


def _reference_line(args, world):
    import oracle

    w = WORKLOADS[args.workload]
    device = "cuda" if torch.cuda.is_available() else "cpu"
    gen_dev = device if w.d * w.h * w.E > (1 << 27) else "cpu"
    inp = make_inputs(w, seed=0, device=gen_dev)
    host, fetch = host_view(inp)
    # Size one step's sample from the cost of one token so the whole run stays short.
    probe = tokens_step(w, host, fetch, [0])
    per_token = max(probe, 1e-4)
    total_steps = args.steps + args.warmup
    target = max(0.05, min(5.0, 150.0 / max(total_steps, 1)))
    S = int(max(1, min(w.T, target / per_token)))
    times = []
    for i in range(total_steps):
        start = (i * S) % w.T
        toks = [(start + q) % w.T for q in range(S)]
        t = tokens_step(w, host, fetch, toks)
        if i >= args.warmup:
            times.append(t)
    med_s = statistics.median(times) if times else probe
    value = S / med_s
    sample = f"{S} consecutive tokens per step of the {w.T}-token workload, whole layer in fp64"
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 3),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(med_s * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "d": w.d, "h": w.h, "E": w.E, "k": w.k,
                   "routing": w.routing,
                   "gate": ["topk_softmax", "softmax_topk_renorm"][w.gate],
                   "capacity_factor": w.capacity_factor, "inputs": input_recipe(w)},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the timed CPU-oracle sample (for quick runs)")
    ap.add_argument("--pass", dest="pass_", default="forward", choices=["forward", "train"],
                    help="forward (default) or train: forward + backward of the layer per step")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the `workloads` map of the other layer configurations")
    ap.add_argument("--fused-gather", action="store_true",
                    help="time the forward with cfg.fused_gather (GEMM1 gathers its token rows "
                         "from x; no expert-ordered copy in the workspace)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.gpus < 1:
        ap.error("--gpus must be at least 1")
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        # One process per GPU: start N ranks of this script and return their status.
        with socket.socket() as s:
            s.bind(("127.0.0.1", 0))
            port = s.getsockname()[1]
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
               f"--nproc-per-node={args.gpus}", "--master-addr", "127.0.0.1", "--master-port",
               str(port), os.path.abspath(__file__), *sys.argv[1:]]
        sys.exit(subprocess.call(cmd))
    world, rank, local = dist_env()
    if world != args.gpus:
        ap.error(f"--gpus {args.gpus} does not match WORLD_SIZE={world}")
    if args.impl == "reference":
        line = run_reference(args, world, rank, local)
    else:
        dist_init(world, local)
        if args.pass_ == "train":
            line = run_train(args, world, rank, local)
        else:
            line = run_ours(args, world, rank, local)
            if args.workload == DEFAULT_WORKLOAD and not args.no_workloads and not args.fused_gather:
                line = run_family(args, world, rank, local, line)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
