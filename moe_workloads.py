"""Seeded synthetic workloads for the top-k MoE FFN forward.

This module is shared by the CUDA-path tests, the oracle tests, ``bench.py`` and
``__graft_entry__.smoke()``.  It holds the workload table and the seeded input
generators only: no routing, expert or combine arithmetic lives here, so neither
side of a parity check can borrow the other's maths through it.

The five workloads are the ones the MoE pages' discussion is built around (an
8-expert top-2 layer, a 128-expert Switch-style top-1 layer with capacity, a
256-expert top-8 fine-grained layer, a decode-sized batch and a tiny fp32 layer).

Distributions.  ``N(0, s)`` is read as mean 0 and *variance* s, so weights drawn
``N(0, 1/fan_in)`` get standard deviation ``1/sqrt(fan_in)`` and biases drawn
``N(0, 0.01)`` get standard deviation 0.1.  Every tensor is drawn in fp32 from one
``torch.Generator`` seeded with ``seed`` in the fixed order x, W_g, W1, b1, W2, b2,
logit bias, then rounded (round-to-nearest-even) to the workload dtype.  The logit
bias is always fp32.

Large weight tensors are drawn one expert at a time so that peak temporary memory
stays at one expert's fp32 copy.  ``device`` selects where the generator runs: CPU
draws are reproducible on any machine; CUDA draws are reproducible for a given GPU
model and are used for the multi-GB workloads.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

GATE_TOPK_SOFTMAX = 0          # G(x) = softmax(TopK(x . W_g))
GATE_SOFTMAX_TOPK_RENORM = 1   # p = softmax(x . W_g); keep top-k of p; divide by their sum


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    h: int
    E: int
    k: int
    dtype: str                 # "f32" or "bf16"
    gate: int                  # GATE_*
    capacity_factor: float     # <= 0: no capacity limit
    x_std: float = 1.0
    bias_std: float = 0.0      # expert biases b1, b2 (0 -> zeros)
    logit_bias: str = "none"   # "none" | "zipf" | "normal1.5"
    wg_std: Optional[float] = None   # default 1/sqrt(d)
    routing: str = "topk"      # "topk" (tokens choose k experts) | "expert_choice"

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads, in the order the performance discussion lists them.
WORKLOADS = {
    # Tiny fp32 layer: softmax-then-topk-then-renormalise, no capacity, biases N(0, 0.01).
    "tiny_f32": Workload("tiny_f32", T=256, d=128, h=256, E=8, k=2, dtype="f32",
                         gate=GATE_SOFTMAX_TOPK_RENORM, capacity_factor=0.0, bias_std=0.1),
    # 8-expert top-2 prefill (Mixtral-shaped sizes), G = softmax(TopK(.)), no drop.
    "mixtral_prefill": Workload("mixtral_prefill", T=4096, d=4096, h=14336, E=8, k=2, dtype="bf16",
                                gate=GATE_TOPK_SOFTMAX, capacity_factor=0.0),
    # 128-expert Switch-style top-1 with capacity factor 1.25 and a Zipf-skewing logit bias.
    "switch_capacity": Workload("switch_capacity", T=8192, d=1024, h=4096, E=128, k=1, dtype="bf16",
                                gate=GATE_SOFTMAX_TOPK_RENORM, capacity_factor=1.25, logit_bias="zipf"),
    # 256-expert top-8 fine-grained routing (DeepSeek-V3-shaped sizes), softmax-topk-renormalise.
    "deepseek_fine": Workload("deepseek_fine", T=8192, d=7168, h=2048, E=256, k=8, dtype="bf16",
                              gate=GATE_SOFTMAX_TOPK_RENORM, capacity_factor=0.0),
    # Decode-sized batch: 64 tokens, 64 experts, top-2, logit bias ~ N(0, 1.5) skews the load.
    "decode": Workload("decode", T=64, d=4096, h=14336, E=64, k=2, dtype="bf16",
                       gate=GATE_TOPK_SOFTMAX, capacity_factor=0.0, logit_bias="normal1.5"),
}

# Same per-expert shape as the 256-expert workload (d=7168, h=2048, top-8, ~256 rows
# per expert) with 32 experts and 1024 tokens: 1.9 GB of weights, small enough for
# multi-pass profiler captures while keeping the weights far larger than L2.
WORKLOADS["deepseek_fine_e32"] = WORKLOADS["deepseek_fine"].scaled(name="deepseek_fine_e32",
                                                                  T=1024, E=32)
# The decode layer's shapes (64 tokens, d=4096, h=14336, top-2, skewing logit bias) with 8
# experts: 1.9 GB of weights, for profiler captures of the decode-sized kernels.
WORKLOADS["decode_e8"] = WORKLOADS["decode"].scaled(name="decode_e8", E=8)

# Expert-choice routing over the same layer shapes: each expert takes C =
# ceil(T * capacity_factor / E) tokens.  A capacity factor of k gives the top-k layer's
# number of expert rows (T*k), so the expert FFN does the same work as its top-k twin.
WORKLOADS["mixtral_prefill_ec"] = WORKLOADS["mixtral_prefill"].scaled(
    name="mixtral_prefill_ec", routing="expert_choice", capacity_factor=2.0)
WORKLOADS["deepseek_fine_ec"] = WORKLOADS["deepseek_fine"].scaled(
    name="deepseek_fine_ec", routing="expert_choice", capacity_factor=8.0)

# Reduced-size variants with each workload's structure (expert count, k, gate, capacity,
# bias recipe) that the oracle evaluates in full in seconds, while still spanning several
# 128-row tiles, several 256-column tiles and a ragged tail.
PARITY_WORKLOADS = {
    "tiny_f32": WORKLOADS["tiny_f32"],
    "mixtral_prefill": WORKLOADS["mixtral_prefill"].scaled(T=777, d=512, h=1024),
    "switch_capacity": WORKLOADS["switch_capacity"].scaled(T=2048, d=256, h=512),
    "deepseek_fine": WORKLOADS["deepseek_fine"].scaled(T=389, d=512, h=256),
    "decode": WORKLOADS["decode"].scaled(d=512, h=768),
}

# Expert-choice parity cases: several capacities (C from 1 row to every token), both
# dtypes, 8 to 256 experts, token counts with a ragged tail.
EC_PARITY_WORKLOADS = {
    "tiny_f32_ec": WORKLOADS["tiny_f32"].scaled(name="tiny_f32_ec", routing="expert_choice",
                                                capacity_factor=2.0),
    "mixtral_prefill_ec": WORKLOADS["mixtral_prefill_ec"].scaled(T=777, d=512, h=1024),
    "switch_ec": WORKLOADS["switch_capacity"].scaled(name="switch_ec", routing="expert_choice",
                                                     T=2048, d=256, h=512, capacity_factor=1.25),
    "deepseek_fine_ec": WORKLOADS["deepseek_fine_ec"].scaled(T=389, d=512, h=256),
    "decode_ec": WORKLOADS["decode"].scaled(name="decode_ec", routing="expert_choice", d=512,
                                            h=768, capacity_factor=1.0),
    # C = 544 rows per expert: the 256-row tile kernel (two full tiles and a half tile).
    "wide_ec": WORKLOADS["mixtral_prefill_ec"].scaled(name="wide_ec", T=1088, E=4, d=256,
                                                       h=512),
}


def capacity_factor_or_none(w: Workload):
    return w.capacity_factor if w.capacity_factor > 0 else None


def _randn(gen, shape, std, device):
    t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


def _draw_stacked(gen, E, rows, cols, std, dtype, device, out_device):
    """Draw E matrices [rows, cols] one at a time (bounded fp32 temporaries)."""
    out = torch.empty((E, rows, cols), dtype=dtype, device=out_device)
    for e in range(E):
        out[e].copy_(_randn(gen, (rows, cols), std, device).to(dtype))
    return out


def make_inputs(w: Workload, seed: int = 0, device: str = "cpu", out_device: Optional[str] = None):
    """Return a dict of the workload's input tensors, drawn in the documented order.

    Keys: x [T,d], w_gate [E,d], w1 [E,h,d], b1 [E,h], w2 [E,d,h], b2 [E,d] (all in the
    workload dtype) and logit_bias [E] fp32 or None.  Weights use the ``nn.Linear``
    orientation [out_features, in_features].
    """
    out_device = out_device or device
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    dt = w.torch_dtype
    x = _randn(gen, (w.T, w.d), w.x_std, device).to(dt).to(out_device)
    wg_std = w.wg_std if w.wg_std is not None else 1.0 / math.sqrt(w.d)
    w_gate = _randn(gen, (w.E, w.d), wg_std, device).to(dt).to(out_device)
    w1 = _draw_stacked(gen, w.E, w.h, w.d, 1.0 / math.sqrt(w.d), dt, device, out_device)
    if w.bias_std > 0:
        b1 = _randn(gen, (w.E, w.h), w.bias_std, device).to(dt).to(out_device)
    else:
        b1 = torch.zeros((w.E, w.h), dtype=dt, device=out_device)
    w2 = _draw_stacked(gen, w.E, w.d, w.h, 1.0 / math.sqrt(w.h), dt, device, out_device)
    if w.bias_std > 0:
        b2 = _randn(gen, (w.E, w.d), w.bias_std, device).to(dt).to(out_device)
    else:
        b2 = torch.zeros((w.E, w.d), dtype=dt, device=out_device)
    if w.logit_bias == "none":
        logit_bias = None
    elif w.logit_bias == "zipf":
        # b_e = 2.0 * log(1 / (e+1)^1.1) with the natural logarithm.
        e = torch.arange(w.E, dtype=torch.float64)
        logit_bias = (2.0 * torch.log(1.0 / (e + 1.0) ** 1.1)).to(torch.float32).to(out_device)
    elif w.logit_bias == "normal1.5":
        logit_bias = _randn(gen, (w.E,), math.sqrt(1.5), device).to(out_device)
    else:
        raise ValueError(f"unknown logit bias recipe {w.logit_bias!r}")
    return dict(x=x, w_gate=w_gate, w1=w1, b1=b1, w2=w2, b2=b2, logit_bias=logit_bias)


def input_recipe(w: Workload) -> str:
    """One-line description of the input recipe, for reports."""
    lb = {"none": "no logit bias", "zipf": "logit bias b_e=2.0*ln(1/(e+1)^1.1)",
          "normal1.5": "logit bias ~N(0,1.5) (std sqrt(1.5))"}[w.logit_bias]
    bias = f"biases ~N(0,{w.bias_std**2:g})" if w.bias_std > 0 else "zero biases"
    head = (f"T={w.T} d={w.d} h={w.h} E={w.E} k={w.k} {w.dtype} gate={w.gate} "
            if w.routing == "topk" else
            f"expert choice T={w.T} d={w.d} h={w.h} E={w.E} {w.dtype} ")
    return head + f"cf={w.capacity_factor:g}; x~N(0,1), weights ~N(0,1/fan_in), {bias}, {lb}"
