"""moe_forward_host: batches in host memory, copies overlapped with the layer.

Every batch's y must be bitwise the y of moe_forward (or moe_expert_choice_forward)
on the same x through the same workspace layout, and one batch is checked against
the oracle as well.  Covers both routings, bf16 and fp32, page-locked and pageable
host buffers, a single batch, more batches than the two device slots, empty batches
and device flags raised by an early batch surviving the later ones; and both ways
the call runs batches: overlapped on three streams (the 777 x 512 and 2048 x 256
bf16 cases, at least 256 KiB of x per batch) and in order on one stream (one batch,
or the 256 x 128 fp32 and 64 x 64 cases).
"""

import numpy as np
import pytest
import torch

import moe_testlib as tl
import oracle
import sparse_mixture_experts_61_b300 as moe
from moe_workloads import PARITY_WORKLOADS, Workload, capacity_factor_or_none, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_mixture_experts_61_b300 import build
    build.build()
    moe.lib()


def batches(w, n, pinned=True):
    """n seeded x batches (seeds 11, 12, ...) sharing the weights of seed 0."""
    weights = tl.to_device({k: v for k, v in make_inputs(w, seed=0).items() if k != "x"})
    xs = [make_inputs(w, seed=11 + i)["x"] for i in range(n)]
    if pinned:
        xs = [x.pin_memory() for x in xs]
    ys = [torch.full_like(x, float("nan")) for x in xs]
    if pinned:
        ys = [y.pin_memory() for y in ys]
    return weights, xs, ys


def device_forward(w, cfg, weights, x, routing):
    """y of the single-batch entry point on the same x."""
    dev = dict(weights, x=x.cuda())
    y = torch.empty((w.T, w.d), dtype=w.torch_dtype, device="cuda")
    aux = torch.empty((1,), dtype=torch.float32, device="cuda")
    if routing == "topk":
        ws = tl.poisoned_workspace(moe.moe_workspace_size(cfg))
        moe.moe_forward(cfg, dev, dict(y=y, aux_loss=aux), ws)
    else:
        ws = tl.poisoned_workspace(moe.moe_expert_choice_workspace_size(cfg))
        moe.moe_expert_choice_forward(cfg, dev, dict(y=y), ws)
    assert moe.moe_device_error(ws) == 0
    return y.cpu(), float(aux.cpu()[0])


@pytest.mark.parametrize("name,n,pinned", [
    ("mixtral_prefill", 5, True),
    ("switch_capacity", 3, True),
    ("tiny_f32", 4, False),
    ("deepseek_fine", 1, True),
])
def test_host_batches_match_device_forward(name, n, pinned):
    w = PARITY_WORKLOADS[name]
    cfg = moe.config_from_workload(w)
    weights, xs, ys = batches(w, n, pinned)
    aux = torch.full((n,), float("nan"), dtype=torch.float32)
    ws = tl.poisoned_workspace(moe.moe_forward_host_workspace_size(cfg))
    moe.moe_forward_host(cfg, weights, xs, ys, ws, aux_loss=aux)
    assert moe.moe_device_error(ws) == 0
    for i in range(n):
        y_ref, aux_ref = device_forward(w, cfg, weights, xs[i], "topk")
        assert torch.equal(ys[i], y_ref), (name, i)
        assert float(aux[i]) == aux_ref, (name, i)
    # the last batch against the oracle, on the routing of the GPU's fp32 logits
    inp = dict(tl.to_host(weights), x=xs[-1])
    r = tl.run_forward(w, tl.to_device(inp))
    assert r["flags"] == 0
    g = tl.host(r["outs"])
    ref = oracle.routed_reference(None, w.k, w.gate, capacity_factor_or_none(w), g["logits"])
    np.testing.assert_array_equal(g["slot_row"], ref["slot_row"])
    y_ref = tl.y_on_routing(inp, ref["idx"], ref["slot_row"], ref["w"])
    assert tl.max_rel_err(ys[-1].float().numpy(), y_ref) <= tl.TOL_Y[w.dtype]


@pytest.mark.parametrize("cf,n", [(2.0, 4), (0.7, 1)])
def test_host_batches_expert_choice(cf, n):
    w = PARITY_WORKLOADS["mixtral_prefill"].scaled(routing="expert_choice", capacity_factor=cf)
    cfg = moe.config_from_workload(w)
    weights, xs, ys = batches(w, n)
    ws = tl.poisoned_workspace(moe.moe_forward_host_workspace_size(cfg, "expert_choice"))
    moe.moe_forward_host(cfg, weights, xs, ys, ws, routing="expert_choice")
    assert moe.moe_device_error(ws) == 0
    for i in range(n):
        y_ref, _ = device_forward(w, cfg, weights, xs[i], "expert_choice")
        assert torch.equal(ys[i], y_ref), i
    # the last batch against the oracle, selecting on the GPU's fp32 probabilities
    inp = dict(tl.to_host(weights), x=xs[-1])
    C = moe.moe_expert_choice_capacity(cfg)
    f32 = dict(dtype=torch.float32, device="cuda")
    outs = dict(y=torch.empty((w.T, w.d), dtype=w.torch_dtype, device="cuda"),
                probs=torch.empty((w.T, w.E), **f32))
    ws1 = tl.poisoned_workspace(moe.moe_expert_choice_workspace_size(cfg))
    moe.moe_expert_choice_forward(cfg, tl.to_device(inp), outs, ws1)
    assert moe.moe_device_error(ws1) == 0
    p = outs["probs"].cpu().numpy().astype(np.float64)
    tok, _ = oracle.expert_choice(p, C)
    p_ref = oracle.softmax(oracle.logits(inp["x"], inp["w_gate"], inp["logit_bias"]))
    w_ref = np.stack([p_ref[tok[e], e] for e in range(w.E)])
    z = np.zeros((w.E * C, w.d))
    for e in range(w.E):
        z[e * C:(e + 1) * C] = oracle.expert_rows(inp["x"][tok[e].tolist()], inp["w1"][e],
                                                  inp["b1"][e], inp["w2"][e], inp["b2"][e])
    y_ref = oracle.combine_expert_choice(w.T, tok, w_ref, z)
    assert tl.max_rel_err(ys[-1].float().numpy(), y_ref) <= tl.TOL_Y[w.dtype]


def test_host_batches_reuse_buffers_in_order():
    """The same host buffers named several times: the copies keep batch order, so each
    y buffer ends with its last batch's result."""
    w = PARITY_WORKLOADS["mixtral_prefill"]
    cfg = moe.config_from_workload(w)
    weights, xs, ys = batches(w, 2)
    seq_x = [xs[0], xs[1], xs[1], xs[0], xs[1]]
    seq_y = [ys[0], ys[1], ys[0], ys[1], ys[0]]
    ws = tl.poisoned_workspace(moe.moe_forward_host_workspace_size(cfg))
    moe.moe_forward_host(cfg, weights, seq_x, seq_y, ws)
    assert moe.moe_device_error(ws) == 0
    y0, _ = device_forward(w, cfg, weights, xs[0], "topk")
    y1, _ = device_forward(w, cfg, weights, xs[1], "topk")
    assert torch.equal(ys[0], y1)   # batch 4 (x1) was the last into ys[0]
    assert torch.equal(ys[1], y0)   # batch 3 (x0) was the last into ys[1]


def test_host_batches_empty():
    w = Workload("empty", T=0, d=64, h=128, E=8, k=2, dtype="bf16", gate=0, capacity_factor=0.0)
    cfg = moe.config_from_workload(w)
    weights = tl.to_device({k: v for k, v in make_inputs(w, seed=0).items() if k != "x"})
    aux = torch.full((3,), float("nan"), dtype=torch.float32)
    ws = tl.poisoned_workspace(moe.moe_forward_host_workspace_size(cfg))
    empty = torch.empty((0, 64), dtype=torch.bfloat16)
    moe.moe_forward_host(cfg, weights, [empty] * 3, [empty] * 3, ws, aux_loss=aux)
    assert moe.moe_device_error(ws) == 0
    assert torch.equal(aux, torch.zeros(3))


def test_host_batches_keep_an_early_flag():
    """A non-finite logit in batch 0 stays flagged after batches 1 and 2 ran clean."""
    w = Workload("nanb", T=64, d=64, h=64, E=8, k=2, dtype="bf16", gate=0, capacity_factor=0)
    cfg = moe.config_from_workload(w)
    weights, xs, ys = batches(w, 3)
    xs[0][7, 3] = float("nan")
    ws = tl.poisoned_workspace(moe.moe_forward_host_workspace_size(cfg))
    moe.moe_forward_host(cfg, weights, xs, ys, ws)
    assert moe.moe_device_error(ws) & moe.MOE_DEVERR_NONFINITE
    for i in (1, 2):
        y_ref, _ = device_forward(w, cfg, weights, xs[i], "topk")
        assert torch.equal(ys[i], y_ref), i
