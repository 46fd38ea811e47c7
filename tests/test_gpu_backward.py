"""Parity of the layer's backward (moe_backward through the C ABI) with the CPU oracle.

The forward runs first and keeps its activations (Xp, H, Yp and the pre-activation A)
in caller buffers; the backward takes them with a seeded dy and a non-zero balance-loss
gradient.  The oracle's backward, itself pinned by central differences of its fp64
forward, runs on the GPU's own fp32 logits (so both sides take the same routing
decisions) and every gradient is compared element by element.
"""

import numpy as np
import pytest
import torch

import moe_testlib as tl
import oracle
import sparse_mixture_experts_61_b300 as moe
from moe_workloads import PARITY_WORKLOADS, Workload, capacity_factor_or_none, make_inputs

pytestmark = pytest.mark.gpu

D_AUX = 0.05
# max |dg - ref| / max |ref| per gradient.  dYp, dA, dXp and dl are rounded to bf16
# before the next contraction (2^-9 each) and dx, dW1, dW2 once more on output, on top
# of the forward's own bf16 roundings of Yp and H that enter dw and dW2: about four
# roundings of 2^-9 plus fp32 accumulation; measured 1.6e-3 to 5.3e-3.
TOL_GRAD = 1.5e-2
BF16_NAMES = [n for n, w in PARITY_WORKLOADS.items() if w.dtype == "bf16"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_mixture_experts_61_b300 import build
    build.build()
    moe.lib()


def forward_saving(w, dev):
    """moe_forward with the activations kept in caller buffers."""
    outs = tl.alloc_outputs(w)
    rows = w.T * w.k
    bf = dict(dtype=w.torch_dtype, device="cuda")
    outs.update(x_perm=torch.full((rows, w.d), float("nan"), **bf),
                h_act=torch.full((rows, w.h), float("nan"), **bf),
                y_perm=torch.full((rows, w.d), float("nan"), **bf),
                h_pre=torch.full((rows, w.h), float("nan"), **bf))
    r = tl.run_forward(w, dev, outs)
    assert r["flags"] == 0
    return r


def run_backward(w, dev, outs, dy, cfg, d_aux=D_AUX):
    f32 = dict(dtype=torch.float32, device="cuda")
    bf = dict(dtype=w.torch_dtype, device="cuda")
    E, d, h = w.E, w.d, w.h
    g = dict(dx=torch.full((w.T, d), float("nan"), **bf),
             dw_gate=torch.full((E, d), float("nan"), **f32),
             dlogit_bias=torch.full((E,), float("nan"), **f32),
             dw1=torch.full((E, h, d), float("nan"), **bf),
             db1=torch.full((E, h), float("nan"), **f32),
             dw2=torch.full((E, d, h), float("nan"), **bf),
             db2=torch.full((E, d), float("nan"), **f32))
    inputs = dict(dy=dy, x=dev["x"], w_gate=dev["w_gate"], w1=dev["w1"], w2=dev["w2"])
    for n in ("logits", "topk_idx", "topk_w", "counts", "offsets", "slot_row", "x_perm", "h_pre",
              "h_act", "y_perm"):
        inputs[n] = outs[n]
    ws = tl.poisoned_workspace(moe.moe_backward_workspace_size(cfg))
    moe.moe_backward(cfg, inputs, g, d_aux, ws)
    return g, moe.moe_device_error(ws)


def seeded_dy(w, seed=1):
    gen = torch.Generator().manual_seed(seed)
    return torch.randn((w.T, w.d), generator=gen).to(w.torch_dtype)


@pytest.mark.parametrize("name", BF16_NAMES)
def test_backward_parity(name):
    w = PARITY_WORKLOADS[name]
    inp = make_inputs(w, seed=0)
    dev = tl.to_device(inp)
    r = forward_saving(w, dev)
    outs = r["outs"]
    dy = seeded_dy(w)
    g, flags = run_backward(w, dev, outs, dy.cuda(), r["cfg"])
    assert flags == 0
    gh = tl.host(g)
    ref = oracle.backward(inp, dy, w.k, w.gate, capacity_factor_or_none(w), D_AUX,
                          logits_in=outs["logits"].cpu().numpy())
    errs = {}
    for key in ("dx", "dw_gate", "dlogit_bias", "dw1", "db1", "dw2", "db2"):
        assert np.all(np.isfinite(gh[key])), key
        errs[key] = tl.max_rel_err(gh[key], ref[key])
    print(name, {k: f"{v:.2e}" for k, v in errs.items()})
    for key, e in errs.items():
        assert e <= TOL_GRAD, (key, e)


def test_forward_saved_activations_are_consistent():
    """Keeping the activations in caller buffers changes nothing in the forward, Xp holds
    exactly the gathered tokens and H = SiLU(A) up to bf16 rounding."""
    w = PARITY_WORKLOADS["mixtral_prefill"]
    dev = tl.to_device(make_inputs(w, seed=0))
    plain = tl.host(tl.run_forward(w, dev)["outs"])
    saved = forward_saving(w, dev)["outs"]
    sv = tl.host(saved)
    np.testing.assert_array_equal(sv["y"], plain["y"])
    M = int(sv["offsets"][-1])
    rt = saved["row_token"][:M].long()
    assert torch.equal(saved["x_perm"][:M], dev["x"][rt])
    a = saved["h_pre"][:M].float()
    assert float((torch.nn.functional.silu(a) - saved["h_act"][:M].float()).abs().max()) <= \
        1e-2 * float(saved["h_act"][:M].float().abs().max())


def test_backward_deterministic():
    w = PARITY_WORKLOADS["deepseek_fine"]
    dev = tl.to_device(make_inputs(w, seed=2))
    r = forward_saving(w, dev)
    dy = seeded_dy(w, 3).cuda()
    a, _ = run_backward(w, dev, r["outs"], dy, r["cfg"])
    b, _ = run_backward(w, dev, r["outs"], dy, r["cfg"])
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_backward_without_upstream_gradient():
    """dy = 0 and d_aux = 0: every gradient is exactly zero."""
    w = PARITY_WORKLOADS["decode"]
    dev = tl.to_device(make_inputs(w, seed=0))
    r = forward_saving(w, dev)
    cfg = r["cfg"]
    dy = torch.zeros((w.T, w.d), dtype=w.torch_dtype, device="cuda")
    g, flags = run_backward(w, dev, r["outs"], dy, cfg, d_aux=0.0)
    assert flags == 0
    for k, v in g.items():
        assert torch.count_nonzero(v) == 0, k


def test_backward_empty_batch():
    w = Workload("bwd_empty", T=0, d=64, h=64, E=8, k=2, dtype="bf16", gate=0,
                 capacity_factor=0.0)
    cfg = moe.config_from_workload(w)
    dev = tl.to_device(make_inputs(w.scaled(T=1), seed=0))
    f32 = dict(dtype=torch.float32, device="cuda")
    g = dict(dw_gate=torch.full((8, 64), 7.0, **f32), dw1=torch.full((8, 64, 64), 7.0,
                                                                     dtype=torch.bfloat16, device="cuda"))
    i32 = dict(dtype=torch.int32, device="cuda")
    inputs = dict(w_gate=dev["w_gate"], w1=dev["w1"], w2=dev["w2"],
                  counts=torch.zeros(8, **i32), offsets=torch.zeros(9, **i32))
    ws = tl.poisoned_workspace(moe.moe_backward_workspace_size(cfg))
    moe.moe_backward(cfg, inputs, g, 0.5, ws)
    assert moe.moe_device_error(ws) == 0
    assert torch.count_nonzero(g["dw_gate"]) == 0 and torch.count_nonzero(g["dw1"]) == 0
