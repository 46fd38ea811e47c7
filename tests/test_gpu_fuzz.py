"""Seeded random shapes through the C ABI against the oracle.

Each case draws a layer (dtype, T, E, k, d, h, gate form, capacity, biases) from a fixed seed,
so a failure names a reproducible configuration.  Widths are multiples of 8 between 8 and 392,
which exercises partial 64-column k-blocks, partial 128/256-column output tiles and ragged row
tails in every GEMM; small T and large E leave many experts empty.
"""

import numpy as np
import pytest
import torch

import moe_testlib as tl
import oracle
import sparse_mixture_experts_61_b300 as moe
from moe_workloads import Workload, capacity_factor_or_none, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_mixture_experts_61_b300 import build
    build.build()
    moe.lib()


def draw(seed, dtype=None, routing="topk"):
    rng = np.random.default_rng(seed)
    k = int(rng.integers(1, 9))
    E = int(rng.integers(max(k, 2), 65))
    T = int(rng.integers(1, 700))
    d = 8 * int(rng.integers(1, 50))
    h = 8 * int(rng.integers(1, 50))
    dt = dtype or ("bf16" if rng.random() < 0.75 else "f32")
    gate = int(rng.integers(0, 2))
    cf = float(rng.choice([0.0, 0.0, round(rng.uniform(0.5, 2.5), 2)]))
    if routing == "expert_choice":
        cf = round(float(rng.uniform(0.3, 3.0)), 2)
    return Workload(f"fuzz{seed}", T=T, d=d, h=h, E=E, k=k, dtype=dt, gate=gate,
                    capacity_factor=cf, bias_std=0.1, logit_bias="none", routing=routing)


@pytest.mark.parametrize("seed", range(16))
def test_fuzz_forward(seed):
    w = draw(seed)
    cf = capacity_factor_or_none(w)
    inp = make_inputs(w, seed=seed)
    r = tl.run_forward(w, tl.to_device(inp))
    assert r["flags"] == 0, w
    g = tl.host(r["outs"])
    lg_ref = oracle.logits(inp["x"], inp["w_gate"], inp["logit_bias"])
    assert float(np.abs(g["logits"] - lg_ref).max()) <= tl.logits_tol(lg_ref), w
    ref = oracle.routed_reference(None, w.k, w.gate, cf, g["logits"])
    tl.check_routing_exact(g, ref)   # indices, counts, kept, offsets, rows, drops, weights, loss, stats
    y_ref = tl.y_on_routing(inp, ref["idx"], ref["slot_row"], ref["w"])
    err = tl.max_rel_err(g["y"], y_ref)
    assert err <= tl.TOL_Y[w.dtype], (w, err)


@pytest.mark.parametrize("seed", range(100, 106))
def test_fuzz_expert_choice(seed):
    w = draw(seed, routing="expert_choice")
    cfg = moe.config(w.T, w.d, w.h, w.E, w.k, w.dtype, w.gate, w.capacity_factor)
    C = moe.moe_expert_choice_capacity(cfg)
    inp = make_inputs(w, seed=seed)
    dev = tl.to_device(inp)
    f32 = dict(dtype=torch.float32, device="cuda")
    i32 = dict(dtype=torch.int32, device="cuda")
    outs = dict(y=torch.empty((w.T, w.d), dtype=w.torch_dtype, device="cuda"),
                logits=torch.empty((w.T, w.E), **f32), probs=torch.empty((w.T, w.E), **f32),
                sel_token=torch.empty((w.E, C), **i32), sel_w=torch.empty((w.E, C), **f32))
    ws = tl.poisoned_workspace(moe.moe_expert_choice_workspace_size(cfg))
    moe.moe_expert_choice_forward(cfg, dev, outs, ws)
    assert moe.moe_device_error(ws) == 0, w
    g = tl.host(outs)
    tok, w_g = oracle.expert_choice(g["probs"].astype(np.float64), C)
    np.testing.assert_array_equal(g["sel_token"], tok)
    p_ref = oracle.softmax(g["logits"])
    w_ref = np.stack([p_ref[tok[e], e] for e in range(w.E)])
    z = np.zeros((w.E * C, w.d))
    for e in range(w.E):
        if C:
            z[e * C:(e + 1) * C] = oracle.expert_rows(inp["x"][tok[e].tolist()], inp["w1"][e],
                                                      inp["b1"][e], inp["w2"][e], inp["b2"][e])
    y_ref = oracle.combine_expert_choice(w.T, tok, w_ref, z)
    err = tl.max_rel_err(g["y"], y_ref)
    assert err <= tl.TOL_Y[w.dtype], (w, err)


@pytest.mark.parametrize("seed", range(200, 206))
def test_fuzz_backward(seed):
    w = draw(seed, dtype="bf16")
    cf = capacity_factor_or_none(w)
    inp = make_inputs(w, seed=seed)
    dev = tl.to_device(inp)
    outs = tl.alloc_outputs(w)
    rows = w.T * w.k
    bf = dict(dtype=torch.bfloat16, device="cuda")
    outs.update(x_perm=torch.empty((rows, w.d), **bf), h_act=torch.empty((rows, w.h), **bf),
                y_perm=torch.empty((rows, w.d), **bf), h_pre=torch.empty((rows, w.h), **bf))
    r = tl.run_forward(w, dev, outs)
    assert r["flags"] == 0
    gen = torch.Generator().manual_seed(seed)
    dy = torch.randn((w.T, w.d), generator=gen).to(torch.bfloat16)
    f32 = dict(dtype=torch.float32, device="cuda")
    E, d, h = w.E, w.d, w.h
    grads = dict(dx=torch.empty((w.T, d), **bf), dw_gate=torch.empty((E, d), **f32),
                 dlogit_bias=torch.empty((E,), **f32), dw1=torch.empty((E, h, d), **bf),
                 db1=torch.empty((E, h), **f32), dw2=torch.empty((E, d, h), **bf),
                 db2=torch.empty((E, d), **f32))
    bin_ = dict(dy=dy.cuda(), x=dev["x"], w_gate=dev["w_gate"], w1=dev["w1"], w2=dev["w2"])
    for n in ("logits", "topk_idx", "topk_w", "counts", "offsets", "slot_row", "x_perm", "h_pre",
              "h_act", "y_perm"):
        bin_[n] = outs[n]
    ws = tl.poisoned_workspace(moe.moe_backward_workspace_size(r["cfg"]))
    moe.moe_backward(r["cfg"], bin_, grads, 0.03, ws)
    assert moe.moe_device_error(ws) == 0
    gh = tl.host(grads)
    ref = oracle.backward(inp, dy, w.k, w.gate, cf, 0.03, logits_in=outs["logits"].cpu().numpy())
    for key in grads:
        err = tl.max_rel_err(gh[key], ref[key])
        assert err <= 1.5e-2, (w, key, err)
