"""Parity of the expert-choice layer (moe_expert_choice_forward) with the CPU oracle.

Each expert takes the C tokens with the largest softmax probability.  The selection
is an integer decision taken on floating-point values, so it is checked exactly
against the oracle's selection run on the GPU's own fp32 probabilities; the
probabilities themselves are checked against the oracle's softmax of the GPU's
logits, and the logits against the oracle's contraction.  The output y is checked
against the oracle's expert path and combine on that selection, and a fully
independent oracle run may differ only where two probabilities are within a near-tie
of the expert's C-th largest.
"""

import numpy as np
import pytest
import torch

import moe_testlib as tl
import oracle
import sparse_mixture_experts_61_b300 as moe
from moe_workloads import EC_PARITY_WORKLOADS, WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu

NEAR_TIE_P = 1e-5   # relative probability gap below which a selection may flip


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_mixture_experts_61_b300 import build
    build.build()
    moe.lib()


def ec_config(w):
    return moe.config(w.T, w.d, w.h, w.E, w.k, w.dtype, w.gate, w.capacity_factor)


def alloc_ec_outputs(w, C, device="cuda"):
    T, E, d = w.T, w.E, w.d
    i32 = dict(dtype=torch.int32, device=device)
    f32 = dict(dtype=torch.float32, device=device)
    return dict(
        y=torch.full((T, d), float("nan"), dtype=w.torch_dtype, device=device),
        logits=torch.full((T, E), float("nan"), **f32),
        probs=torch.full((T, E), float("nan"), **f32),
        sel_token=torch.full((E, C), -7, **i32),
        sel_w=torch.full((E, C), float("nan"), **f32),
        token_experts=torch.full((T,), -7, **i32),
        unrouted=torch.full((1,), -7, **i32),
    )


def run_ec(w, inp_dev, outs=None):
    cfg = ec_config(w)
    C = moe.moe_expert_choice_capacity(cfg)
    if outs is None:
        outs = alloc_ec_outputs(w, C, inp_dev["x"].device)
    ws = tl.poisoned_workspace(moe.moe_expert_choice_workspace_size(cfg), inp_dev["x"].device)
    moe.moe_expert_choice_forward(cfg, inp_dev, outs, ws)
    flags = moe.moe_device_error(ws)
    return dict(outs=outs, ws=ws, flags=flags, C=C, cfg=cfg)


def check_selection_exact(g, C, T):
    """Selection, weights and per-token counts against the oracle run on the GPU's
    own probabilities; returns (sel_token, oracle weights p(fp64 softmax of the GPU
    logits) at the selection)."""
    probs_g = g["probs"].astype(np.float64)
    p_ref = oracle.softmax(g["logits"])
    assert float(np.abs(g["probs"] - p_ref).max()) <= tl.TOL_W
    tok, w_g = oracle.expert_choice(probs_g, C)
    np.testing.assert_array_equal(g["sel_token"], tok)
    np.testing.assert_array_equal(g["sel_w"], w_g.astype(np.float32))   # the very p it chose on
    E = tok.shape[0]
    w_ref = np.stack([p_ref[tok[e], e] for e in range(E)]) if C else np.zeros((E, 0))
    counts = np.bincount(tok.ravel(), minlength=T)
    np.testing.assert_array_equal(g["token_experts"], counts)
    assert int(g["unrouted"][0]) == int((counts == 0).sum())
    return tok, w_ref, counts


def y_on_selection(inp_host, tok, w_ref, tokens=None, fetch=None):
    """Oracle expert path + combine on a given selection, for all tokens or a sample."""
    E, C = tok.shape
    T = inp_host["x"].shape[0]
    d = inp_host["x"].shape[1]
    want = None if tokens is None else set(int(t) for t in tokens)
    z = np.zeros((E * C, d))
    for e in range(E):
        cs = [c for c in range(C) if want is None or int(tok[e, c]) in want]
        if not cs:
            continue
        w1e, b1e, w2e, b2e = fetch(e) if fetch else (inp_host["w1"][e], inp_host["b1"][e],
                                                     inp_host["w2"][e], inp_host["b2"][e])
        rows = inp_host["x"][[int(tok[e, c]) for c in cs]]
        ze = oracle.expert_rows(rows, w1e, b1e, w2e, b2e)
        for q, c in enumerate(cs):
            z[e * C + c] = ze[q]
    return oracle.combine_expert_choice(T, tok, w_ref, z)


@pytest.mark.parametrize("name", list(EC_PARITY_WORKLOADS))
def test_expert_choice_parity(name):
    w = EC_PARITY_WORKLOADS[name]
    inp = make_inputs(w, seed=0)
    r = run_ec(w, tl.to_device(inp))
    assert r["flags"] == 0
    C = r["C"]
    assert C == min(w.T, oracle.capacity(w.T, w.E, w.capacity_factor))
    g = tl.host(r["outs"])

    lg_ref = oracle.logits(inp["x"], inp["w_gate"], inp["logit_bias"])
    assert float(np.abs(g["logits"] - lg_ref).max()) <= tl.logits_tol(lg_ref)
    tok, w_ref, counts = check_selection_exact(g, C, w.T)

    y_ref = y_on_selection(inp, tok, w_ref)
    err = tl.max_rel_err(g["y"], y_ref)
    assert err <= tl.TOL_Y[w.dtype]
    assert np.all(g["y"][counts == 0] == 0.0)

    # Independent oracle run: selections may differ only at near-ties of the C-th value.
    full = oracle.forward_expert_choice(inp, w.capacity_factor)
    p = full["p"]
    flips = 0
    for e in range(w.E):
        a, b = set(full["sel_token"][e].tolist()), set(tok[e].tolist())
        if a == b:
            continue
        kth = np.sort(p[:, e])[::-1][C - 1]
        for t in a ^ b:
            assert abs(p[t, e] - kth) <= NEAR_TIE_P * kth, "a selection flip away from a near-tie"
            flips += 1
    same = np.ones(w.T, bool)
    for e in range(w.E):
        for t in set(full["sel_token"][e].tolist()) ^ set(tok[e].tolist()):
            same[t] = False
    scale = float(np.abs(full["y"]).max())
    assert float(np.abs(g["y"][same] - full["y"][same]).max()) <= tl.TOL_Y[w.dtype] * scale
    print(f"{name}: C={C} unrouted={int(g['unrouted'][0])} max_experts={int(counts.max())} "
          f"y_err={err:.2e} near_tie_flips={flips}")


def test_expert_choice_deterministic():
    w = EC_PARITY_WORKLOADS["switch_ec"]
    dev = tl.to_device(make_inputs(w, seed=3))
    a = tl.host(run_ec(w, dev)["outs"])
    b = tl.host(run_ec(w, dev)["outs"])
    for k in a:
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)


def test_expert_choice_full_capacity_is_dense_mixture():
    """capacity_factor >= E: C = T, every expert takes every token, and the layer is the
    softmax-weighted mixture of all experts."""
    w = Workload("ec_full", T=150, d=64, h=96, E=4, k=1, dtype="f32", gate=0,
                 capacity_factor=6.0, bias_std=0.1, routing="expert_choice")
    inp = make_inputs(w, seed=5)
    r = run_ec(w, tl.to_device(inp))
    assert r["flags"] == 0 and r["C"] == 150
    g = tl.host(r["outs"])
    assert np.all(g["token_experts"] == 4) and int(g["unrouted"][0]) == 0
    np.testing.assert_array_equal(g["sel_token"], np.tile(np.arange(150), (4, 1)))
    full = oracle.forward_expert_choice(inp, 6.0)
    assert tl.max_rel_err(g["y"], full["y"]) <= tl.TOL_Y["f32"]


def test_expert_choice_ties_take_lower_token_first():
    """Ten copies of each of 30 token rows give bitwise-equal probabilities; the
    selection must take equal values in token order."""
    w = Workload("ec_ties", T=300, d=64, h=64, E=8, k=1, dtype="bf16", gate=0,
                 capacity_factor=1.0, routing="expert_choice")
    inp = make_inputs(w, seed=8)
    inp["x"] = inp["x"][:30].repeat(10, 1).contiguous()
    r = run_ec(w, tl.to_device(inp))
    assert r["flags"] == 0
    g = tl.host(r["outs"])
    _, counts_eq = np.unique(g["probs"][:, 0], return_counts=True)
    assert counts_eq.max() >= 10          # ties really are present
    check_selection_exact(g, r["C"], w.T)


@pytest.mark.parametrize("T,E,cf", [(1, 1, 1.0), (1, 8, 1.0), (2, 256, 0.5), (65, 3, 1.0)])
def test_expert_choice_small_shapes(T, E, cf):
    w = Workload("ec_small", T=T, d=16, h=24, E=E, k=1, dtype="bf16", gate=0,
                 capacity_factor=cf, bias_std=0.1, routing="expert_choice")
    inp = make_inputs(w, seed=T + E)
    r = run_ec(w, tl.to_device(inp))
    assert r["flags"] == 0
    g = tl.host(r["outs"])
    tok, w_ref, counts = check_selection_exact(g, r["C"], T)
    y_ref = y_on_selection(inp, tok, w_ref)
    assert tl.max_rel_err(g["y"], y_ref) <= tl.TOL_Y["bf16"]


def test_expert_choice_empty_batch():
    w = Workload("ec_empty", T=0, d=64, h=64, E=8, k=1, dtype="bf16", gate=0,
                 capacity_factor=1.0, routing="expert_choice")
    cfg = ec_config(w)
    assert moe.moe_expert_choice_capacity(cfg) == 0
    dev = tl.to_device(make_inputs(w.scaled(T=1), seed=0))
    inputs = dict(dev, x=None)
    unrouted = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    ws = tl.poisoned_workspace(moe.moe_expert_choice_workspace_size(cfg))
    moe.moe_expert_choice_forward(cfg, inputs, dict(y=None, unrouted=unrouted), ws)
    assert moe.moe_device_error(ws) == 0
    assert int(unrouted.item()) == 0


def test_expert_choice_nonfinite_logit_flag():
    w = Workload("ec_nan", T=64, d=64, h=64, E=8, k=1, dtype="bf16", gate=0,
                 capacity_factor=1.0, routing="expert_choice")
    inp = make_inputs(w, seed=0)
    inp["x"][7, 3] = float("nan")
    r = run_ec(w, tl.to_device(inp))
    assert r["flags"] & moe.MOE_DEVERR_NONFINITE


@pytest.mark.parametrize("name", ["mixtral_prefill_ec", "deepseek_fine_ec"])
def test_expert_choice_full_size_sampled(name):
    """Full workload sizes through the call the benchmark times: the selection exact
    for every expert, logits and y on sampled tokens."""
    w = WORKLOADS[name]
    inp = make_inputs(w, seed=0, device="cuda")
    r = run_ec(w, inp)
    assert r["flags"] == 0
    g = tl.host(r["outs"])
    tok, w_ref, counts = check_selection_exact(g, r["C"], w.T)

    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, w.T - 1], rng.choice(w.T, 48, replace=False)]))
    xs = inp["x"][torch.as_tensor(rows, device="cuda")].cpu()
    lb = inp["logit_bias"].cpu() if inp["logit_bias"] is not None else None
    lg_ref = oracle.logits(xs, inp["w_gate"].cpu(), lb)
    assert float(np.abs(g["logits"][rows] - lg_ref).max()) <= tl.logits_tol(lg_ref)

    toks = np.unique(np.concatenate([[0, w.T - 1], rng.choice(w.T, 12, replace=False)]))
    cache = {}

    def fetch(e):
        if e not in cache:
            cache.clear()
            cache[e] = tuple(inp[n][e].cpu() for n in ("w1", "b1", "w2", "b2"))
        return cache[e]

    y_ref = y_on_selection({"x": inp["x"].cpu()}, tok, w_ref, tokens=toks, fetch=fetch)[toks]
    err = tl.max_rel_err(g["y"][toks], y_ref)
    assert err <= tl.TOL_Y[w.dtype]
    print(f"{name}: C={r['C']} unrouted={int(g['unrouted'][0])} "
          f"max_experts={int(counts.max())} sampled y_err={err:.2e}")
