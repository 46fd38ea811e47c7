"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI, and
evaluate the oracle on the same seeded inputs (and on the GPU's own routing
decisions, so that the floating-point check of the expert path is not confounded
by near-tie routing flips)."""

from __future__ import annotations

import numpy as np
import torch

import oracle
import sparse_mixture_experts_61_b300 as moe

# Tolerances (max |dy| relative to max |y_ref|): bf16 keeps three roundings of the
# expert path (H, Y_perm, y) at 2^-9 each; fp32 keeps fp32 accumulation only.
TOL_Y = {"bf16": 2e-2, "f32": 1e-4}
TOL_W = 2e-6          # gate weights, absolute
TOL_AUX = 1e-5        # balance loss, relative
TOL_STATS = 1e-5      # routing statistics (fp32 output of a double computation), relative
NEAR_TIE = 1e-4       # k-th / (k+1)-th logit gap below which routing may flip


def logits_tol(lg_ref: np.ndarray) -> float:
    return 1e-5 * float(np.abs(lg_ref).max()) + 1e-5


def to_device(inp: dict, device="cuda") -> dict:
    return {k: (None if v is None else v.to(device).contiguous()) for k, v in inp.items()}


def to_host(inp: dict) -> dict:
    return {k: (None if v is None else v.cpu()) for k, v in inp.items()}


def alloc_outputs(w, device="cuda") -> dict:
    T, E, k, d = w.T, w.E, w.k, w.d
    i32 = dict(dtype=torch.int32, device=device)
    f32 = dict(dtype=torch.float32, device=device)
    return dict(
        y=torch.full((T, d), float("nan"), dtype=w.torch_dtype, device=device),
        logits=torch.full((T, E), float("nan"), **f32),
        topk_idx=torch.full((T, k), -7, **i32),
        topk_w=torch.full((T, k), float("nan"), **f32),
        counts=torch.full((E,), -7, **i32),
        aux_loss=torch.full((1,), float("nan"), **f32),
        offsets=torch.full((E + 1,), -7, **i32),
        kept_counts=torch.full((E,), -7, **i32),
        slot_row=torch.full((T, k), -7, **i32),
        row_token=torch.full((T * k,), -7, **i32),
        dropped=torch.full((1,), -7, **i32),
        routing_stats=torch.full((6,), float("nan"), **f32),
    )


def poisoned_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """Workspace filled with 0xFF bytes (NaN for floats, -1 for ints), so that any read
    of a value the kernels did not write shows up as a mismatch."""
    return torch.full((max(nbytes, 16),), 0xFF, dtype=torch.uint8, device=device)


def run_forward(w, inp_dev: dict, outs: dict = None, ws: torch.Tensor = None, cfg=None) -> dict:
    cfg = cfg if cfg is not None else moe.config_from_workload(w)
    if outs is None:
        outs = alloc_outputs(w, inp_dev["x"].device)
    if ws is None:
        ws = poisoned_workspace(moe.moe_workspace_size(cfg), inp_dev["x"].device)
    moe.moe_forward(cfg, inp_dev, outs, ws)
    flags = moe.moe_device_error(ws)
    return dict(outs=outs, ws=ws, flags=flags, cfg=cfg)


def host(outs: dict) -> dict:
    r = {}
    for k, v in outs.items():
        if v.dtype == torch.bfloat16:
            r[k] = v.float().cpu().numpy()
        else:
            r[k] = v.cpu().numpy()
    return r


def expert_outputs(inp_host: dict, idx: np.ndarray, slot_row: np.ndarray, tokens=None,
                   fetch=None) -> np.ndarray:
    """Oracle expert outputs z[t, j, :] for every kept (t, j) among ``tokens`` (all by
    default); dropped slots are zero.  ``fetch(e)`` returns (w1_e, b1_e, w2_e, b2_e) on
    the host (default: slices of inp_host)."""
    T, k = idx.shape
    x = inp_host["x"]
    d = x.shape[1]
    toks = np.arange(T) if tokens is None else np.asarray(tokens)
    z = np.zeros((len(toks), k, d), np.float64)
    by_e = {}
    for a, t in enumerate(toks):
        for j in range(k):
            if slot_row[t, j] >= 0:
                by_e.setdefault(int(idx[t, j]), []).append((a, j, int(t)))
    for e, items in sorted(by_e.items()):
        if fetch is None:
            w1e, b1e, w2e, b2e = (inp_host["w1"][e], inp_host["b1"][e], inp_host["w2"][e],
                                  inp_host["b2"][e])
        else:
            w1e, b1e, w2e, b2e = fetch(e)
        rows = x[[t for _, _, t in items]]
        ze = oracle.expert_rows(rows, w1e, b1e, w2e, b2e)
        for q, (a, j, _) in enumerate(items):
            z[a, j] = ze[q]
    return z


def y_on_routing(inp_host, idx, slot_row, w_ref, tokens=None, fetch=None) -> np.ndarray:
    """Oracle O6-O7 evaluated on given routing decisions (the GPU's)."""
    toks = np.arange(idx.shape[0]) if tokens is None else np.asarray(tokens)
    z = expert_outputs(inp_host, idx, slot_row, toks, fetch)
    return oracle.combine(slot_row[toks], w_ref[toks], z)


def topk_gaps(lg: np.ndarray, k: int) -> np.ndarray:
    """Gap between the k-th and (k+1)-th largest logit of each token (inf when k = E)."""
    if k >= lg.shape[1]:
        return np.full(lg.shape[0], np.inf)
    s = -np.sort(-lg, axis=1)
    return s[:, k - 1] - s[:, k]


def check_routing_exact(g, ref, tol_w=TOL_W):
    """Every routing and indexing output of the GPU (``g``, host arrays) equal to the
    oracle's routing stages run on the GPU's own logits (``ref``); gate weights, the
    balance loss and the routing statistics within their tolerances."""
    np.testing.assert_array_equal(g["topk_idx"], ref["idx"])
    np.testing.assert_array_equal(g["counts"], ref["counts"])
    np.testing.assert_array_equal(g["kept_counts"], ref["kept"])
    np.testing.assert_array_equal(g["offsets"], ref["offsets"])
    np.testing.assert_array_equal(g["slot_row"], ref["slot_row"])
    np.testing.assert_array_equal(g["row_token"], ref["row_token"])
    assert int(g["dropped"][0]) == ref["dropped"]
    assert float(np.abs(g["topk_w"] - ref["w"]).max()) <= tol_w
    assert abs(float(g["aux_loss"][0]) - ref["aux"]) <= TOL_AUX * abs(ref["aux"])
    st = oracle.routing_stats(ref["counts"])
    np.testing.assert_allclose(g["routing_stats"], st, rtol=TOL_STATS, atol=1e-7)


def max_rel_err(a: np.ndarray, ref: np.ndarray) -> float:
    scale = float(np.abs(ref).max())
    return float(np.abs(a - ref).max()) / (scale if scale > 0 else 1.0)
