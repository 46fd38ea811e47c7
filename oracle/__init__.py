"""ctypes front end of the plain CPU oracle of the top-k MoE FFN forward.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py``; the product package never imports it.

Inputs are CPU torch tensors (fp32 or bf16) or numpy arrays; they are handed to
the C oracle as raw fp32 / bf16 bit patterns and widened exactly to double
there.  Outputs are numpy float64 / int32 / int64 arrays.  Each wrapper names the
oracle stage it runs; the formulas and their sources are in ``moe_oracle.cpp``.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int
_D = ctypes.c_double


def lib():
    global _lib
    if _lib is None:
        # MOE_ORACLE_LIB names a prebuilt copy of the oracle instead (the test that plants
        # mistakes in copies of the source and checks that the pins catch each one).
        path = os.environ.get("MOE_ORACLE_LIB") or _build.build()
        L = ctypes.CDLL(path)
        L.orc_num_threads.restype = _I
        L.orc_set_num_threads.argtypes = [_I]
        L.orc_logits.argtypes = [_I64, _I, _I, _I, _P, _P, _P, _P]
        L.orc_softmax.argtypes = [_I64, _I, _P, _P]
        L.orc_topk.argtypes = [_I64, _I, _I, _P, _P]
        L.orc_gate_weights.argtypes = [_I64, _I, _I, _I, _P, _P, _P]
        L.orc_aux_loss.argtypes = [_I64, _I, _I, _P, _P, _P, _P, _P]
        L.orc_aux_loss.restype = _D
        L.orc_routing_stats.argtypes = [_I, _P, _P]
        L.orc_noisy_scores.argtypes = [_I64, _I, _I, _P, _P, _P]
        L.orc_backward.argtypes = [_I64, _I, _I, _I, _I, _I, _I, ctypes.c_double] + [_P] * 8 + \
            [ctypes.c_double] + [_P] * 8
        L.orc_backward.restype = _I
        L.orc_expert_choice.argtypes = [_I64, _I, _I64, _P, _P, _P]
        L.orc_combine_expert_choice.argtypes = [_I64, _I, _I, _I64, _P, _P, _P, _P]
        L.orc_capacity.argtypes = [_I64, _I, _D]
        L.orc_capacity.restype = _I64
        L.orc_dispatch.argtypes = [_I64, _I, _I, _I64, _P, _P, _P, _P, _P, _P]
        L.orc_dispatch.restype = _I
        L.orc_expert_rows.argtypes = [_I, _I, _I, _I64, _P, _P, _P, _P, _P, _P]
        L.orc_combine.argtypes = [_I64, _I, _I, _P, _P, _P, _P]
        L.orc_forward.argtypes = [_I64, _I, _I, _I, _I, _I, _I, _D] + [_P] * 7 + [_P] * 11
        L.orc_forward.restype = _I
        L.orc_forward_dense.argtypes = [_I64, _I, _I, _I, _I, _I, _I, _D] + [_P] * 8
        _lib = L
    return _lib


def num_threads() -> int:
    return lib().orc_num_threads()


def set_num_threads(n: int) -> None:
    lib().orc_set_num_threads(int(n))


def raw(a):
    """Return (contiguous numpy array of raw element bits, dtype code) for a tensor/array.

    dtype code 0 = fp32, 1 = bf16, 2 = fp64.  Accepts CPU torch tensors (fp32/bf16/fp64)
    and numpy float32/float64 arrays."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().contiguous()
            if a.dtype == torch.bfloat16:
                return a.view(torch.int16).numpy(), 1
            if a.dtype == torch.float32:
                return a.numpy(), 0
            if a.dtype == torch.float64:
                return a.numpy(), 2
            raise TypeError(f"unsupported tensor dtype {a.dtype}")
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return a, 0
    if a.dtype == np.float64:
        return a, 2
    if a.dtype in (np.int16, np.uint16):
        return a, 1
    raise TypeError(f"unsupported array dtype {a.dtype}")


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(a):
    if a is None:
        return None
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().float().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(a, dtype=np.float32)


def logits(x, w_gate, logit_bias=None):
    """O1: logits[t,e] = sum_i x[t,i] w_gate[e,i] (+ logit_bias[e])."""
    xr, dt = raw(x)
    wr, dt2 = raw(w_gate)
    assert dt == dt2
    T, d = xr.shape
    E = wr.shape[0]
    out = np.empty((T, E), np.float64)
    lb = _f32(logit_bias)
    lib().orc_logits(T, d, E, dt, _ptr(xr), _ptr(wr), _ptr(lb), _ptr(out))
    return out


def softmax(lg):
    """O2: row-wise softmax of a [T,E] float64 array."""
    lg = np.ascontiguousarray(lg, np.float64)
    T, E = lg.shape
    out = np.empty_like(lg)
    lib().orc_softmax(T, E, _ptr(lg), _ptr(out))
    return out


def topk(lg, k):
    """O3: stable top-k indices [T,k] int32 (value desc, lower index on ties)."""
    lg = np.ascontiguousarray(lg, np.float64)
    T, E = lg.shape
    out = np.empty((T, k), np.int32)
    lib().orc_topk(T, E, k, _ptr(lg), _ptr(out))
    return out


def gate_weights(lg, idx, mode):
    """O3w: kept gate weights [T,k] float64 (mode 0: softmax(TopK); mode 1: renormalised p)."""
    lg = np.ascontiguousarray(lg, np.float64)
    idx = np.ascontiguousarray(idx, np.int32)
    T, E = lg.shape
    k = idx.shape[1]
    out = np.empty((T, k), np.float64)
    lib().orc_gate_weights(T, E, k, int(mode), _ptr(lg), _ptr(idx), _ptr(out))
    return out


def aux_loss(p, idx):
    """O4: (loss, counts[E] int64, f[E], P[E])."""
    p = np.ascontiguousarray(p, np.float64)
    idx = np.ascontiguousarray(idx, np.int32)
    T, E = p.shape
    k = idx.shape[1]
    counts = np.empty(E, np.int64)
    f = np.empty(E, np.float64)
    P = np.empty(E, np.float64)
    loss = lib().orc_aux_loss(T, E, k, _ptr(p), _ptr(idx), _ptr(counts), _ptr(f), _ptr(P))
    return loss, counts, f, P


NOISE_NONE, NOISE_GUMBEL, NOISE_PROB_GAUSS, NOISE_LOGIT_SOFTMAX = 0, 1, 2, 3


def noisy_scores(lg, noise, mode):
    """O2n: selection scores under routing noise `mode` (1 Gumbel on logits from uniform
    draws, 2 Gaussian draws added to probabilities, 3 logits + draws * softmax)."""
    lg = np.ascontiguousarray(lg, np.float64)
    noise = np.ascontiguousarray(noise, np.float32)
    T, E = lg.shape
    out = np.empty_like(lg)
    lib().orc_noisy_scores(T, E, int(mode), _ptr(lg), _ptr(noise), _ptr(out))
    return out


ROUTING_STATS = ("cv", "dead_ratio", "max_over_avg", "entropy", "effective_experts",
                 "count_cv_loss")


def routing_stats(counts):
    """O4s: the six routing statistics of per-expert counts (order: ROUTING_STATS)."""
    counts = np.ascontiguousarray(counts, np.int64)
    out = np.empty(6, np.float64)
    lib().orc_routing_stats(int(counts.shape[0]), _ptr(counts), _ptr(out))
    return out


def capacity(T, E, capacity_factor):
    """O5a: capacity ceil(T*cf/E), or -1 when there is no limit (cf <= 0 or None)."""
    return int(lib().orc_capacity(int(T), int(E), float(capacity_factor or 0.0)))


def dispatch(idx, E, C):
    """O5b: dict(kept[E], offsets[E+1], slot_row[T,k], row_token[T*k], dropped)."""
    idx = np.ascontiguousarray(idx, np.int32)
    T, k = idx.shape
    kept = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    slot_row = np.empty((T, k), np.int32)
    row_token = np.empty(T * k, np.int32)
    dropped = np.zeros(1, np.int64)
    rc = lib().orc_dispatch(T, E, k, int(C), _ptr(idx), _ptr(kept), _ptr(offsets),
                            _ptr(slot_row), _ptr(row_token), _ptr(dropped))
    if rc != 0:
        raise ValueError("expert index out of range")
    return dict(kept=kept, offsets=offsets, slot_row=slot_row, row_token=row_token,
                dropped=int(dropped[0]))


def backward(inp, dy, k, mode, capacity_factor=None, d_aux=0.0, logits_in=None):
    """Gradients of the layer (B1..B7 in moe_oracle.cpp) for dL/dy = dy and dL/daux =
    d_aux: dict dx [T,d], dw_gate [E,d], dlogit_bias [E], dw1 [E,h,d], db1 [E,h],
    dw2 [E,d,h], db2 [E,d], all float64.  dy has the dtype of x.  logits_in [T,E]
    (optional) replaces the recomputed router logits downstream of O1."""
    xr, dt = raw(inp["x"])
    wg, _ = raw(inp["w_gate"])
    w1, _ = raw(inp["w1"])
    w2, _ = raw(inp["w2"])
    b1 = raw(inp["b1"])[0] if inp.get("b1") is not None else None
    b2 = raw(inp["b2"])[0] if inp.get("b2") is not None else None
    g, gdt = raw(dy)
    if gdt != dt:
        raise TypeError("dy must have the dtype of x")
    lb = _f32(inp.get("logit_bias"))
    T, d = xr.shape
    E, h = w1.shape[0], w1.shape[1]
    out = dict(dx=np.empty((T, d)), dw_gate=np.empty((E, d)), dlogit_bias=np.empty(E),
               dw1=np.empty((E, h, d)), db1=np.empty((E, h)), dw2=np.empty((E, d, h)),
               db2=np.empty((E, d)))
    li = None if logits_in is None else np.ascontiguousarray(logits_in, np.float64)
    rc = lib().orc_backward(T, d, h, E, k, int(mode), dt, float(capacity_factor or 0.0),
                            _ptr(xr), _ptr(wg), _ptr(lb), _ptr(w1), _ptr(b1), _ptr(w2), _ptr(b2),
                            _ptr(g), float(d_aux), _ptr(li), _ptr(out["dx"]), _ptr(out["dw_gate"]),
                            _ptr(out["dlogit_bias"]), _ptr(out["dw1"]), _ptr(out["db1"]),
                            _ptr(out["dw2"]), _ptr(out["db2"]))
    if rc != 0:
        raise ValueError("oracle backward failed")
    return out


def expert_choice(p, C):
    """O5e: each expert's C chosen tokens (ascending) and their weights p[t,e]:
    (sel_token [E,C] int32, sel_w [E,C] float64)."""
    p = np.ascontiguousarray(p, np.float64)
    T, E = p.shape
    tok = np.empty((E, C), np.int32)
    w = np.empty((E, C), np.float64)
    lib().orc_expert_choice(T, E, int(C), _ptr(p), _ptr(tok), _ptr(w))
    return tok, w


def combine_expert_choice(T, sel_token, sel_w, z):
    """O7e: y[T,d] = sum over choosing experts (ascending) of w * z; z is [E*C, d]."""
    sel_token = np.ascontiguousarray(sel_token, np.int32)
    sel_w = np.ascontiguousarray(sel_w, np.float64)
    z = np.ascontiguousarray(z, np.float64)
    E, C = sel_token.shape
    d = z.shape[1]
    y = np.empty((T, d), np.float64)
    lib().orc_combine_expert_choice(T, d, E, C, _ptr(sel_token), _ptr(sel_w), _ptr(z), _ptr(y))
    return y


def forward_expert_choice(inp, capacity_factor):
    """Whole expert-choice layer (O1, O2, O5e, O6, O7e) on an input dict."""
    lg = logits(inp["x"], inp["w_gate"], inp.get("logit_bias"))
    T, E = lg.shape
    C = min(T, capacity(T, E, capacity_factor))
    p = softmax(lg)
    tok, w = expert_choice(p, C)
    z = np.zeros((E * C, inp["x"].shape[1]))
    for e in range(E):
        if C:
            z[e * C:(e + 1) * C] = expert_rows(inp["x"][tok[e].tolist()], inp["w1"][e], inp["b1"][e],
                                               inp["w2"][e], inp["b2"][e])
    return dict(y=combine_expert_choice(T, tok, w, z), logits=lg, p=p, sel_token=tok, sel_w=w, C=C)


def expert_rows(x_rows, w1_e, b1_e, w2_e, b2_e):
    """O6: z = W2 SiLU(W1 x + b1) + b2 for each row of x_rows [n,d] (one expert)."""
    xr, dt = raw(x_rows)
    w1r, _ = raw(w1_e)
    w2r, _ = raw(w2_e)
    b1r = raw(b1_e)[0] if b1_e is not None else None
    b2r = raw(b2_e)[0] if b2_e is not None else None
    n, d = xr.shape
    h = w1r.shape[0]
    z = np.empty((n, d), np.float64)
    lib().orc_expert_rows(d, h, dt, n, _ptr(xr), _ptr(w1r), _ptr(b1r), _ptr(w2r), _ptr(b2r), _ptr(z))
    return z


def combine(slot_row, w, z):
    """O7: y[T,d] from slot_row [T,k], weights [T,k] and expert outputs z [T,k,d]."""
    slot_row = np.ascontiguousarray(slot_row, np.int32)
    w = np.ascontiguousarray(w, np.float64)
    z = np.ascontiguousarray(z, np.float64)
    T, k, d = z.shape
    y = np.empty((T, d), np.float64)
    lib().orc_combine(T, d, k, _ptr(slot_row), _ptr(w), _ptr(z), _ptr(y))
    return y


def forward(inp, k, mode, capacity_factor=None):
    """Whole layer O1..O7 on an input dict from ``moe_workloads.make_inputs``.

    Returns a dict with y, logits, idx, w, counts, aux, kept, offsets, slot_row,
    row_token, dropped."""
    xr, dt = raw(inp["x"])
    wg, _ = raw(inp["w_gate"])
    w1, _ = raw(inp["w1"])
    w2, _ = raw(inp["w2"])
    b1 = raw(inp["b1"])[0] if inp.get("b1") is not None else None
    b2 = raw(inp["b2"])[0] if inp.get("b2") is not None else None
    lb = _f32(inp.get("logit_bias"))
    T, d = xr.shape
    E, h = w1.shape[0], w1.shape[1]
    out = dict(y=np.empty((T, d)), logits=np.empty((T, E)), idx=np.empty((T, k), np.int32),
               w=np.empty((T, k)), counts=np.empty(E, np.int64), aux=np.zeros(1),
               kept=np.empty(E, np.int32), offsets=np.empty(E + 1, np.int32),
               slot_row=np.empty((T, k), np.int32), row_token=np.empty(T * k, np.int32),
               dropped=np.zeros(1, np.int64))
    rc = lib().orc_forward(T, d, h, E, k, int(mode), dt, float(capacity_factor or 0.0),
                           _ptr(xr), _ptr(wg), _ptr(lb), _ptr(w1), _ptr(b1), _ptr(w2), _ptr(b2),
                           _ptr(out["y"]), _ptr(out["logits"]), _ptr(out["idx"]), _ptr(out["w"]),
                           _ptr(out["counts"]), _ptr(out["aux"]), _ptr(out["kept"]),
                           _ptr(out["offsets"]), _ptr(out["slot_row"]), _ptr(out["row_token"]),
                           _ptr(out["dropped"]))
    if rc != 0:
        raise ValueError("oracle forward failed")
    out["aux"] = float(out["aux"][0])
    out["dropped"] = int(out["dropped"][0])
    return out


def forward_dense(inp, k, mode, capacity_factor=None):
    """O-BF: dense brute force (all experts on all tokens, masked); tiny inputs only."""
    xr, dt = raw(inp["x"])
    wg, _ = raw(inp["w_gate"])
    w1, _ = raw(inp["w1"])
    w2, _ = raw(inp["w2"])
    b1 = raw(inp["b1"])[0] if inp.get("b1") is not None else None
    b2 = raw(inp["b2"])[0] if inp.get("b2") is not None else None
    lb = _f32(inp.get("logit_bias"))
    T, d = xr.shape
    E, h = w1.shape[0], w1.shape[1]
    y = np.empty((T, d))
    lib().orc_forward_dense(T, d, h, E, k, int(mode), dt, float(capacity_factor or 0.0),
                            _ptr(xr), _ptr(wg), _ptr(lb), _ptr(w1), _ptr(b1), _ptr(w2), _ptr(b2),
                            _ptr(y))
    return y


def noisy_routed_reference(k, mode, capacity_factor, gpu_scores, noise_mode, clean_logits):
    """Routing stages on given fp32 selection scores (the GPU's) under routing noise.

    Top-k, counts, capacity and placement follow the scores exactly.  Gate weights and
    the balance loss's f use the scores as logits for the logit-noise modes (1, 3); for
    noise on the probabilities (mode 2) they use `clean_logits` (double), since the
    noisy scores are not a distribution."""
    sc = np.asarray(gpu_scores, dtype=np.float32).astype(np.float64)
    T, E = sc.shape
    idx = topk(sc, k)
    base = sc if noise_mode in (NOISE_GUMBEL, NOISE_LOGIT_SOFTMAX) else np.asarray(clean_logits,
                                                                                 np.float64)
    w = gate_weights(base, idx, mode)
    aux, counts, f, P = aux_loss(softmax(base), idx)
    C = capacity(T, E, capacity_factor)
    disp = dispatch(idx, E, C)
    return dict(idx=idx, w=w, counts=counts, aux=aux, f=f, P=P, C=C, **disp)


def routed_reference(inp, k, mode, capacity_factor, gpu_logits):
    """Routing stages O2..O5 run on given fp32 logits (normally the GPU's own).

    Returns a dict with idx, w, counts, aux, f, P, kept, offsets, slot_row,
    row_token, dropped, C."""
    lg = np.asarray(gpu_logits, dtype=np.float32).astype(np.float64)
    T, E = lg.shape
    p = softmax(lg)
    idx = topk(lg, k)
    w = gate_weights(lg, idx, mode)
    aux, counts, f, P = aux_loss(p, idx)
    C = capacity(T, E, capacity_factor)
    disp = dispatch(idx, E, C)
    return dict(idx=idx, w=w, counts=counts, aux=aux, f=f, P=P, C=C, **disp)
