"""Python binding of ``libmoe.so``, the sm_103a top-k Mixture-of-Experts FFN forward.

Argument marshalling only: every function here takes torch CUDA tensors (or None
for optional arguments), passes their device pointers and the current CUDA stream
to the C entry point of the same name declared in ``include/moe.h``, and raises
``MoeError`` on a non-OK status.  No step of the layer runs in Python, and there is
no fallback: if ``libmoe.so`` is missing the import of the library fails loudly.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARGUMENT = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_DEVICE = 5

MOE_F32 = 0
MOE_BF16 = 1
MOE_GATE_TOPK_SOFTMAX = 0
MOE_GATE_SOFTMAX_TOPK_RENORM = 1
MOE_NOISE_NONE = 0
MOE_NOISE_GUMBEL = 1
MOE_NOISE_PROB_GAUSS = 2
MOE_NOISE_LOGIT_SOFTMAX = 3

MOE_ROUTING_TOPK = 0
MOE_ROUTING_EXPERT_CHOICE = 1

MOE_DEVERR_BAD_INDEX = 1
MOE_DEVERR_BAD_ROW = 2
MOE_DEVERR_NONFINITE = 4
MOE_DEVERR_TIMEOUT = 8

# Every C symbol include/moe.h declares.
EXPORTED = ("moe_status_str", "moe_capacity", "moe_workspace_size", "moe_stage_workspace_size",
            "moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_forward",
            "moe_device_error", "moe_dispatch_static", "moe_selftest_wait_timeout",
            "moe_expert_choice_capacity", "moe_expert_choice_workspace_size",
            "moe_expert_choice_forward", "moe_backward_workspace_size", "moe_backward",
            "moe_forward_host_workspace_size", "moe_forward_host")

# Table cells of moe_dispatch_static's library-held scratch (include/moe.h).
MOE_DISPATCH_STATIC_MAX_CELLS = 262144


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_str(status)}")


class MoeConfig(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int32), ("h", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("gate", ctypes.c_int32), ("capacity_factor", ctypes.c_double),
                ("noise", ctypes.c_int32), ("fused_gather", ctypes.c_int32)]


class MoeForwardArgs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "x", "w_gate", "logit_bias", "noise", "w1", "b1", "w2", "b2", "y", "logits", "topk_idx",
        "topk_w",
        "counts", "aux_loss", "offsets", "kept_counts", "slot_row", "row_token", "dropped",
        "routing_stats", "x_perm", "h_act", "y_perm", "h_pre")]


BACKWARD_INPUTS = ("dy", "x", "w_gate", "w1", "w2", "logits", "topk_idx", "topk_w", "counts",
                   "offsets", "slot_row", "x_perm", "h_pre", "h_act", "y_perm")
BACKWARD_OUTPUTS = ("dx", "dw_gate", "dlogit_bias", "dw1", "db1", "dw2", "db2")


class MoeBackwardArgs(ctypes.Structure):
    _fields_ = ([(n, ctypes.c_void_p) for n in BACKWARD_INPUTS] + [("d_aux", ctypes.c_float)] +
                [(n, ctypes.c_void_p) for n in BACKWARD_OUTPUTS])


class MoeExpertChoiceArgs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "x", "w_gate", "logit_bias", "w1", "b1", "w2", "b2", "y", "logits", "probs", "sel_token",
        "sel_w", "token_experts", "unrouted")]


WEIGHTS = ("w_gate", "logit_bias", "w1", "b1", "w2", "b2")


class MoeWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in WEIGHTS]


class MoeHostBatches(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int64), ("x", ctypes.POINTER(ctypes.c_void_p)),
                ("y", ctypes.POINTER(ctypes.c_void_p)), ("aux_loss", ctypes.c_void_p)]


_lib = None


def lib():
    """The loaded ``libmoe.so``; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m sparse_mixture_experts_61_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P, S = ctypes.c_void_p, ctypes.c_size_t
        cfg = ctypes.POINTER(MoeConfig)
        L.moe_status_str.argtypes = [ctypes.c_int]
        L.moe_status_str.restype = ctypes.c_char_p
        L.moe_capacity.argtypes = [cfg, ctypes.POINTER(ctypes.c_int64)]
        L.moe_workspace_size.argtypes = [cfg, ctypes.POINTER(S)]
        L.moe_stage_workspace_size.argtypes = [cfg, ctypes.POINTER(S)]
        L.moe_route.argtypes = [cfg, P, P, P, P, P, P, P, P, P, P, P, S, P]
        L.moe_dispatch.argtypes = [cfg, P, P, P, P, P, P, P, P, P, S, P]
        L.moe_expert_ffn.argtypes = [cfg, P, P, P, P, P, P, P, P, P, S, P]
        L.moe_combine.argtypes = [cfg, P, P, P, P, P, S, P]
        L.moe_forward.argtypes = [cfg, ctypes.POINTER(MoeForwardArgs), P, S, P]
        L.moe_device_error.argtypes = [P, P, ctypes.POINTER(ctypes.c_int32)]
        L.moe_dispatch_static.argtypes = [cfg, P, P, P, P, P, P, P, P, P, P]
        L.moe_selftest_wait_timeout.argtypes = [P, ctypes.c_uint64, P]
        L.moe_expert_choice_capacity.argtypes = [cfg, ctypes.POINTER(ctypes.c_int64)]
        L.moe_expert_choice_workspace_size.argtypes = [cfg, ctypes.POINTER(S)]
        L.moe_expert_choice_forward.argtypes = [cfg, ctypes.POINTER(MoeExpertChoiceArgs), P, S, P]
        L.moe_backward_workspace_size.argtypes = [cfg, ctypes.POINTER(S)]
        L.moe_backward.argtypes = [cfg, ctypes.POINTER(MoeBackwardArgs), P, S, P]
        L.moe_forward_host_workspace_size.argtypes = [cfg, ctypes.c_int32, ctypes.POINTER(S)]
        L.moe_forward_host.argtypes = [cfg, ctypes.c_int32, ctypes.POINTER(MoeWeights),
                                       ctypes.POINTER(MoeHostBatches), P, S, P]
        for name in EXPORTED:
            if name != "moe_status_str":
                getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def status_str(status: int) -> str:
    return lib().moe_status_str(int(status)).decode()


def config(T, d, h, E, k, dtype="bf16", gate=0, capacity_factor=0.0, noise=0,
           fused_gather=0) -> MoeConfig:
    dt = {"f32": MOE_F32, "bf16": MOE_BF16}[dtype] if isinstance(dtype, str) else int(dtype)
    return MoeConfig(int(T), int(d), int(h), int(E), int(k), dt, int(gate),
                     float(capacity_factor or 0.0), int(noise), int(fused_gather))


def config_from_workload(w, noise=0, fused_gather=0) -> MoeConfig:
    """Config for an object with T, d, h, E, k, dtype, gate, capacity_factor attributes."""
    return config(w.T, w.d, w.h, w.E, w.k, w.dtype, w.gate, w.capacity_factor, noise,
                  fused_gather)


def _p(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(status: int, where: str) -> None:
    if status != MOE_OK:
        raise MoeError(status, where)


def moe_capacity(cfg: MoeConfig) -> int:
    v = ctypes.c_int64()
    _check(lib().moe_capacity(ctypes.byref(cfg), ctypes.byref(v)), "moe_capacity")
    return v.value


def moe_workspace_size(cfg: MoeConfig) -> int:
    v = ctypes.c_size_t()
    _check(lib().moe_workspace_size(ctypes.byref(cfg), ctypes.byref(v)), "moe_workspace_size")
    return v.value


def moe_stage_workspace_size(cfg: MoeConfig) -> int:
    v = ctypes.c_size_t()
    _check(lib().moe_stage_workspace_size(ctypes.byref(cfg), ctypes.byref(v)),
           "moe_stage_workspace_size")
    return v.value


def moe_route(cfg, x, w_gate, logit_bias, logits, topk_idx, topk_w, counts, aux_loss, ws,
              stream=None, routing_stats=None, noise=None):
    _check(lib().moe_route(ctypes.byref(cfg), _p(x), _p(w_gate), _p(logit_bias), _p(noise),
                           _p(logits),
                           _p(topk_idx), _p(topk_w), _p(counts), _p(aux_loss), _p(routing_stats),
                           _p(ws), ws.numel() * ws.element_size(), _stream(stream)), "moe_route")


def moe_dispatch(cfg, x, topk_idx, offsets, kept_counts, slot_row, row_token, dropped, x_perm, ws,
                 stream=None):
    _check(lib().moe_dispatch(ctypes.byref(cfg), _p(x), _p(topk_idx), _p(offsets),
                              _p(kept_counts), _p(slot_row), _p(row_token), _p(dropped),
                              _p(x_perm), _p(ws), ws.numel() * ws.element_size(),
                              _stream(stream)), "moe_dispatch")


def moe_expert_ffn(cfg, x_perm, offsets, w1, b1, w2, b2, h_buf, y_perm, ws, stream=None):
    _check(lib().moe_expert_ffn(ctypes.byref(cfg), _p(x_perm), _p(offsets), _p(w1), _p(b1),
                                _p(w2), _p(b2), _p(h_buf), _p(y_perm), _p(ws),
                                ws.numel() * ws.element_size(), _stream(stream)),
           "moe_expert_ffn")


def moe_combine(cfg, y_perm, slot_row, topk_w, y, ws, stream=None):
    _check(lib().moe_combine(ctypes.byref(cfg), _p(y_perm), _p(slot_row), _p(topk_w), _p(y),
                             _p(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_combine")


FORWARD_INPUTS = ("x", "w_gate", "logit_bias", "noise", "w1", "b1", "w2", "b2")
FORWARD_OUTPUTS = ("y", "logits", "topk_idx", "topk_w", "counts", "aux_loss", "offsets",
                   "kept_counts", "slot_row", "row_token", "dropped", "routing_stats", "x_perm",
                   "h_act", "y_perm", "h_pre")

# Order of the routing statistics (include/moe.h, MOE_STAT_*).
ROUTING_STATS = ("cv", "dead_ratio", "max_over_avg", "entropy", "effective_experts",
                 "count_cv_loss")


def forward_args(inputs: dict, outputs: dict) -> MoeForwardArgs:
    """Build the moe_forward_args struct from dicts of tensors (missing keys -> NULL)."""
    a = MoeForwardArgs()
    for n in FORWARD_INPUTS:
        setattr(a, n, _p(inputs.get(n)))
    for n in FORWARD_OUTPUTS:
        setattr(a, n, _p(outputs.get(n)))
    return a


def moe_forward(cfg, inputs: dict, outputs: dict, ws, stream=None, args: MoeForwardArgs = None):
    """One call of the whole layer.  ``inputs`` holds x, w_gate, w1, w2 and optionally
    logit_bias, b1, b2; ``outputs`` holds y and any optional outputs to expose."""
    if args is None:
        args = forward_args(inputs, outputs)
    _check(lib().moe_forward(ctypes.byref(cfg), ctypes.byref(args), _p(ws),
                             ws.numel() * ws.element_size(), _stream(stream)), "moe_forward")


def moe_device_error(ws, stream=None) -> int:
    """Waits for the stream and returns the device flag word (0 = clean)."""
    v = ctypes.c_int32()
    s = lib().moe_device_error(_p(ws), _stream(stream), ctypes.byref(v))
    if s not in (MOE_OK, MOE_ERR_DEVICE):
        raise MoeError(s, "moe_device_error")
    return v.value


def moe_dispatch_static(cfg, x, topk_idx, offsets, kept_counts, slot_row, row_token, dropped,
                        x_perm, device_flags=None, stream=None):
    """moe_dispatch for callers that cannot allocate a workspace: the library keeps the
    scratch in its own device array (see include/moe.h for the size limit and the rule
    that overlapping calls must be serialised)."""
    _check(lib().moe_dispatch_static(ctypes.byref(cfg), _p(x), _p(topk_idx), _p(offsets),
                                     _p(kept_counts), _p(slot_row), _p(row_token), _p(dropped),
                                     _p(x_perm), _p(device_flags), _stream(stream)),
           "moe_dispatch_static")


def moe_selftest_wait_timeout(device_flags, limit_ns: int, stream=None) -> None:
    """Runs the bounded pipeline wait on a barrier nothing completes (see moe.h)."""
    _check(lib().moe_selftest_wait_timeout(_p(device_flags), int(limit_ns), _stream(stream)),
           "moe_selftest_wait_timeout")


EC_INPUTS = ("x", "w_gate", "logit_bias", "w1", "b1", "w2", "b2")
EC_OUTPUTS = ("y", "logits", "probs", "sel_token", "sel_w", "token_experts", "unrouted")


def moe_expert_choice_capacity(cfg: MoeConfig) -> int:
    v = ctypes.c_int64()
    _check(lib().moe_expert_choice_capacity(ctypes.byref(cfg), ctypes.byref(v)),
           "moe_expert_choice_capacity")
    return v.value


def moe_expert_choice_workspace_size(cfg: MoeConfig) -> int:
    v = ctypes.c_size_t()
    _check(lib().moe_expert_choice_workspace_size(ctypes.byref(cfg), ctypes.byref(v)),
           "moe_expert_choice_workspace_size")
    return v.value


def expert_choice_args(inputs: dict, outputs: dict) -> MoeExpertChoiceArgs:
    """Build the moe_expert_choice_args struct (missing keys -> NULL)."""
    a = MoeExpertChoiceArgs()
    for n in EC_INPUTS:
        setattr(a, n, _p(inputs.get(n)))
    for n in EC_OUTPUTS:
        setattr(a, n, _p(outputs.get(n)))
    return a


def moe_expert_choice_forward(cfg, inputs: dict, outputs: dict, ws, stream=None,
                              args: MoeExpertChoiceArgs = None):
    """The expert-choice layer: each expert takes its C highest-probability tokens."""
    if args is None:
        args = expert_choice_args(inputs, outputs)
    _check(lib().moe_expert_choice_forward(ctypes.byref(cfg), ctypes.byref(args), _p(ws),
                                           ws.numel() * ws.element_size(), _stream(stream)),
           "moe_expert_choice_forward")


def moe_backward_workspace_size(cfg: MoeConfig) -> int:
    v = ctypes.c_size_t()
    _check(lib().moe_backward_workspace_size(ctypes.byref(cfg), ctypes.byref(v)),
           "moe_backward_workspace_size")
    return v.value


def backward_args(inputs: dict, outputs: dict, d_aux: float) -> MoeBackwardArgs:
    """Build the moe_backward_args struct (missing keys -> NULL)."""
    a = MoeBackwardArgs()
    for n in BACKWARD_INPUTS:
        setattr(a, n, _p(inputs.get(n)))
    a.d_aux = float(d_aux)
    for n in BACKWARD_OUTPUTS:
        setattr(a, n, _p(outputs.get(n)))
    return a


def moe_backward(cfg, inputs: dict, outputs: dict, d_aux: float, ws, stream=None,
                 args: MoeBackwardArgs = None):
    """Gradients of the layer.  ``inputs``: dy and the forward's inputs / saved outputs
    (BACKWARD_INPUTS); ``outputs``: dx and any parameter gradients wanted."""
    if args is None:
        args = backward_args(inputs, outputs, d_aux)
    _check(lib().moe_backward(ctypes.byref(cfg), ctypes.byref(args), _p(ws),
                              ws.numel() * ws.element_size(), _stream(stream)), "moe_backward")


_ROUTING = {"topk": MOE_ROUTING_TOPK, "expert_choice": MOE_ROUTING_EXPERT_CHOICE}


def moe_forward_host_workspace_size(cfg: MoeConfig, routing: str = "topk") -> int:
    v = ctypes.c_size_t()
    _check(lib().moe_forward_host_workspace_size(ctypes.byref(cfg), _ROUTING[routing],
                                                 ctypes.byref(v)),
           "moe_forward_host_workspace_size")
    return v.value


def moe_forward_host(cfg, weights: dict, xs, ys, ws, stream=None, routing: str = "topk",
                     aux_loss=None):
    """The layer over the host batches ``xs[i]`` -> ``ys[i]`` (CPU tensors, page-locked
    for the copies to overlap the layer), weights on the device.  ``aux_loss``: an
    optional CPU fp32 tensor of len(xs) for each batch's balance statistic.  Enqueued
    on ``stream``; synchronise it before reading ``ys``."""
    n = len(xs)
    if len(ys) != n:
        raise ValueError("xs and ys differ in length")
    w = MoeWeights()
    for name in WEIGHTS:
        setattr(w, name, _p(weights.get(name)))
    xa = (ctypes.c_void_p * max(n, 1))(*[_p(t) for t in xs])
    ya = (ctypes.c_void_p * max(n, 1))(*[_p(t) for t in ys])
    b = MoeHostBatches(n, ctypes.cast(xa, ctypes.POINTER(ctypes.c_void_p)),
                       ctypes.cast(ya, ctypes.POINTER(ctypes.c_void_p)), _p(aux_loss))
    _check(lib().moe_forward_host(ctypes.byref(cfg), _ROUTING[routing], ctypes.byref(w),
                                  ctypes.byref(b), _p(ws), ws.numel() * ws.element_size(),
                                  _stream(stream)), "moe_forward_host")
