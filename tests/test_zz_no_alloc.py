"""moe_dispatch_static, the dispatch entry point for callers that cannot allocate.

Some callers of this library cannot pass a workspace: they run under a host framework
that owns all device memory and forbids allocation once it is serving, or they are
plugins handed only their inputs and outputs.  For them moe_dispatch_static keeps the
dispatch scratch in a device array owned by the library.  This test calls it through
the C ABI twice in a row -- a larger batch and then a smaller one with a different
expert count, so the second call runs over the first call's leftover scratch -- and
checks each result against moe_dispatch with a caller workspace.  Dispatch outputs are
integers and copied rows, so they must match bit for bit.  The file is named to be
collected last.
"""

import pytest
import torch

import sparse_mixture_experts_61_b300 as moe
from moe_workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu

CASES = [
    Workload("static_a", T=1000, d=256, h=64, E=16, k=2, dtype="bf16", gate=0,
             capacity_factor=1.0, logit_bias="normal1.5"),
    Workload("static_b", T=300, d=128, h=64, E=64, k=4, dtype="bf16", gate=1,
             capacity_factor=0.0),
]


def _route(w):
    from sparse_mixture_experts_61_b300 import build
    build.build()
    cfg = moe.config_from_workload(w)
    inp = {k: (None if v is None else v.cuda()) for k, v in make_inputs(w, seed=11).items()}
    ws = torch.zeros(moe.moe_stage_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    idx = torch.empty((w.T, w.k), dtype=torch.int32, device="cuda")
    wts = torch.empty((w.T, w.k), dtype=torch.float32, device="cuda")
    moe.moe_route(cfg, inp["x"], inp["w_gate"], inp["logit_bias"], None, idx, wts, None, None, ws)
    return cfg, inp["x"], idx, ws


def _dispatch_outputs(w):
    i32 = dict(dtype=torch.int32, device="cuda")
    return dict(offsets=torch.full((w.E + 1,), -5, **i32), kept=torch.full((w.E,), -5, **i32),
                slot_row=torch.full((w.T, w.k), -5, **i32),
                row_token=torch.full((w.T * w.k,), -5, **i32), dropped=torch.full((1,), -5, **i32),
                x_perm=torch.zeros((w.T * w.k, w.d), dtype=torch.bfloat16, device="cuda"))


def test_dispatch_static_matches_dispatch_twice():
    for w in CASES:
        cfg, x, idx, ws = _route(w)
        ref = _dispatch_outputs(w)
        moe.moe_dispatch(cfg, x, idx, ref["offsets"], ref["kept"], ref["slot_row"], ref["row_token"],
                         ref["dropped"], ref["x_perm"], ws)
        assert moe.moe_device_error(ws) == 0
        got = _dispatch_outputs(w)
        flags = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        moe.moe_dispatch_static(cfg, x, idx, got["offsets"], got["kept"], got["slot_row"],
                                got["row_token"], got["dropped"], got["x_perm"], flags)
        torch.cuda.synchronize()
        assert flags.item() == 0
        for key in ref:
            assert torch.equal(got[key], ref[key]), f"{w.name}: {key} differs"


def test_dispatch_static_without_a_flags_buffer():
    """device_flags = NULL keeps the flag word inside the library's array; the outputs are
    still moe_dispatch's, bit for bit."""
    w = CASES[0]
    cfg, x, idx, ws = _route(w)
    ref = _dispatch_outputs(w)
    moe.moe_dispatch(cfg, x, idx, ref["offsets"], ref["kept"], ref["slot_row"], ref["row_token"],
                     ref["dropped"], ref["x_perm"], ws)
    got = _dispatch_outputs(w)
    moe.moe_dispatch_static(cfg, x, idx, got["offsets"], got["kept"], got["slot_row"],
                            got["row_token"], got["dropped"], got["x_perm"], None)
    torch.cuda.synchronize()
    for key in ref:
        assert torch.equal(got[key], ref[key]), f"{key} differs"


def test_dispatch_static_flags_an_out_of_range_index():
    """Expert indices outside [0, E) (host-written, in-bounds data) are skipped as dropped
    and raise MOE_DEVERR_BAD_INDEX in the caller's flag buffer, as moe_dispatch does."""
    w = CASES[1]
    cfg, x, idx, ws = _route(w)
    idx[5, 1] = w.E
    idx[17, 0] = -3
    ref = _dispatch_outputs(w)
    moe.moe_dispatch(cfg, x, idx, ref["offsets"], ref["kept"], ref["slot_row"], ref["row_token"],
                     ref["dropped"], ref["x_perm"], ws)
    assert moe.moe_device_error(ws) & moe.MOE_DEVERR_BAD_INDEX
    got = _dispatch_outputs(w)
    flags = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    moe.moe_dispatch_static(cfg, x, idx, got["offsets"], got["kept"], got["slot_row"],
                            got["row_token"], got["dropped"], got["x_perm"], flags)
    torch.cuda.synchronize()
    assert flags.item() & moe.MOE_DEVERR_BAD_INDEX
    assert got["slot_row"][5, 1].item() == -1 and got["slot_row"][17, 0].item() == -1
    for key in ref:
        assert torch.equal(got[key], ref[key]), f"{key} differs"


def test_dispatch_static_validates_like_dispatch():
    """A configuration moe_dispatch rejects (here an unknown routing-noise mode) is rejected
    by moe_dispatch_static with the same status, before anything is enqueued."""
    cfg = moe.config(64, 64, 64, 8, 2, "bf16", noise=9)
    buf = torch.zeros(4096, dtype=torch.int32, device="cuda")
    p = buf.data_ptr()
    st_static = moe.lib().moe_dispatch_static(cfg, p, p, p, None, p, p, None, p, None, None)
    st_dispatch = moe.lib().moe_dispatch(cfg, p, p, p, None, p, p, None, p, p, buf.numel() * 4,
                                         None)
    assert st_static == st_dispatch == moe.MOE_ERR_INVALID_ARGUMENT


def test_dispatch_static_rejects_sizes_beyond_its_scratch():
    cells = moe.MOE_DISPATCH_STATIC_MAX_CELLS
    E = 256
    T = (cells // E) * 64 + 1          # one chunk more than the array holds
    cfg = moe.config(T, 64, 64, E, 1, "bf16")
    buf = torch.empty(16, dtype=torch.int32, device="cuda")
    st = moe.lib().moe_dispatch_static(cfg, buf.data_ptr(), buf.data_ptr(), buf.data_ptr(), None,
                                       buf.data_ptr(), buf.data_ptr(), None, buf.data_ptr(), None,
                                       None)
    assert st == moe.MOE_ERR_UNSUPPORTED
