"""Host-side checks of the C ABI (no GPU needed, no kernel launched).

The library is built for sm_103a and loaded; every function include/moe.h declares
must be exported; struct layouts must match the header; and every host-side
validation path must return its documented status before touching the GPU (all
pointers below are fake, 16-byte-aligned integers that are never dereferenced).
"""

import ctypes
import os
import re

import pytest

import oracle
import sparse_mixture_experts_61_b300 as moe
from sparse_mixture_experts_61_b300 import build as moe_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")

FAKE = 0x10000          # aligned fake device address, never dereferenced
FAKE_ODD = 0x10004      # 4-byte aligned but not 16-byte aligned


@pytest.fixture(scope="module")
def L():
    moe_build.build()
    return moe.lib()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:moe_status|const char\*)\s+(moe_\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_forward",
              "moe_workspace_size", "moe_device_error", "moe_status_str"):
        assert n in names
    assert sorted(moe.EXPORTED) == names


def test_library_exports_every_declared_symbol(L):
    for n in declared_functions():
        assert hasattr(L, n), f"{n} not exported"
    # only the C API is visible
    out = os.popen(f"nm -D --defined-only {moe.LIB_PATH}").read()
    exported = sorted(set(re.findall(r" T (moe_\w+)", out)))
    assert exported == declared_functions()


def test_struct_layouts_match_header():
    assert ctypes.sizeof(moe.MoeConfig) == 48
    assert moe.MoeConfig.noise.offset == 40
    assert moe.MoeConfig.capacity_factor.offset == 32
    assert ctypes.sizeof(moe.MoeForwardArgs) == 24 * 8
    assert ctypes.sizeof(moe.MoeBackwardArgs) == 15 * 8 + 8 + 7 * 8
    assert moe.MoeBackwardArgs.d_aux.offset == 15 * 8
    assert moe.MoeBackwardArgs.dx.offset == 16 * 8
    assert ctypes.sizeof(moe.MoeExpertChoiceArgs) == 14 * 8


def test_status_strings(L):
    for s, name in [(0, "MOE_OK"), (1, "MOE_ERR_INVALID_ARGUMENT"), (2, "MOE_ERR_UNSUPPORTED"),
                    (3, "MOE_ERR_WORKSPACE"), (4, "MOE_ERR_CUDA"), (5, "MOE_ERR_DEVICE")]:
        assert moe.status_str(s) == name
    assert moe.status_str(99) == "MOE_ERR_UNKNOWN"


@pytest.mark.parametrize("kw,status", [
    (dict(k=0), moe.MOE_ERR_UNSUPPORTED),
    (dict(k=9, E=16), moe.MOE_ERR_UNSUPPORTED),
    (dict(k=4, E=3), moe.MOE_ERR_UNSUPPORTED),
    (dict(E=257), moe.MOE_ERR_UNSUPPORTED),
    (dict(d=12), moe.MOE_ERR_UNSUPPORTED),
    (dict(h=0), moe.MOE_ERR_UNSUPPORTED),
    (dict(T=-1), moe.MOE_ERR_UNSUPPORTED),
    (dict(T=2**30, k=2), moe.MOE_ERR_UNSUPPORTED),
    (dict(dtype=7), moe.MOE_ERR_INVALID_ARGUMENT),
    (dict(gate=2), moe.MOE_ERR_INVALID_ARGUMENT),
    (dict(capacity_factor=float("nan")), moe.MOE_ERR_INVALID_ARGUMENT),
    (dict(noise=4), moe.MOE_ERR_INVALID_ARGUMENT),
    (dict(noise=-1), moe.MOE_ERR_INVALID_ARGUMENT),
    (dict(fused_gather=2), moe.MOE_ERR_INVALID_ARGUMENT),
    (dict(fused_gather=1, dtype=0), moe.MOE_ERR_UNSUPPORTED),
])
def test_config_validation(L, kw, status):
    base = dict(T=64, d=64, h=128, E=8, k=2, dtype=1, gate=0, capacity_factor=0.0, noise=0,
                fused_gather=0)
    base.update(kw)
    cfg = moe.MoeConfig(base["T"], base["d"], base["h"], base["E"], base["k"], base["dtype"],
                        base["gate"], base["capacity_factor"], base["noise"], base["fused_gather"])
    n = ctypes.c_size_t()
    assert L.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == status
    assert L.moe_route(ctypes.byref(cfg), FAKE, FAKE, None, None, None, FAKE, FAKE, None, None, None, FAKE, 1 << 40, None) == status


def test_null_config_and_outputs(L):
    n = ctypes.c_size_t()
    assert L.moe_workspace_size(None, ctypes.byref(n)) == moe.MOE_ERR_INVALID_ARGUMENT
    cfg = moe.config(64, 64, 128, 8, 2)
    assert L.moe_workspace_size(ctypes.byref(cfg), None) == moe.MOE_ERR_INVALID_ARGUMENT
    assert L.moe_forward(ctypes.byref(cfg), None, FAKE, 1 << 40, None) == moe.MOE_ERR_INVALID_ARGUMENT


def _ws(cfg):
    return moe.moe_stage_workspace_size(cfg), moe.moe_workspace_size(cfg)


def test_workspace_sizes_cover_buffers(L):
    cfg = moe.config(4096, 4096, 14336, 8, 2, "bf16")
    stage, full = _ws(cfg)
    rows = 4096 * 2
    assert full >= stage + rows * (4096 + 14336 + 4096) * 2
    assert stage >= 4096 * 8 * 4       # logits
    assert full % 256 == 0 and stage % 256 == 0
    c32 = moe.config(4096, 4096, 14336, 8, 2, "f32")
    assert moe.moe_workspace_size(c32) > full


def test_fused_gather_drops_the_row_copy_from_the_workspace(L):
    """With fused_gather the forward's workspace holds no expert-ordered copy of the token
    rows: exactly T*k*d*2 bytes less (rounded to the 256-byte region alignment); the stage
    workspace is unchanged, and expert-choice routing refuses the flag."""
    T, d, h, E, k = 8192, 7168, 2048, 256, 8
    plain = moe.config(T, d, h, E, k, "bf16", gate=1)
    fused = moe.config(T, d, h, E, k, "bf16", gate=1, fused_gather=1)
    assert moe.moe_workspace_size(plain) - moe.moe_workspace_size(fused) == T * k * d * 2
    assert moe.moe_stage_workspace_size(plain) == moe.moe_stage_workspace_size(fused)
    ec = moe.config(T, d, h, E, k, "bf16", gate=1, capacity_factor=8.0, fused_gather=1)
    n = ctypes.c_size_t()
    assert L.moe_expert_choice_workspace_size(ctypes.byref(ec), ctypes.byref(n)) == \
        moe.MOE_ERR_UNSUPPORTED


def test_required_pointers_and_alignment(L):
    cfg = moe.config(64, 64, 128, 8, 2)
    big = 1 << 40
    INV = moe.MOE_ERR_INVALID_ARGUMENT
    # moe_route: x, w_gate, topk_idx, topk_w required; x 16-byte aligned
    assert L.moe_route(ctypes.byref(cfg), None, FAKE, None, None, None, FAKE, FAKE, None, None, None, FAKE, big, None) == INV
    assert L.moe_route(ctypes.byref(cfg), FAKE_ODD, FAKE, None, None, None, FAKE, FAKE, None, None, None, FAKE, big, None) == INV
    assert L.moe_route(ctypes.byref(cfg), FAKE, FAKE, None, None, None, None, FAKE, None, None, None, FAKE, big, None) == INV
    # moe_dispatch: x_perm required
    assert L.moe_dispatch(ctypes.byref(cfg), FAKE, FAKE, FAKE, None, FAKE, FAKE, None, None, FAKE, big, None) == INV
    # moe_expert_ffn: w1 required, b1 optional but aligned
    assert L.moe_expert_ffn(ctypes.byref(cfg), FAKE, FAKE, None, None, FAKE, None, FAKE, FAKE, FAKE, big, None) == INV
    assert L.moe_expert_ffn(ctypes.byref(cfg), FAKE, FAKE, FAKE, FAKE_ODD, FAKE, None, FAKE, FAKE, FAKE, big, None) == INV
    # moe_combine: y required
    assert L.moe_combine(ctypes.byref(cfg), FAKE, FAKE, FAKE, None, FAKE, big, None) == INV


def test_workspace_too_small_is_rejected_before_launch(L):
    cfg = moe.config(64, 64, 128, 8, 2)
    stage, full = _ws(cfg)
    WS = moe.MOE_ERR_WORKSPACE
    assert L.moe_route(ctypes.byref(cfg), FAKE, FAKE, None, None, None, FAKE, FAKE, None, None, None, FAKE, stage - 1, None) == WS
    assert L.moe_route(ctypes.byref(cfg), FAKE, FAKE, None, None, None, FAKE, FAKE, None, None, None, None, stage, None) == WS
    assert L.moe_dispatch(ctypes.byref(cfg), FAKE, FAKE, FAKE, None, FAKE, FAKE, None, FAKE, FAKE, stage - 1, None) == WS
    assert L.moe_expert_ffn(ctypes.byref(cfg), FAKE, FAKE, FAKE, None, FAKE, None, FAKE, FAKE, FAKE, 16, None) == WS
    assert L.moe_combine(ctypes.byref(cfg), FAKE, FAKE, FAKE, FAKE, FAKE, 0, None) == WS
    args = moe.MoeForwardArgs(x=FAKE, w_gate=FAKE, w1=FAKE, w2=FAKE, y=FAKE)
    assert L.moe_forward(ctypes.byref(cfg), ctypes.byref(args), FAKE, full - 1, None) == WS
    assert L.moe_device_error(None, None, None) == WS


@pytest.mark.parametrize("T,E,cf", [(8192, 128, 1.25), (1000, 16, 1.25), (3, 4, 1.0), (10, 3, 0.7),
                                    (64, 64, 0.0), (5, 8, -1.0)])
def test_capacity_matches_oracle(L, T, E, cf):
    cfg = moe.config(T, 64, 64, E, 1, "bf16", 1, cf)
    assert moe.moe_capacity(cfg) == oracle.capacity(T, E, cf if cf > 0 else None)


def test_noise_input_required_when_noise_is_on(L):
    cfg = moe.config(64, 64, 128, 8, 2, noise=moe.MOE_NOISE_GUMBEL)
    assert L.moe_route(ctypes.byref(cfg), FAKE, FAKE, None, None, None, FAKE, FAKE, None, None,
                       None, FAKE, 1 << 40, None) == moe.MOE_ERR_INVALID_ARGUMENT
    args = moe.MoeForwardArgs(x=FAKE, w_gate=FAKE, w1=FAKE, w2=FAKE, y=FAKE)
    assert L.moe_forward(ctypes.byref(cfg), ctypes.byref(args), FAKE, 1 << 40,
                         None) == moe.MOE_ERR_INVALID_ARGUMENT


def test_selftest_validation_before_launch(L):
    assert L.moe_selftest_wait_timeout(None, 1000, None) == moe.MOE_ERR_INVALID_ARGUMENT
    assert L.moe_selftest_wait_timeout(FAKE_ODD + 1, 1000, None) == moe.MOE_ERR_INVALID_ARGUMENT
    assert L.moe_selftest_wait_timeout(FAKE, 0, None) == moe.MOE_ERR_INVALID_ARGUMENT
    assert L.moe_selftest_wait_timeout(FAKE, 3 * 10**9, None) == moe.MOE_ERR_INVALID_ARGUMENT


# ---------------------------------------------------------------- expert choice
@pytest.mark.parametrize("kw,status", [
    (dict(capacity_factor=0.0), moe.MOE_ERR_INVALID_ARGUMENT),
    (dict(capacity_factor=-1.0), moe.MOE_ERR_INVALID_ARGUMENT),
    (dict(capacity_factor=float("inf")), moe.MOE_ERR_INVALID_ARGUMENT),
    (dict(noise=1), moe.MOE_ERR_INVALID_ARGUMENT),
    (dict(dtype=3), moe.MOE_ERR_INVALID_ARGUMENT),
    (dict(E=0), moe.MOE_ERR_UNSUPPORTED),
    (dict(E=257), moe.MOE_ERR_UNSUPPORTED),
    (dict(d=4), moe.MOE_ERR_UNSUPPORTED),
    (dict(T=-5), moe.MOE_ERR_UNSUPPORTED),
    (dict(T=2**31), moe.MOE_ERR_UNSUPPORTED),
    (dict(T=2**26, E=256, capacity_factor=64.0), moe.MOE_ERR_UNSUPPORTED),  # E*C >= 2^31
    (dict(k=0, gate=9), moe.MOE_OK),      # k and gate are not read
    (dict(E=1), moe.MOE_OK),
])
def test_expert_choice_config_validation(L, kw, status):
    base = dict(T=64, d=64, h=128, E=8, k=2, dtype="bf16", gate=0, capacity_factor=1.0)
    base.update(kw)
    cfg = moe.config(**base)
    n = ctypes.c_size_t()
    assert L.moe_expert_choice_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == status
    c = ctypes.c_int64()
    assert L.moe_expert_choice_capacity(ctypes.byref(cfg), ctypes.byref(c)) == status


@pytest.mark.parametrize("T,E,cf", [(4096, 8, 2.0), (777, 8, 2.0), (64, 64, 1.0), (10, 3, 0.7),
                                    (5, 8, 100.0), (1, 1, 1.0), (0, 4, 1.0)])
def test_expert_choice_capacity_is_clamped_capacity_rule(L, T, E, cf):
    cfg = moe.config(T, 64, 64, E, 1, "bf16", 0, cf)
    assert moe.moe_expert_choice_capacity(cfg) == min(T, oracle.capacity(T, E, cf))


def test_expert_choice_pointer_and_workspace_checks(L):
    cfg = moe.config(64, 64, 128, 8, 2, capacity_factor=2.0)
    need = moe.moe_expert_choice_workspace_size(cfg)
    C = moe.moe_expert_choice_capacity(cfg)
    # the row buffers alone: E*C rows of d, h and d bf16 elements
    assert need >= 8 * C * (64 + 128 + 64) * 2
    INV, WS = moe.MOE_ERR_INVALID_ARGUMENT, moe.MOE_ERR_WORKSPACE
    ok = dict(x=FAKE, w_gate=FAKE, w1=FAKE, w2=FAKE, y=FAKE)
    f = L.moe_expert_choice_forward
    assert f(ctypes.byref(cfg), None, FAKE, need, None) == INV
    for drop in ok:
        a = moe.MoeExpertChoiceArgs(**{k: v for k, v in ok.items() if k != drop})
        assert f(ctypes.byref(cfg), ctypes.byref(a), FAKE, need, None) == INV, drop
    for odd in ("x", "w1", "y", "b2", "probs"):
        a = moe.MoeExpertChoiceArgs(**dict(ok, **{odd: FAKE_ODD}))
        assert f(ctypes.byref(cfg), ctypes.byref(a), FAKE, need, None) == INV, odd
    a = moe.MoeExpertChoiceArgs(**dict(ok, sel_token=FAKE + 2))
    assert f(ctypes.byref(cfg), ctypes.byref(a), FAKE, need, None) == INV
    a = moe.MoeExpertChoiceArgs(**ok)
    assert f(ctypes.byref(cfg), ctypes.byref(a), FAKE, need - 1, None) == WS
    assert f(ctypes.byref(cfg), ctypes.byref(a), None, need, None) == WS
    assert f(ctypes.byref(cfg), ctypes.byref(a), FAKE_ODD, need, None) == WS


# ---------------------------------------------------------------- backward
@pytest.mark.parametrize("kw,status", [
    (dict(dtype="f32"), moe.MOE_ERR_UNSUPPORTED),
    (dict(noise=1), moe.MOE_ERR_UNSUPPORTED),
    (dict(k=9), moe.MOE_ERR_UNSUPPORTED),
    (dict(gate=5), moe.MOE_ERR_INVALID_ARGUMENT),
    (dict(), moe.MOE_OK),
])
def test_backward_config_validation(L, kw, status):
    base = dict(T=64, d=64, h=128, E=8, k=2, dtype="bf16", gate=0, capacity_factor=0.0)
    base.update(kw)
    cfg = moe.config(**base)
    n = ctypes.c_size_t()
    assert L.moe_backward_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == status


def test_backward_pointer_and_workspace_checks(L):
    cfg = moe.config(64, 64, 128, 8, 2)
    need = moe.moe_backward_workspace_size(cfg)
    assert need >= 64 * 2 * (64 + 128 + 64) * 2  # dYp, dA, dXp row buffers
    INV, WS = moe.MOE_ERR_INVALID_ARGUMENT, moe.MOE_ERR_WORKSPACE
    ok = {n: FAKE for n in moe.BACKWARD_INPUTS}
    ok["dx"] = FAKE
    f = L.moe_backward

    def args(**kw):
        d = dict(ok, **kw)
        a = moe.MoeBackwardArgs()
        for n, v in d.items():
            setattr(a, n, v)
        return a

    assert f(ctypes.byref(cfg), None, FAKE, need, None) == INV
    for drop in list(ok):
        a = args(**{drop: None})
        assert f(ctypes.byref(cfg), ctypes.byref(a), FAKE, need, None) == INV, drop
    a = args(dw1=FAKE_ODD)
    assert f(ctypes.byref(cfg), ctypes.byref(a), FAKE, need, None) == INV
    a = args(d_aux=float("nan"))
    assert f(ctypes.byref(cfg), ctypes.byref(a), FAKE, need, None) == INV
    a = args()
    assert f(ctypes.byref(cfg), ctypes.byref(a), FAKE, need - 1, None) == WS


# ---------------------------------------------------------------- host batches
def test_host_batch_struct_layouts():
    assert ctypes.sizeof(moe.MoeWeights) == 6 * 8
    assert ctypes.sizeof(moe.MoeHostBatches) == 4 * 8
    assert moe.MoeHostBatches.aux_loss.offset == 3 * 8


@pytest.mark.parametrize("routing,cf", [("topk", 0.0), ("topk", 1.25), ("expert_choice", 2.0)])
def test_host_workspace_holds_layer_and_two_slots(L, routing, cf):
    for dt, s in (("bf16", 2), ("f32", 4)):
        cfg = moe.config(300, 64, 128, 8, 2, dt, 0, cf)
        fwd = (moe.moe_workspace_size(cfg) if routing == "topk"
               else moe.moe_expert_choice_workspace_size(cfg))
        need = moe.moe_forward_host_workspace_size(cfg, routing)
        assert need >= fwd + 4 * 300 * 64 * s
        assert need % 256 == 0


def test_host_forward_validation_before_launch(L):
    cfg = moe.config(64, 64, 128, 8, 2)
    need = moe.moe_forward_host_workspace_size(cfg)
    INV, WS, UNS = moe.MOE_ERR_INVALID_ARGUMENT, moe.MOE_ERR_WORKSPACE, moe.MOE_ERR_UNSUPPORTED
    f = L.moe_forward_host
    w = moe.MoeWeights(w_gate=FAKE, w1=FAKE, w2=FAKE)
    ptrs = (ctypes.c_void_p * 2)(FAKE, FAKE)
    pp = ctypes.cast(ptrs, ctypes.POINTER(ctypes.c_void_p))
    b = moe.MoeHostBatches(2, pp, pp, None)
    TOPK, EC = moe.MOE_ROUTING_TOPK, moe.MOE_ROUTING_EXPERT_CHOICE

    def call(cfg=cfg, routing=TOPK, w=w, b=b, ws=FAKE, n=need):
        return f(ctypes.byref(cfg), routing, ctypes.byref(w) if w is not None else None,
                 ctypes.byref(b) if b is not None else None, ws, n, None)

    assert call(routing=7) == INV
    assert call(w=None) == INV
    assert call(b=None) == INV
    assert call(b=moe.MoeHostBatches(0, pp, pp, None)) == INV
    assert call(b=moe.MoeHostBatches(2, None, pp, None)) == INV
    nulls = (ctypes.c_void_p * 2)(FAKE, None)
    np_ = ctypes.cast(nulls, ctypes.POINTER(ctypes.c_void_p))
    assert call(b=moe.MoeHostBatches(2, pp, np_, None)) == INV
    assert call(n=need - 1) == WS
    assert call(ws=None) == WS
    assert call(ws=FAKE_ODD) == WS
    # the layer's own checks of the weights
    assert call(w=moe.MoeWeights(w_gate=FAKE, w1=FAKE)) == INV
    assert call(w=moe.MoeWeights(w_gate=FAKE, w1=FAKE, w2=FAKE_ODD)) == INV
    noisy = moe.config(64, 64, 128, 8, 2, noise=moe.MOE_NOISE_GUMBEL)
    assert call(cfg=noisy, n=moe.moe_forward_host_workspace_size(noisy)) == UNS
    assert call(cfg=moe.config(64, 60, 128, 8, 2)) == UNS
    ec = moe.config(64, 64, 128, 8, 2, capacity_factor=2.0)
    need_ec = moe.moe_forward_host_workspace_size(ec, "expert_choice")
    aux = (ctypes.c_float * 2)()
    assert call(cfg=ec, routing=EC, n=need_ec,
                b=moe.MoeHostBatches(2, pp, pp, ctypes.addressof(aux))) == INV
    assert call(cfg=moe.config(64, 64, 128, 8, 2), routing=EC) == INV  # EC needs cf > 0
