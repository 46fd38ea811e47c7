"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

For each workload: the router logits against the oracle's contraction; every routing
and indexing output bit-exact against the oracle's routing stages run on the GPU's
own fp32 logits; the gate weights and balance loss within their tolerances; the
output y against the oracle's expert path evaluated on those routing decisions; and
a fully independent oracle run, where only near-tie tokens may route differently.
Reduced-size variants run element by element on every token; the full-size
workloads (the sizes the benchmark times, through the same moe_forward call) are
checked exactly on routing and on sampled tokens for y.
"""

import numpy as np
import pytest
import torch

import moe_testlib as tl
import oracle
import sparse_mixture_experts_61_b300 as moe
from moe_workloads import PARITY_WORKLOADS, WORKLOADS, Workload, capacity_factor_or_none, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_mixture_experts_61_b300 import build
    build.build()
    moe.lib()


check_routing_exact = tl.check_routing_exact


@pytest.mark.parametrize("name", list(PARITY_WORKLOADS))
def test_forward_parity(name):
    w = PARITY_WORKLOADS[name]
    cf = capacity_factor_or_none(w)
    inp = make_inputs(w, seed=0)
    r = tl.run_forward(w, tl.to_device(inp))
    assert r["flags"] == 0
    g = tl.host(r["outs"])

    lg_ref = oracle.logits(inp["x"], inp["w_gate"], inp["logit_bias"])
    assert float(np.abs(g["logits"] - lg_ref).max()) <= tl.logits_tol(lg_ref)

    ref = oracle.routed_reference(None, w.k, w.gate, cf, g["logits"])
    check_routing_exact(g, ref)

    y_ref = tl.y_on_routing(inp, ref["idx"], ref["slot_row"], ref["w"])
    assert tl.max_rel_err(g["y"], y_ref) <= tl.TOL_Y[w.dtype]
    all_dropped = np.all(ref["slot_row"] < 0, axis=1)
    assert np.all(g["y"][all_dropped] == 0.0)

    # Fully independent oracle run: only near-tie tokens may route differently.
    full = oracle.forward(inp, w.k, w.gate, cf)
    gaps = tl.topk_gaps(full["logits"], w.k)
    differ = np.any(full["idx"] != g["topk_idx"], axis=1)
    assert np.all(gaps[differ] < tl.NEAR_TIE), "a routing flip away from a near-tie"
    same = ~differ
    if cf is not None:
        same &= np.all((full["slot_row"] >= 0) == (g["slot_row"] >= 0), axis=1)
    scale = float(np.abs(full["y"]).max())
    assert float(np.abs(g["y"][same] - full["y"][same]).max()) <= tl.TOL_Y[w.dtype] * scale
    print(f"{name}: M={int(g['offsets'][-1])} dropped={int(g['dropped'][0])} "
          f"y_err={tl.max_rel_err(g['y'], y_ref):.2e} near_tie_flips={int(differ.sum())}")


@pytest.mark.parametrize("name", list(PARITY_WORKLOADS))
def test_stage_calls_match_forward(name):
    """moe_route -> moe_dispatch -> moe_expert_ffn -> moe_combine reproduce moe_forward
    bit for bit, and the dispatch gather copies exactly x[row_token]."""
    w = PARITY_WORKLOADS[name]
    dev = tl.to_device(make_inputs(w, seed=0))
    r = tl.run_forward(w, dev)
    fw = tl.host(r["outs"])
    cfg = r["cfg"]
    T, k, E, d, h = w.T, w.k, w.E, w.d, w.h
    ws = tl.poisoned_workspace(moe.moe_stage_workspace_size(cfg))
    i32 = dict(dtype=torch.int32, device="cuda")
    f32 = dict(dtype=torch.float32, device="cuda")
    logits = torch.empty((T, E), **f32)
    idx = torch.empty((T, k), **i32)
    wts = torch.empty((T, k), **f32)
    counts = torch.empty((E,), **i32)
    aux = torch.empty((1,), **f32)
    stats = torch.empty((6,), **f32)
    moe.moe_route(cfg, dev["x"], dev["w_gate"], dev["logit_bias"], logits, idx, wts, counts, aux, ws,
                  routing_stats=stats)
    assert moe.moe_device_error(ws) == 0
    # logits kept inside the workspace instead of a caller buffer: same decisions
    idx2 = torch.empty_like(idx)
    wts2 = torch.empty_like(wts)
    moe.moe_route(cfg, dev["x"], dev["w_gate"], dev["logit_bias"], None, idx2, wts2, None, None, ws)
    assert torch.equal(idx, idx2) and torch.equal(wts, wts2)

    offsets = torch.empty((E + 1,), **i32)
    kept = torch.empty((E,), **i32)
    slot_row = torch.empty((T, k), **i32)
    row_token = torch.empty((T * k,), **i32)
    dropped = torch.empty((1,), **i32)
    x_perm = torch.full((T * k, d), float("nan"), dtype=w.torch_dtype, device="cuda")
    moe.moe_dispatch(cfg, dev["x"], idx, offsets, kept, slot_row, row_token, dropped, x_perm, ws)
    assert moe.moe_device_error(ws) == 0
    h_buf = torch.empty((T * k, h), dtype=w.torch_dtype, device="cuda")
    y_perm = torch.empty((T * k, d), dtype=w.torch_dtype, device="cuda")
    moe.moe_expert_ffn(cfg, x_perm, offsets, dev["w1"], dev["b1"], dev["w2"], dev["b2"], h_buf,
                       y_perm, ws)
    y = torch.empty((T, d), dtype=w.torch_dtype, device="cuda")
    moe.moe_combine(cfg, y_perm, slot_row, wts, y, ws)
    assert moe.moe_device_error(ws) == 0

    for key, t in [("logits", logits), ("topk_idx", idx), ("topk_w", wts), ("counts", counts),
                   ("aux_loss", aux), ("routing_stats", stats), ("offsets", offsets),
                   ("kept_counts", kept),
                   ("slot_row", slot_row), ("row_token", row_token), ("dropped", dropped), ("y", y)]:
        got = t.float().cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()
        np.testing.assert_array_equal(got, fw[key], err_msg=key)
    M = int(offsets[-1])
    rt = row_token[:M].long()
    assert torch.equal(x_perm[:M], dev["x"][rt])


def _noise_draws(mode, T, E, seed):
    g = torch.Generator().manual_seed(seed)
    if mode == moe.MOE_NOISE_GUMBEL:
        return torch.rand((T, E), generator=g)                 # uniform draws
    if mode == moe.MOE_NOISE_PROB_GAUSS:
        return 0.1 * torch.randn((T, E), generator=g)          # 0.1 * N(0, 1) on probabilities
    return torch.randn((T, E), generator=g)                    # unit amplitude * N(0, 1)


@pytest.mark.parametrize("noise_mode", [moe.MOE_NOISE_GUMBEL, moe.MOE_NOISE_PROB_GAUSS,
                                        moe.MOE_NOISE_LOGIT_SOFTMAX])
@pytest.mark.parametrize("name", ["tiny_f32", "mixtral_prefill", "switch_capacity", "deepseek_fine"])
def test_noisy_routing_parity(name, noise_mode):
    """Routing noise: the GPU's selection scores match the oracle's (same draws); top-k,
    counts, capacity and placement follow the GPU's scores bit-exactly; y matches."""
    w = PARITY_WORKLOADS[name]
    cf = capacity_factor_or_none(w)
    inp = make_inputs(w, seed=0)
    inp["noise"] = _noise_draws(noise_mode, w.T, w.E, 100 + noise_mode)
    cfg = moe.config_from_workload(w, noise=noise_mode)
    r = tl.run_forward(w, tl.to_device(inp), cfg=cfg)
    assert r["flags"] == 0
    g = tl.host(r["outs"])
    lg_ref = oracle.logits(inp["x"], inp["w_gate"], inp["logit_bias"])
    sc_ref = oracle.noisy_scores(lg_ref, inp["noise"].numpy(), noise_mode)
    assert float(np.abs(g["logits"] - sc_ref).max()) <= tl.logits_tol(sc_ref)
    ref = oracle.noisy_routed_reference(w.k, w.gate, cf, g["logits"], noise_mode, lg_ref)
    # With noise on the probabilities the weights come from the clean logits, which the
    # oracle computes itself: allow the fp32 logit error through the softmax.
    check_routing_exact(g, ref, tl.TOL_W if noise_mode != moe.MOE_NOISE_PROB_GAUSS else 2e-5)
    y_ref = tl.y_on_routing(inp, ref["idx"], ref["slot_row"], ref["w"])
    assert tl.max_rel_err(g["y"], y_ref) <= tl.TOL_Y[w.dtype]
    # the noise actually changed the routing
    clean = oracle.topk(lg_ref, w.k)
    assert np.any(clean != g["topk_idx"])


@pytest.mark.parametrize("name", ["tiny_f32", "mixtral_prefill", "deepseek_fine"])
def test_deterministic(name):
    w = PARITY_WORKLOADS[name]
    dev = tl.to_device(make_inputs(w, seed=1))
    a = tl.host(tl.run_forward(w, dev)["outs"])
    b = tl.host(tl.run_forward(w, dev)["outs"])
    for key in a:
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)


# ----------------------------------------------------------------- edge cases

def _parity_small(w, inp, expect_flags=0):
    r = tl.run_forward(w, tl.to_device(inp))
    assert r["flags"] == expect_flags
    g = tl.host(r["outs"])
    cf = capacity_factor_or_none(w)
    ref = oracle.routed_reference(None, w.k, w.gate, cf, g["logits"])
    check_routing_exact(g, ref)
    y_ref = tl.y_on_routing(inp, ref["idx"], ref["slot_row"], ref["w"])
    assert tl.max_rel_err(g["y"], y_ref) <= tl.TOL_Y[w.dtype]
    return g, ref


EDGE = [
    Workload("one_token_bf16", T=1, d=256, h=512, E=8, k=2, dtype="bf16", gate=0, capacity_factor=0),
    Workload("one_token_f32", T=1, d=64, h=128, E=8, k=2, dtype="f32", gate=1, capacity_factor=0,
             bias_std=0.1),
    Workload("e_equals_k", T=100, d=128, h=256, E=4, k=4, dtype="bf16", gate=1, capacity_factor=0,
             bias_std=0.1),
    Workload("ragged_tail", T=129, d=136, h=264, E=16, k=3, dtype="bf16", gate=0,
             capacity_factor=0, bias_std=0.1),
    Workload("k8_e8_f32", T=70, d=32, h=40, E=8, k=8, dtype="f32", gate=0, capacity_factor=0),
    Workload("tight_capacity_k2", T=300, d=128, h=128, E=8, k=2, dtype="bf16", gate=1,
             capacity_factor=0.5, logit_bias="normal1.5"),
    Workload("narrow_d8", T=77, d=8, h=16, E=32, k=2, dtype="bf16", gate=0, capacity_factor=0),
    # 512 or more rows per expert on average: the 256-row tile kernel, with full tiles, a
    # half-filled last tile, a ragged K tail (264 = 4 x 64 + 8) and a ragged last weight
    # block (520 = 2 x 256 + 8 columns, stored row by row) ...
    Workload("wide_tiles", T=1100, d=264, h=520, E=4, k=2, dtype="bf16", gate=1,
             capacity_factor=0, bias_std=0.1),
    # ... and with a capacity that drops rows (C = 564 of ~1024 per expert).
    Workload("wide_tiles_capacity", T=1024, d=128, h=384, E=2, k=1, dtype="bf16", gate=0,
             capacity_factor=1.1, bias_std=0.1, logit_bias="normal1.5"),
    # Weights-as-M groups of 65-128 rows (C = 100): token tiles of two 64-row boxes, the
    # second partly past the group; top-1, so the combine is folded into the GEMMs.
    Workload("two_token_boxes", T=400, d=192, h=320, E=4, k=1, dtype="bf16", gate=1,
             capacity_factor=1.0, bias_std=0.1),
] + [
    # Shapes whose weights-as-M expert GEMMs split tiles between SMs (on a 148-SM B300):
    # GEMM1 here is 4 tiles of 150 k-blocks cut into ~19 pieces each (several load
    # batches in the finishing CTA's sum) ...
    Workload("split_k_many_pieces", T=48, d=9600, h=256, E=2, k=1, dtype="bf16", gate=1,
             capacity_factor=0, bias_std=0.1),
    # ... and here both GEMMs split: 64 tiles of 150 k-blocks and 150 tiles of 64.
    Workload("split_k_both_gemms", T=64, d=9600, h=4096, E=2, k=1, dtype="bf16", gate=1,
             capacity_factor=0, bias_std=0.1),
]
SPLIT = [w for w in EDGE if w.name.startswith("split_k")]


@pytest.mark.parametrize("w", EDGE, ids=[w.name for w in EDGE])
def test_edge_shapes(w):
    _parity_small(w, make_inputs(w, seed=5))


@pytest.mark.parametrize("w", SPLIT, ids=[w.name for w in SPLIT])
def test_split_tiles_deterministic(w):
    """Tiles computed in pieces by several SMs are summed in a fixed order: two runs,
    and the stage calls, agree bit for bit."""
    dev = tl.to_device(make_inputs(w, seed=6))
    a = tl.host(tl.run_forward(w, dev)["outs"])
    b = tl.host(tl.run_forward(w, dev)["outs"])
    for key in a:
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)
    cfg = moe.config_from_workload(w)
    rows = w.T * w.k
    ws = tl.poisoned_workspace(moe.moe_stage_workspace_size(cfg))
    x_perm = torch.empty((rows, w.d), dtype=w.torch_dtype, device="cuda")
    x_perm[:] = dev["x"][torch.as_tensor(a["row_token"], device="cuda").long().clamp(min=0)]
    offsets = torch.as_tensor(a["offsets"], device="cuda")
    h_buf = torch.empty((rows, w.h), dtype=w.torch_dtype, device="cuda")
    y_perm = torch.empty((rows, w.d), dtype=w.torch_dtype, device="cuda")
    for _ in range(2):
        moe.moe_expert_ffn(cfg, x_perm, offsets, dev["w1"], dev["b1"], dev["w2"], dev["b2"], h_buf,
                           y_perm, ws)
        assert moe.moe_device_error(ws) == 0
        y = torch.empty((w.T, w.d), dtype=w.torch_dtype, device="cuda")
        moe.moe_combine(cfg, y_perm, torch.as_tensor(a["slot_row"], device="cuda"),
                        torch.as_tensor(a["topk_w"], device="cuda"), y, ws)
        np.testing.assert_array_equal(y.float().cpu().numpy(), a["y"])


FUSED = [w for w in list(PARITY_WORKLOADS.values()) + EDGE if w.dtype == "bf16"]


@pytest.mark.parametrize("w", FUSED, ids=[w.name for w in FUSED])
def test_fused_gather_is_bitwise_the_forward(w):
    """cfg.fused_gather: GEMM1 reads the token rows from x through the row -> token map
    (both expert GEMM kernels, split tiles, ragged tails, one-token batches): every output
    is bitwise the default forward's, on a workspace without the row copy."""
    dev = tl.to_device(make_inputs(w, seed=9))
    a = tl.host(tl.run_forward(w, dev)["outs"])
    cfg = moe.config_from_workload(w, fused_gather=1)
    r = tl.run_forward(w, dev, cfg=cfg)
    assert r["flags"] == 0
    assert r["ws"].numel() < moe.moe_workspace_size(moe.config_from_workload(w))
    b = tl.host(r["outs"])
    for key in a:
        np.testing.assert_array_equal(b[key], a[key], err_msg=key)


def test_fused_gather_with_x_perm_output():
    """A fused_gather forward that is given an x_perm buffer fills it (the rows in expert
    order, as the default forward writes them) and returns the same outputs."""
    w = PARITY_WORKLOADS["switch_capacity"]  # capacity drops: fewer rows than T*k
    dev = tl.to_device(make_inputs(w, seed=4))
    outs = tl.alloc_outputs(w, "cuda")
    outs["x_perm"] = torch.full((w.T * w.k, w.d), float("nan"), dtype=w.torch_dtype,
                                device="cuda")
    a = tl.host(tl.run_forward(w, dev, outs=outs)["outs"])
    outs2 = {k: torch.full_like(v, -7 if v.dtype == torch.int32 else float("nan"))
             for k, v in outs.items()}
    r = tl.run_forward(w, dev, outs=outs2, cfg=moe.config_from_workload(w, fused_gather=1))
    assert r["flags"] == 0
    b = tl.host(r["outs"])
    M = int(a["offsets"][-1])
    np.testing.assert_array_equal(b["x_perm"][:M], a["x_perm"][:M])
    for key in a:
        if key != "x_perm":
            np.testing.assert_array_equal(b[key], a[key], err_msg=key)


@pytest.mark.parametrize("name", ["mixtral_prefill", "switch_capacity", "decode"])
def test_fused_gather_full_size(name):
    """The same at the benchmark's sizes: row tiles (prefill) and weights-as-M tiles with
    and without split tiles (Switch, decode)."""
    w = WORKLOADS[name]
    inp = make_inputs(w, seed=0, device="cuda")
    outs = dict(y=torch.empty((w.T, w.d), dtype=w.torch_dtype, device="cuda"))
    ws = torch.empty(moe.moe_workspace_size(moe.config_from_workload(w)), dtype=torch.uint8,
                     device="cuda")
    moe.moe_forward(moe.config_from_workload(w), inp, outs, ws)
    assert moe.moe_device_error(ws) == 0
    y0 = outs["y"].clone()
    cfg = moe.config_from_workload(w, fused_gather=1)
    ws = torch.empty(moe.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    moe.moe_forward(cfg, inp, outs, ws)
    assert moe.moe_device_error(ws) == 0
    assert torch.equal(outs["y"], y0)


TOP1 = [w for w in list(PARITY_WORKLOADS.values()) + EDGE if w.k == 1 and w.dtype == "bf16"]


@pytest.mark.parametrize("w", TOP1, ids=[w.name for w in TOP1])
def test_top1_combine_in_gemm2_is_bitwise_the_combine(w):
    """A bf16 top-1 forward writes y from GEMM2's epilogue and zeroes the rows of tokens
    with no kept slot in the dispatch (split tiles included); a forward asked for y_perm
    runs the separate combine pass instead.  Same bits everywhere, from an all-NaN y."""
    dev = tl.to_device(make_inputs(w, seed=5))
    a = tl.run_forward(w, dev)
    assert a["flags"] == 0
    outs = tl.alloc_outputs(w, "cuda")
    outs["y_perm"] = torch.empty((w.T * w.k, w.d), dtype=w.torch_dtype, device="cuda")
    b = tl.run_forward(w, dev, outs=outs)
    assert b["flags"] == 0
    ya, yb = tl.host(a["outs"])["y"], tl.host(b["outs"])["y"]
    assert not np.isnan(ya).any()
    np.testing.assert_array_equal(ya, yb)
    dropped = (tl.host(a["outs"])["slot_row"] < 0).all(axis=1)
    assert (ya[dropped] == 0).all()


def test_top1_combine_in_gemm2_full_size():
    """The same on the 128-expert Switch layer at the benchmark's size (most tokens
    dropped by the capacity)."""
    w = WORKLOADS["switch_capacity"]
    inp = make_inputs(w, seed=0, device="cuda")
    cfg = moe.config_from_workload(w)
    ws = torch.empty(moe.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    y0 = torch.full((w.T, w.d), float("nan"), dtype=w.torch_dtype, device="cuda")
    moe.moe_forward(cfg, inp, dict(y=y0), ws)
    assert moe.moe_device_error(ws) == 0
    y1 = torch.full_like(y0, float("nan"))
    yp = torch.empty((w.T * w.k, w.d), dtype=w.torch_dtype, device="cuda")
    moe.moe_forward(cfg, inp, dict(y=y1, y_perm=yp), ws)
    assert moe.moe_device_error(ws) == 0
    assert torch.equal(y0, y1)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_all_ties_and_drop_storm(dtype):
    """W_g = 0: every logit ties, so every token picks experts 0..k-1; with capacity 1.25
    the first C tokens of experts 0 and 1 survive (a drop storm), the rest get y = 0."""
    w = Workload("ties", T=500, d=64, h=128, E=16, k=2, dtype=dtype, gate=1,
                 capacity_factor=1.25, bias_std=0.1)
    inp = make_inputs(w, seed=2)
    inp["w_gate"] = torch.zeros_like(inp["w_gate"])
    g, ref = _parity_small(w, inp)
    C = oracle.capacity(w.T, w.E, 1.25)
    assert np.all(g["topk_idx"] == np.array([0, 1])[None, :])
    assert g["kept_counts"].tolist() == [C, C] + [0] * 14
    assert int(g["dropped"][0]) == 2 * (w.T - C)
    assert np.all(g["y"][C:] == 0.0)
    np.testing.assert_array_equal(g["row_token"][:C], np.arange(C))
    assert float(g["aux_loss"][0]) == pytest.approx(2.0, rel=1e-5)   # uniform f: loss = k


def test_one_expert_takes_everything():
    """A dominant logit bias sends every token to expert 3 (top-1, capacity 1.25)."""
    w = Workload("storm", T=1000, d=64, h=64, E=16, k=1, dtype="bf16", gate=1,
                 capacity_factor=1.25)
    inp = make_inputs(w, seed=3)
    inp["logit_bias"] = torch.zeros(16)
    inp["logit_bias"][3] = 100.0
    g, _ = _parity_small(w, inp)
    C = oracle.capacity(w.T, w.E, 1.25)
    assert g["kept_counts"][3] == C and g["kept_counts"].sum() == C
    np.testing.assert_array_equal(g["row_token"][:C], np.arange(C))
    assert np.all(g["row_token"][C:] == -1)


def test_empty_batch():
    w = Workload("empty", T=0, d=64, h=64, E=8, k=2, dtype="bf16", gate=0, capacity_factor=0)
    cfg = moe.config_from_workload(w)
    outs = tl.alloc_outputs(w)
    inp = tl.to_device(make_inputs(w.scaled(T=1), seed=0))
    ws = tl.poisoned_workspace(moe.moe_workspace_size(cfg))
    moe.moe_forward(cfg, inp, outs, ws)
    assert moe.moe_device_error(ws) == 0
    assert outs["counts"].eq(0).all() and outs["offsets"].eq(0).all()
    assert outs["dropped"].item() == 0 and outs["aux_loss"].item() == 0.0
    assert outs["routing_stats"].eq(0).all()


def test_dispatch_flags_out_of_range_index():
    w = Workload("badidx", T=40, d=64, h=64, E=8, k=2, dtype="bf16", gate=0, capacity_factor=0)
    cfg = moe.config_from_workload(w)
    x = make_inputs(w, seed=0)["x"].cuda()
    idx = torch.tensor([[i % 8, (i + 1) % 8] for i in range(40)], dtype=torch.int32, device="cuda")
    idx[5, 1] = 8
    idx[17, 0] = -3
    i32 = dict(dtype=torch.int32, device="cuda")
    offsets, kept = torch.empty(9, **i32), torch.empty(8, **i32)
    slot_row, row_token = torch.empty((40, 2), **i32), torch.empty(80, **i32)
    dropped = torch.empty(1, **i32)
    x_perm = torch.empty((80, 64), dtype=torch.bfloat16, device="cuda")
    ws = tl.poisoned_workspace(moe.moe_stage_workspace_size(cfg))
    moe.moe_dispatch(cfg, x, idx, offsets, kept, slot_row, row_token, dropped, x_perm, ws)
    assert moe.moe_device_error(ws) & moe.MOE_DEVERR_BAD_INDEX
    assert slot_row[5, 1].item() == -1 and slot_row[17, 0].item() == -1
    assert int(offsets[-1]) == 78


def test_combine_flags_out_of_range_row():
    w = Workload("badrow", T=16, d=64, h=64, E=8, k=2, dtype="bf16", gate=0, capacity_factor=0)
    cfg = moe.config_from_workload(w)
    y_perm = torch.ones((32, 64), dtype=torch.bfloat16, device="cuda")
    slot_row = torch.arange(32, dtype=torch.int32, device="cuda").view(16, 2).contiguous()
    slot_row[3, 0] = 32
    wts = torch.full((16, 2), 0.5, device="cuda")
    y = torch.empty((16, 64), dtype=torch.bfloat16, device="cuda")
    ws = tl.poisoned_workspace(moe.moe_stage_workspace_size(cfg))
    moe.moe_combine(cfg, y_perm, slot_row, wts, y, ws)
    assert moe.moe_device_error(ws) & moe.MOE_DEVERR_BAD_ROW
    assert torch.all(y[3] == 0.5) and torch.all(y[4] == 1.0)


def test_nonfinite_logit_is_flagged():
    w = Workload("nan", T=64, d=64, h=64, E=8, k=2, dtype="bf16", gate=0, capacity_factor=0)
    inp = make_inputs(w, seed=0)
    inp["x"][7, 3] = float("nan")
    r = tl.run_forward(w, tl.to_device(inp))
    assert r["flags"] & moe.MOE_DEVERR_NONFINITE


# ----------------------------------------------------------------- full size

FULL = ["mixtral_prefill", "switch_capacity", "deepseek_fine", "decode"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(name):
    """Full workload sizes through the same moe_forward call the benchmark times:
    every routing/indexing output exact on all tokens, logits on sampled tokens, and y
    on sampled tokens that include every non-empty expert's first and last kept row."""
    w = WORKLOADS[name]
    cf = capacity_factor_or_none(w)
    inp = make_inputs(w, seed=0, device="cuda")
    r = tl.run_forward(w, inp)
    assert r["flags"] == 0
    g = tl.host(r["outs"])
    ref = oracle.routed_reference(None, w.k, w.gate, cf, g["logits"])
    check_routing_exact(g, ref)

    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, w.T - 1], rng.choice(w.T, min(w.T, 48), replace=False)]))
    xs = inp["x"][torch.as_tensor(rows, device="cuda")].cpu()
    lb = inp["logit_bias"].cpu() if inp["logit_bias"] is not None else None
    lg_ref = oracle.logits(xs, inp["w_gate"].cpu(), lb)
    assert float(np.abs(g["logits"][rows] - lg_ref).max()) <= tl.logits_tol(lg_ref)

    # y on: every token of a small batch; else the first and last token, 24 random ones,
    # and the tokens of every non-empty expert's first and last kept row, so that each
    # expert's ragged last tile is compared at the full K.
    if w.T <= 256:
        toks = np.arange(w.T)
    else:
        off, rt = g["offsets"], g["row_token"]
        ends = [rt[off[e]] for e in range(w.E) if off[e + 1] > off[e]]
        ends += [rt[off[e + 1] - 1] for e in range(w.E) if off[e + 1] > off[e]]
        toks = np.unique(np.concatenate([[0, w.T - 1], rng.choice(w.T, 24, replace=False),
                                         np.asarray(ends, dtype=np.int64)]))
    host_inp = {"x": inp["x"].cpu()}
    cache = {}

    def fetch(e):
        if e not in cache:
            cache.clear()
            cache[e] = tuple(inp[n][e].cpu() for n in ("w1", "b1", "w2", "b2"))
        return cache[e]

    y_ref = tl.y_on_routing(host_inp, ref["idx"], ref["slot_row"], ref["w"], tokens=toks, fetch=fetch)
    err = tl.max_rel_err(g["y"][toks], y_ref)
    assert err <= tl.TOL_Y[w.dtype]
    print(f"{name}: M={int(g['offsets'][-1])} dropped={int(g['dropped'][0])} "
          f"nonempty={int((g['kept_counts'] > 0).sum())} sampled y_err={err:.2e}")
