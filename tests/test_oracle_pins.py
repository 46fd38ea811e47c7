"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks one oracle stage against something independent: the hand-derived
worked example in tests/golden, a closed form, an invariant the formulas imply, a
library routine evaluating the same definition (numpy matmul, scipy softmax,
torch silu), or brute force on tiny inputs.  The formulas are those of the page
"MoE mixture-of-experts routing mechanism: principles and sparse activation"
(gating formula G(x)=softmax(TopK(x.W_g)), output y = sum G_i E_i(x), the
TopKRouter / Expert / MoELayer listing, the load-balancing loss and the
capacity-factor section).
"""

import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import softmax as scipy_softmax

import oracle
from moe_workloads import PARITY_WORKLOADS, Workload, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_e4_k2_t3.json")


def _hand_inputs(g):
    E, d, h = g["E"], g["d"], g["h"]
    x = torch.tensor(g["x"], dtype=torch.float32)
    w_gate = torch.eye(E, d)
    w1 = torch.stack([torch.eye(h, d) for _ in range(E)])
    w2 = torch.stack([(e + 1) * torch.eye(d, h) for e in range(E)])
    b1 = torch.zeros(E, h)
    b2 = torch.stack([torch.full((d,), float(e)) for e in range(E)])
    return dict(x=x, w_gate=w_gate, w1=w1, b1=b1, w2=w2, b2=b2, logit_bias=None)


@pytest.mark.parametrize("mode", [0, 1])
def test_hand_example_no_capacity(mode):
    g = json.load(open(GOLDEN))
    ref = g["no_capacity"]
    out = oracle.forward(_hand_inputs(g), g["k"], mode, None)
    assert out["idx"].tolist() == ref["idx"]
    np.testing.assert_allclose(out["w"], ref["w"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(out["y"], ref["y"], rtol=1e-14, atol=1e-14)
    assert out["counts"].tolist() == ref["counts"]
    assert out["aux"] == pytest.approx(ref["aux"], rel=1e-14)
    assert out["kept"].tolist() == ref["kept"]
    assert out["offsets"].tolist() == ref["offsets"]
    assert out["slot_row"].tolist() == ref["slot_row"]
    assert out["row_token"].tolist() == ref["row_token"]
    assert out["dropped"] == ref["dropped"]
    _, _, f, _ = oracle.aux_loss(oracle.softmax(out["logits"]), out["idx"])
    np.testing.assert_allclose(f, ref["f"], rtol=1e-14)


@pytest.mark.parametrize("mode", [0, 1])
def test_hand_example_capacity(mode):
    g = json.load(open(GOLDEN))
    ref = g["capacity_factor_1"]
    assert oracle.capacity(g["T"], g["E"], 1.0) == ref["C"]
    out = oracle.forward(_hand_inputs(g), g["k"], mode, 1.0)
    assert out["kept"].tolist() == ref["kept"]
    assert out["offsets"].tolist() == ref["offsets"]
    assert out["slot_row"].tolist() == ref["slot_row"]
    assert out["row_token"].tolist() == ref["row_token"]
    assert out["dropped"] == ref["dropped"]
    np.testing.assert_allclose(out["y"], ref["y"], rtol=1e-14, atol=1e-14)
    assert np.all(out["y"][2] == 0.0)   # fully dropped token: exactly zero MoE output
    assert out["counts"].tolist() == g["no_capacity"]["counts"]   # counts are pre-drop


@pytest.mark.parametrize("E,k", [(8, 2), (64, 2), (128, 1), (256, 8), (4, 4)])
def test_all_ties_pick_lowest_indices(E, k):
    """W_g = 0 makes every logit equal: slot j must hold expert j, each weight is 1/k,
    f is uniform and the balance loss is exactly k."""
    T, d = 37, 16
    x = torch.randn(T, d, generator=torch.Generator().manual_seed(1))
    lg = oracle.logits(x, torch.zeros(E, d))
    assert np.all(lg == 0.0)
    idx = oracle.topk(lg, k)
    assert np.all(idx == np.arange(k)[None, :])
    for mode in (0, 1):
        w = oracle.gate_weights(lg, idx, mode)
        np.testing.assert_allclose(w, 1.0 / k, rtol=1e-15)
    loss, counts, f, P = oracle.aux_loss(oracle.softmax(lg), idx)
    np.testing.assert_allclose(f, 1.0 / E, rtol=1e-14)
    assert loss == pytest.approx(k, rel=1e-13)


def test_signed_zero_ties():
    """-0.0 and +0.0 compare equal, so the lower expert index wins."""
    lg = np.array([[-1.0, -0.0, 0.0, -2.0], [0.0, -5.0, -0.0, -0.0]])
    assert oracle.topk(lg, 2).tolist() == [[1, 2], [0, 2]]


def _brute_topk(row, k):
    order = sorted(range(len(row)), key=lambda e: (-row[e], e))
    return order[:k]


@pytest.mark.parametrize("E,k", [(8, 2), (64, 2), (256, 8), (5, 5)])
def test_topk_matches_sorted_order(E, k):
    rng = np.random.default_rng(7)
    lg = rng.standard_normal((200, E))
    lg[::3] = np.round(lg[::3], 1)       # force many exact ties
    idx = oracle.topk(lg, k)
    for t in range(lg.shape[0]):
        assert idx[t].tolist() == _brute_topk(lg[t].tolist(), k)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_logits_match_library_matmul(dtype):
    w = Workload("t", T=53, d=96, h=32, E=16, k=2, dtype=dtype, gate=0, capacity_factor=0,
                 logit_bias="normal1.5")
    inp = make_inputs(w, seed=3)
    lg = oracle.logits(inp["x"], inp["w_gate"], inp["logit_bias"])
    ref = (inp["x"].double().numpy() @ inp["w_gate"].double().numpy().T
           + inp["logit_bias"].double().numpy()[None, :])
    np.testing.assert_allclose(lg, ref, rtol=1e-13, atol=1e-13)


def test_softmax_matches_library():
    rng = np.random.default_rng(0)
    lg = rng.standard_normal((64, 37)) * 5
    np.testing.assert_allclose(oracle.softmax(lg), scipy_softmax(lg, axis=1), rtol=1e-13)


@pytest.mark.parametrize("k", [1, 2, 8])
def test_gate_modes_agree_and_sum_to_one(k):
    """softmax(TopK(l)) and the renormalised softmax-then-topk are the same function:
    p_i / sum_kept p = e^{l_i} / sum_kept e^{l_j}."""
    rng = np.random.default_rng(11)
    lg = rng.standard_normal((300, 32)) * 3
    idx = oracle.topk(lg, k)
    w0 = oracle.gate_weights(lg, idx, 0)
    w1 = oracle.gate_weights(lg, idx, 1)
    np.testing.assert_allclose(w0.sum(1), 1.0, rtol=0, atol=1e-14)
    np.testing.assert_allclose(w1.sum(1), 1.0, rtol=0, atol=1e-14)
    np.testing.assert_allclose(w0, w1, rtol=0, atol=1e-12)
    # weights are non-increasing along the slots (slot 0 holds the largest logit)
    assert np.all(np.diff(w0, axis=1) <= 1e-15)


def test_mode0_is_softmax_over_masked_logits():
    """mode 0 equals softmax of the logits with non-top-k entries at -inf (the formula)."""
    rng = np.random.default_rng(5)
    lg = rng.standard_normal((50, 16))
    k = 3
    idx = oracle.topk(lg, k)
    masked = np.full_like(lg, -np.inf)
    for t in range(lg.shape[0]):
        masked[t, idx[t]] = lg[t, idx[t]]
    G = scipy_softmax(masked, axis=1)
    w = oracle.gate_weights(lg, idx, 0)
    for t in range(lg.shape[0]):
        np.testing.assert_allclose(w[t], G[t, idx[t]], rtol=1e-13)
        assert np.all(np.delete(G[t], idx[t]) == 0.0)


@pytest.mark.parametrize("E,k", [(8, 2), (128, 1), (256, 8)])
def test_aux_loss_invariants(E, k):
    rng = np.random.default_rng(E + k)
    lg = rng.standard_normal((500, E)) * 2
    p = oracle.softmax(lg)
    idx = oracle.topk(lg, k)
    loss, counts, f, P = oracle.aux_loss(p, idx)
    assert f.sum() == pytest.approx(1.0, abs=1e-12)
    assert P.sum() == pytest.approx(k, abs=1e-12)
    assert counts.sum() == 500 * k
    np.testing.assert_array_equal(counts, np.bincount(idx.ravel(), minlength=E))
    assert loss == pytest.approx(E * float(np.dot(f, P)), rel=1e-14)


@pytest.mark.parametrize("E,k", [(8, 1), (8, 2), (16, 1), (16, 4)])
def test_balanced_routing_gives_loss_k(E, k):
    """Uniform routing (every expert receives exactly T*k/E assignments) gives P_e = k/E,
    hence loss = E * sum_e f_e * k/E = k * sum_e f_e = k (1 for top-1)."""
    d = E
    reps = 5
    T = E * reps
    # Token t prefers experts t, t+1, ..., t+k-1 (mod E) in that order.
    x = torch.zeros(T, d)
    for t in range(T):
        for j in range(k):
            x[t, (t + j) % E] = 10.0 - j
    w_gate = torch.eye(E, d)
    lg = oracle.logits(x, w_gate)
    idx = oracle.topk(lg, k)
    loss, counts, f, P = oracle.aux_loss(oracle.softmax(lg), idx)
    assert np.all(counts == T * k // E)
    assert loss == pytest.approx(float(k), rel=1e-13)


def _brute_dispatch(idx, E, C):
    """Independent placement: sort assignments by (expert, token); keep the first C of each."""
    T, k = idx.shape
    pairs = sorted(((int(idx[t, j]), t, j) for t in range(T) for j in range(k)))
    kept_pairs = []
    seen = {}
    for e, t, j in pairs:
        n = seen.get(e, 0)
        seen[e] = n + 1
        if C < 0 or n < C:
            kept_pairs.append((e, t, j))
    slot_row = -np.ones((T, k), np.int32)
    row_token = -np.ones(T * k, np.int32)
    for row, (e, t, j) in enumerate(kept_pairs):
        slot_row[t, j] = row
        row_token[row] = t
    kept = np.bincount([e for e, _, _ in kept_pairs], minlength=E).astype(np.int32)
    return kept, slot_row, row_token


@pytest.mark.parametrize("E,k,cf", [(8, 2, None), (128, 1, 1.25), (16, 4, 1.0), (4, 2, 0.5)])
def test_dispatch_invariants_and_brute_force(E, k, cf):
    rng = np.random.default_rng(E * 10 + k)
    T = 300
    lg = rng.standard_normal((T, E)) + np.linspace(2, -2, E)[None, :]   # skewed load
    idx = oracle.topk(lg, k)
    C = oracle.capacity(T, E, cf)
    out = oracle.dispatch(idx, E, C)
    counts = np.bincount(idx.ravel(), minlength=E)
    assert out["kept"].sum() == T * k - out["dropped"]
    assert out["offsets"][E] == out["kept"].sum()
    np.testing.assert_array_equal(np.diff(out["offsets"]), out["kept"])
    if C >= 0:
        np.testing.assert_array_equal(out["kept"], np.minimum(counts, C))
    else:
        np.testing.assert_array_equal(out["kept"], counts)
    for e in range(E):
        toks = out["row_token"][out["offsets"][e]:out["offsets"][e + 1]]
        assert np.all(np.diff(toks) > 0)          # stable token order inside each expert
    kept_b, slot_b, rt_b = _brute_dispatch(idx, E, C)
    np.testing.assert_array_equal(out["kept"], kept_b)
    np.testing.assert_array_equal(out["slot_row"], slot_b)
    np.testing.assert_array_equal(out["row_token"], rt_b)


def test_drop_storm_keeps_first_C_tokens():
    """Every token routed to one expert with capacity factor 1.25: exactly C = ceil(T*1.25/E)
    assignments survive, and they are the first C token ids."""
    T, E = 1000, 16
    idx = np.full((T, 1), 5, np.int32)
    C = oracle.capacity(T, E, 1.25)
    assert C == math.ceil(T * 1.25 / E) == 79
    out = oracle.dispatch(idx, E, C)
    assert out["kept"][5] == C and out["kept"].sum() == C
    assert out["dropped"] == T - C
    np.testing.assert_array_equal(out["row_token"][:C], np.arange(C))
    assert np.all(out["slot_row"][C:] == -1)


def test_dispatch_rejects_out_of_range_index():
    with pytest.raises(ValueError):
        oracle.dispatch(np.array([[0, 9]], np.int32), 8, -1)


def test_expert_identity_reduces_to_silu():
    """W1 = I, b1 = 0, W2 = I, b2 = 0 make the expert the textbook SiLU."""
    d = 24
    x = torch.randn(10, d, generator=torch.Generator().manual_seed(2)) * 4
    z = oracle.expert_rows(x, torch.eye(d), None, torch.eye(d), None)
    ref = torch.nn.functional.silu(x.double()).numpy()
    np.testing.assert_allclose(z, ref, rtol=1e-14, atol=1e-15)


def test_expert_scalar_by_hand():
    """d = h = 1: x = 2, w1 = 0.5, b1 = 0 -> a = 1, silu(1) = e/(e+1); w2 = 2, b2 = 0.25."""
    x = torch.tensor([[2.0]])
    z = oracle.expert_rows(x, torch.tensor([[0.5]]), torch.tensor([0.0]),
                           torch.tensor([[2.0]]), torch.tensor([0.25]))
    assert z[0, 0] == pytest.approx(2.0 * math.e / (math.e + 1.0) + 0.25, rel=1e-15)


def test_combine_dropped_token_is_zero_and_k1_weight_one():
    w = Workload("t", T=40, d=16, h=24, E=4, k=1, dtype="f32", gate=1, capacity_factor=0.5,
                 bias_std=0.1)
    inp = make_inputs(w, seed=9)
    out = oracle.forward(inp, 1, 1, 0.5)
    assert out["dropped"] > 0
    np.testing.assert_array_equal(out["w"], 1.0)          # k = 1, mode 1: weight exactly 1
    for t in range(w.T):
        if out["slot_row"][t, 0] < 0:
            assert np.all(out["y"][t] == 0.0)
        else:
            e = out["idx"][t, 0]
            z = oracle.expert_rows(inp["x"][t:t + 1], inp["w1"][e], inp["b1"][e],
                                   inp["w2"][e], inp["b2"][e])
            np.testing.assert_array_equal(out["y"][t], z[0])


TINY = [
    Workload("a", T=13, d=16, h=8, E=8, k=2, dtype="f32", gate=0, capacity_factor=0, bias_std=0.1),
    Workload("b", T=16, d=8, h=16, E=4, k=1, dtype="bf16", gate=1, capacity_factor=1.25,
             bias_std=0.1, logit_bias="zipf"),
    Workload("c", T=11, d=16, h=16, E=8, k=3, dtype="bf16", gate=1, capacity_factor=1.0,
             logit_bias="normal1.5"),
    Workload("d", T=9, d=8, h=8, E=5, k=5, dtype="f32", gate=0, capacity_factor=0),
    Workload("e", T=16, d=12, h=4, E=6, k=2, dtype="f32", gate=1, capacity_factor=0.5,
             bias_std=0.1),
]


@pytest.mark.parametrize("w", TINY, ids=[w.name for w in TINY])
def test_dispatch_path_equals_dense_brute_force(w):
    """The staged oracle (top-k, dispatch, per-slot experts, combine) equals evaluating all
    experts on every token masked by the top-k set and the capacity rule."""
    inp = make_inputs(w, seed=4)
    cf = w.capacity_factor if w.capacity_factor > 0 else None
    y = oracle.forward(inp, w.k, w.gate, cf)["y"]
    y_bf = oracle.forward_dense(inp, w.k, w.gate, cf)
    scale = max(1e-300, float(np.abs(y_bf).max()))
    assert float(np.abs(y - y_bf).max()) <= 1e-12 * scale


def test_parity_workloads_are_finite_and_routing_valid():
    """Seeded inputs feed the oracle cleanly (finite outputs, valid indices) on the smallest
    parity workload."""
    w = PARITY_WORKLOADS["tiny_f32"]
    inp = make_inputs(w, seed=0)
    out = oracle.forward(inp, w.k, w.gate, None)
    assert np.isfinite(out["y"]).all()
    assert out["idx"].min() >= 0 and out["idx"].max() < w.E
    assert all(len(set(r)) == w.k for r in out["idx"].tolist())


@pytest.mark.parametrize("E", [1, 4, 8, 64, 256])
def test_routing_stats_uniform_load(E):
    """Perfectly even counts: CV 0, no dead expert, max/avg 1, entropy ln E, E effective."""
    st = oracle.routing_stats(np.full(E, 37))
    np.testing.assert_allclose(st[[0, 1, 5]], 0.0, atol=1e-12)
    assert st[2] == pytest.approx(1.0, rel=1e-12)
    # entropy = -sum (1/E) ln(1/E + 1e-10) = -ln(1/E + 1e-10)
    assert st[3] == pytest.approx(-math.log(1.0 / E + 1e-10), rel=1e-13)
    assert st[4] == pytest.approx(1.0 / (1.0 / E + 1e-10), rel=1e-12)


@pytest.mark.parametrize("E", [2, 8, 128])
def test_routing_stats_single_expert_takes_all(E):
    """All assignments on one expert: load = (1, 0, ...): sample std 1/sqrt(E), so
    CV = sqrt(E); dead ratio (E-1)/E; max/avg = E; entropy ~ 0; one effective expert."""
    counts = np.zeros(E, np.int64)
    counts[E // 2] = 5000
    st = oracle.routing_stats(counts)
    assert st[0] == pytest.approx(math.sqrt(E), rel=1e-12)
    assert st[1] == pytest.approx((E - 1) / E, rel=1e-12)
    assert st[2] == pytest.approx(E, rel=1e-12)
    assert st[3] == pytest.approx(-math.log(1.0 + 1e-10), abs=1e-15)
    assert st[4] == pytest.approx(1.0, abs=1e-9)
    # counts (N, 0, ...): sample std N/sqrt(E), mean N/E -> (N/sqrt(E)) / (N/E + 1e-6)
    N = 5000.0
    assert st[5] == pytest.approx((N / math.sqrt(E)) / (N / E + 1e-6), rel=1e-12)


def test_routing_stats_match_library_routines():
    rng = np.random.default_rng(3)
    counts = rng.integers(0, 500, 64)
    counts[::7] = 0
    st = oracle.routing_stats(counts)
    load = counts / counts.sum()
    assert st[0] == pytest.approx(np.std(load, ddof=1) / np.mean(load), rel=1e-12)
    assert st[1] == pytest.approx(np.mean(load < 1e-4), rel=1e-12)
    assert st[2] == pytest.approx(load.max() / load.mean(), rel=1e-12)
    from scipy.stats import entropy as scipy_entropy
    assert st[3] == pytest.approx(scipy_entropy(load), rel=1e-7)   # +1e-10 inside the log
    assert st[5] == pytest.approx(np.std(counts, ddof=1) / (np.mean(counts) + 1e-6), rel=1e-12)


def test_routing_stats_empty():
    np.testing.assert_array_equal(oracle.routing_stats(np.zeros(8, np.int64)), 0.0)


def test_gumbel_max_samples_the_softmax():
    """Gumbel-max: argmax_e (l_e + g_e) with g = -log(-log U) is distributed as softmax(l).
    The oracle's Gumbel transform (with the page's 1e-9 guards) must reproduce it."""
    rng = np.random.default_rng(0)
    probs = np.array([0.5, 0.25, 0.15, 0.1])
    lg = np.tile(np.log(probs), (200000, 1))
    u = rng.random(lg.shape, dtype=np.float64).astype(np.float32)
    sc = oracle.noisy_scores(lg, u, oracle.NOISE_GUMBEL)
    freq = np.bincount(oracle.topk(sc, 1)[:, 0], minlength=4) / lg.shape[0]
    np.testing.assert_allclose(freq, probs, atol=4e-3)


def test_gumbel_closed_form_point():
    """u = 1/2: g = -log(-log(1/2 + 1e-9) + 1e-9)."""
    sc = oracle.noisy_scores(np.zeros((1, 2)), np.array([[0.5, 0.5]], np.float32), oracle.NOISE_GUMBEL)
    g = -math.log(-math.log(0.5 + 1e-9) + 1e-9)
    np.testing.assert_allclose(sc, g, rtol=1e-14)
    assert abs(g - (-math.log(math.log(2.0)))) < 1e-8


def test_prob_noise_zero_is_softmax_and_large_noise_wins():
    rng = np.random.default_rng(1)
    lg = rng.standard_normal((20, 8))
    sc = oracle.noisy_scores(lg, np.zeros_like(lg, dtype=np.float32), oracle.NOISE_PROB_GAUSS)
    np.testing.assert_allclose(sc, scipy_softmax(lg, axis=1), rtol=1e-13)
    n = np.zeros_like(lg, dtype=np.float32)
    n[:, 5] = 2.0          # any probability plus 2 beats every probability without it
    assert np.all(oracle.topk(oracle.noisy_scores(lg, n, oracle.NOISE_PROB_GAUSS), 1)[:, 0] == 5)


def test_logit_softmax_noise_closed_forms():
    """Zero draws leave the logits unchanged; with equal logits (p = 1/E) a draw c adds c/E."""
    rng = np.random.default_rng(2)
    lg = rng.standard_normal((10, 6))
    z = oracle.noisy_scores(lg, np.zeros_like(lg, dtype=np.float32), oracle.NOISE_LOGIT_SOFTMAX)
    np.testing.assert_array_equal(z, lg)
    eq = np.full((3, 4), 0.7)
    n = np.array([[0.0, 1.0, 2.0, 3.0]] * 3, np.float32)
    sc = oracle.noisy_scores(eq, n, oracle.NOISE_LOGIT_SOFTMAX)
    np.testing.assert_allclose(sc, 0.7 + n.astype(np.float64) / 4.0, rtol=1e-15)
    assert np.all(oracle.topk(sc, 2) == np.array([3, 2]))


@pytest.mark.parametrize("mode,cf,k", [(0, None, 2), (1, 1.0, 2), (1, 0.75, 3)])
def test_routed_reference_is_the_forward_routing(mode, cf, k):
    """Fed the forward's own logits, the routing reference (what the GPU tests run on the
    GPU's logits) reproduces the whole layer's routing.  x in {-1, 0, 1} and W_g in
    multiples of 1/8 make every logit exact in fp32, so the fp32 hand-off loses nothing,
    and leave many equal logits for the tie rule."""
    g = torch.Generator().manual_seed(40 + k)
    T, d, h, E = 48, 16, 8, 6
    inp = dict(x=torch.randint(-1, 2, (T, d), generator=g).float(),
               w_gate=torch.randint(-8, 9, (E, d), generator=g).float() / 8,
               w1=torch.randn((E, h, d), generator=g), b1=None,
               w2=torch.randn((E, d, h), generator=g), b2=None, logit_bias=None)
    out = oracle.forward(inp, k, mode, cf)
    assert np.array_equal(out["logits"].astype(np.float32).astype(np.float64), out["logits"])
    ref = oracle.routed_reference(None, k, mode, cf, out["logits"].astype(np.float32))
    for key in ("idx", "counts", "kept", "offsets", "slot_row", "row_token"):
        np.testing.assert_array_equal(ref[key], out[key], err_msg=key)
    np.testing.assert_array_equal(ref["w"], out["w"])
    assert ref["aux"] == out["aux"] and ref["dropped"] == out["dropped"]


@pytest.mark.parametrize("name", ["tiny_f32", "switch_capacity"])
def test_expert_path_on_given_routing_is_the_forward_output(name):
    """The GPU tests' expert path on a given routing (the test library's y_on_routing,
    oracle expert rows and combine), fed the forward's own routing, gives the forward's y."""
    import moe_testlib as tl
    w = PARITY_WORKLOADS[name].scaled(T=96, d=32, h=48)
    inp = make_inputs(w, seed=3)
    cf = w.capacity_factor if w.capacity_factor > 0 else None
    out = oracle.forward(inp, w.k, w.gate, cf)
    y = tl.y_on_routing(inp, out["idx"], out["slot_row"], out["w"])
    np.testing.assert_allclose(y, out["y"], rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("noise_mode", [oracle.NOISE_PROB_GAUSS, oracle.NOISE_LOGIT_SOFTMAX])
@pytest.mark.parametrize("mode,cf", [(0, None), (1, 1.0)])
def test_noisy_routing_with_zero_draws_is_clean_routing(noise_mode, mode, cf):
    """Zero draws leave the probabilities (noise on p) or the logits (noise scaled by p)
    unchanged, so the noisy routing reference reduces to the clean one: same selection,
    gate weights, counts, loss and placement."""
    rng = np.random.default_rng(20 + noise_mode)
    lg = rng.standard_normal((40, 8)).astype(np.float32)
    sc = oracle.noisy_scores(lg, np.zeros_like(lg), noise_mode).astype(np.float32)
    noisy = oracle.noisy_routed_reference(2, mode, cf, sc, noise_mode, lg.astype(np.float64))
    clean = oracle.routed_reference(None, 2, mode, cf, lg)
    for key in ("idx", "counts", "slot_row", "offsets", "kept"):
        np.testing.assert_array_equal(noisy[key], clean[key], err_msg=key)
    np.testing.assert_allclose(noisy["w"], clean["w"], rtol=1e-6, atol=1e-7)
    assert abs(noisy["aux"] - clean["aux"]) <= 1e-6 * abs(clean["aux"])


def test_probability_noise_keeps_clean_gate_weights():
    """Noise on the probabilities only picks the experts: the kept experts' weights are
    the clean gate's, a distribution over the kept set, whatever the draws."""
    rng = np.random.default_rng(31)
    lg = rng.standard_normal((40, 8))
    n = (0.3 * rng.standard_normal((40, 8))).astype(np.float32)
    sc = oracle.noisy_scores(lg, n, oracle.NOISE_PROB_GAUSS).astype(np.float32)
    for mode in (0, 1):
        r = oracle.noisy_routed_reference(2, mode, None, sc, oracle.NOISE_PROB_GAUSS, lg)
        np.testing.assert_array_equal(r["w"], oracle.gate_weights(lg, r["idx"], mode))
        np.testing.assert_allclose(r["w"].sum(axis=1), 1.0, rtol=1e-12)
        # the noise moved some selections away from the clean top-2
        assert np.any(r["idx"] != oracle.topk(lg, 2))


@pytest.mark.parametrize("T,E,C", [(50, 4, 13), (64, 8, 1), (7, 3, 7), (100, 16, 0)])
def test_expert_choice_matches_rank_brute_force(T, E, C):
    """Token t is chosen by expert e iff fewer than C tokens rank above it in column e,
    where t' ranks above t when p[t',e] > p[t,e], or they are equal and t' < t."""
    rng = np.random.default_rng(T + E)
    # Scores from a few values, so every column holds runs of equal scores and the rule
    # for equal values decides which tokens straddling the C-th place are taken.
    p = rng.integers(1, 5, size=(T, E)) / 8.0
    tok, w = oracle.expert_choice(p, C)
    for e in range(E):
        above = [sum(1 for q in range(T) if p[q, e] > p[t, e] or (p[q, e] == p[t, e] and q < t))
                 for t in range(T)]
        chosen = [t for t in range(T) if above[t] < C]
        assert tok[e].tolist() == chosen                 # exactly C, ascending token order
        np.testing.assert_array_equal(w[e], p[chosen, e])


def test_expert_choice_full_capacity_is_the_dense_mixture():
    """With C = T every expert takes every token, so the layer is the softmax-weighted
    mixture of all experts: y_t = sum_e softmax(l_t)_e E_e(x_t)."""
    w = Workload("ec", T=12, d=8, h=12, E=4, k=1, dtype="f32", gate=1, capacity_factor=4.0,
                 bias_std=0.1)
    inp = make_inputs(w, seed=6)
    out = oracle.forward_expert_choice(inp, 4.0)           # C = ceil(12 * 4 / 4) = 12 = T
    assert out["C"] == 12
    p = scipy_softmax(inp["x"].double().numpy() @ inp["w_gate"].double().numpy().T, axis=1)
    dense = np.zeros((12, 8))
    for e in range(4):
        dense += p[:, e:e + 1] * oracle.expert_rows(inp["x"], inp["w1"][e], inp["b1"][e],
                                                    inp["w2"][e], inp["b2"][e])
    np.testing.assert_allclose(out["y"], dense, rtol=1e-12, atol=1e-13)


def test_expert_choice_unchosen_tokens_get_zero():
    """C = 1 with 8 experts and 40 tokens: at most 8 tokens are chosen, the rest get 0."""
    w = Workload("ec1", T=40, d=8, h=8, E=8, k=1, dtype="f32", gate=1, capacity_factor=0.2)
    inp = make_inputs(w, seed=7)
    out = oracle.forward_expert_choice(inp, 0.2)           # C = ceil(40 * 0.2 / 8) = 1
    assert out["C"] == 1
    chosen = set(out["sel_token"].ravel().tolist())
    for t in range(40):
        assert np.any(out["y"][t] != 0.0) == (t in chosen)


# ----------------------------------------------------------------- backward (B1..B7)
def _tiny_f64_layer(rng, T=6, d=5, h=7, E=4):
    return dict(x=rng.standard_normal((T, d)), w_gate=rng.standard_normal((E, d)),
                w1=rng.standard_normal((E, h, d)) / 2, b1=rng.standard_normal((E, h)) * 0.1,
                w2=rng.standard_normal((E, d, h)) / 2, b2=rng.standard_normal((E, d)) * 0.1,
                logit_bias=None)


@pytest.mark.parametrize("mode,cf,k", [(0, None, 2), (1, None, 2), (0, 1.0, 2), (1, 0.5, 3),
                                       (1, None, 4)])
def test_backward_matches_central_differences(mode, cf, k):
    """Every gradient of L = <G, y> + d_aux * aux equals the central difference of the
    oracle's own fp64 forward (step 1e-6), with and without capacity drops and with
    k = E (softmax over every expert)."""
    rng = np.random.default_rng(10 * mode + k)
    inp = _tiny_f64_layer(rng)
    G = rng.standard_normal(inp["x"].shape)
    d_aux = 0.7

    def loss():
        o = oracle.forward(inp, k, mode, cf)
        return float((o["y"] * G).sum() + d_aux * o["aux"])

    base = oracle.forward(inp, k, mode, cf)
    g = oracle.backward(inp, G, k, mode, cf, d_aux)
    eps = 1e-6
    for name, key in [("x", "dx"), ("w_gate", "dw_gate"), ("w1", "dw1"), ("b1", "db1"),
                      ("w2", "dw2"), ("b2", "db2")]:
        a = inp[name]
        fd = np.zeros_like(a)
        for ix in np.ndindex(a.shape):
            old = a[ix]
            a[ix] = old + eps
            lp = loss()
            a[ix] = old - eps
            lm = loss()
            a[ix] = old
            fd[ix] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(g[key], fd, rtol=1e-6, atol=1e-7, err_msg=name)
    # the perturbations never crossed a routing decision
    assert np.array_equal(oracle.forward(inp, k, mode, cf)["idx"], base["idx"])


def test_backward_logit_bias_equals_constant_feature_router_weight():
    """With a constant-one input feature, the router weight on that feature acts exactly
    as a logit bias, so its gradient is the logit-bias gradient."""
    rng = np.random.default_rng(3)
    inp = _tiny_f64_layer(rng, T=9)
    inp["x"][:, -1] = 1.0
    G = rng.standard_normal(inp["x"].shape)
    g = oracle.backward(inp, G, 2, 1, 1.0, 0.3)
    np.testing.assert_allclose(g["dlogit_bias"], g["dw_gate"][:, -1], rtol=1e-12, atol=1e-13)


def test_backward_without_upstream_gradient_is_the_balance_loss_gradient():
    """dy = 0: no expert weight receives gradient, and d_aux = 0 makes every gradient 0."""
    rng = np.random.default_rng(4)
    inp = _tiny_f64_layer(rng)
    zero = np.zeros_like(inp["x"])
    g = oracle.backward(inp, zero, 2, 0, None, 1.0)
    for key in ("dw1", "db1", "dw2", "db2"):
        assert np.all(g[key] == 0.0), key
    assert np.abs(g["dw_gate"]).max() > 0
    g0 = oracle.backward(inp, zero, 2, 0, None, 0.0)
    for key, v in g0.items():
        assert np.all(v == 0.0), key


def test_backward_on_given_logits_equals_recomputed():
    """Passing the layer's own logits in reproduces the self-contained backward exactly."""
    rng = np.random.default_rng(5)
    inp = _tiny_f64_layer(rng)
    G = rng.standard_normal(inp["x"].shape)
    lg = oracle.forward(inp, 2, 1, 1.0)["logits"]
    a = oracle.backward(inp, G, 2, 1, 1.0, 0.2)
    b = oracle.backward(inp, G, 2, 1, 1.0, 0.2, logits_in=lg)
    for key in a:
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)
