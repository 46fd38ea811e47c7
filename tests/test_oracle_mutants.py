"""The oracle's pins catch planted mistakes.

Each case copies ``oracle/moe_oracle.cpp``, plants one plausible mistake in the copy
(a wrong tie-break, a wrong normaliser, an off-by-one capacity test, a dropped term, a
sign, a transposed operand, a missing weight, a wrong derivative, in the top-k, expert-choice
and noisy-routing stages), compiles it with the
oracle's own flags and runs ``tests/test_oracle_pins.py`` against it in a subprocess: at
least one pin must fail.  The unchanged copy, compiled the same way, must pass them all,
so a failure is the mistake's and not the harness's.  The mistakes live only in
temporary copies; the oracle itself is never modified.
"""

import concurrent.futures as cf
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "moe_oracle.cpp")

# name -> [(text in the oracle, planted replacement)]; each text occurs exactly once.  Every
# mistake keeps memory accesses in bounds, so a copy fails by its results, not by a crash.
MUTANTS = {
    "topk_tie_to_higher_index": [
        ("if (best < 0 || l[e] > l[best]) best = e;", "if (best < 0 || l[e] >= l[best]) best = e;")],
    "P_over_T_times_k": [
        ("pe = (double)c[e] / (double)T;", "pe = (double)c[e] / ((double)T * k);")],
    "capacity_keeps_C_plus_one": [
        ("if (C < 0 || pos[t * k + j] < C) nkept[e] += 1;",
         "if (C < 0 || pos[t * k + j] <= C) nkept[e] += 1;"),
        ("if (C < 0 || q < C) {", "if (C < 0 || q <= C) {")],
    "softmax_denominator_drops_expert_0": [
        ("for (int e = 0; e < E; ++e) s += std::exp(l[e] - m);",
         "for (int e = 1; e < E; ++e) s += std::exp(l[e] - m);")],
    "b2_subtracted": [
        ("if (b2) acc += elem(b2, dtype, o);", "if (b2) acc -= elem(b2, dtype, o);")],
    "silu_sign": [
        ("double silu(double a) { return a / (1.0 + std::exp(-a)); }",
         "double silu(double a) { return a / (1.0 + std::exp(a)); }")],
    "w1_transposed": [
        ("a += elem(w1, dtype, (int64_t)i * d + c) * elem(x_rows, dtype, r * d + c);",
         "a += elem(w1, dtype, (int64_t)c * h + i) * elem(x_rows, dtype, r * d + c);")],
    "combine_ignores_gate_weight": [
        ("for (int o = 0; o < d; ++o) y[t * d + o] += w[t * k + j] * zz[o];",
         "for (int o = 0; o < d; ++o) y[t * d + o] += zz[o];")],
    "silu_grad_missing_term": [
        ("return sg * (1.0 + a * (1.0 - sg));", "return sg * (1.0 + a * sg);")],
    "expert_choice_ties_to_higher_token": [
        ("for (int64_t t = 0; t < T; ++t) order[t] = t;",
         "for (int64_t t = 0; t < T; ++t) order[t] = T - 1 - t;")],
    "expert_choice_combine_ignores_weight": [
        ("for (int o = 0; o < d; ++o) y[t * d + o] += sel_w[e * C + c] * zz[o];",
         "for (int o = 0; o < d; ++o) y[t * d + o] += zz[o];")],
    "gumbel_sign": [
        ("v = l[e] - std::log(-std::log((double)n[e] + 1e-9) + 1e-9);",
         "v = l[e] + std::log(-std::log((double)n[e] + 1e-9) + 1e-9);")],
    "logit_noise_not_scaled": [
        ("v = l[e] + (double)n[e] * p[e];", "v = l[e] + (double)n[e];")],
    "renorm_gate_not_renormalised": [
        ("for (int j = 0; j < k; ++j) w[t * k + j] = p[idx[t * k + j]] / den;",
         "for (int j = 0; j < k; ++j) w[t * k + j] = p[idx[t * k + j]];")],
    "loss_missing_factor_E": [
        ("return (double)E * loss;", "return loss;")],
    "stats_population_std": [
        ("const double lstd = E > 1 ? std::sqrt(lvar / (E - 1)) : 0.0;",
         "const double lstd = E > 1 ? std::sqrt(lvar / E) : 0.0;")],
    "stats_entropy_sign": [
        ("ent -= load[e] * std::log(load[e] + 1e-10);", "ent += load[e] * std::log(load[e] + 1e-10);")],
    "capacity_rounds_down": [
        ("return (int64_t)std::ceil((double)T * capacity_factor / (double)E);",
         "return (int64_t)std::floor((double)T * capacity_factor / (double)E);")],
    "dispatch_slot_major_priority": [
        ("""  for (int64_t t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      int e = idx[t * k + j];
      pos[t * k + j] = next[e]++;""",
         """  for (int j = 0; j < k; ++j)
    for (int64_t t = 0; t < T; ++t) {
      int e = idx[t * k + j];
      pos[t * k + j] = next[e]++;""")],
    "gate_jacobian_without_mean_term": [
        ("dl[t * E + idx[t * k + j]] += w[t * k + j] * (dw[t * k + j] - inner);",
         "dl[t * E + idx[t * k + j]] += w[t * k + j] * dw[t * k + j];")],
    "gate_jacobian_skips_dropped_slots": [
        ("""    for (int j = 0; j < k; ++j)
      dl[t * E + idx[t * k + j]] += w[t * k + j] * (dw[t * k + j] - inner);""",
         """    for (int j = 0; j < k; ++j)
      if (slot_row[t * k + j] >= 0)
        dl[t * E + idx[t * k + j]] += w[t * k + j] * (dw[t * k + j] - inner);""")],
    "balance_gradient_without_mean_term": [
        ("((double)counts[c] / (double)T - pp);", "((double)counts[c] / (double)T);")],
    "logit_bias_ignored": [
        ("if (logit_bias) acc += (double)logit_bias[e];", "(void)logit_bias;")],
    "b1_ignored": [
        ("if (b1) a += elem(b1, dtype, i);", "(void)b1;")],
    "kept_counts_include_drops": [
        ("kept[e] = (int32_t)nkept[e];", "kept[e] = (int32_t)next[e];")],
    "row_token_holds_slot": [
        ("row_token[row] = (int32_t)t;", "row_token[row] = (int32_t)j;")],
    "dx_missing_router_term": [
        ("""      for (int e = 0; e < E; ++e) acc += dl[t * E + e] * elem(wg, dtype, (int64_t)e * d + c);
      dx[t * d + c] += acc;""",
         """      for (int e = 0; e < E; ++e) acc += dl[t * E + e] * elem(wg, dtype, (int64_t)e * d + c);
      (void)acc;""")],
}

FLAGS = ["g++", "-std=c++17", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp",
         "-shared", "-fPIC"]


def _build(tmp, name, edits):
    text = open(SRC).read()
    for old, new in edits:
        assert text.count(old) == 1, (name, old)
        text = text.replace(old, new)
    src = os.path.join(tmp, f"{name}.cpp")
    lib = os.path.join(tmp, f"lib{name}.so")
    with open(src, "w") as f:
        f.write(text)
    subprocess.run(FLAGS + [src, "-o", lib], check=True)
    return lib


def _pins(lib):
    env = dict(os.environ, MOE_ORACLE_LIB=lib, OMP_NUM_THREADS="2")
    return subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle_pins.py", "-x", "-q",
                           "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True,
                          text=True, timeout=600)


@pytest.fixture(scope="module")
def runs(tmp_path_factory):
    """Every copy built and its pin run done, several at a time."""
    tmp = str(tmp_path_factory.mktemp("oracle_mutants"))
    cases = dict(MUTANTS, unchanged=[])
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        futs = {name: ex.submit(lambda n, e: _pins(_build(tmp, n, e)), name, edits)
                for name, edits in cases.items()}
        return {name: f.result() for name, f in futs.items()}


def test_unchanged_copy_passes_every_pin(runs):
    r = runs["unchanged"]
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(runs, name):
    r = runs[name]
    assert r.returncode == 1 and " failed" in r.stdout, (name, r.stdout[-2000:])
