"""Plant plausible mistakes in a copy of the oracle (CPU only) and check that the pins
fail on each. This shows the pins can tell a right oracle from a wrong one."""
import os

import numpy as np
import pytest

from test_oracle_verify import lossless_error, pq_error

MUTANTS = {
    "residual sign q-p": (
        "r[v] = p[v] - q[v] > 0.0 ? p[v] - q[v] : 0.0;",
        "r[v] = q[v] - p[v] > 0.0 ? q[v] - p[v] : 0.0;"),
    "accept ratio inverted": ("if (uk * qx < px) {", "if (uk * px < qx) {"),
    "temperature multiplies": (
        "p[v] = exp((logit_at(base, dtype, off + (size_t)v) - M) / T);",
        "p[v] = exp((logit_at(base, dtype, off + (size_t)v) - M) * T);"),
    "bonus from the wrong row": (
        "row_softmax(tgt, dtype, (trow0 + L) * (size_t)V, V, T, Mt[L], p);",
        "row_softmax(tgt, dtype, (trow0 + L - 1) * (size_t)V, V, T, Mt[L - 1], p);"),
    "terminal sample reuses the accept uniform": (
        "const double uK = u[(size_t)b * (K + 1) + K];",
        "const double uK = u[(size_t)b * (K + 1) + k];"),
    "inverse CDF one bucket late": ("            return v;\n", "            return v + 1 < V ? v + 1 : v;\n"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_lossless_pin_catches(oracle_mod, tmp_path, name):
    old, new = MUTANTS[name]
    src = oracle_mod.source()
    assert src.count(old) == 1, name
    lib = oracle_mod.build_variant(src.replace(old, new), str(tmp_path / "mutant.so"))
    T = 0.5 if "temperature" in name else 1.0
    assert lossless_error(oracle_mod, T, 0, lib=lib) > 1e-3


# Slips confined to the block that writes the diagnostic p_k(x_k), q_k(x_k): the
# decisions (and so the losslessness pin) are untouched, the probability pin is not.
PQ_MUTANTS = {
    "p and q outputs swapped": (
        "if (out_p) out_p[(size_t)b * K + k] = p[x];\n            if (out_q) out_q[(size_t)b * K + k] = q[x];",
        "if (out_p) out_p[(size_t)b * K + k] = q[x];\n            if (out_q) out_q[(size_t)b * K + k] = p[x];"),
    "p from target row k+1": (
        "row_softmax(tgt, dtype, (trow0 + k) * (size_t)V, V, T, Mt[k], p);\n"
        "            row_softmax(drf, dtype, (drow0 + k) * (size_t)V, V, T, Md[k], q);\n"
        "            if (out_p)",
        "row_softmax(tgt, dtype, (trow0 + k + 1) * (size_t)V, V, T, Mt[k + 1], p);\n"
        "            row_softmax(drf, dtype, (drow0 + k) * (size_t)V, V, T, Md[k], q);\n"
        "            if (out_p)"),
    "temperature dropped in the diagnostic block": (
        "row_softmax(drf, dtype, (drow0 + k) * (size_t)V, V, T, Md[k], q);\n            if (out_p)",
        "row_softmax(drf, dtype, (drow0 + k) * (size_t)V, V, 1.0, Md[k], q);\n            if (out_p)"),
}


@pytest.mark.parametrize("name", sorted(PQ_MUTANTS))
def test_probability_pin_catches(oracle_mod, tmp_path, name):
    old, new = PQ_MUTANTS[name]
    src = oracle_mod.source()
    assert src.count(old) == 1, name
    lib = oracle_mod.build_variant(src.replace(old, new), str(tmp_path / "mutant.so"))
    assert pq_error(oracle_mod, lib=lib) > 1e-3
    assert lossless_error(oracle_mod, 1.0, 0, lib=lib) < 1e-9  # decisions unchanged


SCHED_MUTANTS = {
    "strict tau comparison": ("if (run >= th) n = k + 1;", "if (run > th) n = k + 1;"),
    "no floor of one": ("if (n < 1) n = 1;", "if (n < 0) n = 1;"),
    "tie-break on k reversed": ("if (a->k != b->k) return a->k < b->k ? -1 : 1;",
                                "if (a->k != b->k) return a->k > b->k ? -1 : 1;"),
    "survival ascending": ("if (a->s != b->s) return a->s > b->s ? -1 : 1;",
                           "if (a->s != b->s) return a->s < b->s ? -1 : 1;"),
    "floors never first": ("int floor_first = token_budget >= B;", "int floor_first = 0;"),
}


@pytest.mark.parametrize("name", sorted(SCHED_MUTANTS))
def test_schedule_pins_catch(oracle_mod, tmp_path, name):
    import test_oracle_schedule as ts

    old, new = SCHED_MUTANTS[name]
    src = oracle_mod.source()
    assert src.count(old) == 1, name
    lib = oracle_mod.build_variant(src.replace(old, new), str(tmp_path / "mutant.so"))

    class Shim:
        def __getattr__(self, a):
            return getattr(oracle_mod, a)

        def schedule(self, conf, tau, budget):
            return oracle_mod.schedule(conf, tau, budget, lib=lib)

    shim = Shim()
    failed = 0
    tests = [lambda: ts.test_golden_variable_length_draft(shim),
             lambda: ts.test_truncation_rule_of_the_guide_sketch(shim),
             lambda: ts.test_tie_break_prefers_earlier_positions_then_lower_requests(shim)]
    tests += [lambda s=s: ts.test_budget_trim_bruteforce(shim, s) for s in range(40)]
    tests += [lambda s=s: ts.test_budget_invariants(shim, s) for s in range(20)]
    for t in tests:
        try:
            t()
        except AssertionError:
            failed += 1
    assert failed > 0, name


CALIB_MUTANTS = {
    "temperature multiplies the logit": ("double z = (log(c) - log1p(-c)) / T;",
                                         "double z = (log(c) - log1p(-c)) * T;"),
    "logit sign flipped": ("return 1.0 / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(z));"),
    "load weights swapped": ("double lf = 0.6 * (Q / Qmax) + 0.4 * (M / Mmax);",
                             "double lf = 0.4 * (Q / Qmax) + 0.6 * (M / Mmax);"),
    "load factor not squared": ("return tau_min + (tau_max - tau_min) * (lf * lf);",
                                "return tau_min + (tau_max - tau_min) * lf;"),
    "rejected position not counted": ("for (int k = 0; k < L && k <= j; k++) {",
                                      "for (int k = 0; k < L && k < j; k++) {"),
    "update sign reversed": ("double t = (double)temps[k] + lr * err;",
                             "double t = (double)temps[k] - lr * err;"),
    "ECE without the bin weights": ("if (ece_out) *ece_out = N > 0.0 ? gap / N : 0.0;",
                                    "if (ece_out) *ece_out = N > 0.0 ? gap / ORC_CALIB_BINS : 0.0;"),
}


@pytest.mark.parametrize("name", sorted(CALIB_MUTANTS))
def test_calibration_pins_catch(oracle_mod, tmp_path, name):
    import test_oracle_calib as tc

    old, new = CALIB_MUTANTS[name]
    src = oracle_mod.source()
    assert src.count(old) == 1, name
    lib = oracle_mod.build_variant(src.replace(old, new), str(tmp_path / "mutant.so"))
    failed = 0
    for t in tc.PINS:
        try:
            t(lib)
        except AssertionError:
            failed += 1
    assert failed > 0, name


MARKOV_MUTANTS = {
    "correction subtracted": ("double z = bf16_value(L[row + v]) + c;",
                              "double z = bf16_value(L[row + v]) - c;"),
    "U and Vm swapped": ("for (int j = 0; j < r; j++) c += bf16_value(U[(size_t)v * r + j]) * x[j];",
                         "for (int j = 0; j < r; j++) c += bf16_value(Vm[(size_t)v * r + j]) * bf16_value(U[(size_t)y * r + j]);"),
    "previous token never advances": ("            y = best;\n", "            (void)best;\n"),
    "argmax keeps the last tie": ("if (best < 0 || stored > bestv) {", "if (best < 0 || stored >= bestv) {"),
    "rounding truncates": ("if (frac > 0.5 || (frac == 0.5 && fmod(lo, 2.0) != 0.0)) q = lo + 1.0;",
                           "if (0) q = lo + 1.0;"),
}


@pytest.mark.parametrize("name", sorted(MARKOV_MUTANTS))
def test_markov_pins_catch(oracle_mod, tmp_path, name):
    import test_oracle_markov as tm

    old, new = MARKOV_MUTANTS[name]
    src = oracle_mod.source()
    assert src.count(old) == 1, name
    lib = oracle_mod.build_variant(src.replace(old, new), str(tmp_path / "mutant.so"))
    failed = 0
    for t in tm.PINS:
        try:
            t(lib)
        except AssertionError:
            failed += 1
    assert failed > 0, name


CURVE_MUTANTS = {
    "step time ignores the batch size": (
        "double g = ((double)B + a) * curve_at(curve_x, curve_y, n_pts, x) / x;",
        "double g = ((double)B + a) * curve_at(curve_x, curve_y, n_pts, x);"),
    "floor survivals left out": ("if (floors && k == 0) a_floor += s;",
                                 "if (floors && k == 0) a_floor += 0.0;"),
    "interpolation from the wrong end": ("return y0 + (y1 - y0) * ((x - x0) / (x1 - x0));",
                                         "return y1 + (y0 - y1) * ((x - x0) / (x1 - x0));"),
    "competing survivals ascending": ("return (a < b) - (a > b);", "return (a > b) - (a < b);"),
}


@pytest.mark.parametrize("name", sorted(CURVE_MUTANTS))
def test_curve_pins_catch(oracle_mod, tmp_path, name):
    import test_oracle_curve as tc

    old, new = CURVE_MUTANTS[name]
    src = oracle_mod.source()
    assert src.count(old) == 1, name
    lib = oracle_mod.build_variant(src.replace(old, new), str(tmp_path / "mutant.so"))
    failed = 0
    for t in tc.PINS:
        try:
            t(lib)
        except AssertionError:
            failed += 1
    assert failed > 0, name


TREE_MUTANTS = {
    "tree: residual never updated": ("for (int v = 0; v < V; v++) r[v] = w[v] / Z;",
                                     "for (int v = 0; v < V; v++) r[v] = r[v];"),
    "tree: residual ignores q": ("w[v] = r[v] - q[v] > 0.0 ? r[v] - q[v] : 0.0;",
                                 "w[v] = r[v] > 0.0 ? r[v] : 0.0;"),
    "tree: terminal sample from p": ("int y = inverse_cdf(wlast, V, u[base], &Z, &gap);",
                                     "int y = inverse_cdf(p, V, u[base], &Z, &gap);"),
    "tree: non-children tested": ("if (par[base + n] != c) continue;",
                                  "if (par[base + n] < 0) continue;"),
    "tree: test uses the parent's uniform": ("const double un = u[base + n];",
                                             "const double un = u[base + c];"),
    "tree: greedy takes the last matching child": (
        "for (int n = c + 1; n < nn && next < 0; n++)",
        "for (int n = c + 1; n < nn; n++)"),
    "tree: leaf bonus uses a test uniform": (
        "int y = inverse_cdf(p, V, u[base], &Z, &gap);\n            if (gap < NEAR_TIE) out_flags[b] |= ORC_FLAG_CDF_EDGE;\n            if (gap < margin) margin = gap;\n            if (out_margin)",
        "int y = inverse_cdf(p, V, u[base + c], &Z, &gap);\n            if (gap < NEAR_TIE) out_flags[b] |= ORC_FLAG_CDF_EDGE;\n            if (gap < margin) margin = gap;\n            if (out_margin)"),
    "tree: accept test against q": ("if (un * qx < rx) {\n                next = n;",
                                    "if (un * rx < qx) {\n                next = n;"),
}


@pytest.mark.parametrize("name", sorted(TREE_MUTANTS))
def test_tree_pins_catch(oracle_mod, tmp_path, name):
    import test_oracle_tree as tt

    old, new = TREE_MUTANTS[name]
    src = oracle_mod.source()
    assert src.count(old) == 1, name
    lib = oracle_mod.build_variant(src.replace(old, new), str(tmp_path / "mutant.so"))
    failed = 0
    for t in tt.PINS:
        try:
            t(lib)
        except AssertionError:
            failed += 1
    assert failed > 0, name
