"""Pins for the oracle's confidence schedule (CPU only)."""
import itertools
import json
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_golden_variable_length_draft(oracle_mod):
    with open(os.path.join(GOLDEN, "schedule_variable_length.json")) as f:
        g = json.load(f)
    r = oracle_mod.schedule(np.array(g["conf"], np.float32), g["tau"], g["token_budget"])
    assert r["status"] == 0
    assert r["out_len"].tolist() == g["expected_out_len"]


def test_truncation_rule_of_the_guide_sketch(oracle_mod):
    """DSpark Guide, '2. Confidence-Scheduled Dynamic Verification' and its
    'Hands-On Implementation' sketch: truncate at the first position whose cumulative
    survival falls below tau, keep at least one token, keep all K when none does; the
    comparison is C_k >= tau (a product exactly equal to tau survives)."""
    conf = np.array([[0.5, 0.5, 0.5, 0.5],   # C = .5 .25 .125 .0625, tau .25 -> 2 (inclusive)
                     [0.1, 0.9, 0.9, 0.9],   # C_1 < tau -> floor 1
                     [1.0, 1.0, 1.0, 1.0],   # never below -> K
                     [0.0, 1.0, 1.0, 1.0]],  # zero confidence -> floor 1
                    np.float32)
    r = oracle_mod.schedule(conf, 0.25, 1000)
    assert r["out_len"].tolist() == [2, 1, 4, 1]
    assert r["l0"].tolist() == [2, 1, 4, 1]


def test_survival_is_running_product(oracle_mod):
    rng = np.random.default_rng(0)
    conf = rng.random((50, 16)).astype(np.float32)
    r = oracle_mod.schedule(conf, 0.3, 10_000)
    np.testing.assert_array_equal(r["surv"], np.cumprod(conf.astype(np.float64), axis=1))
    assert (np.diff(r["surv"], axis=1) <= 0).all()


def _expected_accepted(surv, lens):
    """sum_b sum_{k<len_b} S_{b,k}: with calibrated confidences the expected number of
    accepted tokens, since P(accepted length >= k+1) = C_{k+1} (DSpark Guide,
    '1. The Mathematics of Suffix Decay')."""
    return sum(float(surv[b, :l].sum()) for b, l in enumerate(lens))


@pytest.mark.parametrize("seed", range(40))
def test_budget_trim_bruteforce(oracle_mod, seed):
    """The budget trim spends the verify budget where survival is highest
    (DSpark Deep Dive, 'The Optimization Logic'): among all per-request prefix lengths
    with 0 <= len_b <= L0_b, len_b >= 1 when budget >= B, and
    sum len_b = min(budget, sum L0_b), it maximises the expected accepted tokens.
    Distinct confidences make the maximiser unique; it is found by enumeration."""
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 5))
    K = int(rng.integers(1, 5))
    conf = rng.uniform(0.3, 1.0, size=(B, K)).astype(np.float32)
    tau = float(rng.uniform(0.0, 0.6))
    l0 = oracle_mod.schedule(conf, tau, 10 ** 6)["l0"]
    budget = int(rng.integers(0, int(l0.sum()) + 2))
    r = oracle_mod.schedule(conf, tau, budget)
    surv = r["surv"]
    need = min(budget, int(l0.sum()))
    best, best_lens = -1.0, None
    for lens in itertools.product(*[range(0, l + 1) for l in l0]):
        if sum(lens) != need:
            continue
        if budget >= B and min(lens) < 1:
            continue
        v = _expected_accepted(surv, lens)
        if v > best + 1e-12:
            best, best_lens = v, lens
    assert best_lens is not None, "no feasible length vector: the floor was not honoured"
    assert r["out_len"].tolist() == list(best_lens), (conf, tau, budget)


@pytest.mark.parametrize("seed", range(20))
def test_budget_invariants(oracle_mod, seed):
    rng = np.random.default_rng(100 + seed)
    B, K = int(rng.integers(1, 300)), int(rng.integers(1, 17))
    conf = (rng.beta(8, 2, size=(B, K)) * 0.93 ** np.arange(1, K + 1)).astype(np.float32)
    if seed % 4 == 0:
        conf[:, :] = conf[:, :1]  # many exact ties in survival across requests
    tau = float(rng.uniform(0.0, 0.5))
    l0 = oracle_mod.schedule(conf, tau, 10 ** 9)["l0"]
    for budget in [0, 1, B - 1, B, B + 3, int(l0.sum()) // 2, int(l0.sum()), int(l0.sum()) + 5]:
        if budget < 0:
            continue
        r = oracle_mod.schedule(conf, tau, budget)
        L = r["out_len"]
        assert L.sum() == min(budget, l0.sum())
        assert (L <= l0).all() and (L >= 0).all()
        if budget >= B:
            assert (L >= 1).all()
        # nothing dropped outranks anything kept (floor positions aside when budget >= B)
        s = r["surv"]
        lo = 1 if budget >= B else 0
        kept = [s[b, k] for b in range(B) for k in range(lo, L[b])]
        dropped = [s[b, k] for b in range(B) for k in range(max(lo, L[b]), l0[b])]
        if kept and dropped:
            assert max(dropped) <= min(kept)


def test_tie_break_prefers_earlier_positions_then_lower_requests(oracle_mod):
    """Equal survival: the smaller position k wins, then the lower request index b.
    With confidences 1.0 every survival equals 1."""
    conf = np.ones((3, 3), np.float32)
    assert oracle_mod.schedule(conf, 0.5, 7)["out_len"].tolist() == [3, 2, 2]
    assert oracle_mod.schedule(conf, 0.5, 2)["out_len"].tolist() == [1, 1, 0]
    assert oracle_mod.schedule(conf, 0.5, 4)["out_len"].tolist() == [2, 1, 1]
    # Rows of unequal tau-length: request 0 has two positions of survival 1, requests 1
    # and 2 one each. With budget 2 < B the floors compete; (0,0) and (1,0) outrank (0,1).
    conf2 = np.array([[1.0, 1.0], [1.0, 0.1], [1.0, 0.1]], np.float32)
    assert oracle_mod.schedule(conf2, 0.5, 2)["out_len"].tolist() == [1, 1, 0]
    assert oracle_mod.schedule(conf2, 0.5, 1)["out_len"].tolist() == [1, 0, 0]


def test_invalid_schedule_inputs(oracle_mod):
    conf = np.full((2, 3), 0.5, np.float32)
    bad = conf.copy()
    bad[1, 2] = np.nan
    assert oracle_mod.schedule(bad, 0.3, 10)["status"] == oracle_mod.ERR_INPUT
    bad[1, 2] = 1.5
    assert oracle_mod.schedule(bad, 0.3, 10)["status"] == oracle_mod.ERR_INPUT
    assert oracle_mod.schedule(conf, 1.5, 10)["status"] == oracle_mod.ERR_ARG
    assert oracle_mod.schedule(conf, 0.3, -1)["status"] == oracle_mod.ERR_ARG
