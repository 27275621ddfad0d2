"""Pins for the oracle's throughput-curve schedule (CPU only).

Source: DSpark Deep Dive, "The Throughput Curve" and "The Optimization Logic". The budget
is the smallest N maximising (B + A(N)) T(B + N) / (B + N), A(N) the sum of the N best
survivals in the budget-trim order, T the curve (linear between points, flat outside).
Pins: a brute-force re-implementation with numpy.interp (an independent interpolation
routine) and sorted survivals; the two regimes the page describes (throughput growing
with the batch: verify every tau-survivor; a flat curve: only tokens whose survival
beats the running average are worth their slot); and the page's example table.
"""
import numpy as np
import pytest

import oracle

F32 = np.float32
# [DD] "The Throughput Curve": batch size -> tokens/s (example table on the page).
PAGE_X = np.array([1, 2, 4, 8, 16, 32, 64, 128], F32)
PAGE_Y = np.array([35, 67, 125, 220, 360, 520, 650, 720], F32)


def _bf(conf, tau, budget, cx, cy):
    B, K = conf.shape
    S = np.cumprod(conf.astype(np.float64), axis=1)
    L0 = np.maximum(1, (S >= tau).sum(axis=1))
    total = int(L0.sum())
    n_hi = min(total, budget)
    floors = budget >= B
    n_lo = B if floors else 0
    a0 = sum(S[b, 0] for b in range(B)) if floors else 0.0
    comp = sorted((S[b, k] for b in range(B) for k in range(L0[b]) if not (floors and k == 0)),
                  reverse=True)
    best, best_n = -1.0, n_lo
    for n in range(n_lo, n_hi + 1):
        a = a0 + sum(comp[:n - n_lo])
        x = B + n
        g = (B + a) * np.interp(x, cx.astype(np.float64), cy.astype(np.float64)) / x
        if g > best * (1 + 1e-12):
            best, best_n = g, n
    return best_n, best


def pin_bruteforce(lib=None):
    rng = np.random.default_rng(5)
    for seed in range(40):
        B, K = int(rng.integers(1, 10)), int(rng.integers(1, 7))
        conf = rng.beta(6, 2, size=(B, K)).astype(F32)
        cx = np.sort(rng.choice(np.arange(1, 200), size=int(rng.integers(2, 7)), replace=False)).astype(F32)
        cy = np.maximum.accumulate(rng.uniform(10, 100, size=cx.size)).astype(F32)
        budget = int(rng.integers(0, B * K + 2))
        r = oracle.schedule_curve(conf, None, None, 0.2, 0.2, 0.75, cx, cy, budget, lib=lib)
        assert r["status"] == 0
        n, g = _bf(conf, float(F32(0.2)), budget, cx, cy)
        assert r["n"] == n, (seed, r["n"], n)
        assert abs(r["g"] - g) <= 1e-9 * g
        plain = oracle.schedule(conf, 0.2, n, lib=lib)["out_len"]
        assert np.array_equal(r["out_len"], plain)


def pin_regimes(lib=None):
    rng = np.random.default_rng(9)
    conf = rng.beta(8, 2, size=(16, 8)).astype(F32)
    l0 = oracle.schedule(conf, 0.1, 10 ** 6, lib=lib)["l0"]
    # Throughput proportional to the batch: every token adds output at no cost.
    lin = oracle.schedule_curve(conf, None, None, 0.1, 0.2, 0.75, np.array([1, 1e6], F32),
                                np.array([1, 1e6], F32), 10 ** 6, lib=lib)
    assert lin["n"] == int(l0.sum()) and np.array_equal(lin["out_len"], l0)
    # A flat curve: goodput (B + A) / (B + N) grows only while the next survival beats it.
    flat = oracle.schedule_curve(conf, None, None, 0.1, 0.2, 0.75, np.array([1, 2], F32),
                                 np.array([100, 100], F32), 10 ** 6, lib=lib)
    S = np.cumprod(conf.astype(np.float64), axis=1)
    comp = np.sort(np.concatenate([S[b, 1:l0[b]] for b in range(16)]))[::-1]
    a, n = S[:, 0].sum(), 16
    while n - 16 < comp.size and comp[n - 16] > (16 + a) / (16 + n):
        a += comp[n - 16]
        n += 1
    assert flat["n"] == n
    assert flat["n"] < lin["n"]


def pin_page_table(lib=None):
    """With the page's curve, a lightly loaded batch verifies more per request than a
    heavily loaded one (its tokens/s still grow steeply at small batches)."""
    conf = np.tile(np.array([[0.95, 0.9, 0.8, 0.7, 0.6, 0.5, 0.45, 0.4]], F32), (1, 1))
    small = oracle.schedule_curve(np.tile(conf, (2, 1)), None, None, 0.0, 0.2, 0.75, PAGE_X,
                                  PAGE_Y, 10 ** 6, lib=lib)
    large = oracle.schedule_curve(np.tile(conf, (48, 1)), None, None, 0.0, 0.2, 0.75, PAGE_X,
                                  PAGE_Y, 10 ** 6, lib=lib)
    assert small["n"] / 2 > large["n"] / 48


PINS = [pin_bruteforce, pin_regimes, pin_page_table]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(None)


def test_invalid_curve():
    conf = np.full((2, 3), 0.5, F32)
    bad = oracle.schedule_curve(conf, None, None, 0.3, 0.2, 0.75, np.array([2, 1], F32),
                                np.array([1, 1], F32), 6)
    assert bad["status"] == -5 and not bad["out_len"].any()
    bad = oracle.schedule_curve(conf, None, None, 0.3, 0.2, 0.75, np.array([1, 2], F32),
                                np.array([1, 0], F32), 6)
    assert bad["status"] == -5
