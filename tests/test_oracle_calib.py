"""Pins for the oracle's calibration prologue, load-aware threshold and online
calibration loop (CPU only).

Each pin checks the oracle against something other than itself: the power form of
temperature scaling, c' = c^(1/T) / (c^(1/T) + (1-c)^(1/T)) (an algebraic identity of
sigmoid(logit(c)/T)), its fixed points, the end points and weights of the load factor,
brute-force re-implementations in plain Python, and hand-computed cases.
Sources: DSpark Deep Dive, "Sequential Temperature Scaling", "Online Adaptation",
"The Calibration Loop in Practice", "The Raw Confidence Problem"; DSpark Guide,
"Dynamic Verification Scheduling Algorithm".
"""
import numpy as np
import pytest

import oracle

F32 = np.float32


def _power_form(c, T):
    a, b = c ** (1.0 / T), (1.0 - c) ** (1.0 / T)
    return a / (a + b)


def pin_power_form(lib=None):
    rng = np.random.default_rng(1)
    for _ in range(200):
        c = float(F32(rng.uniform(0.001, 0.999)))
        T = float(rng.uniform(0.25, 4.0))
        got = oracle.calibrate(c, T, lib=lib)
        assert abs(got - _power_form(c, T)) <= 1e-12 * max(got, 1e-300), (c, T, got)


def pin_fixed_points(lib=None):
    for c in (0.05, 0.3, 0.77, 0.999):
        assert abs(oracle.calibrate(c, 1.0, lib=lib) - c) <= 1e-15
    for T in (0.3, 1.0, 7.0):
        assert oracle.calibrate(0.5, T, lib=lib) == 0.5
        assert oracle.calibrate(0.0, T, lib=lib) == 0.0
        assert oracle.calibrate(1.0, T, lib=lib) == 1.0


def pin_symmetry_and_direction(lib=None):
    for c in (0.1, 0.6, 0.93):
        for T in (0.5, 2.0):
            s = oracle.calibrate(c, T, lib=lib) + oracle.calibrate(1.0 - c, T, lib=lib)
            assert abs(s - 1.0) <= 1e-15
    # A temperature above 1 pulls an overconfident score toward 1/2; below 1 sharpens it.
    assert oracle.calibrate(0.9, 2.0, lib=lib) < 0.9 < oracle.calibrate(0.9, 0.5, lib=lib)
    assert oracle.calibrate(0.2, 2.0, lib=lib) > 0.2 > oracle.calibrate(0.2, 0.5, lib=lib)


def pin_load_tau(lib=None):
    lo, hi = 0.2, 0.75
    d = hi - lo
    cases = [((0, 10, 0, 64), lo), ((10, 10, 64, 64), hi), ((5, 10, 32, 64), lo + 0.25 * d),
             ((10, 10, 0, 64), lo + 0.36 * d), ((0, 10, 64, 64), lo + 0.16 * d),
             ((40, 10, 64, 64), hi)]
    for load, want in cases:
        got = oracle.load_tau(np.array(load, F32), lo, hi, lib=lib)
        assert abs(got - want) <= 1e-15, (load, got, want)
    for bad in ((1, 0, 1, 1), (1, 1, 1, -1), (float("nan"), 1, 1, 1), (-1, 1, 1, 1)):
        assert oracle.load_tau(np.array(bad, F32), lo, hi, lib=lib) == -1.0


def _bf_schedule(cal, tau, budget):
    """Brute force: survival products, tau-truncation with a floor of one, and the
    budget trim by sorting all kept positions."""
    B, K = cal.shape
    S = np.cumprod(cal, axis=1)
    L0 = np.maximum(1, (S >= tau).sum(axis=1))
    if L0.sum() <= budget:
        return L0.astype(np.int32), S
    floor_first = budget >= B
    cand = [((0 if (floor_first and k == 0) else 1), -S[b, k], k, b)
            for b in range(B) for k in range(L0[b])]
    cand.sort()
    out = np.zeros(B, np.int32)
    for c in cand[:budget]:
        out[c[3]] += 1
    return out, S


def pin_schedule_ex_bruteforce(lib=None):
    rng = np.random.default_rng(7)
    checked = 0
    for seed in range(60):
        B, K = int(rng.integers(1, 9)), int(rng.integers(1, 7))
        conf = rng.beta(8, 2, size=(B, K)).astype(F32) * F32(0.95)
        temps = rng.uniform(0.5, 2.5, size=K).astype(F32)
        load = np.array([rng.uniform(0, 12), 10, rng.uniform(0, 80), 80], F32)
        budget = int(rng.integers(0, B * K + 2))
        r = oracle.schedule_ex(conf, temps, load, 0.3, 0.2, 0.75, budget, lib=lib)
        assert r["status"] == 0
        cal = np.array([[_power_form(float(conf[b, k]), float(temps[k])) for k in range(K)]
                        for b in range(B)])
        lf = min(1.0, 0.6 * float(load[0]) / float(load[1]) + 0.4 * float(load[2]) / float(load[3]))
        tmin, tmax = float(F32(0.2)), float(F32(0.75))  # the call passes them as float32
        tau = tmin + (tmax - tmin) * lf * lf
        want, S = _bf_schedule(cal, tau, budget)
        # Skip draws where rounding could decide: a survival within 1e-9 of tau, or two
        # competing survivals within 1e-9 of each other.
        flat = np.sort(S.ravel())
        if np.min(np.abs(S - tau)) < 1e-9 or (flat.size > 1 and np.min(np.diff(flat)) < 1e-9):
            continue
        checked += 1
        assert abs(r["tau"] - tau) <= 1e-15
        assert np.array_equal(r["out_len"], want), (seed, r["out_len"], want)
        assert np.allclose(r["surv"], S, rtol=1e-12, atol=0)
        assert np.allclose(r["cal"], cal.astype(F32), rtol=2 ** -23, atol=0)
    assert checked >= 40


def pin_schedule_ex_plain_path(lib=None):
    """No temperatures and no load: exactly the plain schedule."""
    rng = np.random.default_rng(3)
    for _ in range(20):
        B, K = int(rng.integers(1, 12)), int(rng.integers(1, 9))
        conf = rng.uniform(0.3, 1.0, size=(B, K)).astype(F32)
        budget = int(rng.integers(0, B * K + 1))
        a = oracle.schedule(conf, 0.35, budget, lib=lib)
        b = oracle.schedule_ex(conf, None, None, 0.35, 0.2, 0.75, budget, lib=lib)
        assert np.array_equal(a["out_len"], b["out_len"]) and np.array_equal(a["surv"], b["surv"])


def _bf_observe(cal, vlen, acc, K):
    st = np.zeros(oracle.calib_stats_len(K))
    nb = oracle.CALIB_BINS
    for b in range(cal.shape[0]):
        L, j = int(vlen[b]), int(acc[b])
        if j < 0:
            continue
        for k in range(K):
            if k < L and k <= j:
                c = float(cal[b, k])
                a = 1.0 if k < j else 0.0
                st[3 * k:3 * k + 3] += (c, 1.0, a)
                bi = min(nb - 1, int(np.floor(c * nb)))
                st[3 * K + 3 * bi:3 * K + 3 * bi + 3] += (1.0, c, a)
    return st


def pin_observe_bruteforce(lib=None):
    rng = np.random.default_rng(11)
    for _ in range(30):
        B, K = int(rng.integers(1, 20)), int(rng.integers(1, 9))
        cal = rng.uniform(0, 1, size=(B, K)).astype(F32)
        vlen = rng.integers(0, K + 1, size=B).astype(np.int32)
        acc = np.array([rng.integers(0, v + 1) for v in vlen], np.int32)
        acc[rng.uniform(size=B) < 0.1] = -1
        st = np.zeros(oracle.calib_stats_len(K))
        assert oracle.calib_observe(cal, vlen, acc, st, lib=lib) == 0
        assert np.allclose(st, _bf_observe(cal, vlen, acc, K), rtol=1e-14, atol=0)


def _hand_stats(lib=None):
    # Values well inside their bins (0.9 as float32 is just below 0.9, in bin 8).
    cal = np.array([[0.95, 0.85, 0.75], [0.65, 0.55, 0.45]], F32)
    st = np.zeros(oracle.calib_stats_len(3))
    assert oracle.calib_observe(cal, np.array([3, 2], np.int32), np.array([1, 2], np.int32), st,
                                lib=lib) == 0
    return cal, st


def pin_observe_hand(lib=None):
    cal, st = _hand_stats(lib)
    c = cal.astype(np.float64)
    assert np.array_equal(st[0:3], [c[0, 0] + c[1, 0], 2, 2])
    assert np.array_equal(st[3:6], [c[0, 1] + c[1, 1], 2, 1])
    assert np.array_equal(st[6:9], [0, 0, 0])
    bins = st[9:].reshape(-1, 3)
    assert np.array_equal(bins[9], [1, c[0, 0], 1]) and np.array_equal(bins[8], [1, c[0, 1], 0])
    assert np.array_equal(bins[6], [1, c[1, 0], 1]) and np.array_equal(bins[5], [1, c[1, 1], 1])
    assert bins[[0, 1, 2, 3, 4, 7]].sum() == 0


def pin_update_hand(lib=None):
    cal, st = _hand_stats(lib)
    c = cal.astype(np.float64)
    temps = np.ones(3, F32)
    rc, ece = oracle.calib_update(st, temps, 0.1, 0.05, lib=lib)
    assert rc == 0
    e0 = (c[0, 0] + c[1, 0]) / 2 - 1.0
    e1 = (c[0, 1] + c[1, 1]) / 2 - 0.5
    assert temps[0] == F32(1.0 + 0.1 * e0) and temps[1] == F32(1.0 + 0.1 * e1) and temps[2] == 1.0
    assert temps[0] < 1.0 < temps[1]  # under- then overconfident position
    want = (abs(1 - c[0, 0]) + abs(0 - c[0, 1]) + abs(1 - c[1, 0]) + abs(1 - c[1, 1])) / 4
    assert abs(ece - want) <= 1e-15
    assert not st.any()  # the window starts over


def pin_ece_limits(lib=None):
    K = 2
    st = np.zeros(oracle.calib_stats_len(K))
    bins = st[3 * K:].reshape(-1, 3)
    bins[7] = (100, 70.0, 70)  # predicted 0.7, 70 of 100 accepted
    bins[2] = (10, 2.5, 2.5)
    rc, ece = oracle.calib_update(st, np.ones(K, F32), 0.01, 0.05, lib=lib)
    assert rc == 0 and ece == 0.0
    st = np.zeros(oracle.calib_stats_len(K))
    st[3 * K + 3 * 9:3 * K + 3 * 9 + 3] = (50, 47.5, 0)  # confident and always wrong
    st[3 * K + 3 * 1:3 * K + 3 * 1 + 3] = (50, 7.5, 50)
    rc, ece = oracle.calib_update(st, np.ones(K, F32), 0.01, 0.05, lib=lib)
    assert abs(ece - (47.5 + 42.5) / 100) <= 1e-15


def pin_update_floor_and_idle(lib=None):
    K = 2
    st = np.zeros(oracle.calib_stats_len(K))
    st[0:3] = (0.0, 10, 10)  # error -1 at position 0
    temps = np.array([0.3, 2.0], F32)
    oracle.calib_update(st, temps, 0.5, 0.1, lib=lib)
    assert temps[0] == F32(0.1) and temps[1] == F32(2.0)  # floored; untested position kept


PINS = [pin_power_form, pin_fixed_points, pin_symmetry_and_direction, pin_load_tau,
        pin_schedule_ex_bruteforce, pin_schedule_ex_plain_path, pin_observe_bruteforce,
        pin_observe_hand, pin_update_hand, pin_ece_limits, pin_update_floor_and_idle]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(None)


def test_invalid_inputs():
    conf = np.full((2, 3), 0.5, F32)
    assert oracle.schedule_ex(conf, np.array([1, 0, 1], F32), None, 0.3, 0.2, 0.75, 6)["status"] == -5
    assert oracle.schedule_ex(conf, None, np.array([1, 0, 1, 1], F32), 0.3, 0.2, 0.75, 6)["status"] == -5
    conf[1, 2] = 1.5
    r = oracle.schedule_ex(conf, None, None, 0.3, 0.2, 0.75, 6)
    assert r["status"] == -5 and not r["out_len"].any()
