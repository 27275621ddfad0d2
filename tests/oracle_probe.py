"""Helpers that measure the oracle's decisions as functions of its uniforms.

The verification outcome is a step function of each uniform. These helpers locate
the steps by a grid scan plus bisection (to about 1e-14), so a test can integrate
the oracle's behaviour over u exactly instead of sampling it.
"""
import numpy as np

GRID = 2048
TOL = 1e-14


def intervals(f, grid=GRID, tol=TOL):
    """Partition [0,1) by the value of f(u). Returns {value: total length}."""
    us = np.linspace(0.0, 1.0, grid + 1)
    us[-1] = 1.0 - 1e-16
    vals = [f(float(u)) for u in us]
    cuts = []  # (position, value to the right)

    def split(lo, hi, flo, fhi):
        if flo == fhi:
            return
        if hi - lo < tol:
            cuts.append((0.5 * (lo + hi), fhi))
            return
        mid = 0.5 * (lo + hi)
        fm = f(mid)
        split(lo, mid, flo, fm)
        split(mid, hi, fm, fhi)

    for i in range(grid):
        split(us[i], us[i + 1], vals[i], vals[i + 1])
    cuts.sort()
    mass = {}
    pos, cur = 0.0, vals[0]
    for c, v in cuts:
        mass[cur] = mass.get(cur, 0.0) + (c - pos)
        pos, cur = c, v
    mass[cur] = mass.get(cur, 0.0) + (1.0 - pos)
    return mass


def softmax64(z, T):
    """Reference softmax of the (already rounded) logits in float64, numpy."""
    z = np.asarray(z, dtype=np.float64) / T
    e = np.exp(z - z.max())
    return e / e.sum()


def intervals_batch(fb, grid=GRID, tol=TOL):
    """intervals() for a function evaluated on many uniforms at once: fb maps a float64
    array of uniforms to an integer array of values. Returns {value: total length}."""
    us = np.linspace(0.0, 1.0, grid + 1)
    us[-1] = 1.0 - 1e-16
    vals = np.asarray(fb(us))
    step = np.nonzero(vals[:-1] != vals[1:])[0]
    active = [(us[i], us[i + 1], vals[i], vals[i + 1]) for i in step]
    cuts = []  # (position, value to the right)
    while active:
        mids = np.array([0.5 * (lo + hi) for lo, hi, _, _ in active])
        fm = np.asarray(fb(mids))
        nxt = []
        for (lo, hi, flo, fhi), mid, v in zip(active, mids, fm):
            for a, b, fa, fb_ in ((lo, mid, flo, v), (mid, hi, v, fhi)):
                if fa == fb_:
                    continue
                if b - a < tol:
                    cuts.append((0.5 * (a + b), fb_))
                else:
                    nxt.append((a, b, fa, fb_))
        active = nxt
    cuts.sort()
    mass = {}
    pos, cur = 0.0, vals[0]
    for c, v in cuts:
        mass[cur] = mass.get(cur, 0.0) + (c - pos)
        pos, cur = c, v
    mass[cur] = mass.get(cur, 0.0) + (1.0 - pos)
    return {int(k): v for k, v in mass.items()}
