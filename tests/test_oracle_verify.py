"""Pins for the oracle's verification (CPU only).

Each test checks the oracle against something other than itself: the losslessness
theorem (exact, by integrating the oracle's own decisions over its uniforms), the
greedy special case (numpy argmax), the q == p closed form, the closed-form
acceptance rate, and hand-derived cases.
"""
import itertools

import numpy as np
import pytest

from oracle_probe import intervals, softmax64

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _one(oracle_mod, t, d, tok, L, u, T, u64=True, lib=None):
    """Run the oracle on a single request; returns (out_tok row, accepted)."""
    r = oracle_mod.verify(t[None], None if d is None else d[None], np.asarray(tok)[None],
                          np.array([L]), None if u is None else np.asarray(u)[None], T,
                          diag=False, u64=u64, lib=lib)
    return r["out_tok"][0], int(r["out_accepted"][0])


def _random_rows(rng, rows, V, scale):
    return (rng.normal(0.0, scale, size=(rows, V))).astype(np.float32)


def lossless_error(oracle_mod, T, seed, lib=None):
    """Largest |P(m-th emitted token = v | first m emitted were accepted drafts) - p_m(v)|
    over m and v, computed exactly for V=8, K=3 (see test_lossless_bruteforce_V8_K3)."""
    V, K = 8, 3
    rng = np.random.default_rng(seed)
    t = _random_rows(rng, K + 1, V, 1.5)
    d = (t[:K] + rng.normal(0.0, 1.0, size=(K, V))).astype(np.float32)
    P = [softmax64(t[k], T) for k in range(K + 1)]
    Q = [softmax64(d[k], T) for k in range(K)]

    def run(tok, u):
        return _one(oracle_mod, t, d, tok, K, u, T, lib=lib)

    # a[k][x]: probability over u_k that the oracle accepts draft x at position k.
    a = np.zeros((K, V))
    # R[k][x]: distribution of the token the oracle emits after rejecting x at k.
    R = np.zeros((K, V, V))
    for k in range(K):
        for x in range(V):
            tok = [0] * K
            tok[k] = x

            def acc(uk, k=k, tok=tok):
                u = np.zeros(K + 1)
                u[k] = uk
                u[k + 1:] = 0.5
                return int(run(tok, u)[1] > k)

            a[k, x] = intervals(acc).get(1, 0.0)
            if a[k, x] < 1.0 - 1e-12:
                def term(uK, k=k, tok=tok):
                    u = np.zeros(K + 1)
                    u[k] = 1.0 - 1e-12
                    u[K] = uK
                    out, j = run(tok, u)
                    return int(out[k]) if j == k else -2

                for v, m in intervals(term).items():
                    if 0 <= v < V:
                        R[k, x, v] += m

    def bonus(uK):
        u = np.zeros(K + 1)
        u[K] = uK
        out, j = run([0] * K, u)
        return int(out[K]) if j == K else -2

    Bn = np.zeros(V)
    for v, m in intervals(bonus).items():
        if 0 <= v < V:
            Bn[v] += m

    err = 0.0
    for m in range(K + 1):
        joint = np.zeros(V)
        pe = 0.0
        for xs in itertools.product(range(V), repeat=K):
            w = np.prod([Q[k][xs[k]] for k in range(K)])
            reach = w * np.prod([a[i, xs[i]] for i in range(m)])
            pe += reach
            if m < K:
                x = xs[m]
                joint[x] += reach * a[m, x]
                joint += reach * (1.0 - a[m, x]) * R[m, x]
            else:
                joint += reach * Bn
        err = max(err, float(np.abs(joint / pe - P[m]).max()))
    return err


@pytest.mark.parametrize("T,seed", [(1.0, 0), (0.5, 1), (2.0, 2), (1.0, 3)])
def test_lossless_bruteforce_V8_K3(oracle_mod, T, seed):
    """Losslessness, exactly: the m-th emitted token, given that the first m emitted
    tokens were accepted drafts, is distributed as softmax(target_m / T).

    Pages: 'Verified by the target' (perchy.ai Technology: outputs follow the target
    distribution exactly); DSpark Deep Dive, 'The Speculative Decoding Solution'
    (rejection sampling keeps the target distribution). Drafts x_k ~ q_k independently;
    every draft tuple of V**K = 512 is enumerated with weight prod q_k(x_k); the
    oracle's accept/reject branches and terminal samples are integrated over the
    uniforms by locating the steps of its output (grid + bisection)."""
    assert lossless_error(oracle_mod, T, seed) < 1e-9


def test_accept_rule_orientation(oracle_mod):
    """The accept probability of draft x is min(1, p(x)/q(x)) and not its inverse
    (DSpark Deep Dive, 'The Speculative Decoding Solution')."""
    V, K = 8, 1
    rng = np.random.default_rng(7)
    t = _random_rows(rng, 2, V, 2.0)
    d = (t[:1] + rng.normal(0.0, 1.5, size=(1, V))).astype(np.float32)
    p, q = softmax64(t[0], 1.0), softmax64(d[0], 1.0)
    for x in range(V):
        def acc(u0, x=x):
            return int(_one(oracle_mod, t, d, [x], 1, [u0, 0.5], 1.0)[1] > 0)

        np.testing.assert_allclose(intervals(acc).get(1, 0.0), min(1.0, p[x] / q[x]), atol=1e-9)


def test_greedy_is_argmax_matching(oracle_mod):
    """At T=0 verification reduces to argmax matching; ties go to the lowest index
    (numpy argmax returns the first occurrence)."""
    rng = np.random.default_rng(11)
    B, K, V = 64, 6, 50
    t = rng.integers(-4, 5, size=(B, K + 1, V)).astype(np.float32)  # many exact ties
    am = t.argmax(axis=-1)
    tok = np.where(rng.random((B, K)) < 0.7, am[:, :K], rng.integers(0, V, (B, K))).astype(np.int32)
    vlen = rng.integers(0, K + 1, size=B).astype(np.int32)
    r = oracle_mod.verify(t, None, tok, vlen, None, 0.0, diag=False)
    assert r["status"] == 0
    for b in range(B):
        L = vlen[b]
        j = 0
        while j < L and tok[b, j] == am[b, j]:
            j += 1
        assert r["out_accepted"][b] == j
        np.testing.assert_array_equal(r["out_tok"][b, :j], tok[b, :j])
        assert r["out_tok"][b, j] == am[b, j]
        assert (r["out_tok"][b, j + 1:] == -1).all()


def test_q_equals_p_accepts_everything(oracle_mod):
    """With draft == target logits, p == q and every draft is accepted (u < 1); the
    emitted tokens are the drafts followed by a bonus sample."""
    rng = np.random.default_rng(5)
    B, K, V = 16, 5, 300
    t = _random_rows(rng, B * (K + 1), V, 2.0).reshape(B, K + 1, V)
    d = t[:, :K].copy()
    tok = rng.integers(0, V, size=(B, K)).astype(np.int32)
    u = rng.random((B, K + 1)).astype(np.float32)
    u[:, :K] = np.maximum(u[:, :K], np.float32(0.999999))  # hardest case: u close to 1
    r = oracle_mod.verify(t, d, tok, np.full(B, K, np.int32), u, 1.0)
    assert r["status"] == 0
    assert (r["out_accepted"] == K).all()
    np.testing.assert_array_equal(r["out_tok"][:, :K], tok)
    np.testing.assert_array_equal(r["p"], r["q"])


def test_acceptance_length_matches_product_formula(oracle_mod):
    """P(accepted length >= m) = prod_{k<m} sum_v min(p_k(v), q_k(v)) when drafts are
    drawn from q (DSpark Guide, '1. The Mathematics of Suffix Decay': the prefix
    survives with the product of per-position acceptance probabilities). Monte Carlo
    over 40,000 requests, 5-sigma binomial bounds."""
    rng = np.random.default_rng(21)
    K, V, N = 4, 16, 40_000
    t = _random_rows(rng, K + 1, V, 1.0)
    d = (t[:K] + rng.normal(0.0, 0.8, size=(K, V))).astype(np.float32)
    P = [softmax64(t[k], 1.0) for k in range(K + 1)]
    Q = [softmax64(d[k], 1.0) for k in range(K)]
    alpha = [np.minimum(P[k], Q[k]).sum() for k in range(K)]
    tok = np.stack([rng.choice(V, size=N, p=Q[k]) for k in range(K)], axis=1).astype(np.int32)
    u = rng.random((N, K + 1)).astype(np.float32)
    tt = np.broadcast_to(t, (N, K + 1, V)).copy()
    dd = np.broadcast_to(d, (N, K, V)).copy()
    r = oracle_mod.verify(tt, dd, tok, np.full(N, K, np.int32), u, 1.0, diag=False, nthreads=4)
    acc = r["out_accepted"]
    for m in range(1, K + 1):
        expect = float(np.prod(alpha[:m]))
        got = float((acc >= m).mean())
        assert abs(got - expect) < 5 * np.sqrt(expect * (1 - expect) / N) + 1e-12, (m, got, expect)


def test_hand_cases(oracle_mod):
    """Hand-derived single-position cases (V=3, L=1).

    target row 0 = log[0.5, 0.3, 0.2], draft row 0 = log[0.2, 0.5, 0.3],
    target row 1 = log[0.1, 0.6, 0.3].
      x=1: p/q = 0.6.  u0=0.59 accepts; bonus from row 1: u=0.05 -> 0, 0.5 -> 1, 0.95 -> 2.
           u0=0.61 rejects; residual max(0,p-q) = [0.3,0,0] -> token 0 for any u.
      x=0: p/q = 2.5, accepted for every u0 < 1.
      x=2: p/q = 2/3.  u0=0.66 accepts, u0=0.67 rejects -> token 0.
    At T=2 the same decisions hold for doubled logits (softmax(z/T) with z = 2 log p)."""
    def rows(ps):
        return np.log(np.array(ps, np.float64)).astype(np.float32)

    t = np.stack([rows([0.5, 0.3, 0.2]), rows([0.1, 0.6, 0.3])])
    d = rows([0.2, 0.5, 0.3])[None]
    cases = [
        (1, 0.59, 0.05, 1, [1, 0]), (1, 0.59, 0.5, 1, [1, 1]), (1, 0.59, 0.95, 1, [1, 2]),
        (1, 0.61, 0.99, 0, [0, -1]), (1, 0.61, 0.01, 0, [0, -1]),
        (0, 0.999, 0.5, 1, [0, 1]), (2, 0.66, 0.95, 1, [2, 2]), (2, 0.67, 0.4, 0, [0, -1]),
    ]
    for T, scale in [(1.0, 1.0), (2.0, 2.0)]:
        for x, u0, uK, acc, out in cases:
            ot, j = _one(oracle_mod, t * scale, d * scale, [x], 1, np.array([u0, uK], np.float32),
                         T, u64=False)
            assert j == acc, (T, x, u0, uK)
            assert list(ot) == out, (T, x, u0, uK, ot)
    # Residual with two positive buckets: target [0.5,0.4,0.1], draft [0.2,0.3,0.5],
    # x=2 (p/q = 0.2), u0=0.5 rejects; residual [0.3,0.1,0] (Z=0.4):
    # u=0.7 -> 0.28 < 0.3 -> token 0; u=0.8 -> 0.32 -> token 1.
    t2 = np.stack([rows([0.5, 0.4, 0.1]), rows([0.1, 0.6, 0.3])])
    d2 = rows([0.2, 0.3, 0.5])[None]
    for uK, y in [(0.7, 0), (0.8, 1)]:
        ot, j = _one(oracle_mod, t2, d2, [2], 1, np.array([0.5, uK], np.float32), 1.0, u64=False)
        assert j == 0 and ot[0] == y


def test_decision_margin_hand_case(oracle_mod):
    """The margin diagnostic is the smaller of |u_0 - min(1, p/q)| at the tested position
    and the terminal sample's distance to the nearer edge of its CDF bucket (normalised),
    derived by hand here for V=3, L=1 (accepted -> bonus from p_1; rejected -> residual)."""
    def rows(ps):
        return np.log(np.array(ps, np.float64)).astype(np.float32)

    t = np.stack([rows([0.5, 0.3, 0.2]), rows([0.1, 0.6, 0.3])])
    d = rows([0.2, 0.5, 0.3])[None]
    p0, q0, p1 = softmax64(t[0], 1.0), softmax64(d[0], 1.0), softmax64(t[1], 1.0)
    # (u0, uK): accept margin 0.01 / bonus gap 0.05; accept margin 0.05 / bonus gap 0.01;
    # reject (margin 0.01) with residual [0.3, 0, 0] whose single bucket gives gap 0.5.
    for u0, uK in [(0.59, 0.65), (0.55, 0.69), (0.61, 0.5)]:
        u = np.array([u0, uK], np.float32)
        r = oracle_mod.verify(t[None], d[None], np.array([[1]]), np.array([1]), u[None], 1.0,
                              diag=False)
        accept_margin = abs(float(u[0]) - min(1.0, p0[1] / q0[1]))
        w = p1 if float(u[0]) * q0[1] < p0[1] else np.maximum(p0 - q0, 0.0)
        cum = np.cumsum(w)
        target = float(u[1]) * cum[-1]
        y = int(np.searchsorted(cum, target, side="right"))
        gap = min(target - (cum[y] - w[y]), cum[y] - target) / cum[-1]
        assert abs(r["margin"][0] - min(accept_margin, gap)) < 1e-12, (u0, uK)


def test_zero_length_block_is_plain_sampling(oracle_mod):
    """L = 0: nothing to verify; the call emits one token sampled from p_0 (greedy: argmax)."""
    t = np.log(np.array([[0.25, 0.25, 0.5], [1 / 3, 1 / 3, 1 / 3]])).astype(np.float32)
    for uK, y in [(0.1, 0), (0.3, 1), (0.6, 2)]:
        ot, j = _one(oracle_mod, t, np.zeros((1, 3), np.float32), [0], 0,
                     np.array([0.5, uK], np.float32), 1.0, u64=False)
        assert j == 0 and list(ot) == [y, -1]
    ot, j = _one(oracle_mod, t, None, [0], 0, None, 0.0, u64=False)
    assert j == 0 and list(ot) == [2, -1]


def test_masked_tokens_never_sampled(oracle_mod):
    """-inf logits are masked tokens: probability 0, never accepted or emitted."""
    rng = np.random.default_rng(3)
    B, K, V = 200, 3, 12
    t = _random_rows(rng, B * (K + 1), V, 1.0).reshape(B, K + 1, V)
    t[:, :, ::2] = -np.inf
    d = (t[:, :K] + rng.normal(0, 1.0, (B, K, V))).astype(np.float32)
    d[:, :, 1::4] = -np.inf
    tok = rng.integers(0, V, size=(B, K)).astype(np.int32)
    u = rng.random((B, K + 1)).astype(np.float32)
    r = oracle_mod.verify(t, d, tok, np.full(B, K, np.int32), u, 1.0)
    assert r["status"] == 0
    for b in range(B):
        j = r["out_accepted"][b]
        assert r["out_tok"][b, j] % 2 == 1


def test_invalid_inputs_flagged(oracle_mod):
    """Invalid requests give out_accepted = -1, a row of -1, the INVALID flag and a
    non-zero status; valid requests in the same batch are unaffected."""
    rng = np.random.default_rng(9)
    B, K, V = 8, 3, 20
    t = _random_rows(rng, B * (K + 1), V, 1.0).reshape(B, K + 1, V)
    d = (t[:, :K] + rng.normal(0, 1.0, (B, K, V))).astype(np.float32)
    tok = rng.integers(0, V, size=(B, K)).astype(np.int32)
    vlen = np.full(B, K, np.int32)
    u = rng.random((B, K + 1)).astype(np.float32)
    t[1, 2, 5] = np.nan
    d[2, 0, 3] = np.inf
    t[3, 1, :] = -np.inf
    tok[4, 1] = V
    vlen[5] = K + 1
    u[6, 0] = 1.0
    ref = oracle_mod.verify(t, d, tok, vlen, u, 1.0)
    assert ref["status"] == oracle_mod.ERR_INPUT
    for b in range(1, 7):
        assert ref["out_accepted"][b] == -1 and (ref["out_tok"][b] == -1).all()
        assert ref["flags"][b] & oracle_mod.FLAG_INVALID
    for b in (0, 7):
        assert ref["out_accepted"][b] >= 0 and not ref["flags"][b] & oracle_mod.FLAG_INVALID


def _bf16_round(x):
    """float32 array -> (bf16 bit patterns, their exact float64 values), round to
    nearest even, written out with integer arithmetic (no torch)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)
    return b, (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def pq_error(oracle_mod, lib=None):
    """Largest relative error of the oracle's diagnostic outputs p_k(x_k), q_k(x_k)
    against numpy's float64 softmax of the same (exactly representable) logits, over
    fp32 and bf16 inputs, T in {0.5, 1, 2}, ragged verify lengths and drafted tokens
    spread over the row; inf when a position k >= L_b is not NaN or a tested one is."""
    worst = 0.0
    for i, dt in enumerate(("f32", "bf16")):
        for j, T in enumerate((0.5, 1.0, 2.0)):
            rng = np.random.default_rng(100 + 10 * i + j)
            B, K, V = 6, 5, 700
            t = rng.normal(0.0, 2.5, size=(B, K + 1, V)).astype(np.float32)
            d = (t[:, :K] + rng.normal(0.0, 1.0, size=(B, K, V))).astype(np.float32)
            if dt == "bf16":
                (tb, tv), (db, dv) = _bf16_round(t), _bf16_round(d)
                targ, darg = tb, db
            else:
                tv, dv = t.astype(np.float64), d.astype(np.float64)
                targ, darg = t, d
            tok = rng.integers(0, V, size=(B, K)).astype(np.int32)
            L = np.array([0, 1, 3, 5, 2, 4], np.int32)
            u = rng.random((B, K + 1)).astype(np.float32)
            r = oracle_mod.verify(targ, darg, tok, L, u, T, lib=lib)
            for b in range(B):
                for k in range(K):
                    if k >= L[b]:
                        if not (np.isnan(r["p"][b, k]) and np.isnan(r["q"][b, k])):
                            return np.inf
                        continue
                    pk = softmax64(tv[b, k], T)[tok[b, k]]
                    qk = softmax64(dv[b, k], T)[tok[b, k]]
                    for got, want in ((r["p"][b, k], pk), (r["q"][b, k], qk)):
                        if not np.isfinite(got):
                            return np.inf
                        worst = max(worst, abs(got - want) / want)
    return worst


def test_diag_probabilities_are_softmax_at_drafted_token(oracle_mod):
    """The oracle's p_k(x_k) and q_k(x_k) outputs (the reference for the GPU's
    probability parity) against numpy's float64 softmax of target row k and draft row
    k at temperature T, evaluated at the drafted token [DSpark Deep Dive, 'The
    Speculative Decoding Solution': p and q are the softmax distributions of the target
    and draft logits]. Both sides sum V = 700 exponentials in float64 in different
    orders (sequential against pairwise) and round (z - M)/T against z/T - max(z/T),
    so they agree to a few ulps (measured 2e-15): 1e-14 relative. NaN beyond each
    request's verify length."""
    assert pq_error(oracle_mod) < 1e-14
