"""Pins for the oracle's tree (multi-candidate) verification (CPU only).

Each test checks the oracle against something other than its own code: the chain
oracle on chain-shaped trees (pinned on its own in test_oracle_verify.py), the
losslessness theorem integrated exactly over the oracle's uniforms at the root and one
level down, greedy invariants from numpy's argmax, hand-derived cases, and input
validation.
"""
import itertools

import numpy as np
import pytest

from oracle_probe import intervals_batch, softmax64

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

U_REJECT = 1.0 - 1e-16  # the largest uniform below 1: rejects unless acceptance is certain


def _rows(rng, n, V, scale=1.5):
    return rng.normal(0.0, scale, size=(n, V)).astype(np.float32)


def _batch(oracle_mod, t, d, par, tok, U, T, lib=None):
    """One tree, many uniform vectors: U [M, N] float64."""
    M, N = U.shape
    rep = lambda a: np.ascontiguousarray(np.repeat(a[None], M, axis=0))
    return oracle_mod.verify_tree(rep(t), None if d is None else rep(d), rep(par), rep(tok),
                                  np.full(M, N, np.int32), U, T, u64=True, lib=lib)


# ----------------------------------------------------------------------------------
# Chain-shaped trees reduce to the chain.
# ----------------------------------------------------------------------------------

def chain_mismatches(oracle_mod, seed, T, dtype_bits=False, lib=None):
    """Random chain requests run through both oracles; returns the number of requests
    whose outputs differ."""
    rng = np.random.default_rng(seed)
    B, K, V = 24, 5, 37
    t = _rows(rng, B * (K + 1), V, 2.0).reshape(B, K + 1, V)
    d = (t[:, :K] + rng.normal(0.0, 1.0, size=(B, K, V))).astype(np.float32)
    if dtype_bits:  # round to bf16 and pass bit patterns
        t = (t.view(np.uint32) >> 16).astype(np.uint16)
        d = (d.view(np.uint32) >> 16).astype(np.uint16)
        tf = (t.astype(np.uint32) << 16).view(np.float32)
    else:
        tf = t
    L = rng.integers(0, K + 1, size=B).astype(np.int32)
    tok = rng.integers(0, V, size=(B, K)).astype(np.int32)
    # Make some drafts the target's argmax so that greedy chains run deep.
    am = tf[:, :K].argmax(-1).astype(np.int32)
    pick = rng.random((B, K)) < 0.6
    tok[pick] = am[pick]
    u = rng.random((B, K + 1)).astype(np.float32)
    ref = oracle_mod.verify(t, d if T > 0 else None, tok, L, u if T > 0 else None, T,
                            diag=False, lib=lib)
    N = K + 1
    par = np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1))
    ttok = np.zeros((B, N), np.int32)
    ttok[:, 1:] = tok
    tu = np.zeros((B, N), np.float32)
    tu[:, 1:] = u[:, :K]
    tu[:, 0] = u[:, K]
    td = np.zeros_like(t)
    td[:, :K] = d
    got = oracle_mod.verify_tree(t, td if T > 0 else None, par, ttok, L + 1,
                                 tu if T > 0 else None, T, lib=lib)
    bad = (got["out_accepted"] != ref["out_accepted"]) | (got["out_tok"] != ref["out_tok"]).any(1)
    # The path of a chain is nodes 1..j.
    for b in range(B):
        j = got["out_accepted"][b]
        want = [n + 1 for n in range(j)] + [-1] * (N - j)
        if list(got["out_path"][b]) != want:
            bad[b] = True
    return int(bad.sum())


@pytest.mark.parametrize("T", [0.0, 0.6, 1.0, 2.5])
@pytest.mark.parametrize("seed", range(4))
def test_chain_tree_equals_chain(oracle_mod, seed, T):
    assert chain_mismatches(oracle_mod, seed, T) == 0


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_chain_tree_equals_chain_bf16(oracle_mod, T):
    assert chain_mismatches(oracle_mod, 7, T, dtype_bits=True) == 0


# ----------------------------------------------------------------------------------
# Losslessness, exactly: integrate the oracle's decisions over its uniforms.
# ----------------------------------------------------------------------------------

def level_distribution(oracle_mod, t, d, par, tok_fixed, level_node, children, T,
                       forced=None, lib=None):
    """Distribution of the token emitted at the walk's step from ``level_node``, with
    the children's tokens drawn i.i.d. from q = softmax(d[level_node]/T), computed by
    exact integration over the children's uniforms and the terminal uniform.

    forced: {node: uniform} fixed for every evaluation (used to steer the walk to
    ``level_node``); the depth of ``level_node`` is len(forced)."""
    V = t.shape[1]
    N = len(par)
    forced = forced or {}
    depth = len(forced)
    q = softmax64(d[level_node], T)
    out = np.zeros(V)
    m = len(children)
    for xs in itertools.product(range(V), repeat=m):
        w = float(np.prod([q[x] for x in xs]))
        tok = np.array(tok_fixed, np.int32).copy()
        for n, x in zip(children, xs):
            tok[n] = x

        def base(M):
            U = np.full((M, N), U_REJECT)
            U[:, 0] = 0.5
            for n, un in forced.items():
                U[:, n] = un
            return U

        reach = 1.0
        for i, n in enumerate(children):
            def fb(us, n=n):
                U = base(len(us))
                U[:, n] = us
                r = _batch(oracle_mod, t, d, par, tok, U, T, lib=lib)
                return r["out_path"][:, depth]

            a = intervals_batch(fb).get(n, 0.0)
            out[xs[i]] += w * reach * a
            reach *= 1.0 - a
            if reach <= 0.0:
                break
        if reach > 0.0:
            def fterm(us):
                U = base(len(us))
                U[:, 0] = us
                r = _batch(oracle_mod, t, d, par, tok, U, T, lib=lib)
                return np.where(r["out_accepted"] == depth, r["out_tok"][:, depth], -2)

            for v, mass in intervals_batch(fterm).items():
                if 0 <= v < V:
                    out[v] += w * reach * mass
    return out


def root_lossless_error(oracle_mod, m, T, seed, V=4, lib=None):
    rng = np.random.default_rng(seed)
    N = m + 1
    t = _rows(rng, N, V)
    d = (t + rng.normal(0.0, 1.2, size=(N, V))).astype(np.float32)
    par = np.array([-1] + [0] * m, np.int32)
    got = level_distribution(oracle_mod, t, d, par, np.zeros(N, np.int32), 0,
                             list(range(1, N)), T, lib=lib)
    return float(np.abs(got - softmax64(t[0], T)).max())


@pytest.mark.parametrize("m,T,seed", [(1, 1.0, 0), (2, 1.0, 1), (3, 1.0, 2), (3, 0.6, 3),
                                      (2, 2.0, 4)])
def test_lossless_root(oracle_mod, m, T, seed):
    """First emitted token ~ p_0 when the root's m children are i.i.d. draws from q_0."""
    assert root_lossless_error(oracle_mod, m, T, seed) < 1e-10


def test_lossless_second_level(oracle_mod):
    """After the walk accepts node 1, the next token ~ p_1 (node 1's own rows, children
    and uniforms)."""
    rng = np.random.default_rng(11)
    V, T = 4, 1.0
    par = np.array([-1, 0, 0, 1, 1, 2], np.int32)
    N = len(par)
    t = _rows(rng, N, V)
    d = (t + rng.normal(0.0, 1.2, size=(N, V))).astype(np.float32)
    tok = np.array([0, 2, 1, 0, 0, 3], np.int32)
    # u_1 = 0 accepts node 1 whenever p_0(x_1) > 0, which softmax guarantees.
    got = level_distribution(oracle_mod, t, d, par, tok, 1, [3, 4], T, forced={1: 0.0})
    assert np.abs(got - softmax64(t[1], T)).max() < 1e-10


# ----------------------------------------------------------------------------------
# Greedy verification: invariants from numpy's argmax.
# ----------------------------------------------------------------------------------

def greedy_violations(oracle_mod, seed, lib=None):
    rng = np.random.default_rng(seed)
    B, N, V = 40, 12, 9
    t = _rows(rng, B * N, V).reshape(B, N, V)
    par = np.zeros((B, N), np.int32)
    par[:, 0] = -1
    for n in range(1, N):
        par[:, n] = np.where(rng.random(B) < 0.5, n - 1, rng.integers(0, n, size=B))
    am = t.argmax(-1)
    tok = rng.integers(0, V, size=(B, N)).astype(np.int32)
    take = rng.random((B, N)) < 0.6  # a child often drafts its parent's argmax
    for b in range(B):
        for n in range(1, N):
            if take[b, n]:
                tok[b, n] = am[b, par[b, n]]
    tok[:, 0] = 0
    nn = rng.integers(1, N + 1, size=B).astype(np.int32)
    r = oracle_mod.verify_tree(t, None, par, tok, nn, None, 0.0, lib=lib)
    bad = 0
    for b in range(B):
        j = r["out_accepted"][b]
        path = r["out_path"][b]
        c = 0
        ok = j >= 0
        for i in range(max(j, 0)):
            # the lowest-index child of c drafting c's argmax
            kids = [n for n in range(c + 1, nn[b]) if par[b, n] == c and tok[b, n] == am[b, c]]
            ok &= bool(kids) and path[i] == kids[0] and r["out_tok"][b, i] == am[b, c]
            c = kids[0] if kids else c
        kids = [n for n in range(c + 1, nn[b]) if par[b, n] == c and tok[b, n] == am[b, c]]
        ok &= not kids and r["out_tok"][b, j] == am[b, c]
        ok &= (r["out_tok"][b, j + 1:] == -1).all() and (path[j:] == -1).all()
        bad += not ok
    return bad


@pytest.mark.parametrize("seed", range(3))
def test_greedy_walk(oracle_mod, seed):
    assert greedy_violations(oracle_mod, seed) == 0


# ----------------------------------------------------------------------------------
# Hand-derived cases. V = 3, T = 1, target logits log(0.5, 0.3, 0.2) and draft logits
# log(0.2, 0.2, 0.6) at the root; every child is a leaf whose target row is uniform.
#   r0 = p = (0.5, 0.3, 0.2).  Token 2: r0/q = 1/3.  Token 1: 1.5.  Token 0: 2.5.
#   After a rejection: r1 = max(0, p - q)/0.4 = (0.75, 0.25, 0).
#   After another:     r2 = max(0, r1 - q)/0.6 = (11/12, 1/12, 0).
# ----------------------------------------------------------------------------------

P0 = np.log(np.array([0.5, 0.3, 0.2]))
Q0 = np.log(np.array([0.2, 0.2, 0.6]))

HAND = [
    # (children tokens, uniforms of children, terminal uniform, out_tok, path)
    # child 1 (token 2): 0.2 < 1/3 accepts; the bonus at the uniform leaf with u0 = 0.5
    # is token 1 (CDF 1/3, 2/3, 1).
    ((2, 1), (0.2, 0.99), 0.5, [2, 1], [1]),
    # child 1 rejected (0.5 >= 1/3); child 2 (token 1) against r1: 0.25/0.2 >= 1 accepts.
    # In reversed order child 2 would be tested against p (1.5) and token 1 taken too,
    # so the next case separates the orders.
    ((2, 1), (0.5, 0.99), 0.9, [1, 2], [2]),
    # order matters: child 1 (token 2) accepted at 0.2; child 2 (token 1) never tested.
    ((2, 1), (0.2, 0.0), 0.1, [2, 0], [1]),
    # token 2 rejected twice (second time r1(2) = 0); terminal from r2 = (11/12, 1/12, 0)
    # at u0 = 0.95 -> target 0.95 > 11/12 -> token 1.
    ((2, 2), (0.5, 0.0), 0.95, [1], []),
    # the same at u0 = 0.5 -> token 0.
    ((2, 2), (0.5, 0.0), 0.5, [0], []),
    # one child rejected: terminal from r1 = (0.75, 0.25, 0) at u0 = 0.8 -> token 1.
    ((2,), (0.9,), 0.8, [1], []),
    # three children: 2 rejected, 2 rejected, then token 0 against r2: (11/12)/0.2 > 1.
    ((2, 2, 0), (0.5, 0.3, 0.999), 0.5, [0, 1], [3]),
]


def hand_case(oracle_mod, case, lib=None):
    kids, uk, u0, want_tok, want_path = HAND[case]
    m = len(kids)
    N = m + 1
    V = 3
    t = np.zeros((N, V), np.float32)
    d = np.zeros((N, V), np.float32)
    t[0] = P0
    d[0] = Q0
    par = np.array([-1] + [0] * m, np.int32)
    tok = np.array((0,) + kids, np.int32)
    u = np.array((u0,) + uk, np.float64)
    r = oracle_mod.verify_tree(t[None], d[None], par[None], tok[None], np.array([N]), u[None],
                               1.0, u64=True, lib=lib)
    j = len(want_path)
    assert r["out_accepted"][0] == j
    assert list(r["out_tok"][0, :j + 1]) == want_tok
    assert list(r["out_path"][0, :j]) == want_path
    assert (r["out_tok"][0, j + 1:] == -1).all() and (r["out_path"][0, j:] == -1).all()


@pytest.mark.parametrize("case", range(len(HAND)))
def test_hand_cases(oracle_mod, case):
    hand_case(oracle_mod, case)


def test_no_residual_mass_restarts_from_p(oracle_mod):
    """p == q with a child drafting a token of probability 0 under both: the rejection
    leaves no residual mass, and the sample is taken from p (the chain's reading)."""
    t = np.array([[0.0, 0.0, -np.inf], [0.0, 0.0, 0.0]], np.float32)
    d = t.copy()
    par = np.array([-1, 0], np.int32)
    tok = np.array([0, 2], np.int32)
    for u0, want in ((0.3, 0), (0.7, 1)):
        r = oracle_mod.verify_tree(t[None], d[None], par[None], tok[None], np.array([2]),
                                   np.array([[u0, 0.5]]), 1.0, u64=True)
        assert r["out_accepted"][0] == 0 and r["out_tok"][0, 0] == want
        assert r["flags"][0] & oracle_mod.FLAG_SMALL_RESIDUAL


# ----------------------------------------------------------------------------------
# What is read, and validation.
# ----------------------------------------------------------------------------------

def test_unreached_rows_are_not_read(oracle_mod):
    rng = np.random.default_rng(5)
    V, N = 6, 4
    par = np.array([-1, 0, 0, 1], np.int32)
    t = _rows(rng, N, V)
    d = _rows(rng, N, V)
    tok = np.array([0, 1, 2, 3], np.int32)
    # u_1 = 0 accepts node 1; node 1's child 3 is tested with u_3 = 0 and accepted;
    # node 3 is a leaf. Node 2 is never reached.
    u = np.array([0.4, 0.0, 0.5, 0.0])
    base = oracle_mod.verify_tree(t[None], d[None], par[None], tok[None], np.array([N]),
                                  u[None], 1.0, u64=True)
    assert base["out_accepted"][0] == 2
    t2, d2 = t.copy(), d.copy()
    t2[2] = np.nan
    d2[2] = np.nan
    d2[3] = np.nan  # a leaf's draft row is never read
    r = oracle_mod.verify_tree(t2[None], d2[None], par[None], tok[None], np.array([N]),
                               u[None], 1.0, u64=True)
    assert r["status"] == 0 and (r["out_tok"] == base["out_tok"]).all()
    t3 = t.copy()
    t3[3, 1] = np.inf  # a reached row with +inf is invalid
    r = oracle_mod.verify_tree(t3[None], d[None], par[None], tok[None], np.array([N]),
                               u[None], 1.0, u64=True)
    assert r["out_accepted"][0] == -1 and r["flags"][0] & oracle_mod.FLAG_INVALID


@pytest.mark.parametrize("what", ["parent_self", "parent_neg", "tok_high", "tok_neg",
                                  "nn_zero", "nn_big", "u_one", "u_neg"])
def test_invalid_requests(oracle_mod, what):
    rng = np.random.default_rng(3)
    B, N, V = 3, 4, 5
    t = _rows(rng, B * N, V).reshape(B, N, V)
    d = _rows(rng, B * N, V).reshape(B, N, V)
    par = np.tile(np.array([-1, 0, 1, 1], np.int32), (B, 1))
    tok = rng.integers(0, V, size=(B, N)).astype(np.int32)
    nn = np.full(B, N, np.int32)
    u = rng.random((B, N)).astype(np.float32)
    ok = oracle_mod.verify_tree(t, d, par, tok, nn, u, 1.0)
    assert ok["status"] == 0
    if what == "parent_self":
        par[1, 2] = 2
    elif what == "parent_neg":
        par[1, 3] = -1
    elif what == "tok_high":
        tok[1, 2] = V
    elif what == "tok_neg":
        tok[1, 1] = -3
    elif what == "nn_zero":
        nn[1] = 0
    elif what == "nn_big":
        nn[1] = N + 1
    elif what == "u_one":
        u[1, 0] = 1.0
    else:
        u[1, 3] = -0.25
    r = oracle_mod.verify_tree(t, d, par, tok, nn, u, 1.0)
    assert r["status"] == oracle_mod.ERR_INPUT
    assert r["out_accepted"][1] == -1 and (r["out_tok"][1] == -1).all()
    assert r["flags"][1] == oracle_mod.FLAG_INVALID
    for b in (0, 2):
        assert (r["out_tok"][b] == ok["out_tok"][b]).all()


def _pins():
    """The pins above as functions of a compiled oracle (the mutant tests run them on
    copies with planted mistakes)."""
    import oracle as om

    def check(ok):
        assert ok

    pins = []
    for seed in range(4):
        for T in (0.0, 0.6, 1.0, 2.5):
            pins.append(lambda lib, s=seed, T=T: check(chain_mismatches(om, s, T, lib=lib) == 0))
    for m, T, seed in [(1, 1.0, 0), (2, 1.0, 1), (3, 1.0, 2)]:
        pins.append(lambda lib, m=m, T=T, s=seed: check(root_lossless_error(om, m, T, s, lib=lib)
                                                        < 1e-10))
    for seed in range(3):
        pins.append(lambda lib, s=seed: check(greedy_violations(om, s, lib=lib) == 0))
    for case in range(len(HAND)):
        pins.append(lambda lib, c=case: hand_case(om, c, lib=lib))
    return pins


PINS = _pins()


def test_tree_path_bytes_counts_the_walk():
    """The benchmark's algorithmic bytes for a tree call: target rows of the root, the
    accepted nodes (the stop node is the last of them), and draft rows of those with
    children (none at T == 0). Hand case: tree16 parents, path 0 -> 1 -> 5."""
    import synth

    par = np.array([synth.TREE16_PARENTS, synth.TREE16_PARENTS], np.int32)
    path = np.full((2, 16), -1, np.int32)
    path[0, :2] = [1, 5]  # request 0 accepted nodes 1 and 5 (node 5 has children 11, 12)
    acc = np.array([2, -1], np.int32)  # request 1 invalid: nothing counted
    V, e = 10, 2
    # target rows of nodes 0, 1, 5; draft rows of 0, 1, 5 (all three have children)
    assert synth.tree_path_bytes(path, acc, par, V, e) == 6 * V * e
    assert synth.tree_path_bytes(path, acc, par, V, e, greedy=True) == 3 * V * e
    path[0, :2] = [4, -1]  # node 4 is a leaf: its draft row is not read
    acc[0] = 1
    assert synth.tree_path_bytes(path, acc, par, V, e) == 3 * V * e
