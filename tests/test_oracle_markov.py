"""Pins for the oracle's Markov logit-bias drafting loop (CPU only).

Source: DSpark Guide, "1. The Markov Logit-Bias Head" (L'_k = L_k + U V[y_{k-1}]^T with
U, V of shape [vocab, rank]) and "Hands-On Implementation" (greedy drafting, each token
feeding the next position's correction). The pins use cases whose answers are fixed
independently of the oracle's code: a zero correction, a hand-built chain with small
integers (exact in bf16), the defining properties of round-to-nearest-even and of a
lowest-index argmax, and a float64 matrix product from numpy.
"""
import numpy as np
import pytest

import oracle


def bf16_bits(x):
    """float32 values that are exactly representable in bf16 -> bf16 bits."""
    a = np.asarray(x, np.float32)
    bits = a.view(np.uint32)
    assert not (bits & 0xFFFF).any(), "value not exact in bf16"
    return (bits >> 16).astype(np.uint16)


def bf16_float(h):
    return (np.asarray(h, np.uint32) << 16).view(np.float32).astype(np.float64)


def _random_bf16(rng, shape, scale):
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)  # truncate to bf16


def pin_zero_correction(lib=None):
    rng = np.random.default_rng(0)
    B, K, V, r = 3, 4, 50, 8
    L = _random_bf16(rng, (B, K, V), 2.0)
    U = np.zeros((V, r), np.uint16)
    Vm = _random_bf16(rng, (V, r), 1.0)
    res = oracle.markov_draft(L, U, Vm, np.array([1, 2, 3], np.int32), lib=lib)
    assert res["status"] == 0
    assert np.array_equal(res["corrected"], L)
    assert np.array_equal(res["tok"], np.argmax(bf16_float(L), axis=2))


def pin_hand_chain(lib=None):
    """V = 4, r = 2. Row v of U is the correction's response to the two features of the
    previous token's row of Vm. The chain: prev = 0 -> y_0 -> y_1 -> y_2."""
    U = bf16_bits([[1, 0], [0, 1], [2, 0], [0, -3]])
    Vm = bf16_bits([[0, 1], [1, 0], [0, 0], [2, 2]])
    L = bf16_bits(np.zeros((1, 3, 4), np.float32) + np.array([0.5, 0.25, 0.0, 2.0], np.float32))
    res = oracle.markov_draft(L, U, Vm, np.array([0], np.int32), lib=lib)
    # k=0: prev 0, x = (0,1): correction (0, 1, 0, -3) -> (0.5, 1.25, 0, -1) -> y0 = 1
    # k=1: prev 1, x = (1,0): correction (1, 0, 2, 0) -> (1.5, 0.25, 2, 2) -> y1 = 2 (first max)
    # k=2: prev 2, x = (0,0): no correction -> (0.5, 0.25, 0, 2) -> y2 = 3
    assert res["tok"].tolist() == [[1, 2, 3]]
    want = np.array([[[0.5, 1.25, 0, -1], [1.5, 0.25, 2, 2], [0.5, 0.25, 0, 2]]])
    assert np.array_equal(bf16_float(res["corrected"]), want)


def pin_rounding_and_argmax_properties(lib=None):
    rng = np.random.default_rng(4)
    B, K, V, r = 2, 3, 300, 32
    L = _random_bf16(rng, (B, K, V), 3.0)
    U = _random_bf16(rng, (V, r), 0.1)
    Vm = _random_bf16(rng, (V, r), 0.1)
    prev = np.array([5, 299], np.int32)
    res = oracle.markov_draft(L, U, Vm, prev, lib=lib)
    Uf, Vf, Lf = bf16_float(U), bf16_float(Vm), bf16_float(L)
    got = bf16_float(res["corrected"])
    y = prev.copy()
    for k in range(K):
        z = Lf[:, k, :] + (Uf @ Vf[y].T).T  # exact inputs, float64 product
        # round to nearest: |stored - z| <= half the bf16 spacing at z; ties to even
        e = np.floor(np.log2(np.abs(z))) - 7
        spacing = np.exp2(e)
        assert (np.abs(got[:, k, :] - z) <= spacing / 2 * (1 + 1e-12)).all()
        tie = np.isclose(np.abs(got[:, k, :] - z), spacing / 2, rtol=1e-12, atol=0)
        if tie.any():
            mant = (res["corrected"][:, k, :][tie].astype(np.uint32) & 1)
            assert not mant.any()
        # greedy: the first index of the row maximum of the stored values
        assert np.array_equal(res["tok"][:, k], np.argmax(got[:, k, :], axis=1))
        y = res["tok"][:, k]


PINS = [pin_zero_correction, pin_hand_chain, pin_rounding_and_argmax_properties]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(None)


def test_rejects_bad_previous_token():
    res = oracle.markov_draft(np.zeros((1, 1, 4), np.uint16), np.zeros((4, 2), np.uint16),
                              np.zeros((4, 2), np.uint16), np.array([4], np.int32))
    assert res["status"] == -5
