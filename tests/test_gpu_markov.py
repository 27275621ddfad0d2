"""GPU parity of sv_markov_draft (Markov logit-bias head + greedy drafting) against the
float64 oracle.

The kernel forms the correction U Vm[y]^T on the tensor cores with fp32 accumulation;
the oracle in float64. For each element, 2^-24 (r sum_j |U_vj x_j| + |z|) bounds the
kernel's error before its single rounding to bf16, so the stored values must be equal
except where the exact value z lies within that bound of a bf16 rounding midpoint, and
there they may differ by one bf16 step. A drafted token must be equal unless the two
largest exact values of the row are within one bf16 step plus twice the bound (a near
tie); after a near tie the request's later positions follow different tokens and are
not compared."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu
needs_cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verification_79_gb300 as m

    m.load()
    return m


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _f(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _spacing(z):
    e = np.floor(np.log2(np.maximum(np.abs(z), 1e-300)))
    return np.exp2(e - 7)


def _compare(inp, got_corr, got_tok):
    L, U, Vm, prev = (_bits(inp["logits"]), _bits(inp["U"]), _bits(inp["Vm"]),
                      inp["prev"].numpy())
    ref = oracle.markov_draft(L, U, Vm, prev)
    assert ref["status"] == 0
    B, K, V = L.shape
    r = U.shape[1]
    Uf, Vf, Lf = _f(U), _f(Vm), _f(L)
    Ua = np.abs(Uf)
    near_ties = flagged = 0
    for b in range(B):
        y = int(prev[b])
        for k in range(K):
            x = Vf[y]
            terms = Ua @ np.abs(x)
            z = Lf[b, k] + Uf @ x
            bound = 2.0 ** -24 * (r * terms + np.abs(z)) * 2
            sp = _spacing(z)
            frac = np.abs(z) / sp
            mid_dist = np.abs((frac - np.floor(frac)) - 0.5) * sp
            risky = mid_dist <= bound
            want = _f(ref["corrected"][b, k])
            have = _f(got_corr[b, k])
            diff = have != want
            assert not (diff & ~risky).any(), (b, k, np.nonzero(diff & ~risky)[0][:5])
            # within the bound of z before rounding, then one rounding on each side: where
            # L and the correction nearly cancel, the bound spans several bf16 steps at z
            sp_big = _spacing(np.maximum(np.abs(have), np.abs(want)))
            assert (np.abs(have - want)[diff] <= (bound + sp_big)[diff] * 1.0000001).all()
            flagged += int(diff.sum())
            order = np.argsort(-z, kind="stable")
            gap = z[order[0]] - z[order[1]] if V > 1 else np.inf
            if gap <= sp[order[0]] + 2 * bound[order[0]] + 2 * bound[order[1]]:
                near_ties += 1
                break  # later positions of this request may follow another token
            assert got_tok[b, k] == ref["tok"][b, k], (b, k)
            y = int(ref["tok"][b, k])
    return flagged, near_ties


CASES = [(1, 1, 1000, 16), (3, 4, 1003, 128), (64, 4, 4096, 256), (65, 2, 2048, 64),
         (16, 8, 777, 32), (130, 1, 512, 256), (8, 3, 2048, 192), (130, 3, 1000, 64)]


@needs_cuda
@pytest.mark.parametrize("B,K,V,r", CASES)
def test_markov_parity(sv, B, K, V, r):
    inp = synth.markov_inputs(B, K, V, r, seed=B + K + V + r)
    ws = sv.Workspace(min(B, 4096), K, 16)
    d = {k: v.cuda() for k, v in inp.items()}
    corr, tok = sv.sv_markov_draft(d["logits"], d["U"], d["Vm"], d["prev"], ws)
    assert ws.status(clear=True) == sv.SV_OK
    flagged, ties = _compare(inp, _bits(corr.cpu()), tok.cpu().numpy())
    print(f"[markov] B={B} K={K} V={V} r={r}: {flagged} elements one bf16 step apart at "
          f"rounding midpoints, {ties} near-tie tokens")


@needs_cuda
@pytest.mark.parametrize("r", [128, 256])
def test_markov_parity_benchmarked_shape(sv, r):
    """The shape the drafting kernel is timed at: B=64 requests, K=8 positions, the
    151,936-entry vocabulary, ranks 128 and 256 ([GD] "1. The Markov Logit-Bias Head"):
    every request and position against the oracle."""
    test_markov_parity(sv, 64, 8, synth.QWEN3_VOCAB, r)


@needs_cuda
def test_markov_zero_correction_and_invalid_prev(sv):
    inp = synth.markov_inputs(5, 3, 600, 64, seed=2)
    inp["U"].zero_()
    inp["prev"][2] = 600  # out of range
    ws = sv.Workspace(5, 3, 16)
    d = {k: v.cuda() for k, v in inp.items()}
    corr, tok = sv.sv_markov_draft(d["logits"], d["U"], d["Vm"], d["prev"], ws)
    assert ws.status(clear=True) == sv.SV_ERR_DEVICE_INPUT
    tok = tok.cpu().numpy()
    L = inp["logits"].float().numpy()
    for b in range(5):
        if b == 2:
            assert (tok[b] == -1).all()
            continue
        assert torch.equal(corr[b].cpu(), inp["logits"][b])
        assert np.array_equal(tok[b], np.argmax(L[b], axis=1))


@needs_cuda
def test_markov_deterministic(sv):
    inp = synth.markov_inputs(64, 4, 8192, 256, seed=7)
    ws = sv.Workspace(64, 4, 16)
    d = {k: v.cuda() for k, v in inp.items()}
    a = sv.sv_markov_draft(d["logits"], d["U"], d["Vm"], d["prev"], ws)
    b = sv.sv_markov_draft(d["logits"], d["U"], d["Vm"], d["prev"], ws)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@needs_cuda
def test_markov_shared_workspace_across_calls(sv):
    """One workspace for calls of different shapes in a row: at most 128 requests all
    positions run in one launch whose CTAs meet at a grid barrier counted in the
    workspace header, and every call must leave that count at zero for the next (also
    after a call that takes one launch per position, or reports invalid input)."""
    ws = sv.Workspace(256, 8, 16)
    shapes = [(8, 3, 2048, 64, 11), (64, 4, 4096, 128, 12), (130, 2, 1024, 64, 13),
              (3, 5, 1000, 32, 14), (64, 4, 4096, 128, 12)]
    for B, K, V, r, seed in shapes:
        inp = synth.markov_inputs(B, K, V, r, seed=seed)
        d = {k: v.cuda() for k, v in inp.items()}
        corr, tok = sv.sv_markov_draft(d["logits"], d["U"], d["Vm"], d["prev"], ws)
        assert ws.status(clear=True) == sv.SV_OK, (B, K, V, r)
        _compare(inp, _bits(corr.cpu()), tok.cpu().numpy())
    # A call with an invalid previous token reports it; the next call is unaffected.
    inp = synth.markov_inputs(5, 3, 600, 64, seed=2)
    inp["prev"][1] = -3
    d = {k: v.cuda() for k, v in inp.items()}
    sv.sv_markov_draft(d["logits"], d["U"], d["Vm"], d["prev"], ws)
    assert ws.status(clear=True) == sv.SV_ERR_DEVICE_INPUT
    inp = synth.markov_inputs(16, 6, 2048, 128, seed=15)
    d = {k: v.cuda() for k, v in inp.items()}
    corr, tok = sv.sv_markov_draft(d["logits"], d["U"], d["Vm"], d["prev"], ws)
    assert ws.status(clear=True) == sv.SV_OK
    _compare(inp, _bits(corr.cpu()), tok.cpu().numpy())
