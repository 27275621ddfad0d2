"""GPU parity of sv_schedule_curve (the throughput-curve budget) against the float64
oracle. Without calibration the survival products are bit-identical on both sides; the
sums A(N) differ only by summation order (a block scan against a sequential sum), so the
chosen N must match unless the two largest goodputs over distinct N are within 1e-12
(relative) of each other, which is flagged and then only required to be near-optimal.
With calibration (fp32 on the device) the window is 1e-4."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu
needs_cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")

# [DD] "The Throughput Curve": batch size -> tokens/s (example table on the page).
PAGE = torch.tensor([[1, 2, 4, 8, 16, 32, 64, 128], [35, 67, 125, 220, 360, 520, 650, 720]],
                    dtype=torch.float32)


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verification_79_gb300 as m

    m.load()
    return m


def _goodputs(conf, temps, load, tau, budget, curve):
    """G(N) for every admissible N from the oracle's own survivals (numpy.interp)."""
    ex = oracle.schedule_ex(conf, temps, load, tau, 0.2, 0.75, 10 ** 9)
    S, l0 = ex["surv"], ex["l0"]
    B = S.shape[0]
    floors = budget >= B
    n_lo = B if floors else 0
    n_hi = min(int(l0.sum()), budget)
    a = S[:, 0].sum() if floors else 0.0
    comp = np.sort(np.concatenate([S[b, (1 if floors else 0):l0[b]] for b in range(B)]))[::-1]
    ns = np.arange(n_lo, n_hi + 1)
    A = a + np.concatenate([[0.0], np.cumsum(comp)])[: ns.size]
    x = B + ns
    cx, cy = curve[0].numpy().astype(np.float64), curve[1].numpy().astype(np.float64)
    return ns, (B + A) * np.interp(x, cx, cy) / x


def _check(sv, conf, temps, load, tau, budget, curve, window):
    B, K = conf.shape
    ws = sv.Workspace(min(B, 4096), K, 16)
    dev = lambda a: None if a is None else a.cuda()  # noqa: E731
    out_len, n, g = sv.sv_schedule_curve(dev(conf), dev(temps), dev(load), tau, 0.2, 0.75,
                                         curve.cuda(), budget, ws)
    assert ws.status(clear=True) == sv.SV_OK
    ref = oracle.schedule_curve(conf.numpy(), None if temps is None else temps.numpy(),
                                None if load is None else load.numpy(), tau, 0.2, 0.75,
                                curve[0].numpy(), curve[1].numpy(), budget)
    assert ref["status"] == 0
    ns, G = _goodputs(conf.numpy(), None if temps is None else temps.numpy(),
                      None if load is None else load.numpy(), tau, budget, curve)
    n_gpu = int(n.cpu()[0])
    top = np.sort(G)[::-1]
    tie = top.size > 1 and top[0] - top[1] <= window * top[0]
    if tie:
        # near-optimal: the device's N is within the window of the best goodput
        assert G[ns == n_gpu][0] >= top[0] * (1 - window), (n_gpu, ref["n"])
        return 1
    assert n_gpu == ref["n"], (B, K, budget, n_gpu, ref["n"])
    # goodputs agree to the summation order, or (fp32 calibration) to ~1e-6 in S
    assert abs(float(g.cpu()[0]) - ref["g"]) <= (1e-12 if temps is None else 1e-5) * ref["g"]
    if temps is None:
        assert np.array_equal(out_len.cpu().numpy(), ref["out_len"])
    else:
        assert out_len.cpu().numpy().sum() == ref["out_len"].sum()
    return 0


@needs_cuda
@pytest.mark.parametrize("seed", range(10))
def test_curve_schedule(sv, seed):
    rng = np.random.default_rng(seed)
    B = int(rng.choice([1, 5, 64, 256, 1024]))
    K = int(rng.choice([4, 8]))
    conf = synth.confidences(B, K, seed=seed)
    curve = PAGE if seed % 3 == 0 else synth.throughput_curve(int(rng.integers(2, 12)), seed=seed)
    ties = 0
    for budget in sorted({B * K * 2, B, max(0, B - 1), B + (B * K) // 3}):
        ties += _check(sv, conf, None, None, 0.2, budget, curve, 1e-12)
    print(f"[curve] seed {seed}: {ties} near-tie budgets")


@needs_cuda
def test_curve_regimes_and_calibration(sv):
    conf = synth.confidences(64, 8, seed=3)
    lin = torch.tensor([[1.0, 1e6], [1.0, 1e6]], dtype=torch.float32)
    flat = torch.tensor([[1.0, 2.0], [100.0, 100.0]], dtype=torch.float32)
    ws = sv.Workspace(64, 8, 16)
    l0 = oracle.schedule(conf.numpy(), 0.1, 10 ** 6)["l0"]
    out, n, _ = sv.sv_schedule_curve(conf.cuda(), None, None, 0.1, 0.2, 0.75, lin.cuda(), 10 ** 6, ws)
    assert int(n.cpu()[0]) == int(l0.sum()) and np.array_equal(out.cpu().numpy(), l0)
    _, n2, _ = sv.sv_schedule_curve(conf.cuda(), None, None, 0.1, 0.2, 0.75, flat.cuda(), 10 ** 6, ws)
    assert int(n2.cpu()[0]) < int(l0.sum())
    _check(sv, conf, synth.temperatures(8, seed=3), synth.load_state(seed=3), 0.2, 10 ** 6, PAGE, 1e-4)


@needs_cuda
def test_invalid_curve(sv):
    conf = synth.confidences(8, 4, seed=1).cuda()
    ws = sv.Workspace(8, 4, 16)
    bad = torch.tensor([[2.0, 1.0], [10.0, 10.0]]).cuda()
    out, _, _ = sv.sv_schedule_curve(conf, None, None, 0.2, 0.2, 0.75, bad, 32, ws)
    assert ws.status(clear=True) == sv.SV_ERR_DEVICE_INPUT and not out.cpu().any()
