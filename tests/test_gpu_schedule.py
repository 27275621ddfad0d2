"""GPU parity of sv_schedule against the oracle: bit-exact lengths."""
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


def _run(sv, conf, tau, budget, ws=None):
    B, K = conf.shape
    ws = ws or sv.Workspace(min(B, 4096), K, 16)
    out = sv.sv_schedule(torch.from_numpy(conf).cuda(), tau, budget, ws).cpu().numpy()
    return out, ws.status(clear=True)


@needs_cuda
@pytest.mark.parametrize("seed", range(30))
def test_random_schedules(sv, seed):
    rng = np.random.default_rng(seed)
    B = int(rng.choice([1, 3, 17, 100, 256, 1000, 4096, 8192]))
    K = int(rng.integers(1, min(32, 16384 // B) + 1))
    conf = (rng.beta(8, 2, size=(B, K)) * 0.93 ** np.arange(1, K + 1)).astype(np.float32)
    if seed % 5 == 0:
        conf[:] = conf[:, :1]  # ties across positions and requests
    if seed % 7 == 0:
        conf[rng.random((B, K)) < 0.05] = 1.0
    tau = float(rng.choice([0.0, 0.1, 0.3, 0.5, 1.0]))
    l0 = oracle.schedule(conf, tau, 10 ** 9)["l0"]
    for budget in sorted({0, 1, max(0, B - 1), B, B + 5, int(l0.sum()) // 3, int(l0.sum())}):
        got, st = _run(sv, conf, tau, budget)
        ref = oracle.schedule(conf, tau, budget)
        assert st == sv.SV_OK
        assert np.array_equal(got, ref["out_len"]), (B, K, tau, budget)


@needs_cuda
def test_ragged_config_schedule(sv):
    conf = synth.confidences(256, 16, seed=0).numpy()
    for budget in (1024, 256, 200):
        got, _ = _run(sv, conf, 0.3, budget)
        assert np.array_equal(got, oracle.schedule(conf, 0.3, budget)["out_len"])


@needs_cuda
def test_golden_variable_length(sv):
    conf = np.array([[0.95, 0.90, 0.80, 0.70, 0.60, 0.50, 0.50, 0.50]], np.float32)
    got, _ = _run(sv, conf, 0.20, 8)
    assert got.tolist() == [5]


@needs_cuda
def test_invalid_confidence(sv):
    conf = np.full((4, 4), 0.5, np.float32)
    conf[2, 1] = np.nan
    got, st = _run(sv, conf, 0.3, 100)
    assert st == sv.SV_ERR_DEVICE_INPUT and (got == 0).all()
    conf[2, 1] = 1.01
    got, st = _run(sv, conf, 0.3, 100)
    assert st == sv.SV_ERR_DEVICE_INPUT and (got == 0).all()
