"""GPU parity of the calibration prologue (sv_schedule_cal), the load-aware threshold,
and the online calibration loop (sv_calib_observe, sv_calib_update) against the
float64 oracle.

The kernel calibrates in fp32 and the oracle in float64, so calibrated confidences
agree to a few fp32 ulps and a schedule decision can differ only where the oracle's
survival product lies within 1e-5 (relative) of the threshold or of the budget cut:
such requests are flagged as near-ties and every other length must match exactly.
The window statistics, temperatures and ECE must match exactly on identical inputs
(the sums are exact in float64 for these inputs)."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu
needs_cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")

# Error of the fp32 calibration: z = logit(c) / T carries an absolute error of at most
# about 2 ulps of |logit(c)| plus the rounding of the ratio c / (1 - c), so
# |dc'| <= c'(1 - c') |dz| + 4 ulps(c'). A survival product of K <= 32 such factors
# is then within K * 2e-6 (relative) of the oracle's for temperatures >= 0.5 and
# |logit| <= 17: decisions within NEAR of tau or of the budget cut are near-ties.
NEAR = 5e-5


def _cal_tolerance(conf, temps, cal_ref):
    c = conf.astype(np.float64)
    inner = (c > 0) & (c < 1)
    lg = np.zeros_like(c)
    lg[inner] = np.abs(np.log(c[inner] / (1 - c[inner])))
    dz = (2.0 * 2.0 ** -23 * np.maximum(lg, 1.0) + 2.0 ** -23) / temps[None, :].astype(np.float64)
    cr = cal_ref.astype(np.float64)
    return cr * (1 - cr) * dz + 4 * 2.0 ** -24 * cr

@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verification_79_gb300 as m

    m.load()
    return m


def _near_tie_requests(ref, tau, budget):
    """Requests whose length could flip under fp32 calibration: a survival within NEAR
    of tau, or, when the budget binds, the kept and the dropped key on either side of
    the cut within NEAR of each other (then every key that close to the cut)."""
    S = ref["surv"]
    B, K = S.shape
    flag = (np.abs(S - tau) <= NEAR * max(tau, 1e-30)).any(axis=1)
    l0 = ref["l0"]
    if l0.sum() > budget:
        floor_first = budget >= B
        lo = 1 if floor_first else 0
        r = budget - B if floor_first else budget
        comp = np.sort(np.concatenate([S[b, lo:l0[b]] for b in range(B)]))[::-1]
        if 0 < r < comp.size:
            kept, dropped = comp[r - 1], comp[r]
            if kept - dropped <= NEAR * kept:
                flag |= (np.abs(S - kept) <= NEAR * kept).any(axis=1)
    return flag


def _check(sv, conf, temps, load, tau, budget, tmin=0.2, tmax=0.75):
    B, K = conf.shape
    ws = sv.Workspace(min(B, 4096), K, 16)
    dev = lambda a: None if a is None else a.cuda()  # noqa: E731
    out_len, cal, tau_out = sv.sv_schedule_cal(dev(conf), dev(temps), dev(load), tau, tmin, tmax,
                                               budget, ws)
    got = out_len.cpu().numpy()
    st = ws.status(clear=True)
    ref = oracle.schedule_ex(conf.numpy(), None if temps is None else temps.numpy(),
                             None if load is None else load.numpy(), tau, tmin, tmax, budget)
    assert st == sv.SV_OK and ref["status"] == 0
    assert float(tau_out.cpu()[0]) == ref["tau"]
    calg = cal.cpu().numpy()
    if temps is None:
        assert np.array_equal(calg, conf.numpy())
    else:
        tol = _cal_tolerance(conf.numpy(), temps.numpy(), ref["cal"])
        err = np.abs(calg.astype(np.float64) - ref["cal"].astype(np.float64))
        assert (err <= tol).all(), float((err / np.maximum(tol, 1e-300)).max())
    flag = _near_tie_requests(ref, ref["tau"], budget)
    assert np.array_equal(got[~flag], ref["out_len"][~flag]), (B, K, tau, budget)
    assert got.sum() == ref["out_len"].sum()
    return int(flag.sum())


@needs_cuda
@pytest.mark.parametrize("seed", range(12))
def test_calibrated_schedule(sv, seed):
    rng = np.random.default_rng(seed)
    B = int(rng.choice([1, 5, 64, 256, 1000]))
    K = int(rng.choice([4, 8, 16]))
    conf = synth.confidences(B, K, seed=seed)
    temps = synth.temperatures(K, seed=seed)
    load = synth.load_state(seed=seed) if seed % 2 else None
    tau = float(rng.choice([0.1, 0.3, 0.5]))
    l0 = oracle.schedule_ex(conf.numpy(), temps.numpy(), None if load is None else load.numpy(),
                            tau, 0.2, 0.75, 10 ** 9)["l0"]
    flagged = 0
    for budget in sorted({0, max(0, B - 1), B, int(l0.sum()) // 2, int(l0.sum())}):
        flagged += _check(sv, conf, temps, load, tau, budget)
    print(f"[calib] seed {seed}: {flagged} near-tie requests")


@needs_cuda
def test_calibrated_ragged_config(sv):
    """The confidence-scheduled ragged batch (B=256, K=16, tau 0.3) with per-position
    temperatures that grow along the block, at budgets 1024, 256 and 200."""
    conf = synth.confidences(256, 16, seed=0)
    temps = torch.linspace(1.0, 2.5, 16, dtype=torch.float32)
    for budget in (1024, 256, 200):
        _check(sv, conf, temps, None, 0.3, budget)
        _check(sv, conf, temps, synth.load_state(seed=3), 0.3, budget)


@needs_cuda
def test_plain_path_is_the_schedule(sv):
    """No temperatures, no load: bit-exact with the plain schedule."""
    conf = synth.confidences(300, 12, seed=5)
    ws = sv.Workspace(300, 12, 16)
    for budget in (0, 299, 300, 1000, 10 ** 6):
        a = sv.sv_schedule(conf.cuda(), 0.3, budget, ws).cpu().numpy()
        b, cal, _ = sv.sv_schedule_cal(conf.cuda(), None, None, 0.3, 0.2, 0.75, budget, ws)
        assert np.array_equal(a, b.cpu().numpy())
        assert np.array_equal(a, oracle.schedule(conf.numpy(), 0.3, budget)["out_len"])
        assert torch.equal(cal.cpu(), conf)


@needs_cuda
def test_load_threshold_end_points(sv):
    conf = torch.full((4, 8), 0.9, dtype=torch.float32)
    ws = sv.Workspace(4, 8, 16)
    for load, want in (([0, 64, 0, 80], np.float32(0.2)), ([64, 64, 80, 80], np.float32(0.75)),
                       ([640, 64, 800, 80], np.float32(0.75))):
        _, _, t = sv.sv_schedule_cal(conf.cuda(), None, torch.tensor(load, dtype=torch.float32).cuda(),
                                     0.5, 0.2, 0.75, 32, ws)
        assert float(t.cpu()[0]) == float(want)


@needs_cuda
def test_invalid_calibration_inputs(sv):
    conf = synth.confidences(8, 4, seed=1).cuda()
    ws = sv.Workspace(8, 4, 16)
    bad_temps = torch.tensor([1.0, 0.0, 1.0, 1.0]).cuda()
    out, _, _ = sv.sv_schedule_cal(conf, bad_temps, None, 0.3, 0.2, 0.75, 32, ws)
    assert ws.status(clear=True) == sv.SV_ERR_DEVICE_INPUT and not out.cpu().any()
    bad_load = torch.tensor([1.0, 0.0, 1.0, 1.0]).cuda()
    out, _, _ = sv.sv_schedule_cal(conf, None, bad_load, 0.3, 0.2, 0.75, 32, ws)
    assert ws.status(clear=True) == sv.SV_ERR_DEVICE_INPUT and not out.cpu().any()
    out, _, _ = sv.sv_schedule_cal(conf, None, None, 0.3, 0.2, 0.75, 32, ws)
    assert ws.status(clear=True) == sv.SV_OK and out.cpu().sum() > 0


def _same_window(got, want, K):
    """Counts exact; sums of c' to 1e-14 relative (float64 sums of fp32 values are
    exact unless a value is below 2^-14, where the summation order can round)."""
    g, w = got.reshape(-1, 3), want.reshape(-1, 3)
    pos, bins = slice(0, K), slice(K, None)
    assert np.array_equal(g[pos, 1:], w[pos, 1:]) and np.array_equal(g[bins, 0], w[bins, 0])
    assert np.array_equal(g[bins, 2], w[bins, 2])
    assert np.allclose(g[pos, 0], w[pos, 0], rtol=1e-14, atol=0)
    assert np.allclose(g[bins, 1], w[bins, 1], rtol=1e-14, atol=0)


@needs_cuda
@pytest.mark.parametrize("B,K", [(1, 1), (7, 4), (64, 8), (256, 16), (4096, 32)])
def test_calibration_loop(sv, B, K):
    """Rounds of observe, with a window update every third round: window statistics,
    temperatures and ECE identical to the oracle's on the same inputs."""
    n = sv.sv_calib_stats_len(K)
    stats_d = torch.zeros(n, dtype=torch.float64, device="cuda")
    stats_h = np.zeros(n)
    temps0 = synth.temperatures(K, seed=B)
    temps_d = temps0.clone().cuda()
    temps_h = temps0.numpy().copy()
    for r in range(7):
        c, vl, acc = synth.calib_round(B, K, seed=100 * B + r)
        sv.sv_calib_observe(c.cuda(), vl.cuda(), acc.cuda(), stats_d)
        assert oracle.calib_observe(c.numpy(), vl.numpy(), acc.numpy(), stats_h) == 0
        _same_window(stats_d.cpu().numpy(), stats_h, K)
        if r % 3 == 2:
            ece_d = sv.sv_calib_update(stats_d, temps_d, 0.01, 0.05)
            rc, ece_h = oracle.calib_update(stats_h, temps_h, float(np.float32(0.01)),
                                            float(np.float32(0.05)))
            assert rc == 0
            assert np.array_equal(temps_d.cpu().numpy(), temps_h)
            assert abs(float(ece_d.cpu()[0]) - ece_h) <= 1e-13 * max(ece_h, 1e-300)
            assert not stats_d.cpu().any()


@needs_cuda
def test_overconfidence_raises_temperature(sv):
    """End to end on the device (schedule -> verify -> observe -> update): confidences
    far above the real acceptance rate push every tested position's temperature up,
    as the oracle chain does on the same inputs."""
    B, K, V = 64, 4, 1024
    inp = synth.verify_inputs(B, K, V, dtype=torch.float32, temperature=1.0, target_sigma=2.0,
                              draft_sigma=2.0, seed=9)
    conf = torch.full((B, K), 0.97, dtype=torch.float32)
    temps = torch.ones(K, dtype=torch.float32)
    ws = sv.Workspace(B, K, V)
    out_len, cal, _ = sv.sv_schedule_cal(conf.cuda(), temps.cuda(), None, 0.0, 0.2, 0.75, B * K, ws)
    d = {k: v.cuda() for k, v in inp.items()}
    out_tok, acc = sv.sv_verify(d["target"], d["draft"], d["draft_tok"], out_len, d["uniforms"], 1.0, ws)
    stats = torch.zeros(sv.sv_calib_stats_len(K), dtype=torch.float64, device="cuda")
    sv.sv_calib_observe(cal, out_len, acc, stats)
    t_d = temps.clone().cuda()
    ece = float(sv.sv_calib_update(stats, t_d, 0.01, 0.05).cpu()[0])
    # the oracle chain on the same seeded inputs
    ref_s = oracle.schedule_ex(conf.numpy(), temps.numpy(), None, 0.0, 0.2, 0.75, B * K)
    ref_v = oracle.verify(synth.to_oracle(inp["target"]), synth.to_oracle(inp["draft"]),
                          inp["draft_tok"].numpy(), ref_s["out_len"], inp["uniforms"].numpy(), 1.0)
    st = np.zeros(oracle.calib_stats_len(K))
    oracle.calib_observe(ref_s["cal"], ref_s["out_len"], ref_v["out_accepted"], st)
    t_h = temps.numpy().copy()
    _, ece_h = oracle.calib_update(st, t_h, float(np.float32(0.01)), float(np.float32(0.05)))
    assert np.array_equal(out_len.cpu().numpy(), ref_s["out_len"])
    assert (t_d.cpu().numpy() > 1.0).all() and (t_h > 1.0).all()
    assert np.allclose(t_d.cpu().numpy(), t_h, rtol=1e-6) and abs(ece - ece_h) < 1e-3
