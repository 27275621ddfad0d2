"""GPU parity of sv_verify against the float64 oracle (bit-exact decisions outside
flagged near-ties; p(x), q(x) within 1e-5 relative)."""
import numpy as np
import pytest
import torch

import gpu_util
import oracle
import synth
from gpu_util import account, compare, run_gpu, run_oracle, to_dev

pytestmark = pytest.mark.gpu

needs_cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verification_79_gb300 as m

    m.load()
    return m


@needs_cuda
@pytest.mark.parametrize("T", [1.0, 0.0])
def test_tiny_fp32(sv, T):
    inp = synth.verify_inputs(4, 4, 1024, dtype=torch.float32, temperature=T, target_sigma=2.0,
                              draft_sigma=0.5, seed=0)
    gpu = run_gpu(sv, to_dev(inp), T)
    res = compare(gpu, run_oracle(inp, T), T, inp["verify_len"].numpy())
    assert gpu["status"] == sv.SV_OK
    account(f"tiny T={T}", *res)


SMALL = [
    (dt, V, T)
    for dt in (torch.bfloat16, torch.float32)
    for V in (1, 2, 7, 100, 2047, 2048, 2049, 4095, 4096, 4097, 12345)
    for T in (0.0, 0.5, 1.0, 3.0)
]


@needs_cuda
@pytest.mark.parametrize("dt,V,T", SMALL)
def test_small_shapes(sv, dt, V, T):
    """Several pieces per row and ragged tails; random verify lengths in [0, K]."""
    B, K = 12, 5
    inp = synth.verify_inputs(B, K, V, dtype=dt, temperature=T, target_sigma=2.0,
                              draft_sigma=1.0, seed=V * 7 + int(T * 10),
                              verify_len=list(np.random.default_rng(V).integers(0, K + 1, B)))
    gpu = run_gpu(sv, to_dev(inp), T)
    compare(gpu, run_oracle(inp, T), T, inp["verify_len"].numpy())
    assert gpu["status"] == sv.SV_OK


@needs_cuda
@pytest.mark.parametrize("T", [0.0, 1.0])
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_unaligned_rows(sv, T, dt):
    """Odd V and a base pointer one element past an allocation boundary: rows start at
    every 16-byte phase, so the direct head/tail paths and the direct job path run."""
    B, K, V = 6, 4, 4099
    inp = synth.verify_inputs(B, K, V, dtype=dt, temperature=T, seed=11)
    g = to_dev(inp)
    for key, shape in (("target", (B, K + 1, V)), ("draft", (B, K, V))):
        big = torch.empty(g[key].numel() + 1, dtype=dt, device="cuda")
        big[1:] = g[key].reshape(-1)
        g[key] = big[1:].view(shape)
    gpu = run_gpu(sv, g, T)
    compare(gpu, run_oracle(inp, T), T, inp["verify_len"].numpy())


@needs_cuda
@pytest.mark.parametrize("T", [1.0, 0.0])
def test_qwen3_vocab(sv, T):
    """B=32, K=8, V=151,936 bf16, peaked target rows, draft noise 1.0: full parity."""
    inp = synth.qwen3_verify(T, seed=0, device="cuda")
    gpu = run_gpu(sv, inp, T)
    account(f"qwen3 T={T}",
            *compare(gpu, run_oracle(inp, T), T, inp["verify_len"].cpu().numpy()))


@needs_cuda
@pytest.mark.parametrize("budget", [1024, 256, 200])
def test_ragged_schedule_then_verify(sv, budget):
    """B=256, K=16: schedule (tau 0.3) then verify the ragged prefixes, all on device."""
    inp = synth.ragged_schedule(seed=0, device="cuda")
    B, K, V = 256, 16, synth.QWEN3_VOCAB
    ws = sv.Workspace(B, K, V)
    out_len = sv.sv_schedule(inp["conf"], 0.3, budget, ws)
    ref_s = oracle.schedule(inp["conf"].cpu().numpy(), 0.3, budget)
    assert np.array_equal(out_len.cpu().numpy(), ref_s["out_len"])
    inp["verify_len"] = out_len
    gpu = run_gpu(sv, inp, 1.0, ws=ws)
    account(f"ragged budget={budget}",
            *compare(gpu, run_oracle(inp, 1.0), 1.0, ref_s["out_len"]))
    print(f"sum L = {ref_s['out_len'].sum()}, sum L0 = {ref_s['l0'].sum()}")


@needs_cuda
def test_large_batch(sv):
    """B=512, K=8, V=129,280 bf16, T=0.7, verify lengths U{1..8} (the DeepSeek-V4
    vocabulary of [DD] "The Low-Rank Trick"): every request against the oracle."""
    inp = synth.large_batch(seed=0, device="cuda")
    gpu = run_gpu(sv, inp, 0.7)
    ref = run_oracle(inp, 0.7)
    account("large batch", *compare(gpu, ref, 0.7, inp["verify_len"].cpu().numpy()))
    acc = gpu["out_accepted"]
    L = inp["verify_len"].cpu().numpy()
    assert ((acc >= 0) & (acc <= L)).all()
    assert (gpu["out_tok"][np.arange(512), acc] >= 0).all()


@needs_cuda
def test_bench_workload(sv):
    """The benchmarked launch: B=64, K=8, V=151,936 bf16, T=1, draft noise 1.0."""
    inp = synth.sweep_point(64, 8, seed=0, device="cuda")
    gpu = run_gpu(sv, inp, 1.0)
    account("bench workload",
            *compare(gpu, run_oracle(inp, 1.0), 1.0, inp["verify_len"].cpu().numpy()))


@needs_cuda
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_q_equals_p(sv, dt):
    inp = synth.verify_inputs(32, 6, 5000, dtype=dt, temperature=1.0, seed=3)
    inp["draft"] = inp["target"][:, :6].clone()
    inp["uniforms"][:, :6] = torch.clamp(inp["uniforms"][:, :6], min=0.9999)
    gpu = run_gpu(sv, to_dev(inp), 1.0)
    assert (gpu["out_accepted"] == 6).all()
    assert np.array_equal(gpu["p"], gpu["q"])
    compare(gpu, run_oracle(inp, 1.0), 1.0, inp["verify_len"].numpy())


@needs_cuda
@pytest.mark.parametrize("T", [1.0, 0.0])
def test_invalid_inputs(sv, T):
    """Invalid device data marks the request (-1) and sets the status word; the other
    requests are verified normally. Same rules as the oracle."""
    B, K, V = 10, 3, 3000
    inp = synth.verify_inputs(B, K, V, dtype=torch.bfloat16, temperature=T, seed=5)
    inp["target"][1, 2, 5] = float("nan")
    inp["draft"][2, 0, 3] = float("inf")
    inp["target"][3, 1, :] = float("-inf")
    inp["draft_tok"][4, 1] = V
    inp["verify_len"][5] = K + 1
    inp["uniforms"][6, 0] = 1.0
    inp["verify_len"][7] = -1
    inp["target"][8, 0, :7] = float("-inf")  # some masked entries: valid
    gpu = run_gpu(sv, to_dev(inp), T)
    ref = run_oracle(inp, T)
    compare(gpu, ref, T, inp["verify_len"].numpy())
    assert gpu["status"] == sv.SV_ERR_DEVICE_INPUT
    bad = ref["out_accepted"] < 0
    assert bad.sum() >= 4
    assert (gpu["out_accepted"][bad] == -1).all()


@needs_cuda
def test_deterministic_and_workspace_reuse(sv):
    """Identical inputs give identical outputs; one workspace serves calls of several
    shapes and temperatures back to back."""
    ws = sv.Workspace(64, 8, 151936)
    a = to_dev(synth.verify_inputs(64, 8, 20000, seed=1))
    b = to_dev(synth.verify_inputs(7, 3, 151936, dtype=torch.float32, seed=2))
    r1 = run_gpu(sv, a, 1.0, ws=ws)
    r2 = run_gpu(sv, b, 0.0, ws=ws)
    r3 = run_gpu(sv, b, 0.8, ws=ws)
    r4 = run_gpu(sv, a, 1.0, ws=ws)
    for r in (r1, r2, r3, r4):
        assert r["status"] == sv.SV_OK
    for k in ("out_tok", "out_accepted", "p", "q"):
        assert np.array_equal(r1[k], r4[k], equal_nan=True), k
    bc = {k: v.cpu() for k, v in b.items()}
    compare(r2, run_oracle(bc, 0.0), 0.0, bc["verify_len"])
    compare(r3, run_oracle(bc, 0.8), 0.8, bc["verify_len"])
    ac = {k: v.cpu() for k, v in a.items()}
    compare(r4, run_oracle(ac, 1.0), 1.0, ac["verify_len"])


@needs_cuda
def test_zero_lengths_and_k32(sv):
    """verify_len 0 (plain sampling of one token) and K = 32."""
    inp = synth.verify_inputs(8, 32, 3000, temperature=1.0, seed=9, verify_len=[0] * 4 + [32] * 4)
    inp["draft"][4:] = inp["target"][4:, :32]  # all 32 accepted for the last four
    for T in (1.0, 0.0):
        gpu = run_gpu(sv, to_dev(inp), T)
        compare(gpu, run_oracle(inp, T), T, inp["verify_len"].numpy())
    assert (gpu["out_accepted"][:4] == 0).all()


@needs_cuda
def test_emitted_distribution_matches_target(sv):
    """Losslessness on the GPU, statistically: 20,480 copies of one request (5 calls of
    4,096) with fresh uniforms and drafts from q; the first emitted token follows p_0
    (chi-square, 15 degrees of freedom)."""
    B, K, V, calls = 4096, 2, 16, 5
    rng = np.random.default_rng(4)
    t = (rng.normal(0, 1.0, (K + 1, V))).astype(np.float32)
    d = (t[:K] + rng.normal(0, 1.0, (K, V))).astype(np.float32)
    q = [np.exp(d[k] - d[k].max()) / np.exp(d[k] - d[k].max()).sum() for k in range(K)]
    p0 = np.exp(t[0] - t[0].max()) / np.exp(t[0] - t[0].max()).sum()
    ws = sv.Workspace(B, K, V)
    counts = np.zeros(V)
    for _ in range(calls):
        tok = np.stack([rng.choice(V, size=B, p=q[k]) for k in range(K)], 1).astype(np.int32)
        g = {"target": torch.from_numpy(np.broadcast_to(t, (B, K + 1, V)).copy()).cuda(),
             "draft": torch.from_numpy(np.broadcast_to(d, (B, K, V)).copy()).cuda(),
             "draft_tok": torch.from_numpy(tok).cuda(),
             "verify_len": torch.full((B,), K, dtype=torch.int32, device="cuda"),
             "uniforms": torch.from_numpy(rng.random((B, K + 1)).astype(np.float32)).cuda()}
        gpu = run_gpu(sv, g, 1.0, ws=ws, diag=False)
        counts += np.bincount(gpu["out_tok"][:, 0], minlength=V)
    exp = p0 * B * calls
    chi2 = float(((counts - exp) ** 2 / exp).sum())
    assert chi2 < 50.0, chi2  # p < 1e-5 under the null


@needs_cuda
def test_acceptance_counters(sv):
    inp = synth.verify_inputs(40, 6, 3000, temperature=1.0, seed=12, verify_len="uniform")
    g = to_dev(inp)
    ws = sv.Workspace(40, 6, 3000)
    acc_c = torch.zeros(6, dtype=torch.int32, device="cuda")
    tst_c = torch.zeros(6, dtype=torch.int32, device="cuda")
    tok, acc = sv.sv_verify(g["target"], g["draft"], g["draft_tok"], g["verify_len"],
                            g["uniforms"], 1.0, ws, accept_count=acc_c, tested_count=tst_c)
    acc = acc.cpu().numpy()
    L = inp["verify_len"].numpy()
    k = np.arange(6)[None, :]
    assert np.array_equal(acc_c.cpu().numpy(), (k < acc[:, None]).sum(0))
    assert np.array_equal(tst_c.cpu().numpy(), ((k <= acc[:, None]) & (k < L[:, None])).sum(0))


@needs_cuda
def test_cuda_graph_replay(sv):
    """Schedule + verify captured once in a CUDA graph and replayed on new data written
    into the same buffers (the max-length buffers + masking pattern)."""
    B, K, V = 48, 8, 30000
    ws = sv.Workspace(B, K, V)
    g = to_dev(synth.verify_inputs(B, K, V, seed=20))
    conf = synth.confidences(B, K, seed=20).cuda()
    out_len = torch.empty(B, dtype=torch.int32, device="cuda")
    out_tok = torch.empty((B, K + 1), dtype=torch.int32, device="cuda")
    out_acc = torch.empty(B, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())

    def body():
        sv.sv_schedule(conf, 0.3, 200, ws, out_len=out_len, stream=s)
        sv.sv_verify(g["target"], g["draft"], g["draft_tok"], out_len, g["uniforms"], 1.0, ws,
                     out_tok=out_tok, out_accepted=out_acc, stream=s)

    with torch.cuda.stream(s):  # warm-up outside capture
        body()
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        body()
    for seed in (21, 22):
        nxt = synth.verify_inputs(B, K, V, seed=seed)
        c2 = synth.confidences(B, K, seed=seed)
        for k in ("target", "draft", "draft_tok", "uniforms"):
            g[k].copy_(nxt[k])
        conf.copy_(c2)
        graph.replay()
        torch.cuda.synchronize()
        ref_s = oracle.schedule(c2.numpy(), 0.3, 200)
        assert np.array_equal(out_len.cpu().numpy(), ref_s["out_len"])
        nxt["verify_len"] = torch.from_numpy(ref_s["out_len"])
        compare({"out_tok": out_tok.cpu().numpy(), "out_accepted": out_acc.cpu().numpy()},
                run_oracle(nxt, 1.0), 1.0, ref_s["out_len"], check_p=False)


@needs_cuda
def test_timeout_then_clean_call(sv):
    """Every wait of a verify call for another warp's result is bounded. With the bound
    cut to 300 clock cycles (a testing aid), waits that normally last microseconds (the
    producers waiting for the last decisions, warps waiting for published words) run
    out: the call gives up, SV_ERR_TIMEOUT is reported, and the kernel returns. The
    next call on the same workspace, with the status still set, must match the oracle
    exactly: the abort of one call does not leak into the next."""
    inp = synth.sweep_point(64, 8, seed=3, device="cuda")
    ws = sv.Workspace(64, 8, synth.QWEN3_VOCAB)
    prev = sv.set_wait_limit(300)
    try:
        sv.sv_verify(inp["target"], inp["draft"], inp["draft_tok"], inp["verify_len"],
                     inp["uniforms"], 1.0, ws)
        torch.cuda.synchronize()
    finally:
        sv.set_wait_limit(prev)
    assert ws.status() == sv.SV_ERR_TIMEOUT
    for _ in range(2):
        tok, acc, p, q, fl = sv.sv_verify(inp["target"], inp["draft"], inp["draft_tok"],
                                          inp["verify_len"], inp["uniforms"], 1.0, ws, diag=True)
        torch.cuda.synchronize()
        gpu = {"out_tok": tok.cpu().numpy(), "out_accepted": acc.cpu().numpy(),
               "p": p.cpu().numpy(), "q": q.cpu().numpy(), "flags": fl.cpu().numpy()}
        compare(gpu, run_oracle(inp, 1.0), 1.0, inp["verify_len"].cpu().numpy())
    assert ws.status(clear=True) == sv.SV_ERR_TIMEOUT  # the report stays until cleared
    assert ws.status() == sv.SV_OK


@needs_cuda
def test_near_tie_summary():
    """Reading of the near-tie rule. Outside the oracle's 1e-5 near-tie windows every
    decision above was bit-exact. At V = 151,936 the mean inverse-CDF bucket (6.6e-6) is
    narrower than that window, so a few percent of terminal samples are flagged whatever
    the arithmetic; inside the window a decision may differ from the oracle only where
    the oracle's own margin is below the GPU's fp32 resolution (MARGIN_RESOLUTION), which
    every comparison above asserted. Reported here: flagged requests, differing
    decisions, and the largest margin among those."""
    t = gpu_util.TOTALS
    if t["positions"] == 0:
        pytest.skip("no full-size parity test ran")
    print(f"[near-ties] total: {t['flagged']} flagged requests "
          f"({t['flagged'] / t['positions']:.2e} of {t['positions']} positions), "
          f"{t['mismatch']} decided differently ({t['mismatch'] / t['positions']:.2e}), "
          f"largest oracle margin among them {t['max_margin']:.2e}")
    print(f"[near-ties] by kind: accept test within 1e-5 of its ratio in {t['accept_tie']} "
          f"requests ({t['accept_tie'] / t['positions']:.2e} of positions); terminal sample "
          f"within 1e-5 of a CDF edge in {t['cdf_edge']} of {t['requests']} requests; "
          f"degenerate (tiny probabilities, empty residual) in {t['degenerate']}")
    f = gpu_util.FLAG_COUNTS
    if f["requests"]:
        print(f"[near-ties] GPU flags (accept ties and CDF edges): {f['gpu_flagged']} of "
              f"{f['requests']} valid requests ({f['gpu_flagged'] / t['positions']:.2e} of "
              f"positions); {f['in_band']} requests had an oracle margin within 2e-6 of the "
              f"1e-5 window, where the GPU's flag may differ")
    assert t["max_margin"] < gpu_util.MARGIN_RESOLUTION
