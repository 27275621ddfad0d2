"""Helpers for the GPU parity tests: run the CUDA path and the oracle on the same
seeded inputs and compare them element by element."""
import os

import numpy as np
import torch

import oracle
import synth

NTHREADS = max(1, min(32, os.cpu_count() or 1))

# Probabilities p_k(x_k), q_k(x_k): the kernel works in fp32 on the same (exactly
# widened) inputs as the float64 oracle, so both dtypes are held to 1e-5 relative,
# the bound stated for fp32 inputs (bf16's stated bound, 2e-3, is looser).
P_RTOL = 1e-5

# Resolution of the GPU's decisions: its probabilities carry fp32 rounding (p, q within
# ~5e-7 relative, CDF positions within ~1e-7), so a decision whose oracle margin (the
# distance |u - min(1, p/q)|, or the terminal sample's distance to a CDF edge) is below
# this may come out differently. Differing decisions with a larger margin fail.
MARGIN_RESOLUTION = 2e-6

# Running totals over the full-size parity tests: verified positions, requests flagged
# as near-ties by the oracle (windows of 1e-5 on the accept ratio and on the inverse-CDF
# position), flagged requests on which the GPU actually decided differently, and the
# largest oracle margin among those.
TOTALS = {"positions": 0, "flagged": 0, "mismatch": 0, "max_margin": 0.0,
          "requests": 0, "accept_tie": 0, "cdf_edge": 0, "degenerate": 0}
# The flag kinds of the last comparison (added to TOTALS by account()): requests with
# an accept test within 1e-5 of its ratio, a terminal sample within 1e-5 of a CDF
# bucket edge, and degenerate cases (both probabilities below 1e-30, or a residual
# with less than 1e-5 of mass).
LAST = {"requests": 0, "accept_tie": 0, "cdf_edge": 0, "degenerate": 0}


def to_dev(inp, device="cuda"):
    return {k: (v.to(device) if torch.is_tensor(v) else v) for k, v in inp.items()}


def run_gpu(sv, g, T, ws=None, diag=True):
    B, K1, V = g["target"].shape
    ws = ws or sv.Workspace(B, K1 - 1, V, device=g["target"].device)
    out = sv.sv_verify(g["target"], g["draft"] if T > 0 else None, g["draft_tok"],
                       g["verify_len"], g["uniforms"] if T > 0 else None, T, ws, diag=diag)
    torch.cuda.synchronize()
    res = {"out_tok": out[0].cpu().numpy(), "out_accepted": out[1].cpu().numpy()}
    if diag:
        res["p"] = out[2].cpu().numpy()
        res["q"] = out[3].cpu().numpy()
        res["flags"] = out[4].cpu().numpy()
    res["status"] = ws.status(clear=True)
    return res


def run_oracle(inp, T, idx=None, diag=True):
    sel = (lambda t: t[idx]) if idx is not None else (lambda t: t)
    return oracle.verify(synth.to_oracle(sel(inp["target"])),
                         synth.to_oracle(sel(inp["draft"])) if T > 0 else None,
                         sel(inp["draft_tok"]).cpu().numpy(), sel(inp["verify_len"]).cpu().numpy(),
                         sel(inp["uniforms"]).cpu().numpy() if T > 0 else None, T,
                         nthreads=NTHREADS, diag=diag)


def compare(gpu, ref, T, verify_len, idx=None, check_p=True):
    """Bit-exact decisions outside flagged near-ties; p/q within P_RTOL.
    Returns (flagged requests, verified positions, flagged requests that differ)."""
    acc, tok = gpu["out_accepted"], gpu["out_tok"]
    if idx is not None:
        acc, tok = acc[idx], tok[idx]
    L = np.asarray(verify_len)
    flagged = (ref["flags"] & oracle.NEAR_TIE_MASK) != 0
    ok = ~flagged
    bad = np.nonzero(ok & (acc != ref["out_accepted"]))[0]
    assert bad.size == 0, (f"accepted mismatch at requests {bad[:10]}: gpu {acc[bad[:10]]} "
                           f"ref {ref['out_accepted'][bad[:10]]}")
    rows = np.nonzero(ok & (tok != ref["out_tok"]).any(axis=1))[0]
    assert rows.size == 0, (f"token mismatch at requests {rows[:10]}: gpu {tok[rows[:3]]} "
                            f"ref {ref['out_tok'][rows[:3]]}")
    if check_p and T > 0 and "p" in gpu:
        gp, gq = gpu["p"], gpu["q"]
        if idx is not None:
            gp, gq = gp[idx], gq[idx]
        valid = (ref["flags"] & oracle.FLAG_INVALID) == 0
        K = gp.shape[1]
        mask = (np.arange(K)[None, :] < np.clip(L, 0, K)[:, None]) & valid[:, None]
        for name, g, r in (("p", gp, ref["p"]), ("q", gq, ref["q"])):
            err = np.abs(g.astype(np.float64) - r)
            lim = P_RTOL * np.abs(r) + 1e-30
            badm = mask & ~(err <= lim)
            if badm.any():
                rel = np.where(badm, err / (np.abs(r) + 1e-300), 0)
                bb, kk = np.unravel_index(np.argmax(rel), rel.shape)
                raise AssertionError(
                    f"{name} rel err {rel[bb, kk]:.3e} at request {bb} position {kk}: gpu "
                    f"{g[bb, kk]:.9e} ref {r[bb, kk]:.9e} (other: gpu p {gp[bb, kk]:.6e} "
                    f"q {gq[bb, kk]:.6e}; ref p {ref['p'][bb, kk]:.6e} q {ref['q'][bb, kk]:.6e}); "
                    f"{int(badm.sum())} elements over")
    if "flags" in gpu:
        check_flags(gpu["flags"] if idx is None else gpu["flags"][idx], ref, T)
    positions = int((np.clip(L, 0, None) + 1).sum())
    fl = ref["flags"]
    LAST.update(requests=int(fl.size), accept_tie=int(((fl & oracle.FLAG_ACCEPT_TIE) != 0).sum()),
                cdf_edge=int(((fl & oracle.FLAG_CDF_EDGE) != 0).sum()),
                degenerate=int(((fl & (oracle.FLAG_TINY_PROB | oracle.FLAG_SMALL_RESIDUAL)) != 0).sum()))
    differ = flagged & ((acc != ref["out_accepted"]) | (tok != ref["out_tok"]).any(axis=1))
    margins = ref["margin"][differ] if "margin" in ref else np.zeros(0)
    for b in np.nonzero(differ)[0][:5]:
        print(f"[near-ties] differs: request {b} flags {ref['flags'][b]} margin "
              f"{ref['margin'][b]:.2e} gpu acc {acc[b]} tok {tok[b].tolist()} ref acc "
              f"{ref['out_accepted'][b]} tok {ref['out_tok'][b].tolist()}")
    assert (margins < MARGIN_RESOLUTION).all(), (
        f"decisions differ at oracle margins {margins.tolist()}, above the GPU's resolution")
    return int(flagged.sum()), positions, int(differ.sum()), float(margins.max(initial=0.0))


# Near-tie flags from the GPU against the oracle's: the accept-test and CDF-edge kinds
# together are raised exactly when a request's smallest decision margin is below 1e-5,
# so they must agree wherever the oracle's margin is outside [1e-5 - 2e-6, 1e-5 + 2e-6]
# (the GPU's flags come from its own fp32 values); the invalid bit must agree always.
FLAG_BAND = MARGIN_RESOLUTION
FLAG_COUNTS = {"requests": 0, "gpu_flagged": 0, "in_band": 0}


def check_flags(gflags, ref, T):
    rf = ref["flags"]
    inv_g = (gflags & oracle.FLAG_INVALID) != 0
    inv_r = (rf & oracle.FLAG_INVALID) != 0
    assert np.array_equal(inv_g, inv_r), f"invalid flags differ at {np.nonzero(inv_g != inv_r)[0][:10]}"
    if T == 0:
        assert (gflags[~inv_g] == 0).all()
        return
    tie_mask = oracle.FLAG_ACCEPT_TIE | oracle.FLAG_CDF_EDGE
    g = ((gflags & tie_mask) != 0) & ~inv_g
    r = ((rf & tie_mask) != 0) & ~inv_r
    m = ref["margin"]
    band = np.abs(m - 1e-5) <= FLAG_BAND
    bad = np.nonzero((g != r) & ~band & ~inv_r)[0]
    assert bad.size == 0, (f"near-tie flags differ at requests {bad[:10]}: gpu {gflags[bad[:10]]} "
                           f"oracle {rf[bad[:10]]} margins {m[bad[:10]]}")
    FLAG_COUNTS["requests"] += int((~inv_r).sum())
    FLAG_COUNTS["gpu_flagged"] += int(g.sum())
    FLAG_COUNTS["in_band"] += int((band & ~inv_r).sum())


def account(name, nf, npos, nmis, max_margin=0.0):
    TOTALS["positions"] += npos
    TOTALS["flagged"] += nf
    TOTALS["mismatch"] += nmis
    TOTALS["max_margin"] = max(TOTALS["max_margin"], max_margin)
    for k in ("requests", "accept_tie", "cdf_edge", "degenerate"):
        TOTALS[k] += LAST[k]
    print(f"[near-ties] {name}: {nf} flagged requests, {nmis} of them decided differently, "
          f"{npos} positions")
