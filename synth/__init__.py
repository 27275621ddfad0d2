"""Seeded synthetic inputs for batched speculative verification.

This module is shared by the tests, the benchmark and the smoke check; it feeds the
same tensors to the CUDA library and to the CPU oracle. It holds none of the
method's arithmetic: no softmax, no acceptance test, no survival product. Draft
tokens are drawn from softmax(draft/T) with the Gumbel-max construction
(argmax of logits/T plus Gumbel noise), which needs no normaliser.

Workload shapes follow the DSpark pages' serving settings: Qwen3-8B's vocabulary of
151,936 entries and DeepSeek-V4's 129,280, 1-512 concurrent requests, draft blocks of
4-16 tokens. No benchmark dataset is involved; every value is drawn here from a seed.
"""
from __future__ import annotations

import numpy as np
import torch

QWEN3_VOCAB = 151_936
DSV4_VOCAB = 129_280

_CHUNK_ELEMS = 1 << 26  # bound on the temporaries of one generation chunk


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def verify_inputs(B, K, V, *, dtype=torch.bfloat16, temperature=1.0, target_sigma=3.0,
                  draft_sigma=1.0, peak_prob=0.0, peak_height=12.0, verify_len="full",
                  seed=0, device="cpu"):
    """Inputs of one verification call.

    target [B,K+1,V] ~ N(0, target_sigma^2); each target row independently gets
    +peak_height at one uniform index with probability peak_prob. draft [B,K,V] =
    target rows 0..K-1 (before rounding) + N(0, sigma_b^2), sigma_b = draft_sigma (a
    scalar or a length-B sequence). Both are rounded to ``dtype``. draft_tok[b,k] is a
    sample of softmax(draft[b,k]/T) from the rounded draft logits (argmax at T == 0).
    verify_len: "full" (= K), "uniform" (U{1..K}), or an int sequence of length B.
    uniforms [B,K+1] ~ U[0,1) float32.
    """
    g = _gen(device, seed)
    sig = torch.as_tensor(draft_sigma, dtype=torch.float32).reshape(-1)
    if sig.numel() == 1:
        sig = sig.expand(B)
    assert sig.numel() == B
    sig = sig.to(device)
    target = torch.empty((B, K + 1, V), dtype=dtype, device=device)
    draft = torch.empty((B, K, V), dtype=dtype, device=device)
    tok = torch.empty((B, K), dtype=torch.int32, device=device)
    rb = max(1, _CHUNK_ELEMS // ((K + 1) * V))
    for b0 in range(0, B, rb):
        b1 = min(B, b0 + rb)
        n = b1 - b0
        t32 = torch.randn((n, K + 1, V), generator=g, device=device) * target_sigma
        if peak_prob > 0.0:
            hit = torch.rand((n, K + 1), generator=g, device=device) < peak_prob
            where = torch.randint(0, V, (n, K + 1), generator=g, device=device)
            t32.scatter_add_(2, where.unsqueeze(-1), (hit.float() * peak_height).unsqueeze(-1))
        noise = torch.randn((n, K, V), generator=g, device=device) * sig[b0:b1].view(n, 1, 1)
        d32 = t32[:, :K, :] + noise
        del noise
        target[b0:b1] = t32.to(dtype)
        draft[b0:b1] = d32.to(dtype)
        del t32, d32
        d = draft[b0:b1].float()
        if temperature > 0.0:
            e = torch.rand((n, K, V), generator=g, device=device).clamp_min_(1e-30)
            gumbel = -torch.log(-torch.log(e))
            del e
            tok[b0:b1] = torch.argmax(d / temperature + gumbel, dim=-1).to(torch.int32)
            del gumbel
        else:
            tok[b0:b1] = torch.argmax(d, dim=-1).to(torch.int32)
        del d
    if isinstance(verify_len, str) and verify_len == "full":
        vlen = torch.full((B,), K, dtype=torch.int32, device=device)
    elif isinstance(verify_len, str) and verify_len == "uniform":
        vlen = torch.randint(1, K + 1, (B,), generator=g, device=device).to(torch.int32)
    else:
        vlen = torch.as_tensor(list(verify_len), dtype=torch.int32).to(device)
        assert vlen.numel() == B
    uniforms = torch.rand((B, K + 1), generator=g, device=device, dtype=torch.float32)
    return {"target": target, "draft": draft, "draft_tok": tok, "verify_len": vlen,
            "uniforms": uniforms}


def confidences(B, K, *, a=8.0, b=2.0, decay=0.93, seed=0):
    """Per-position draft confidences c[b,k] = Beta(a,b) draw * decay**(k+1), float32.

    Positions are 1-based in the exponent (the first position is scaled by decay once).
    """
    rng = np.random.default_rng(int(seed))
    draws = rng.beta(a, b, size=(B, K))
    scale = decay ** np.arange(1, K + 1, dtype=np.float64)
    return torch.from_numpy((draws * scale[None, :]).astype(np.float32))


def to_oracle(t):
    """torch tensor -> numpy array in the form the oracle takes (bf16 as uint16 bits)."""
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


# ----------------------------------------------------------------------------------
# Named workloads. Each returns (kwargs for verify_inputs, extra) for a seed.
# ----------------------------------------------------------------------------------

def tiny_fp32(seed=0, device="cpu"):
    """B=4, K=4, V=1024, fp32; target N(0,2^2), draft noise N(0,0.5^2); T=1; L=K."""
    return verify_inputs(4, 4, 1024, dtype=torch.float32, temperature=1.0, target_sigma=2.0,
                         draft_sigma=0.5, seed=seed, device=device)


def qwen3_verify(temperature, seed=0, device="cpu", B=32, K=8):
    """B=32, K=8, V=151,936 bf16; target N(0,3^2) with rows peaked (+12) w.p. 0.2;
    draft noise N(0,1); L=K."""
    return verify_inputs(B, K, QWEN3_VOCAB, dtype=torch.bfloat16, temperature=temperature,
                         target_sigma=3.0, draft_sigma=1.0, peak_prob=0.2, peak_height=12.0,
                         seed=seed, device=device)


def ragged_sigmas(B):
    """Draft noise 0.5 for the first half of the requests, 1.5 for the second."""
    return [0.5 if b < B // 2 else 1.5 for b in range(B)]


def ragged_schedule(seed=0, device="cpu", B=256, K=16):
    """B=256, K=16, V=151,936 bf16, T=1; confidences Beta(8,2)*0.93^k; draft noise 0.5
    for the first half of the requests and 1.5 for the second. The verify lengths come
    from the schedule, so the caller supplies them; the inputs here carry L=K."""
    inp = verify_inputs(B, K, QWEN3_VOCAB, dtype=torch.bfloat16, temperature=1.0,
                        target_sigma=3.0, draft_sigma=ragged_sigmas(B), seed=seed,
                        device=device)
    inp["conf"] = confidences(B, K, seed=seed).to(device)
    return inp


def large_batch(seed=0, device="cpu", B=512):
    """B=512, K=8, V=129,280 bf16, T=0.7; target N(0,3^2), draft noise N(0,1);
    verify lengths U{1..8}."""
    return verify_inputs(B, 8, DSV4_VOCAB, dtype=torch.bfloat16, temperature=0.7,
                         target_sigma=3.0, draft_sigma=1.0, verify_len="uniform", seed=seed,
                         device=device)


def sweep_point(B, K, seed=0, device="cpu"):
    """Roofline sweep point: V=151,936 bf16, T=1, draft noise 1.0, full-length blocks."""
    return verify_inputs(B, K, QWEN3_VOCAB, dtype=torch.bfloat16, temperature=1.0,
                         target_sigma=3.0, draft_sigma=1.0, seed=seed, device=device)


SWEEP_B = (1, 4, 8, 16, 32, 64, 128)
SWEEP_K = (4, 8, 16)


def logit_bytes(verify_len, V, elem_bytes, greedy=False):
    """Algorithmic logit bytes one verification call must read: per request (L+1)
    target rows, plus L draft rows unless greedy."""
    L = torch.as_tensor(verify_len).to(torch.int64).clamp_min(0)
    rows = (L + 1) if greedy else (2 * L + 1)
    return int(rows.sum().item()) * V * elem_bytes



# ----------------------------------------------------------------------------------
# Calibration-loop inputs (random numbers only).
# ----------------------------------------------------------------------------------

def temperatures(K, *, lo=0.5, hi=2.5, seed=0):
    """Per-position temperatures [K] float32, uniform in [lo, hi]."""
    rng = np.random.default_rng(int(seed) + 1000)
    return torch.from_numpy(rng.uniform(lo, hi, size=K).astype(np.float32))


def load_state(*, seed=0, q_max=64.0, m_max=80.0):
    """{Q, Q_max, M_gpu, M_max} float32: queue depth and memory use, each up to a bit
    past its maximum (so the load factor's clamp is reached now and then)."""
    rng = np.random.default_rng(int(seed) + 2000)
    q = rng.uniform(0.0, 1.2 * q_max)
    m = rng.uniform(0.0, 1.1 * m_max)
    return torch.tensor([q, q_max, m, m_max], dtype=torch.float32)


def calib_round(B, K, *, seed=0):
    """One verification round as the calibration loop sees it: calibrated confidences
    [B,K] float32 in [0,1] (some exactly 0, 1 or on a bin boundary of tenths), verify
    lengths [B] in [0,K] and accepted counts [B] in [0, L_b], a few -1 (invalid)."""
    rng = np.random.default_rng(int(seed) + 3000)
    c = rng.uniform(0.0, 1.0, size=(B, K)).astype(np.float32)
    pick = rng.random((B, K))
    c[pick < 0.02] = 0.0
    c[(pick >= 0.02) & (pick < 0.04)] = 1.0
    edges = (rng.integers(1, 10, size=(B, K)) / 10.0).astype(np.float32)
    c[(pick >= 0.04) & (pick < 0.08)] = edges[(pick >= 0.04) & (pick < 0.08)]
    vlen = rng.integers(0, K + 1, size=B).astype(np.int32)
    acc = np.array([rng.integers(0, v + 1) for v in vlen], np.int32)
    acc[rng.random(B) < 0.05] = -1
    return torch.from_numpy(c), torch.from_numpy(vlen), torch.from_numpy(acc)



def markov_inputs(B, K, V, r, *, seed=0, logit_sigma=3.0):
    """Drafting-side inputs: raw logits [B,K,V] ~ N(0, logit_sigma^2) and low-rank factors
    U, Vm [V,r] ~ N(0, r^-1/2) (so a correction U Vm[y]^T is of order 1), all bf16, and
    previous tokens [B] ~ U{0..V-1}."""
    g = torch.Generator().manual_seed(int(seed))
    L = (torch.randn((B, K, V), generator=g) * logit_sigma).to(torch.bfloat16)
    s = float(r) ** -0.25
    U = (torch.randn((V, r), generator=g) * s).to(torch.bfloat16)
    Vm = (torch.randn((V, r), generator=g) * s).to(torch.bfloat16)
    prev = torch.randint(0, V, (B,), generator=g, dtype=torch.int32)
    return {"logits": L, "U": U, "Vm": Vm, "prev": prev}


def throughput_curve(n, *, seed=0, x_max=4096.0):
    """A throughput curve [2, n] float32: batch sizes in tokens (ascending, from 1 to
    about x_max) and tokens/s rising with a falling slope (memory-bound, then flat)."""
    rng = np.random.default_rng(int(seed) + 4000)
    x = np.unique(np.round(np.geomspace(1.0, x_max, n) * rng.uniform(0.9, 1.1, n)).astype(np.float64))
    x = np.maximum.accumulate(x)
    x = np.unique(x)
    knee = rng.uniform(16.0, 512.0)
    y = 30.0 * x / (1.0 + x / knee) + rng.uniform(0.0, 5.0)
    return torch.tensor(np.stack([x, y]), dtype=torch.float32)


# ----------------------------------------------------------------------------------
# Tree verification inputs.
# ----------------------------------------------------------------------------------

# A 16-node draft tree of the kind tree drafters expand (several candidates for the
# first token, fewer deeper down): node 0 is the committed context, parent links below.
# Depths: nodes 1-4 at 1, 5-10 at 2, 11-13 at 3, 14-15 at 4.
TREE16_PARENTS = (-1, 0, 0, 0, 0, 1, 1, 1, 2, 2, 3, 5, 5, 8, 11, 13)


def tree_parents(B, N, shape="tree16", *, seed=0):
    """Parent links [B, N] int32 (entry 0 is -1; 0 <= parent[n] < n).

    shape: "tree16" (TREE16_PARENTS, N == 16), "chain" (parent n-1), "star" (every node
    a child of the root), "random" (per request: parent n-1 with probability 1/2, else
    uniform over 0..n-1), or an explicit sequence of N links shared by every request.
    """
    if isinstance(shape, str):
        if shape == "tree16":
            assert N == len(TREE16_PARENTS)
            par = np.tile(np.array(TREE16_PARENTS, np.int32), (B, 1))
        elif shape == "chain":
            par = np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1))
        elif shape == "star":
            par = np.zeros((B, N), np.int32)
            par[:, 0] = -1
        elif shape == "random":
            rng = np.random.default_rng(int(seed) + 5000)
            par = np.zeros((B, N), np.int32)
            par[:, 0] = -1
            for n in range(1, N):
                deep = rng.random(B) < 0.5
                par[:, n] = np.where(deep, n - 1, rng.integers(0, n, size=B))
        else:
            raise ValueError(shape)
    else:
        par = np.tile(np.asarray(shape, np.int32).reshape(1, N), (B, 1))
    return torch.from_numpy(np.ascontiguousarray(par))


def tree_inputs(B, N, V, *, dtype=torch.bfloat16, temperature=1.0, target_sigma=3.0,
                draft_sigma=1.0, peak_prob=0.0, peak_height=12.0, shape="tree16",
                n_nodes="full", seed=0, device="cpu"):
    """Inputs of one tree verification call.

    target [B,N,V] ~ N(0, target_sigma^2), each row peaked (+peak_height at one uniform
    index) with probability peak_prob; draft [B,N,V] = target + N(0, draft_sigma^2),
    both rounded to ``dtype``. parent [B,N] from ``tree_parents``. The token of node n
    is an independent sample of softmax(draft[b, parent[n]] / T') from the rounded
    draft logits (Gumbel-max), T' = temperature, or 1 at T == 0 so that siblings differ.
    n_nodes: "full" (= N), "uniform" (U{1..N}), or an int sequence of length B.
    uniforms [B,N] ~ U[0,1) float32.
    """
    g = _gen(device, seed)
    par = tree_parents(B, N, shape, seed=seed).to(device)
    target = torch.empty((B, N, V), dtype=dtype, device=device)
    draft = torch.empty((B, N, V), dtype=dtype, device=device)
    tok = torch.zeros((B, N), dtype=torch.int32, device=device)
    t_draw = temperature if temperature > 0.0 else 1.0
    rb = max(1, _CHUNK_ELEMS // (N * V))
    for b0 in range(0, B, rb):
        b1 = min(B, b0 + rb)
        n = b1 - b0
        t32 = torch.randn((n, N, V), generator=g, device=device) * target_sigma
        if peak_prob > 0.0:
            hit = torch.rand((n, N), generator=g, device=device) < peak_prob
            where = torch.randint(0, V, (n, N), generator=g, device=device)
            t32.scatter_add_(2, where.unsqueeze(-1), (hit.float() * peak_height).unsqueeze(-1))
        d32 = t32 + torch.randn((n, N, V), generator=g, device=device) * draft_sigma
        target[b0:b1] = t32.to(dtype)
        draft[b0:b1] = d32.to(dtype)
        del t32, d32
        # Row of the parent of every node (node 0 reads its own row; its token is unused).
        src = par[b0:b1].clamp_min(0).long()
        d = torch.gather(draft[b0:b1].float(), 1, src.unsqueeze(-1).expand(n, N, V))
        e = torch.rand((n, N, V), generator=g, device=device).clamp_min_(1e-30)
        d = d / t_draw - torch.log(-torch.log(e))
        del e
        tok[b0:b1] = torch.argmax(d, dim=-1).to(torch.int32)
        del d
    tok[:, 0] = 0
    if isinstance(n_nodes, str) and n_nodes == "full":
        nn = torch.full((B,), N, dtype=torch.int32, device=device)
    elif isinstance(n_nodes, str) and n_nodes == "uniform":
        nn = torch.randint(1, N + 1, (B,), generator=g, device=device).to(torch.int32)
    else:
        nn = torch.as_tensor(list(n_nodes), dtype=torch.int32).to(device)
        assert nn.numel() == B
    uniforms = torch.rand((B, N), generator=g, device=device, dtype=torch.float32)
    return {"target": target, "draft": draft, "parent": par, "draft_tok": tok,
            "n_nodes": nn, "uniforms": uniforms}


def tree_qwen3(temperature, seed=0, device="cpu", B=64):
    """B trees (64 by default) of 16 nodes (TREE16_PARENTS), V=151,936 bf16; target N(0,3^2) with
    rows peaked (+12) w.p. 0.2; draft noise N(0,1)."""
    return tree_inputs(B, 16, QWEN3_VOCAB, dtype=torch.bfloat16, temperature=temperature,
                       target_sigma=3.0, draft_sigma=1.0, peak_prob=0.2, peak_height=12.0,
                       shape="tree16", seed=seed, device=device)


def tree_path_bytes(out_path, out_accepted, parent, V, elem_bytes, greedy=False):
    """Logit bytes a tree walk must read: the target row of every node on the accepted
    path plus the stop node, and (unless greedy) the draft row of each of those nodes
    that has children."""
    par = torch.as_tensor(parent).cpu().numpy()
    path = torch.as_tensor(out_path).cpu().numpy()
    acc = torch.as_tensor(out_accepted).cpu().numpy()
    rows = 0
    for b in range(par.shape[0]):
        if acc[b] < 0:
            continue
        nodes = [0] + [int(x) for x in path[b, :acc[b]]]
        rows += len(nodes)
        if not greedy:
            rows += sum(1 for c in nodes if (par[b, c + 1:] == c).any())
    return rows * V * elem_bytes
