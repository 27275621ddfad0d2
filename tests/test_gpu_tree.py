"""GPU parity of sv_verify_tree against the float64 oracle: the accepted path, its
node indices and the terminal token bit-exact outside flagged near-ties (whose
margins must stay below the GPU's resolution)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import MARGIN_RESOLUTION, NTHREADS

pytestmark = pytest.mark.gpu

needs_cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verification_79_gb300 as m

    m.load()
    return m


@pytest.fixture(scope="module")
def ws(sv):
    return sv.Workspace(1, 1, 1)


def run_gpu(sv, ws, g, T):
    out = sv.sv_verify_tree(g["target"], g["draft"] if T > 0 else None, g["parent"],
                            g["draft_tok"], g["n_nodes"], g["uniforms"] if T > 0 else None,
                            T, ws)
    torch.cuda.synchronize()
    return {"out_tok": out[0].cpu().numpy(), "out_accepted": out[1].cpu().numpy(),
            "out_path": out[2].cpu().numpy(), "status": ws.status(clear=True)}


def run_oracle(inp, T):
    return oracle.verify_tree(synth.to_oracle(inp["target"]),
                              synth.to_oracle(inp["draft"]) if T > 0 else None,
                              inp["parent"].cpu().numpy(), inp["draft_tok"].cpu().numpy(),
                              inp["n_nodes"].cpu().numpy(),
                              inp["uniforms"].cpu().numpy() if T > 0 else None, T,
                              nthreads=NTHREADS)


def compare(gpu, ref):
    """Returns (flagged requests, flagged requests decided differently)."""
    flagged = (ref["flags"] & oracle.NEAR_TIE_MASK) != 0
    differ = ((gpu["out_accepted"] != ref["out_accepted"])
              | (gpu["out_tok"] != ref["out_tok"]).any(1)
              | (gpu["out_path"] != ref["out_path"]).any(1))
    bad = np.nonzero(differ & ~flagged)[0]
    assert bad.size == 0, (
        f"requests {bad[:5]}: gpu acc {gpu['out_accepted'][bad[:5]]} tok "
        f"{gpu['out_tok'][bad[:3]]} path {gpu['out_path'][bad[:3]]}; ref acc "
        f"{ref['out_accepted'][bad[:5]]} tok {ref['out_tok'][bad[:3]]} path "
        f"{ref['out_path'][bad[:3]]}")
    margins = ref["margin"][differ & flagged]
    assert (margins < MARGIN_RESOLUTION).all(), margins
    return int(flagged.sum()), int((differ & flagged).sum())


def check(sv, ws, inp, T, expect_ok=True):
    g = {k: (v.to("cuda") if torch.is_tensor(v) else v) for k, v in inp.items()}
    gpu = run_gpu(sv, ws, g, T)
    ref = run_oracle(inp, T)
    nf, nd = compare(gpu, ref)
    if expect_ok:
        assert gpu["status"] == sv.SV_OK
        assert ref["status"] == oracle.OK
    return gpu, ref, nf, nd


SMALL = [(dt, V, T, shape)
         for dt in (torch.bfloat16, torch.float32)
         for V in (1, 7, 100, 2049, 4097, 12345)
         for T in (0.0, 0.6, 1.0, 2.5)
         for shape in ("random", "star")]


@needs_cuda
@pytest.mark.parametrize("dt,V,T,shape", SMALL)
def test_small_shapes(sv, ws, dt, V, T, shape):
    """Random and star trees, ragged node counts, rows of every alignment phase."""
    B, N = 12, 9
    inp = synth.tree_inputs(B, N, V, dtype=dt, temperature=T, target_sigma=2.0,
                            draft_sigma=1.5, shape=shape, n_nodes="uniform",
                            seed=V * 13 + int(T * 10) + (shape == "star"))
    check(sv, ws, inp, T)


@needs_cuda
@pytest.mark.parametrize("T", [0.0, 1.0])
@pytest.mark.parametrize("B", [1, 3, 40, 200])
def test_batch_sizes(sv, ws, B, T):
    """Cluster sizes 8 down to 1 (chosen from the batch), tree16 shape."""
    inp = synth.tree_inputs(B, 16, 3001, dtype=torch.bfloat16, temperature=T, seed=B)
    check(sv, ws, inp, T)


@needs_cuda
@pytest.mark.parametrize("T", [0.7, 1.0])
def test_many_rejections(sv, ws, T):
    """A star of 63 children with a draft far from the target: long rejection runs, so
    the residual passes and the residual sample dominate."""
    inp = synth.tree_inputs(16, 64, 5000, dtype=torch.float32, temperature=T, target_sigma=2.0,
                            draft_sigma=4.0, shape="star", seed=int(T * 10))
    gpu, ref, nf, nd = check(sv, ws, inp, T)
    assert (ref["out_accepted"] == 0).sum() > 0  # some requests reject every child


@needs_cuda
@pytest.mark.parametrize("T", [0.0, 1.0])
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_unaligned_rows(sv, ws, T, dt):
    """Odd V, and target and draft bases one element past different boundaries, so the
    draft rows fall off the target's 16-byte grid."""
    B, N, V = 6, 7, 4099
    inp = synth.tree_inputs(B, N, V, dtype=dt, temperature=T, shape="random", seed=5)
    g = {k: (v.to("cuda") if torch.is_tensor(v) else v) for k, v in inp.items()}
    for key, shift in (("target", 1), ("draft", 2)):
        big = torch.empty(g[key].numel() + shift, dtype=dt, device="cuda")
        big[shift:] = g[key].reshape(-1)
        g[key] = big[shift:].view(B, N, V)
    gpu = run_gpu(sv, ws, g, T)
    compare(gpu, run_oracle(inp, T))


@needs_cuda
@pytest.mark.parametrize("T", [1.0, 0.0])
def test_chain_tree_matches_sv_verify(sv, ws, T):
    """A chain-shaped tree gives what sv_verify gives on the same rows."""
    B, K, V = 32, 6, 20000
    inp = synth.verify_inputs(B, K, V, dtype=torch.bfloat16, temperature=T, seed=3,
                              verify_len="uniform", device="cuda")
    wsv = sv.Workspace(B, K, V)
    ot, oa = sv.sv_verify(inp["target"], inp["draft"] if T > 0 else None, inp["draft_tok"],
                          inp["verify_len"], inp["uniforms"] if T > 0 else None, T, wsv)
    N = K + 1
    par = torch.arange(-1, N - 1, dtype=torch.int32, device="cuda").repeat(B, 1)
    tok = torch.zeros((B, N), dtype=torch.int32, device="cuda")
    tok[:, 1:] = inp["draft_tok"]
    u = torch.zeros((B, N), dtype=torch.float32, device="cuda")
    u[:, 1:] = inp["uniforms"][:, :K]
    u[:, 0] = inp["uniforms"][:, K]
    drf = torch.zeros_like(inp["target"])
    drf[:, :K] = inp["draft"]
    tt, ta, tp = sv.sv_verify_tree(inp["target"], drf if T > 0 else None, par, tok,
                                   inp["verify_len"] + 1, u if T > 0 else None, T, ws)
    torch.cuda.synchronize()
    ref = oracle.verify(synth.to_oracle(inp["target"]), synth.to_oracle(inp["draft"]),
                        inp["draft_tok"].cpu().numpy(), inp["verify_len"].cpu().numpy(),
                        inp["uniforms"].cpu().numpy(), T, nthreads=NTHREADS, diag=False)
    clean = (ref["flags"] & oracle.NEAR_TIE_MASK) == 0
    assert (ta.cpu().numpy()[clean] == oa.cpu().numpy()[clean]).all()
    assert (tt.cpu().numpy()[clean] == ot.cpu().numpy()[clean]).all()


@needs_cuda
@pytest.mark.parametrize("T", [1.0, 0.0])
def test_qwen3_tree16(sv, ws, T):
    """B=64 trees of 16 nodes, V=151,936 bf16: the workload the benchmark times."""
    inp = synth.tree_qwen3(T, seed=1, device="cuda")
    gpu, ref, nf, nd = check(sv, ws, inp, T)
    print(f"[tree] T={T}: mean accepted {ref['out_accepted'].mean():.2f}, {nf} flagged, "
          f"{nd} decided differently")


@needs_cuda
def test_invalid_and_unread_rows(sv, ws):
    """NaN in a reached row invalidates only that request (status set); NaN in rows the
    walk never reaches changes nothing."""
    B, N, V = 6, 5, 3000
    inp = synth.tree_inputs(B, N, V, dtype=torch.float32, temperature=1.0, shape="star",
                            seed=9)
    # Request 0: links 0 -> 1 -> 2 with accepting tests (u = 0 accepts whenever p(x) > 0),
    # so the walk ends at leaf 2 and never reaches nodes 3 and 4 (also children of 0).
    inp["parent"][0] = torch.tensor([-1, 0, 1, 0, 0], dtype=torch.int32)
    inp["uniforms"][0, 1:] = 0.0
    inp["target"][0, 3] = float("nan")
    inp["draft"][0, 4] = float("nan")
    inp["draft"][0, 2] = float("nan")  # leaf's draft row: never read
    inp["target"][2, 0, 17] = float("nan")  # root row of request 2: invalid
    inp["n_nodes"][4] = 0  # invalid
    g = {k: v.to("cuda") for k, v in inp.items()}
    gpu = run_gpu(sv, ws, g, 1.0)
    ref = run_oracle(inp, 1.0)
    compare(gpu, ref)
    assert gpu["out_accepted"][0] == 2
    assert gpu["out_accepted"][2] == -1 and gpu["out_accepted"][4] == -1
    assert (gpu["out_tok"][2] == -1).all() and (gpu["out_path"][4] == -1).all()
    assert gpu["status"] == sv.SV_ERR_DEVICE_INPUT


@needs_cuda
def test_graph_capture_and_repeat(sv, ws):
    """The call captures into a CUDA graph and replays with the same results."""
    inp = synth.tree_inputs(8, 16, 5000, dtype=torch.bfloat16, temperature=1.0, seed=4,
                            device="cuda")
    ref = run_gpu(sv, ws, inp, 1.0)
    st = torch.cuda.Stream()
    outs = [torch.empty((8, 16), dtype=torch.int32, device="cuda"),
            torch.empty(8, dtype=torch.int32, device="cuda"),
            torch.empty((8, 16), dtype=torch.int32, device="cuda")]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(st):
        sv.sv_verify_tree(inp["target"], inp["draft"], inp["parent"], inp["draft_tok"],
                          inp["n_nodes"], inp["uniforms"], 1.0, ws, *outs, stream=st)
        st.synchronize()
        with torch.cuda.graph(graph, stream=st):
            sv.sv_verify_tree(inp["target"], inp["draft"], inp["parent"], inp["draft_tok"],
                              inp["n_nodes"], inp["uniforms"], 1.0, ws, *outs, stream=st)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert (outs[0].cpu().numpy() == ref["out_tok"]).all()
    assert (outs[1].cpu().numpy() == ref["out_accepted"]).all()
    assert (outs[2].cpu().numpy() == ref["out_path"]).all()


@needs_cuda
def test_large_batch_dsv4_vocab(sv, ws):
    """B=512 random trees of 8 nodes at DeepSeek-V4's vocabulary (129,280, bf16), T=0.7:
    one CTA per request, several waves; every request against the oracle."""
    inp = synth.tree_inputs(512, 8, synth.DSV4_VOCAB, dtype=torch.bfloat16, temperature=0.7,
                            target_sigma=3.0, draft_sigma=1.0, shape="random",
                            n_nodes="uniform", seed=12, device="cuda")
    gpu = run_gpu(sv, ws, inp, 0.7)
    nf, nd = compare(gpu, run_oracle(inp, 0.7))
    assert gpu["status"] == sv.SV_OK
    print(f"[tree] B=512 V=129280: {nf} flagged, {nd} decided differently")
