"""sv_verify_static, the entry point for callers that cannot allocate device memory
(plugins whose host application owns every device allocation, runtimes that plan all
their memory up front): it keeps its scratch in a fixed device array inside the
library.

Called through the C-ABI and checked against sv_verify (the workspace entry point) on
two calls in a row with different inputs: the decisions must be identical, the bar of
every parity test here. This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu
needs_cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


def _static_fn(lib):
    fn = lib.sv_verify_static
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [vp, vp, i32, vp, vp, vp, i32, i32, i32, ctypes.c_float, vp, vp, vp]
    fn.restype = i32
    return fn


@needs_cuda
def test_static_scratch_matches_workspace_entry_point():
    import speculative_decoding_verification_79_gb300 as sv

    lib = sv.load()
    fn = _static_fn(lib)
    stream = torch.cuda.current_stream()
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    cases = [(32, 8, synth.QWEN3_VOCAB, torch.bfloat16, 1.0, 5), (16, 5, 30000, torch.float32, 0.7, 6),
             (24, 8, 50000, torch.bfloat16, 0.0, 7)]
    for B, K, V, dt, T, seed in cases:
        g = synth.verify_inputs(B, K, V, dtype=dt, temperature=T, seed=seed, device="cuda",
                                verify_len="uniform")
        ws = sv.Workspace(B, K, V)
        ref_tok, ref_acc = sv.sv_verify(g["target"], g["draft"], g["draft_tok"], g["verify_len"],
                                        g["uniforms"], T, ws)
        for _ in range(2):  # two calls in a row on the shared array
            out_tok = torch.full((B, K + 1), -7, dtype=torch.int32, device="cuda")
            out_acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
            rc = fn(P(g["target"]), P(g["draft"] if T > 0 else None),
                    1 if dt == torch.bfloat16 else 0, P(g["draft_tok"]), P(g["verify_len"]),
                    P(g["uniforms"] if T > 0 else None), B, K, V, T, P(out_tok), P(out_acc),
                    ctypes.c_void_p(stream.cuda_stream))
            assert rc == sv.SV_OK, sv.status_string(rc)
            torch.cuda.synchronize()
            assert np.array_equal(out_acc.cpu().numpy(), ref_acc.cpu().numpy())
            assert np.array_equal(out_tok.cpu().numpy(), ref_tok.cpu().numpy())


@needs_cuda
def test_static_scratch_rejects_oversized_shapes():
    import speculative_decoding_verification_79_gb300 as sv

    lib = sv.load()
    fn = _static_fn(lib)
    limit = lib.sv_workspace_bytes(4096, 32, 1 << 20)
    assert limit > (16 << 20)
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    d = ctypes.c_void_p(dummy.data_ptr())
    rc = fn(d, d, 1, d, d, d, 4096, 32, 1 << 20, 1.0, d, d, None)
    assert rc == sv.SV_ERR_WORKSPACE


@needs_cuda
def test_static_scratch_after_invalid_device_data():
    """A call with invalid device data (a drafted token outside [0, V)) marks that
    request -1; the next call on the shared array must again match sv_verify."""
    import speculative_decoding_verification_79_gb300 as sv

    lib = sv.load()
    fn = _static_fn(lib)
    stream = torch.cuda.current_stream()
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    B, K, V = 16, 6, 40000
    bad = synth.verify_inputs(B, K, V, dtype=torch.bfloat16, temperature=1.0, seed=31,
                              device="cuda", verify_len="uniform")
    bad["draft_tok"][3, 0] = V
    bad["verify_len"][3] = K
    good = synth.verify_inputs(B, K, V, dtype=torch.bfloat16, temperature=1.0, seed=32,
                               device="cuda", verify_len="uniform")
    ws = sv.Workspace(B, K, V)
    ref_tok, ref_acc = sv.sv_verify(good["target"], good["draft"], good["draft_tok"],
                                    good["verify_len"], good["uniforms"], 1.0, ws)
    for g, check in ((bad, False), (good, True)):
        out_tok = torch.full((B, K + 1), -7, dtype=torch.int32, device="cuda")
        out_acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        rc = fn(P(g["target"]), P(g["draft"]), 1, P(g["draft_tok"]), P(g["verify_len"]),
                P(g["uniforms"]), B, K, V, 1.0, P(out_tok), P(out_acc),
                ctypes.c_void_p(stream.cuda_stream))
        assert rc == sv.SV_OK, sv.status_string(rc)
        torch.cuda.synchronize()
        if not check:
            assert int(out_acc[3]) == -1 and (out_tok[3] == -1).all()
            continue
        assert np.array_equal(out_acc.cpu().numpy(), ref_acc.cpu().numpy())
        assert np.array_equal(out_tok.cpu().numpy(), ref_tok.cpu().numpy())
