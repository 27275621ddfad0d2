"""Python binding of libspecverify (GB300 / sm_103a).

Argument marshalling only: every step of the schedule and of verification runs in the
CUDA kernels of libspecverify.so, called through its C-ABI (include/specverify.h).
PyTorch provides device memory and streams. There is no CPU fallback: without the
built library, or without a CUDA device, calls raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

_lib = None

SV_OK, SV_ERR_ARG, SV_ERR_SHAPE, SV_ERR_DTYPE = 0, -1, -2, -3
SV_ERR_CUDA, SV_ERR_DEVICE_INPUT, SV_ERR_TIMEOUT, SV_ERR_WORKSPACE = -4, -5, -6, -7
SV_F32, SV_BF16 = 0, 1
SV_MAX_B, SV_MAX_K = 4096, 32


class SpecVerifyError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        super().__init__(f"{fn} failed: {status_string(code)} ({code})")


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Open libspecverify.so (building it first when it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing and not _build.up_to_date():
        _build.build()
    if not os.path.exists(_build.LIB):
        raise RuntimeError("libspecverify.so is not built; run __graft_entry__.build()")
    lib = ctypes.CDLL(_build.LIB)
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.sv_workspace_bytes.argtypes = [i32, i32, i32]
    lib.sv_workspace_bytes.restype = sz
    lib.sv_workspace_init.argtypes = [vp, sz, vp]
    lib.sv_workspace_init.restype = i32
    lib.sv_schedule.argtypes = [vp, i32, i32, f32, i32, vp, vp, sz, vp]
    lib.sv_schedule.restype = i32
    lib.sv_schedule_cal.argtypes = [vp, vp, vp, f32, f32, f32, i32, i32, i32, vp, vp, vp, vp, sz,
                                    vp]
    lib.sv_schedule_cal.restype = i32
    lib.sv_schedule_curve.argtypes = [vp, vp, vp, f32, f32, f32, vp, i32, i32, i32, i32, vp, vp,
                                      vp, vp, vp, vp, sz, vp]
    lib.sv_schedule_curve.restype = i32
    lib.sv_calib_stats_len.argtypes = [i32]
    lib.sv_calib_stats_len.restype = sz
    lib.sv_calib_observe.argtypes = [vp, vp, vp, i32, i32, vp, vp]
    lib.sv_calib_observe.restype = i32
    lib.sv_calib_update.argtypes = [vp, vp, i32, f32, f32, vp, vp]
    lib.sv_calib_update.restype = i32
    lib.sv_markov_keys_len.argtypes = [i32, i32]
    lib.sv_markov_keys_len.restype = sz
    lib.sv_markov_draft.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, sz, vp]
    lib.sv_markov_draft.restype = i32
    lib.sv_verify.argtypes = [vp, vp, i32, vp, vp, vp, i32, i32, i32, f32, vp, vp, vp, sz, vp]
    lib.sv_verify.restype = i32
    lib.sv_verify_diag.argtypes = [vp, vp, i32, vp, vp, vp, i32, i32, i32, f32, vp, vp, vp, vp,
                                   vp, vp, vp, vp, sz, vp]
    lib.sv_set_wait_limit.argtypes = [ctypes.c_longlong]
    lib.sv_set_wait_limit.restype = ctypes.c_longlong
    lib.sv_verify_diag.restype = i32
    lib.sv_verify_tree.argtypes = [vp, vp, i32, vp, vp, vp, vp, i32, i32, i32, f32, vp, vp, vp,
                                   vp, sz, vp]
    lib.sv_verify_tree.restype = i32
    lib.sv_get_status.argtypes = [vp, vp, i32, ctypes.POINTER(ctypes.c_int32)]
    lib.sv_get_status.restype = i32
    lib.sv_status_string.argtypes = [i32]
    lib.sv_status_string.restype = ctypes.c_char_p
    lib.sv_version.argtypes = []
    lib.sv_version.restype = i32
    _lib = lib
    return lib


load_lib = load  # the library loader, for functions whose arguments shadow `load`


def status_string(code: int) -> str:
    return load().sv_status_string(int(code)).decode()


def _check(fn, code):
    if code != SV_OK:
        raise SpecVerifyError(fn, code)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t, name, dtype=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t


class Workspace:
    """Device workspace for shapes up to (B, K, V); zeroed once at creation (the
    constructor waits for the zeroing, so the workspace can be used on any stream)."""

    def __init__(self, B, K, V, device=None, stream=None):
        self.nbytes = int(load().sv_workspace_bytes(int(B), int(K), int(V)))
        if self.nbytes == 0:
            raise ValueError(f"unsupported workspace shape B={B} K={K} V={V}")
        self.buf = torch.empty(self.nbytes + 256, dtype=torch.uint8, device=device or "cuda")
        off = (-self.buf.data_ptr()) % 256
        self.t = self.buf[off: off + self.nbytes]
        _check("sv_workspace_init",
               load().sv_workspace_init(_ptr(self.t), self.nbytes, _stream(stream)))
        # The zeroing must be complete before a call on any other stream uses it.
        torch.cuda.synchronize(self.t.device)

    def status(self, stream=None, clear=False) -> int:
        out = ctypes.c_int32(0)
        _check("sv_get_status", load().sv_get_status(_ptr(self.t), _stream(stream), int(clear),
                                                     ctypes.byref(out)))
        return int(out.value)


def sv_schedule(conf, tau, token_budget, ws: Workspace, out_len=None, stream=None):
    """Verify lengths [B] int32 from confidences [B,K] float32 (see specverify.h)."""
    conf = _dev(conf, "conf", torch.float32)
    B, K = conf.shape
    if out_len is None:
        out_len = torch.empty(B, dtype=torch.int32, device=conf.device)
    _dev(out_len, "out_len", torch.int32)
    _check("sv_schedule", load().sv_schedule(_ptr(conf), B, K, float(tau), int(token_budget),
                                             _ptr(out_len), _ptr(ws.t), ws.nbytes,
                                             _stream(stream)))
    return out_len


def sv_schedule_cal(conf, temps, load, tau, tau_min, tau_max, token_budget, ws: Workspace,
                    out_len=None, conf_cal=None, tau_out=None, stream=None):
    """sv_schedule on calibrated confidences, optionally with the load-aware threshold
    (see specverify.h). temps [K] float32 or None; load [4] float32 or None. Returns
    (out_len, conf_cal, tau_out); conf_cal [B,K] float32 and tau_out [1] float64 are
    allocated when not given."""
    conf = _dev(conf, "conf", torch.float32)
    B, K = conf.shape
    if temps is not None:
        _dev(temps, "temps", torch.float32)
    if load is not None:
        _dev(load, "load", torch.float32)
    if out_len is None:
        out_len = torch.empty(B, dtype=torch.int32, device=conf.device)
    if conf_cal is None:
        conf_cal = torch.empty(B, K, dtype=torch.float32, device=conf.device)
    if tau_out is None:
        tau_out = torch.empty(1, dtype=torch.float64, device=conf.device)
    _dev(out_len, "out_len", torch.int32)
    _dev(conf_cal, "conf_cal", torch.float32)
    _dev(tau_out, "tau_out", torch.float64)
    _check("sv_schedule_cal", load_lib().sv_schedule_cal(
        _ptr(conf), _ptr(temps), _ptr(load), float(tau), float(tau_min), float(tau_max), B, K,
        int(token_budget), _ptr(out_len), _ptr(conf_cal), _ptr(tau_out), _ptr(ws.t), ws.nbytes,
        _stream(stream)))
    return out_len, conf_cal, tau_out


def sv_schedule_curve(conf, temps, load, tau, tau_min, tau_max, curve, token_budget,
                      ws: Workspace, out_len=None, stream=None):
    """Schedule whose budget is chosen from a throughput curve (see specverify.h).
    curve: [2, n_pts] float32 (tokens, tokens/s). Returns (out_len, n [1] int32,
    goodput [1] float64)."""
    conf = _dev(conf, "conf", torch.float32)
    B, K = conf.shape
    curve = _dev(curve, "curve", torch.float32)
    if curve.dim() != 2 or curve.shape[0] != 2:
        raise ValueError("curve must be [2, n_pts]")
    if temps is not None:
        _dev(temps, "temps", torch.float32)
    if load is not None:
        _dev(load, "load", torch.float32)
    dev = conf.device
    if out_len is None:
        out_len = torch.empty(B, dtype=torch.int32, device=dev)
    n_out = torch.empty(1, dtype=torch.int32, device=dev)
    g_out = torch.empty(1, dtype=torch.float64, device=dev)
    _check("sv_schedule_curve", load_lib().sv_schedule_curve(
        _ptr(conf), _ptr(temps), _ptr(load), float(tau), float(tau_min), float(tau_max),
        _ptr(curve), curve.shape[1], B, K, int(token_budget), _ptr(out_len), None, None,
        _ptr(n_out), _ptr(g_out), _ptr(ws.t), ws.nbytes, _stream(stream)))
    return out_len, n_out, g_out


def sv_calib_stats_len(K: int) -> int:
    """Length (float64) of the calibration window buffer for K positions."""
    return int(load_lib().sv_calib_stats_len(int(K)))


def sv_calib_observe(conf_cal, verify_len, accepted, stats, stream=None):
    """Add one verification round to the window stats (float64, in place)."""
    conf_cal = _dev(conf_cal, "conf_cal", torch.float32)
    B, K = conf_cal.shape
    _dev(verify_len, "verify_len", torch.int32)
    _dev(accepted, "accepted", torch.int32)
    _dev(stats, "stats", torch.float64)
    if stats.numel() != sv_calib_stats_len(K):
        raise ValueError("stats has the wrong length")
    _check("sv_calib_observe", load_lib().sv_calib_observe(
        _ptr(conf_cal), _ptr(verify_len), _ptr(accepted), B, K, _ptr(stats), _stream(stream)))


def sv_calib_update(stats, temps, lr, temp_floor, ece=None, stream=None):
    """Close the window: update temps [K] float32 in place, write the ECE into ece [1]
    float64 (allocated when not given) and zero stats. Returns ece."""
    _dev(stats, "stats", torch.float64)
    _dev(temps, "temps", torch.float32)
    K = temps.numel()
    if stats.numel() != sv_calib_stats_len(K):
        raise ValueError("stats has the wrong length")
    if ece is None:
        ece = torch.empty(1, dtype=torch.float64, device=temps.device)
    _dev(ece, "ece", torch.float64)
    _check("sv_calib_update", load_lib().sv_calib_update(
        _ptr(stats), _ptr(temps), K, float(lr), float(temp_floor), _ptr(ece), _stream(stream)))
    return ece


def sv_markov_draft(logits, U, Vm, prev_tok, ws: Workspace, corrected=None, draft_tok=None,
                    keys=None, stream=None):
    """Markov logit-bias head + greedy drafting loop (see specverify.h). logits [B,K,V]
    bf16, U and Vm [V,r] bf16, prev_tok [B] int32. Returns (corrected [B,K,V] bf16,
    draft_tok [B,K] int32)."""
    logits = _dev(logits, "logits", torch.bfloat16)
    U = _dev(U, "U", torch.bfloat16)
    Vm = _dev(Vm, "Vm", torch.bfloat16)
    prev_tok = _dev(prev_tok, "prev_tok", torch.int32)
    B, K, V = logits.shape
    r = U.shape[1]
    if tuple(U.shape) != (V, r) or tuple(Vm.shape) != (V, r):
        raise ValueError("U and Vm must be [V, r]")
    dev = logits.device
    if corrected is None:
        corrected = torch.empty_like(logits)
    if draft_tok is None:
        draft_tok = torch.empty((B, K), dtype=torch.int32, device=dev)
    if keys is None:
        keys = torch.empty(max(1, B * K), dtype=torch.int64, device=dev)
    _dev(corrected, "corrected", torch.bfloat16)
    _dev(draft_tok, "draft_tok", torch.int32)
    _dev(keys, "keys", torch.int64)
    _check("sv_markov_draft", load_lib().sv_markov_draft(
        _ptr(logits), _ptr(U), _ptr(Vm), _ptr(prev_tok), B, K, V, r, _ptr(corrected),
        _ptr(draft_tok), _ptr(keys), _ptr(ws.t), ws.nbytes, _stream(stream)))
    return corrected, draft_tok


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return SV_BF16
    if t.dtype == torch.float32:
        return SV_F32
    raise ValueError(f"logits must be bfloat16 or float32, got {t.dtype}")


def sv_verify(target, draft, draft_tok, verify_len, uniforms, temperature, ws: Workspace,
              out_tok=None, out_accepted=None, diag=False, accept_count=None,
              tested_count=None, stream=None):
    """Rejection-sampling verification (see specverify.h).

    target [B,K+1,V], draft [B,K,V] (bf16 or fp32; draft/uniforms may be None at T=0),
    draft_tok [B,K] int32, verify_len [B] int32, uniforms [B,K+1] float32.
    Returns (out_tok [B,K+1], out_accepted [B]) and, with diag=True, also (p, q) [B,K]
    and the near-tie flags [B] int32.
    """
    target = _dev(target, "target")
    B, K1, V = target.shape
    K = K1 - 1
    draft = _dev(draft, "draft", target.dtype)
    draft_tok = _dev(draft_tok, "draft_tok", torch.int32)
    verify_len = _dev(verify_len, "verify_len", torch.int32)
    uniforms = _dev(uniforms, "uniforms", torch.float32)
    dev = target.device
    if out_tok is None:
        out_tok = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    if out_accepted is None:
        out_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    lib = load()
    if diag or accept_count is not None or tested_count is not None:
        p = torch.empty((B, K), dtype=torch.float32, device=dev) if diag else None
        q = torch.empty((B, K), dtype=torch.float32, device=dev) if diag else None
        flags = torch.empty(B, dtype=torch.int32, device=dev) if diag else None
        rc = lib.sv_verify_diag(_ptr(target), _ptr(draft), _dtype_code(target), _ptr(draft_tok),
                                _ptr(verify_len), _ptr(uniforms), B, K, V, float(temperature),
                                _ptr(out_tok), _ptr(out_accepted), _ptr(p), _ptr(q),
                                _ptr(accept_count), _ptr(tested_count), _ptr(flags), _ptr(ws.t),
                                ws.nbytes, _stream(stream))
        _check("sv_verify_diag", rc)
        return (out_tok, out_accepted, p, q, flags) if diag else (out_tok, out_accepted)
    rc = lib.sv_verify(_ptr(target), _ptr(draft), _dtype_code(target), _ptr(draft_tok),
                       _ptr(verify_len), _ptr(uniforms), B, K, V, float(temperature),
                       _ptr(out_tok), _ptr(out_accepted), _ptr(ws.t), ws.nbytes, _stream(stream))
    _check("sv_verify", rc)
    return out_tok, out_accepted


def set_wait_limit(cycles: int) -> int:
    """Bound (GPU clock cycles) on a verify call's waits for other warps' results;
    cycles <= 0 restores the default. Returns the previous bound (a testing aid)."""
    return int(load().sv_set_wait_limit(int(cycles)))


def sv_verify_tree(target, draft, parent, draft_tok, n_nodes, uniforms, temperature,
                   ws: Workspace, out_tok=None, out_accepted=None, out_path=None,
                   want_path=True, stream=None):
    """Tree (multi-candidate) verification (see specverify.h).

    target, draft [B,N,V] (bf16 or fp32; draft/uniforms may be None at T=0), parent and
    draft_tok [B,N] int32, n_nodes [B] int32, uniforms [B,N] float32. Any workspace works
    (only its status word is used). Returns (out_tok [B,N], out_accepted [B], out_path
    [B,N] or None).
    """
    target = _dev(target, "target")
    B, N, V = target.shape
    draft = _dev(draft, "draft", target.dtype)
    parent = _dev(parent, "parent", torch.int32)
    draft_tok = _dev(draft_tok, "draft_tok", torch.int32)
    n_nodes = _dev(n_nodes, "n_nodes", torch.int32)
    uniforms = _dev(uniforms, "uniforms", torch.float32)
    dev = target.device
    if out_tok is None:
        out_tok = torch.empty((B, N), dtype=torch.int32, device=dev)
    if out_accepted is None:
        out_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    if out_path is None and want_path:
        out_path = torch.empty((B, N), dtype=torch.int32, device=dev)
    rc = load().sv_verify_tree(_ptr(target), _ptr(draft), _dtype_code(target), _ptr(parent),
                               _ptr(draft_tok), _ptr(n_nodes), _ptr(uniforms), B, N, V,
                               float(temperature), _ptr(out_tok), _ptr(out_accepted),
                               _ptr(out_path), _ptr(ws.t), ws.nbytes, _stream(stream))
    _check("sv_verify_tree", rc)
    return out_tok, out_accepted, out_path
