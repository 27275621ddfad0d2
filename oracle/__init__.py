"""Plain float64 CPU oracle for batched speculative verification (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package. The CUDA library never touches it, and it never touches
the CUDA library: the two share no code. The arithmetic lives in ``sv_oracle.c``
(sequential float64 loops, one element at a time); this module compiles it with
gcc and marshals numpy arrays through ctypes.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
(brute-force output distribution at small V, greedy argmax, q == p, closed-form
acceptance rate, hand-computed golden cases, schedule invariants and brute force;
calibration by the power-form identity and its fixed points, the load-aware threshold
by its end points, the window statistics by brute-force counting and hand cases).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

FLAG_ACCEPT_TIE = 1
FLAG_CDF_EDGE = 2
FLAG_TINY_PROB = 4
FLAG_SMALL_RESIDUAL = 8
FLAG_INVALID = 16
NEAR_TIE_MASK = FLAG_ACCEPT_TIE | FLAG_CDF_EDGE | FLAG_TINY_PROB | FLAG_SMALL_RESIDUAL

OK, ERR_ARG, ERR_INPUT = 0, -1, -5


def build(force: bool = False) -> str:
    """Compile sv_oracle.c into liboracle.so (plain C, -O2, OpenMP over requests)."""
    with _lock:
        if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
        ):
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", _SRC, "-o", tmp, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path):
    """Open a compiled oracle and declare its signatures."""
    lib = ctypes.CDLL(path)
    vp, i32p, f64p, f32p = (ctypes.c_void_p,) * 4
    lib.oracle_schedule.argtypes = [f32p, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                    ctypes.c_longlong, i32p, f64p, i32p]
    lib.oracle_schedule.restype = ctypes.c_int
    common = [vp, vp, ctypes.c_int, i32p, i32p]
    tail = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
    outs = [i32p, i32p, f64p, f64p, i32p, ctypes.c_int]
    lib.oracle_verify.argtypes = common + [f32p] + tail + [ctypes.c_float] + outs
    lib.oracle_verify.restype = ctypes.c_int
    lib.oracle_verify_u64.argtypes = common + [f64p] + tail + [ctypes.c_double] + outs
    lib.oracle_verify_u64.restype = ctypes.c_int
    outs_m = [i32p, i32p, f64p, f64p, i32p, f64p, ctypes.c_int]
    lib.oracle_verify_m.argtypes = common + [f32p] + tail + [ctypes.c_float] + outs_m
    lib.oracle_verify_m.restype = ctypes.c_int
    lib.oracle_verify_u64m.argtypes = common + [f64p] + tail + [ctypes.c_double] + outs_m
    lib.oracle_verify_u64m.restype = ctypes.c_int
    lib.oracle_calibrate.argtypes = [ctypes.c_double, ctypes.c_double]
    lib.oracle_calibrate.restype = ctypes.c_double
    lib.oracle_load_tau.argtypes = [f32p, ctypes.c_double, ctypes.c_double]
    lib.oracle_load_tau.restype = ctypes.c_double
    lib.oracle_schedule_ex.argtypes = [f32p, f32p, f32p, ctypes.c_float, ctypes.c_float,
                                       ctypes.c_float, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_longlong, i32p, f64p, i32p, f32p, f64p]
    lib.oracle_schedule_ex.restype = ctypes.c_int
    lib.oracle_calib_observe.argtypes = [f32p, i32p, i32p, ctypes.c_int, ctypes.c_int, f64p]
    lib.oracle_calib_observe.restype = ctypes.c_int
    lib.oracle_calib_update.argtypes = [f64p, f32p, ctypes.c_int, ctypes.c_double,
                                        ctypes.c_double, f64p]
    lib.oracle_calib_update.restype = ctypes.c_int
    lib.oracle_markov_draft.argtypes = [vp, vp, vp, i32p, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, vp, i32p, f64p, f64p]
    lib.oracle_markov_draft.restype = ctypes.c_int
    lib.oracle_schedule_curve.argtypes = [f32p, f32p, f32p, ctypes.c_float, ctypes.c_float,
                                          ctypes.c_float, f32p, f32p, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_longlong, i32p, i32p, f64p]
    lib.oracle_schedule_curve.restype = ctypes.c_int
    tree = [vp, vp, ctypes.c_int, i32p, i32p, i32p]
    tree_outs = [i32p, i32p, i32p, i32p, f64p, ctypes.c_int]
    lib.oracle_verify_tree.argtypes = tree + [f32p] + tail + [ctypes.c_float] + tree_outs
    lib.oracle_verify_tree.restype = ctypes.c_int
    lib.oracle_verify_tree_u64.argtypes = tree + [f64p] + tail + [ctypes.c_double] + tree_outs
    lib.oracle_verify_tree_u64.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _bind(_LIB_PATH)
    return _lib


def build_variant(source_text: str, path: str):
    """Compile a modified copy of the oracle source to ``path`` and open it. Used only
    by the tests that plant a mistake in the oracle to show that the pins catch it."""
    src = path + ".c"
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", src, "-o", path,
                    "-lm"], check=True)
    return _bind(path)


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def schedule(conf, tau: float, token_budget: int, lib=None):
    """Confidence schedule. conf: [B,K] float32 in [0,1].

    Returns dict(out_len [B] int32, surv [B,K] float64, l0 [B] int32, status int).
    """
    conf = np.ascontiguousarray(conf, dtype=np.float32)
    B, K = conf.shape
    out_len = np.zeros(B, np.int32)
    surv = np.zeros((B, K), np.float64)
    l0 = np.zeros(B, np.int32)
    rc = (lib or _load()).oracle_schedule(_ptr(conf), B, K, float(tau), int(token_budget),
                                          _ptr(out_len), _ptr(surv), _ptr(l0))
    return {"out_len": out_len, "surv": surv, "l0": l0, "status": rc}


CALIB_BINS = 10


def calib_stats_len(K: int) -> int:
    """Length (float64) of the calibration window statistics for K positions."""
    return 3 * K + 3 * CALIB_BINS


def calibrate(c: float, T: float, lib=None) -> float:
    """One calibrated confidence sigmoid(logit(c) / T), float64."""
    return (lib or _load()).oracle_calibrate(float(c), float(T))


def load_tau(load, tau_min: float, tau_max: float, lib=None) -> float:
    """Load-aware threshold from {Q, Q_max, M_gpu, M_max} (float32); -1 if invalid."""
    ld = np.ascontiguousarray(load, dtype=np.float32)
    return (lib or _load()).oracle_load_tau(_ptr(ld), float(tau_min), float(tau_max))


def schedule_ex(conf, temps, load, tau: float, tau_min: float, tau_max: float,
                token_budget: int, lib=None):
    """Schedule on calibrated confidences (temps [K] or None) with an optional
    load-aware threshold (load [4] or None). Returns dict(out_len, surv, l0, cal, tau,
    status)."""
    conf = np.ascontiguousarray(conf, dtype=np.float32)
    B, K = conf.shape
    t = None if temps is None else np.ascontiguousarray(temps, dtype=np.float32)
    ld = None if load is None else np.ascontiguousarray(load, dtype=np.float32)
    out_len = np.zeros(B, np.int32)
    surv = np.zeros((B, K), np.float64)
    l0 = np.zeros(B, np.int32)
    cal = np.zeros((B, K), np.float32)
    tau_used = np.zeros(1, np.float64)
    rc = (lib or _load()).oracle_schedule_ex(
        _ptr(conf), _ptr(t), _ptr(ld), float(tau), float(tau_min), float(tau_max), B, K,
        int(token_budget), _ptr(out_len), _ptr(surv), _ptr(l0), _ptr(cal), _ptr(tau_used))
    return {"out_len": out_len, "surv": surv, "l0": l0, "cal": cal, "tau": float(tau_used[0]),
            "status": rc}


def calib_observe(conf_cal, verify_len, accepted, stats, lib=None):
    """Add one verification round to the window statistics (in place)."""
    c = np.ascontiguousarray(conf_cal, dtype=np.float32)
    B, K = c.shape
    vl = np.ascontiguousarray(verify_len, dtype=np.int32)
    ac = np.ascontiguousarray(accepted, dtype=np.int32)
    assert stats.dtype == np.float64 and stats.size == calib_stats_len(K)
    return (lib or _load()).oracle_calib_observe(_ptr(c), _ptr(vl), _ptr(ac), B, K, _ptr(stats))


def calib_update(stats, temps, lr: float, temp_floor: float, lib=None):
    """Window update of temps (float32 [K], in place); returns (status, ece)."""
    assert stats.dtype == np.float64 and temps.dtype == np.float32
    ece = np.zeros(1, np.float64)
    rc = (lib or _load()).oracle_calib_update(_ptr(stats), _ptr(temps), temps.size, float(lr),
                                              float(temp_floor), _ptr(ece))
    return rc, float(ece[0])


def schedule_curve(conf, temps, load, tau, tau_min, tau_max, curve_x, curve_y, token_budget,
                   lib=None):
    """Schedule whose budget is chosen from a throughput curve (curve_x ascending tokens,
    curve_y tokens/s). Returns dict(out_len, n, g, status)."""
    conf = np.ascontiguousarray(conf, dtype=np.float32)
    B, K = conf.shape
    t = None if temps is None else np.ascontiguousarray(temps, dtype=np.float32)
    ld = None if load is None else np.ascontiguousarray(load, dtype=np.float32)
    cx = np.ascontiguousarray(curve_x, dtype=np.float32)
    cy = np.ascontiguousarray(curve_y, dtype=np.float32)
    out_len = np.zeros(B, np.int32)
    n = np.zeros(1, np.int32)
    g = np.zeros(1, np.float64)
    rc = (lib or _load()).oracle_schedule_curve(
        _ptr(conf), _ptr(t), _ptr(ld), float(tau), float(tau_min), float(tau_max), _ptr(cx),
        _ptr(cy), cx.size, B, K, int(token_budget), _ptr(out_len), _ptr(n), _ptr(g))
    return {"out_len": out_len, "n": int(n[0]), "g": float(g[0]), "status": rc}


def markov_draft(logits, U, Vm, prev, lib=None):
    """Markov logit-bias drafting loop. logits [B,K,V], U and Vm [V,r]: bf16 as uint16
    bits; prev [B] int32. Returns dict(corrected [B,K,V] uint16 bits, tok [B,K] int32,
    edge [B,K], gap [B,K], status)."""
    L = np.ascontiguousarray(logits, dtype=np.uint16)
    Um = np.ascontiguousarray(U, dtype=np.uint16)
    Wm = np.ascontiguousarray(Vm, dtype=np.uint16)
    pv = np.ascontiguousarray(prev, dtype=np.int32)
    B, K, V = L.shape
    r = Um.shape[1]
    assert Um.shape == (V, r) and Wm.shape == (V, r) and pv.shape == (B,)
    corr = np.zeros_like(L)
    tok = np.zeros((B, K), np.int32)
    edge = np.zeros((B, K), np.float64)
    gap = np.zeros((B, K), np.float64)
    rc = (lib or _load()).oracle_markov_draft(_ptr(L), _ptr(Um), _ptr(Wm), _ptr(pv), B, K, V, r,
                                              _ptr(corr), _ptr(tok), _ptr(edge), _ptr(gap))
    return {"corrected": corr, "tok": tok, "edge": edge, "gap": gap, "status": rc}


def _logits(a):
    """numpy float32 -> (array, dtype 0); numpy uint16/int16 bf16 bits -> (array, 1)."""
    if a is None:
        return None, None
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return a, 0
    if a.dtype in (np.uint16, np.int16):
        return a.view(np.uint16), 1
    raise TypeError(f"logits must be float32 or bf16 bits (uint16), got {a.dtype}")


def verify(target, draft, draft_tok, verify_len, uniforms, temperature: float,
           nthreads: int = 1, diag: bool = True, u64: bool = False, lib=None):
    """Batched verification.

    target [B,K+1,V] and draft [B,K,V]: float32, or bf16 given as uint16 bit patterns.
    draft_tok [B,K] int32, verify_len [B] int32, uniforms [B,K+1] float32 (float64 when
    ``u64``; only the brute-force tests use that). Returns dict(out_tok, out_accepted,
    p, q, flags, margin, status); margin [B] is each request's smallest decision margin
    (the quantity the near-tie flags threshold).
    """
    t, dt = _logits(target)
    d, dd = _logits(draft)
    if d is not None and dd != dt:
        raise TypeError("target and draft logits must share a dtype")
    B, K1, V = t.shape
    K = K1 - 1
    tok = np.ascontiguousarray(draft_tok, dtype=np.int32)
    vlen = np.ascontiguousarray(verify_len, dtype=np.int32)
    u = None
    if uniforms is not None:
        u = np.ascontiguousarray(uniforms, dtype=np.float64 if u64 else np.float32)
    out_tok = np.zeros((B, K + 1), np.int32)
    out_acc = np.zeros(B, np.int32)
    p = np.zeros((B, K), np.float64) if diag else None
    q = np.zeros((B, K), np.float64) if diag else None
    flags = np.zeros(B, np.int32)
    margin = np.zeros(B, np.float64)
    lib = lib or _load()
    fn = lib.oracle_verify_u64m if u64 else lib.oracle_verify_m
    rc = fn(_ptr(t), _ptr(d), dt, _ptr(tok), _ptr(vlen), _ptr(u), B, K, V, float(temperature),
            _ptr(out_tok), _ptr(out_acc), _ptr(p), _ptr(q), _ptr(flags), _ptr(margin),
            int(nthreads))
    return {"out_tok": out_tok, "out_accepted": out_acc, "p": p, "q": q, "flags": flags,
            "margin": margin, "status": rc}


def verify_tree(target, draft, parent, draft_tok, n_nodes, uniforms, temperature: float,
                nthreads: int = 1, u64: bool = False, lib=None):
    """Batched tree verification (multi-candidate rejection sampling).

    target, draft [B,N,V]: float32, or bf16 as uint16 bit patterns (draft may be None
    at T == 0). parent, draft_tok [B,N] int32; n_nodes [B] int32; uniforms [B,N]
    float32 (float64 when ``u64``). Returns dict(out_tok [B,N], out_accepted [B],
    out_path [B,N], flags [B], margin [B], status).
    """
    t, dt = _logits(target)
    d, dd = _logits(draft)
    if d is not None and dd != dt:
        raise TypeError("target and draft logits must share a dtype")
    B, N, V = t.shape
    par = np.ascontiguousarray(parent, dtype=np.int32)
    tok = np.ascontiguousarray(draft_tok, dtype=np.int32)
    nn = np.ascontiguousarray(n_nodes, dtype=np.int32)
    u = None
    if uniforms is not None:
        u = np.ascontiguousarray(uniforms, dtype=np.float64 if u64 else np.float32)
    out_tok = np.zeros((B, N), np.int32)
    out_acc = np.zeros(B, np.int32)
    out_path = np.zeros((B, N), np.int32)
    flags = np.zeros(B, np.int32)
    margin = np.zeros(B, np.float64)
    lib = lib or _load()
    fn = lib.oracle_verify_tree_u64 if u64 else lib.oracle_verify_tree
    rc = fn(_ptr(t), _ptr(d), dt, _ptr(par), _ptr(tok), _ptr(nn), _ptr(u), B, N, V,
            float(temperature), _ptr(out_tok), _ptr(out_acc), _ptr(out_path), _ptr(flags),
            _ptr(margin), int(nthreads))
    return {"out_tok": out_tok, "out_accepted": out_acc, "out_path": out_path,
            "flags": flags, "margin": margin, "status": rc}
