"""CPU checks of the C-ABI library: it builds, loads without a GPU, and exports every
function that include/*.h declares; host-side argument checks reject bad calls before
anything touches a device."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(sv_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    import speculative_decoding_verification_79_gb300 as sv

    return sv.load()


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("sv_schedule", "sv_verify", "sv_verify_diag", "sv_workspace_bytes",
              "sv_workspace_init", "sv_get_status", "sv_status_string", "sv_version",
              "sv_schedule_cal", "sv_calib_stats_len", "sv_calib_observe", "sv_calib_update",
              "sv_markov_keys_len", "sv_markov_draft", "sv_schedule_curve", "sv_verify_tree",
              "sv_verify_static", "sv_set_wait_limit"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    import speculative_decoding_verification_79_gb300 as sv

    out = subprocess.run(["nm", "-D", "--defined-only", sv.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if ln.strip()}
    missing = _declared() - exported
    assert not missing, missing
    for n in _declared():
        assert hasattr(lib, n)


def test_host_argument_checks(lib):
    """Rejected before any device work; no GPU is needed for these."""
    import speculative_decoding_verification_79_gb300 as sv

    assert lib.sv_workspace_bytes(64, 8, 151936) > 0
    assert lib.sv_workspace_bytes(-1, 8, 10) == 0
    assert lib.sv_workspace_bytes(4, 0, 10) == 0
    assert lib.sv_workspace_bytes(4, 33, 10) == 0
    fake = ctypes.c_void_p(256)  # never dereferenced: every call below fails its checks first
    n = lib.sv_workspace_bytes(4, 4, 100)
    args = lambda dt=1, B=4, K=4, V=100, T=1.0, ws=fake, nb=n, tgt=fake, drf=fake: (  # noqa: E731
        tgt, drf, dt, fake, fake, fake, B, K, V, T, fake, fake, ws, nb, None)
    assert lib.sv_verify(*args(dt=7)) == sv.SV_ERR_DTYPE
    assert lib.sv_verify(*args(K=0)) == sv.SV_ERR_SHAPE
    assert lib.sv_verify(*args(K=33)) == sv.SV_ERR_SHAPE
    assert lib.sv_verify(*args(B=5000)) == sv.SV_ERR_SHAPE
    for T in (-1.0, float("nan"), float("inf"), 1e-9):
        assert lib.sv_verify(*args(T=T)) == sv.SV_ERR_ARG
    assert lib.sv_verify(*args(nb=n - 1)) == sv.SV_ERR_WORKSPACE
    assert lib.sv_verify(*args(ws=ctypes.c_void_p(264))) == sv.SV_ERR_WORKSPACE
    assert lib.sv_verify(*args(tgt=None)) == sv.SV_ERR_ARG
    assert lib.sv_verify(*args(drf=None)) == sv.SV_ERR_ARG
    assert lib.sv_verify(*args(dt=0, tgt=ctypes.c_void_p(258))) == sv.SV_ERR_ARG
    assert lib.sv_verify(*args(B=0)) == sv.SV_OK
    diag = lambda flags=fake: (fake, fake, 1, fake, fake, fake, 4, 4, 100, 1.0, fake, fake,  # noqa: E731
                               None, None, None, None, flags, fake, n, None)
    assert lib.sv_verify_diag(*diag(flags=ctypes.c_void_p(258))) == sv.SV_ERR_ARG
    assert lib.sv_schedule(fake, 4, 4, 1.5, 10, fake, fake, n, None) == sv.SV_ERR_ARG
    assert lib.sv_schedule(fake, 4, 4, float("nan"), 10, fake, fake, n, None) == sv.SV_ERR_ARG
    assert lib.sv_schedule(fake, 4, 4, 0.3, -1, fake, fake, n, None) == sv.SV_ERR_ARG
    assert lib.sv_schedule(fake, 9000, 1, 0.3, 10, fake, fake, n, None) == sv.SV_ERR_SHAPE
    assert lib.sv_schedule(fake, 4096, 8, 0.3, 10, fake, fake, n, None) == sv.SV_ERR_SHAPE
    assert lib.sv_schedule(fake, 4, 4, 0.3, 10, fake, None, n, None) == sv.SV_ERR_WORKSPACE
    assert lib.sv_schedule(fake, 0, 4, 0.3, 10, fake, fake, n, None) == sv.SV_OK
    assert sv.status_string(sv.SV_ERR_TIMEOUT) == "device wait timed out"


def test_workspace_fits_every_smaller_shape(lib):
    """A workspace sized for (B, K, V) holds the layout of any call with B' <= B,
    K' <= K, V' <= V (calls of different shapes may share it)."""
    import itertools

    shapes = list(itertools.product((1, 7, 64, 512, 4096), (1, 3, 8, 32), (1, 999, 151936)))
    size = {sh: lib.sv_workspace_bytes(*sh) for sh in shapes}
    for a in shapes:
        for b in shapes:
            if all(x <= y for x, y in zip(a, b)):
                assert size[a] <= size[b], (a, b)


def test_static_entry_and_wait_limit_host_side(lib):
    """sv_verify_static checks its arguments before any device work (an empty batch
    needs no GPU); sv_set_wait_limit returns the previous bound."""
    import speculative_decoding_verification_79_gb300 as sv

    fn = lib.sv_verify_static
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [vp, vp, i32, vp, vp, vp, i32, i32, i32, ctypes.c_float, vp, vp, vp]
    fn.restype = i32
    fake = ctypes.c_void_p(256)
    args = lambda dt=1, B=4, K=4, V=100, T=1.0: (  # noqa: E731
        fake, fake, dt, fake, fake, fake, B, K, V, T, fake, fake, None)
    assert fn(*args(B=0)) == sv.SV_OK
    assert fn(*args(B=0, dt=7)) == sv.SV_ERR_DTYPE
    assert fn(*args(B=0, T=-1.0)) == sv.SV_ERR_ARG
    assert fn(*args(K=33)) == sv.SV_ERR_SHAPE
    assert fn(*args(B=4096, K=32, V=1 << 20)) == sv.SV_ERR_WORKSPACE
    prev = lib.sv_set_wait_limit(12345)
    assert lib.sv_set_wait_limit(prev) == 12345
    assert lib.sv_set_wait_limit(0) == prev
    assert lib.sv_set_wait_limit(0) == 4000000000


def test_no_fallback_without_cuda():
    """The product path fails loudly when CUDA is unavailable (no CPU fallback)."""
    import torch

    import speculative_decoding_verification_79_gb300 as sv

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(Exception):
        sv.Workspace(4, 4, 100)


def test_calibration_host_checks(lib):
    """The calibration entry points reject bad calls before any device work."""
    import speculative_decoding_verification_79_gb300 as sv

    fake = ctypes.c_void_p(256)
    n = lib.sv_workspace_bytes(4, 4, 100)
    assert lib.sv_calib_stats_len(8) == 3 * 8 + 3 * 10
    assert lib.sv_calib_stats_len(0) == 0 and lib.sv_calib_stats_len(33) == 0
    cal = lambda tau=0.3, tmin=0.2, tmax=0.75, load=None, B=4, K=4, ws=fake: (  # noqa: E731
        fake, None, load, tau, tmin, tmax, B, K, 10, fake, None, None, ws, n, None)
    assert lib.sv_schedule_cal(*cal(tau=1.5)) == sv.SV_ERR_ARG
    assert lib.sv_schedule_cal(*cal(load=fake, tmax=1.5)) == sv.SV_ERR_ARG
    assert lib.sv_schedule_cal(*cal(load=fake, tmin=float("nan"))) == sv.SV_ERR_ARG
    assert lib.sv_schedule_cal(*cal(K=33)) == sv.SV_ERR_SHAPE
    assert lib.sv_schedule_cal(*cal(ws=None)) == sv.SV_ERR_WORKSPACE
    assert lib.sv_schedule_cal(*cal(B=0)) == sv.SV_OK
    assert lib.sv_calib_observe(fake, fake, fake, 4, 0, fake, None) == sv.SV_ERR_SHAPE
    assert lib.sv_calib_observe(fake, fake, fake, 5000, 4, fake, None) == sv.SV_ERR_SHAPE
    assert lib.sv_calib_observe(None, fake, fake, 4, 4, fake, None) == sv.SV_ERR_ARG
    assert lib.sv_calib_observe(fake, fake, fake, 0, 4, fake, None) == sv.SV_OK
    assert lib.sv_calib_update(fake, fake, 4, 0.01, 0.0, None, None) == sv.SV_ERR_ARG
    assert lib.sv_calib_update(fake, fake, 4, float("inf"), 0.05, None, None) == sv.SV_ERR_ARG
    assert lib.sv_calib_update(fake, None, 4, 0.01, 0.05, None, None) == sv.SV_ERR_ARG
    assert lib.sv_calib_update(fake, fake, 40, 0.01, 0.05, None, None) == sv.SV_ERR_SHAPE


def test_markov_host_checks(lib):
    import speculative_decoding_verification_79_gb300 as sv

    fake = ctypes.c_void_p(256)
    n = lib.sv_workspace_bytes(4, 4, 100)
    args = lambda B=4, K=4, V=100, r=64, lg=fake, ws=fake: (  # noqa: E731
        lg, fake, fake, fake, B, K, V, r, fake, fake, fake, ws, n, None)
    assert lib.sv_markov_keys_len(64, 8) == 512 and lib.sv_markov_keys_len(64, 0) == 0
    assert lib.sv_markov_draft(*args(r=24)) == sv.SV_ERR_SHAPE
    assert lib.sv_markov_draft(*args(r=512)) == sv.SV_ERR_SHAPE
    assert lib.sv_markov_draft(*args(K=0)) == sv.SV_ERR_SHAPE
    assert lib.sv_markov_draft(*args(ws=None)) == sv.SV_ERR_WORKSPACE
    assert lib.sv_markov_draft(*args(lg=None)) == sv.SV_ERR_ARG
    assert lib.sv_markov_draft(*args(lg=ctypes.c_void_p(264))) == sv.SV_ERR_ARG
    assert lib.sv_markov_draft(*args(B=0)) == sv.SV_OK


def test_curve_host_checks(lib):
    import speculative_decoding_verification_79_gb300 as sv

    fake = ctypes.c_void_p(256)
    n = lib.sv_workspace_bytes(4, 4, 100)
    args = lambda curve=fake, npts=4, B=4, K=4: (  # noqa: E731
        fake, None, None, 0.3, 0.2, 0.75, curve, npts, B, K, 10, fake, None, None, None, None,
        fake, n, None)
    assert lib.sv_schedule_curve(*args(curve=None)) == sv.SV_ERR_ARG
    assert lib.sv_schedule_curve(*args(npts=0)) == sv.SV_ERR_SHAPE
    assert lib.sv_schedule_curve(*args(npts=65)) == sv.SV_ERR_SHAPE
    assert lib.sv_schedule_curve(*args(B=4096, K=4)) == sv.SV_ERR_SHAPE
    assert lib.sv_schedule_curve(*args(B=0)) == sv.SV_OK


def test_tree_host_checks(lib):
    import speculative_decoding_verification_79_gb300 as sv

    fake = ctypes.c_void_p(256)
    args = lambda dt=1, B=4, N=16, V=100, T=1.0, tgt=fake, drf=fake, uni=fake, ws=fake, nb=256, \
        path=fake: (tgt, drf, dt, fake, fake, fake, uni, B, N, V, T, fake, fake, path, ws, nb,
                    None)  # noqa: E731
    assert lib.sv_verify_tree(*args(dt=5)) == sv.SV_ERR_DTYPE
    assert lib.sv_verify_tree(*args(N=0)) == sv.SV_ERR_SHAPE
    assert lib.sv_verify_tree(*args(N=65)) == sv.SV_ERR_SHAPE
    assert lib.sv_verify_tree(*args(V=0)) == sv.SV_ERR_SHAPE
    assert lib.sv_verify_tree(*args(B=5000)) == sv.SV_ERR_SHAPE
    for T in (-1.0, float("nan"), float("inf"), 1e-9):
        assert lib.sv_verify_tree(*args(T=T)) == sv.SV_ERR_ARG
    assert lib.sv_verify_tree(*args(nb=255)) == sv.SV_ERR_WORKSPACE
    assert lib.sv_verify_tree(*args(ws=ctypes.c_void_p(264))) == sv.SV_ERR_WORKSPACE
    assert lib.sv_verify_tree(*args(tgt=None)) == sv.SV_ERR_ARG
    assert lib.sv_verify_tree(*args(drf=None)) == sv.SV_ERR_ARG
    assert lib.sv_verify_tree(*args(uni=None)) == sv.SV_ERR_ARG
    assert lib.sv_verify_tree(*args(dt=0, tgt=ctypes.c_void_p(258))) == sv.SV_ERR_ARG
    assert lib.sv_verify_tree(*args(path=ctypes.c_void_p(258))) == sv.SV_ERR_ARG
    assert lib.sv_verify_tree(*args(B=0)) == sv.SV_OK
