"""The C-ABI library loads without a GPU, exports every symbol the header
declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rd.h")

RD_OK, RD_ERR_INVALID_ARG, RD_ERR_UNSUPPORTED, RD_ERR_CUDA = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    from expert_ffn_ragged_gb300 import build

    path = build.build()
    return ctypes.CDLL(path)


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rd_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_abi():
    assert _declared() == sorted([
        "rd_glu_bwd", "rd_glu_fwd", "rd_ragged_dot", "rd_ragged_dot_trans_rhs",
        "rd_get_tuning", "rd_ragged_dot_trans_rhs_glu_bwd", "rd_set_tuning", "rd_status_string",
        "rd_trans_ragged_dot", "rd_trans_ragged_dot_f32", "rd_trans_ragged_dot_no_alloc",
        "rd_trans_ragged_dot_workspace_size", "rd_unsort_bwd_rows"])


class _Tuning(ctypes.Structure):
    _fields_ = [("gemm_variant", ctypes.c_int32), ("band_rows", ctypes.c_int32),
                ("wait_timeout_ns", ctypes.c_uint64), ("reserved", ctypes.c_int32 * 2)]


def test_tuning_overrides_on_the_host(lib):
    """rd_set_tuning / rd_get_tuning need no GPU: set, read back, reject, reset."""
    lib.rd_set_tuning.restype = lib.rd_get_tuning.restype = ctypes.c_int
    lib.rd_set_tuning.argtypes = lib.rd_get_tuning.argtypes = [ctypes.c_void_p]
    t = _Tuning(2, 512, 99)
    assert lib.rd_set_tuning(ctypes.byref(t)) == RD_OK
    back = _Tuning()
    assert lib.rd_get_tuning(ctypes.byref(back)) == RD_OK
    assert (back.gemm_variant, back.band_rows, back.wait_timeout_ns) == (2, 512, 99)
    assert lib.rd_set_tuning(ctypes.byref(_Tuning(3, 0, 0))) == RD_ERR_INVALID_ARG
    assert lib.rd_set_tuning(ctypes.byref(_Tuning(0, -4, 0))) == RD_ERR_INVALID_ARG
    bad = _Tuning(0, 0, 0)
    bad.reserved[1] = 1
    assert lib.rd_set_tuning(ctypes.byref(bad)) == RD_ERR_INVALID_ARG
    assert lib.rd_get_tuning(ctypes.byref(back)) == RD_OK and back.band_rows == 512
    assert lib.rd_get_tuning(None) == RD_ERR_INVALID_ARG
    assert lib.rd_set_tuning(None) == RD_OK
    assert lib.rd_get_tuning(ctypes.byref(back)) == RD_OK
    assert (back.gemm_variant, back.band_rows, back.wait_timeout_ns) == (0, 0, 0)


def test_library_reads_no_environment():
    """No knob of the library hides in an environment variable (all are in rd.h)."""
    import glob
    for path in glob.glob(os.path.join(ROOT, "expert_ffn_ragged_gb300", "csrc", "*")):
        assert "getenv" not in open(path).read(), path


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True, text=True)
    exported = set(re.findall(r"\bT (rd_[a-z0-9_]+)\b", out.stdout))
    for name in _declared():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_status_strings(lib):
    lib.rd_status_string.restype = ctypes.c_char_p
    for code in range(4):
        assert lib.rd_status_string(code).startswith(b"RD_")
    assert b"unknown" in lib.rd_status_string(99)


def _gd(lib, *args):
    f = lib.rd_ragged_dot
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int64] * 3 + [ctypes.c_void_p] + \
        [ctypes.c_int32] * 3 + [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    return f(*args)


P = 0x10000   # fake, 16-byte aligned "device" addresses: never dereferenced on these paths


def test_forward_argument_checks(lib):
    ok = dict(lhs=P, rhs=P * 0x100, out=P * 0x10000, m=16, k=64, n=64, gs=P * 0x1000000,
              g_total=4, off=0, gl=4, limit=None, epi=0, status=None)

    def call(**kw):
        a = dict(ok, **kw)
        return _gd(lib, a["lhs"], a["rhs"], a["out"], a["m"], a["k"], a["n"], a["gs"], a["g_total"],
                   a["off"], a["gl"], a["limit"], a["epi"], a["status"], None)

    assert call(m=-1) == RD_ERR_INVALID_ARG
    assert call(gs=None) == RD_ERR_INVALID_ARG
    assert call(lhs=None) == RD_ERR_INVALID_ARG
    assert call(out=None) == RD_ERR_INVALID_ARG
    assert call(off=-1) == RD_ERR_INVALID_ARG
    assert call(off=2, gl=3) == RD_ERR_INVALID_ARG      # off + g_local > g_total
    assert call(gl=0) == RD_ERR_INVALID_ARG
    assert call(epi=7) == RD_ERR_INVALID_ARG
    assert call(out=ok["lhs"]) == RD_ERR_INVALID_ARG    # output aliases lhs
    assert call(k=12) == RD_ERR_UNSUPPORTED             # not a multiple of 8
    assert call(n=20) == RD_ERR_UNSUPPORTED
    assert call(lhs=P + 8) == RD_ERR_UNSUPPORTED        # misaligned
    assert call(g_total=2000, gl=4) == RD_ERR_UNSUPPORTED
    assert call(epi=1, n=24) == RD_ERR_UNSUPPORTED       # GLU half width 12 not a multiple of 8


def test_other_entry_points_check_arguments(lib):
    v, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    f = lib.rd_ragged_dot_trans_rhs
    f.restype = ctypes.c_int
    f.argtypes = [v, v, v, i64, i64, i64, v, i32, i32, i32, v, v, v]
    assert f(P, P * 0x100, P * 0x10000, 16, 64, 64, None, 4, 0, 4, None, None, None) == RD_ERR_INVALID_ARG
    assert f(P, P * 0x100, P * 0x10000, 16, 60, 64, P * 0x1000000, 4, 0, 4, None, None, None) == RD_ERR_UNSUPPORTED
    assert f(P, P * 0x100, P, 16, 64, 64, P * 0x1000000, 4, 0, 4, None, None, None) == RD_ERR_INVALID_ARG
    sz = ctypes.c_size_t
    f = lib.rd_trans_ragged_dot
    f.restype = ctypes.c_int
    f.argtypes = [v, v, v, i64, i64, i64, v, i32, i32, i32, v, v, sz, v, v]
    assert f(P, P * 0x100, P * 0x10000, 16, 64, 64, None, 4, 0, 4, None, None, 0, None, None) == RD_ERR_INVALID_ARG
    assert f(P, P * 0x100, P * 0x10000, 16, 60, 64, P * 0x1000000, 4, 0, 4, None, None, 0, None, None) == RD_ERR_UNSUPPORTED
    assert f(P, P * 0x100, P, 16, 64, 64, P * 0x1000000, 4, 0, 4, None, None, 0, None, None) == RD_ERR_INVALID_ARG
    # a workspace must be 128-byte aligned
    assert f(P, P * 0x100, P * 0x10000, 16, 64, 64, P * 0x1000000, 4, 0, 4, None, P * 0x3000 + 64, 1 << 20,
             None, None) == RD_ERR_UNSUPPORTED
    f = lib.rd_trans_ragged_dot_no_alloc
    f.restype = ctypes.c_int
    f.argtypes = [v, v, v, i64, i64, i64, v, i32, i32, i32, v, v, v]
    assert f(P, P * 0x100, P * 0x10000, 16, 64, 64, None, 4, 0, 4, None, None, None) == RD_ERR_INVALID_ARG
    assert f(P, P * 0x100, P * 0x10000, 16, 60, 64, P * 0x1000000, 4, 0, 4, None, None, None) == RD_ERR_UNSUPPORTED
    lib.rd_trans_ragged_dot_workspace_size.restype = ctypes.c_int
    lib.rd_trans_ragged_dot_workspace_size.argtypes = [v]
    assert lib.rd_trans_ragged_dot_workspace_size(None) == RD_ERR_INVALID_ARG
    f = lib.rd_ragged_dot_trans_rhs_glu_bwd
    f.restype = ctypes.c_int
    f.argtypes = [v, v, v, v, i64, i64, i64, v, i32, i32, i32, v, v, v]
    assert f(P, P * 0x100, None, P * 0x10000, 16, 64, 64, P * 0x1000000, 4, 0, 4, None, None, None) == RD_ERR_INVALID_ARG
    assert f(P, P * 0x100, P * 0x200, P * 0x200, 16, 64, 64, P * 0x1000000, 4, 0, 4, None, None, None) == RD_ERR_INVALID_ARG
    assert f(P, P * 0x100, P * 0x200, P * 0x10000, 16, 60, 64, P * 0x1000000, 4, 0, 4, None, None, None) == RD_ERR_UNSUPPORTED
    f = lib.rd_trans_ragged_dot_f32
    f.restype = ctypes.c_int
    f.argtypes = [v, v, v, i64, i64, i64, v, i32, i32, i32, v, i32, v, sz, v, v]
    assert f(P, P * 0x100, P * 0x10000, 16, 64, 64, P * 0x1000000, 4, 0, 4, None, 2, None, 0, None, None) == RD_ERR_INVALID_ARG
    assert f(P, P * 0x100, P * 0x10000, 16, 60, 64, P * 0x1000000, 4, 0, 4, None, 1, None, 0, None, None) == RD_ERR_UNSUPPORTED
    lib.rd_glu_fwd.restype = ctypes.c_int
    lib.rd_glu_fwd.argtypes = [v, v, i64, i64, v, v]
    assert lib.rd_glu_fwd(P, P * 0x100, 16, 12, None, None) == RD_ERR_UNSUPPORTED
    assert lib.rd_glu_fwd(None, P * 0x100, 16, 16, None, None) == RD_ERR_INVALID_ARG
    assert lib.rd_glu_fwd(P, P + 16, 16, 16, None, None) == RD_ERR_INVALID_ARG   # overlap
    lib.rd_glu_bwd.restype = ctypes.c_int
    lib.rd_glu_bwd.argtypes = [v, v, v, i64, i64, v, v]
    assert lib.rd_glu_bwd(P, P * 0x100, P, 16, 16, None, None) == RD_ERR_INVALID_ARG
    assert lib.rd_glu_bwd(P, P * 0x100, P * 0x10000, -1, 16, None, None) == RD_ERR_INVALID_ARG
    f = lib.rd_unsort_bwd_rows
    f.restype = ctypes.c_int
    f.argtypes = [v, v, v, v, v, i64, i64, v, v]
    assert f(P, P * 0x100, P * 0x200, P * 0x10000, P * 0x20000, 16, 12, None, None) == RD_ERR_UNSUPPORTED
    assert f(P, P * 0x100, None, P * 0x10000, P * 0x20000, 16, 16, None, None) == RD_ERR_INVALID_ARG
    assert f(P, P * 0x100, P * 0x200, P, P * 0x20000, 16, 16, None, None) == RD_ERR_INVALID_ARG
