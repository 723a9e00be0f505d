"""Comparison rules between the CUDA path and the float64 oracle.

GEMM outputs:  |gpu - ref| <= 2 ulp_bf16(ref) + 1e-3 * sqrt(kc) * max|a| * max|b|
               (kc the contraction length, maxima over the whole operands);
               rows in [0, L) outside the local groups must be +0 bit for bit;
               rows >= L must keep the buffer's prior bits.
GLU epilogue:  1 ulp_bf16(ref) + |d glu/d g| * E + |d glu/d u| * E, E the GEMM
               absolute term, the derivatives taken in float64 at the oracle's
               gate and up; where exp(-g) overflows binary32 (g < -88.72) the
               result is a signed zero by the op sequence and compared as such.
Standalone GLU: within 1 ulp_bf16 of the float64 value where both are finite
               and exp(-g) stays finite in binary32; everywhere else the bits
               of the float32 op-sequence restatement (NaN matches any NaN).
"""
from __future__ import annotations

import math

import numpy as np

from oracle import bf16 as obf


def gemm_tol(ref, kc, amax, bmax):
    return 2.0 * obf.ulp(ref) + 1e-3 * math.sqrt(max(kc, 1)) * amax * bmax


def assert_close(got, ref, tol, what="", max_report=8):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    ok = (err <= tol) | (np.isnan(got) & np.isnan(ref)) | ((got == ref) & np.isinf(ref))
    if not np.all(ok):
        idx = np.argwhere(~ok)[:max_report]
        lines = [f"{tuple(i)}: got {got[tuple(i)]!r} ref {ref[tuple(i)]!r} tol {np.broadcast_to(tol, ref.shape)[tuple(i)]!r}"
                 for i in idx]
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} outside tolerance\n" + "\n".join(lines))


def exp_overflows_f32(g):
    with np.errstate(over="ignore", invalid="ignore"):
        return np.isinf(np.exp(-np.asarray(g, np.float64)).astype(np.float32))


def glu_epilogue_tol(g64, u64, E):
    """Tolerance of the fused GLU epilogue at the oracle's float64 gate/up values."""
    from oracle import glu as oglu

    ref = oglu.glu_fwd_f64(g64, u64)
    dg, du = oglu.glu_bwd_f64(g64, u64, 1.0)   # d glu / d g, d glu / d u (= silu)
    with np.errstate(invalid="ignore"):
        tol = obf.ulp(ref) + np.abs(dg) * E + np.abs(du) * E
    return ref, np.nan_to_num(tol, nan=np.inf, posinf=np.inf)
