"""SiLU-GLU forward and backward for the oracle (test infrastructure only).

Source: MaxText PR #5760, "MoE wo FSDP sharding and valid-rows-only MoE
kernels", commit message, kernels/ragged/glu_rows.py: silu(gate) * up over
the rows below ``limit``, gate and up read in place from the fused
[gate | up] buffer, computed in f32 with XLA's op sequence (negate, exp, +1,
divide, multiply) and rounded only at the output; the backward writes
[d_gate | d_up] in one pass with "the -0 -> +0 fix".

Two forms of each:

* ``*_f64`` -- the mathematical value in float64 (what results are compared
  against, with a bf16-ulp tolerance);
* ``*_f32`` -- the float32 op sequence that the page fixes for the forward
  and that this library fixes for the backward (the page gives no backward
  formula), rounded once to bf16.  It defines the special values (NaN, +-inf,
  signed zeros) that the GPU must reproduce bit for bit.

Readings: silu(g) = g / (1 + exp(-g)) with a single
divide; the backward uses sig = 1/(1+exp(-g)), d_up = d * silu(g) and
d_gate = (d*u) * (sig * (1 + g*(1 - sig))); the "-0 -> +0 fix" turns every
backward output that rounds to -0 into +0.  ``exp`` in the f32 form is the
float64 exponential rounded to float32 (a correctly rounded f32 exp except
for vanishingly rare double-rounding cases).
"""
from __future__ import annotations

import numpy as np

from .bf16 import bits_to_f32, round_f32_to_bf16_bits


def _exp_f32(x32: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore", under="ignore", invalid="ignore"):
        return np.exp(x32.astype(np.float64)).astype(np.float32)


def glu_fwd_f64(gate, up) -> np.ndarray:
    """silu(gate) * up in float64: gate / (1 + exp(-gate)) * up."""
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        g = np.asarray(gate, dtype=np.float64)
        u = np.asarray(up, dtype=np.float64)
        return g / (1.0 + np.exp(-g)) * u


def glu_bwd_f64(gate, up, d):
    """Gradients of silu(gate) * up for an output gradient d, in float64.

    Returns (d_gate, d_up) with d_up = d * silu(g) and
    d_gate = d * u * sig(g) * (1 + g * (1 - sig(g))), sig the logistic.
    """
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        g = np.asarray(gate, dtype=np.float64)
        u = np.asarray(up, dtype=np.float64)
        dd = np.asarray(d, dtype=np.float64)
        sig = 1.0 / (1.0 + np.exp(-g))
        d_up = dd * (g * sig)
        d_gate = dd * u * (sig * (1.0 + g * (1.0 - sig)))
    return d_gate, d_up


def glu_fwd_f32(gate, up):
    """The float32 op sequence of the GLU forward, rounded once to bf16.

    e = exp(-g); den = 1 + e; s = g / den; r = s * u; bf16(r).
    Returns (bf16 bits as uint16, the bf16 values as float32).
    """
    g = np.asarray(gate, dtype=np.float32)
    u = np.asarray(up, dtype=np.float32)
    with np.errstate(over="ignore", invalid="ignore", divide="ignore", under="ignore"):
        e = _exp_f32(-g)
        den = np.float32(1.0) + e
        s = g / den
        r = s * u
    bits = round_f32_to_bf16_bits(r)
    return bits, bits_to_f32(bits)


def glu_bwd_f32(gate, up, d):
    """The float32 op sequence of the GLU backward, rounded once to bf16.

    e = exp(-g); den = 1 + e; sig = 1 / den; silu = g / den;
    d_up = d * silu; dsil = sig * (1 + g * (1 - sig)); d_gate = (d * u) * dsil;
    each result rounded to bf16, then -0 -> +0.
    Returns ((d_gate bits, d_up bits), (d_gate f32, d_up f32)).
    """
    g = np.asarray(gate, dtype=np.float32)
    u = np.asarray(up, dtype=np.float32)
    dd = np.asarray(d, dtype=np.float32)
    one = np.float32(1.0)
    with np.errstate(over="ignore", invalid="ignore", divide="ignore", under="ignore"):
        e = _exp_f32(-g)
        den = one + e
        sig = one / den
        silu = g / den
        d_up = dd * silu
        dsil = sig * (one + g * (one - sig))
        d_gate = (dd * u) * dsil
    out_bits = []
    for r in (d_gate, d_up):
        bits = round_f32_to_bf16_bits(r)
        bits = np.where(bits == np.uint16(0x8000), np.uint16(0), bits).astype(np.uint16)
        out_bits.append(bits)
    return (out_bits[0], out_bits[1]), (bits_to_f32(out_bits[0]), bits_to_f32(out_bits[1]))
