"""Oracle for the valid-rows unsort backward (test infrastructure only).

Source: MaxText PR #5760, "MoE wo FSDP sharding and valid-rows-only MoE
kernels", commit message (kernels/ragged/unsort_bwd_rows.py) and the review
comments on ``_unsort_bwd_rows_kernel``: for every row r below ``limit`` of the
packed buffer, the weighted gradient grad[r] = bf16(f32(g[r]) * w[r]) and the
f32 routing-weight row dot dot[r] = sum_c f32(g[r, c]) * f32(y[r, c]), where g
is the gathered output gradient, y the sorted tokens and w the per-row
routing weight.

Readings: rows at or past L = min(limit, rows) are
neither read nor written (the page's TPU kernel also zeroes the rest of
limit's 1024-row block, an artefact of its blocking that this library does
not copy); the dot is compared in float64 with the worst-case bound of any f32
summation order, since each product of two bf16 values is exact in f32.
"""
from __future__ import annotations

from typing import Optional

import numpy as np

from .bf16 import bits_to_f32, round_f32_to_bf16_bits


def unsort_bwd_rows(g, y, w, limit: Optional[int] = None):
    """Weighted gradient (bf16 bits) and row dot (float64) for rows below L.

    g, y: [rows, hidden] (bf16 values as float32/float64), w: [rows] float32.
    Returns (grad_bits uint16 [L, hidden], grad float32 [L, hidden],
    dot float64 [L]).
    """
    g32 = np.asarray(g, dtype=np.float32)
    y32 = np.asarray(y, dtype=np.float32)
    w32 = np.asarray(w, dtype=np.float32)
    rows = g32.shape[0]
    L = rows if limit is None else max(0, min(int(limit), rows))
    with np.errstate(over="ignore", invalid="ignore"):
        prod = g32[:L] * w32[:L, None]          # one f32 multiply per element
    bits = round_f32_to_bf16_bits(prod)       # one rounding to bf16
    dot = (g32[:L].astype(np.float64) * y32[:L].astype(np.float64)).sum(axis=1)
    return bits, bits_to_f32(bits), dot


def dot_tolerance(g, y, limit: Optional[int] = None):
    """Worst-case error of an f32 sum of the exact products, any order: gamma_n * sum|g*y|."""
    g64 = np.asarray(g, dtype=np.float64)
    y64 = np.asarray(y, dtype=np.float64)
    rows, hidden = g64.shape
    L = rows if limit is None else max(0, min(int(limit), rows))
    u = 2.0 ** -24
    gamma = hidden * u / (1.0 - hidden * u)
    return gamma * np.abs(g64[:L] * y64[:L]).sum(axis=1)
