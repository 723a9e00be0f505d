"""float64 oracle for the grouped GEMMs of the ragged_dot hot path.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources:

* SkyRL PR #867, "Integrate ragged_dot pallas kernel with group_offset
  support" -- review comment with the suggested ``fast_ragged_dot`` body
  (group boundaries from a cumulative sum with an initial zero, a valid-row
  mask for the local groups, zeros elsewhere), the ``trans_ragged_dot``
  backward fix (dx = ragged_dot(y, do, trans_rhs=True), dy = ragged_dot(x, do)),
  and ``_gpu_trans_ragged_dot_fwd`` (x [m,k], y [m,n], f32 accumulation).
* MaxText PR #5760, "MoE wo FSDP sharding and valid-rows-only MoE kernels" --
  commit message: only rows [0, limit) of the packed buffer hold tokens; the
  grouped matmuls skip the rest, and rows left unwritten are never read.

Readings taken where the pages are silent:

* L = min(limit, m) (limit absent => m).  Group boundaries are the exclusive
  prefix of the sizes, negative sizes taken as 0, every boundary clamped to L.
* Rows in [0, L) that are not in a local group are written as +0; rows >= L
  keep the output buffer's prior contents.
* A trans_ragged_dot group with no rows gives an all-zero block.
"""
from __future__ import annotations

from typing import Optional

import numpy as np

from .glu import glu_bwd_f64, glu_fwd_f64


def group_bounds(group_sizes, m: int, limit: Optional[int] = None):
    """Row boundaries of every group and the valid-row count L.

    Returns ``(b, L)`` with ``b[i] = min(sum(max(sizes[:i], 0)), L)`` for
    i = 0..g_total, i.e. the cumulative sum with an initial zero used by
    fast_ragged_dot, clamped to the valid rows.  Group i owns rows
    [b[i], b[i+1]).
    """
    L = m if limit is None else max(0, min(int(limit), m))
    sizes = np.maximum(np.asarray(group_sizes, dtype=np.int64), 0)
    b = np.concatenate([[0], np.cumsum(sizes)])
    return np.minimum(b, L), L


def _prior(out_prior, shape) -> np.ndarray:
    if out_prior is None:
        return np.full(shape, np.nan, dtype=np.float64)
    out = np.array(out_prior, dtype=np.float64, copy=True)
    assert out.shape == tuple(shape)
    return out


def ragged_dot(lhs, rhs, group_sizes, group_offset: int = 0, limit: Optional[int] = None,
               glu: bool = False, out_prior=None) -> np.ndarray:
    """Grouped forward: out[i] = lhs[i] @ rhs[group(i) - group_offset].

    lhs [m, k]; rhs [g_local, k, n]; group_sizes [g_total].  Only the local
    groups group_offset .. group_offset+g_local-1 are computed, against
    rhs[0..g_local); the other rows below L are zero.  With ``glu`` the
    fused [gate | up] result of width n is reduced to
    silu(gate) * up of width n/2 (float64).

    Returns the float64 output, unrounded; rows >= L are ``out_prior``
    (NaN when no prior buffer is given).
    """
    a = np.asarray(lhs, dtype=np.float64)
    w = np.asarray(rhs, dtype=np.float64)
    m, k = a.shape
    g_local, k2, n = w.shape
    assert k == k2
    g_total = len(group_sizes)
    assert 0 <= group_offset and group_offset + g_local <= g_total
    b, L = group_bounds(group_sizes, m, limit)
    n_out = n // 2 if glu else n
    out = _prior(out_prior, (m, n_out))
    out[:L] = 0.0
    for j in range(g_local):
        lo, hi = b[group_offset + j], b[group_offset + j + 1]
        if hi <= lo:
            continue
        acc = a[lo:hi] @ w[j]
        out[lo:hi] = glu_fwd_f64(acc[:, :n_out], acc[:, n_out:]) if glu else acc
    return out


def ragged_dot_trans_rhs(lhs, rhs, group_sizes, group_offset: int = 0,
                         limit: Optional[int] = None, out_prior=None) -> np.ndarray:
    """The trans_rhs form: out[i] = lhs[i] @ rhs[group(i) - group_offset]^T.

    lhs [m, n] (e.g. the output gradient), rhs [g_local, k, n] -> out [m, k].
    Same local-group, zero and limit rules as ``ragged_dot``.
    """
    a = np.asarray(lhs, dtype=np.float64)
    w = np.asarray(rhs, dtype=np.float64)
    m, n = a.shape
    g_local, k, n2 = w.shape
    assert n == n2
    b, L = group_bounds(group_sizes, m, limit)
    out = _prior(out_prior, (m, k))
    out[:L] = 0.0
    for j in range(g_local):
        lo, hi = b[group_offset + j], b[group_offset + j + 1]
        if hi <= lo:
            continue
        out[lo:hi] = a[lo:hi] @ w[j].T
    return out


def trans_ragged_dot(x, y, group_sizes, group_offset: int = 0, g_local: Optional[int] = None,
                     limit: Optional[int] = None) -> np.ndarray:
    """Per-group weight gradient: out[j] = x[rows_j]^T @ y[rows_j].

    x [m, k], y [m, n] -> out [g_local, k, n], float64.  rows_j are the rows
    of local group j (clamped to L); a group without rows gives zeros.
    """
    xa = np.asarray(x, dtype=np.float64)
    ya = np.asarray(y, dtype=np.float64)
    m, k = xa.shape
    m2, n = ya.shape
    assert m == m2
    g_total = len(group_sizes)
    if g_local is None:
        g_local = g_total - group_offset
    b, _ = group_bounds(group_sizes, m, limit)
    out = np.zeros((g_local, k, n), dtype=np.float64)
    for j in range(g_local):
        lo, hi = b[group_offset + j], b[group_offset + j + 1]
        if hi > lo:
            out[j] = xa[lo:hi].T @ ya[lo:hi]
    return out


def ragged_dot_adjusted(lhs, rhs, group_sizes, group_offset: int = 0) -> np.ndarray:
    """Second formulation of the offset forward, as fast_ragged_dot builds it.

    SkyRL PR #867, suggested fast_ragged_dot body: the tokens before the
    shard are folded into the first local group and the tokens after it into
    the last, a ragged_dot over all m rows runs with those adjusted sizes,
    and a valid-row mask then zeroes everything outside the shard.  No
    ``limit`` here (the page has none).  Used only to cross-check
    ``ragged_dot``.
    """
    a = np.asarray(lhs, dtype=np.float64)
    w = np.asarray(rhs, dtype=np.float64)
    m = a.shape[0]
    g_local = w.shape[0]
    sizes = np.asarray(group_sizes, dtype=np.int64)
    cum = np.concatenate([[0], np.cumsum(sizes)])
    shard_start, shard_end = cum[group_offset], cum[group_offset + g_local]
    adjusted = sizes[group_offset:group_offset + g_local].copy()
    adjusted[0] += shard_start
    adjusted[-1] += m - shard_end
    # plain ragged_dot over all rows with the adjusted sizes (no offset)
    full = ragged_dot(a, w, adjusted, 0, None)
    rows = np.arange(m)
    valid = (rows >= shard_start) & (rows < shard_end)
    return np.where(valid[:, None], full, 0.0)


def ragged_dot_trans_rhs_glu_bwd(d_out, rhs, fused, group_sizes, group_offset: int = 0,
                                 limit: Optional[int] = None):
    """SiLU-GLU backward of an expert FFN, through its down projection.

    Forward of the layer (per local group j): h = silu(gate) * up with
    [gate | up] = fused [m, 2f], then out = h @ rhs[j] with rhs [g_local, f, n].
    Given the output gradient d_out [m, n]: dh = d_out @ rhs[j]^T (the
    trans_rhs form, SkyRL PR #867 backward fix) and the GLU backward of
    MaxText PR #5760 (commit message: [d_gate | d_up] in one pass, recomputing
    the forward from the saved fused buffer).  Returns float64 [m, 2f]:
    [d_gate | d_up] on local rows, 0 on the other rows below L, NaN at or past L.
    """
    a = np.asarray(d_out, dtype=np.float64)
    fz = np.asarray(fused, dtype=np.float64)
    m, f2 = fz.shape
    f = f2 // 2
    dh = ragged_dot_trans_rhs(a, rhs, group_sizes, group_offset, limit)
    b, L = group_bounds(group_sizes, m, limit)
    g_local = np.asarray(rhs).shape[0]
    out = np.full((m, 2 * f), np.nan)
    out[:L] = 0.0
    lo, hi = b[group_offset], b[group_offset + g_local]
    if hi > lo:
        d_gate, d_up = glu_bwd_f64(fz[lo:hi, :f], fz[lo:hi, f:], dh[lo:hi])
        out[lo:hi, :f] = d_gate
        out[lo:hi, f:] = d_up
    return out


def trans_ragged_dot_f32(x, y, group_sizes, group_offset: int = 0, g_local: Optional[int] = None,
                         limit: Optional[int] = None, out_prior=None) -> np.ndarray:
    """trans_ragged_dot kept in f32 precision, optionally accumulated into a prior buffer.

    The page's _gpu_trans_ragged_dot_fwd takes ``acc_dtype`` (f32) separately
    from the compute dtype (SkyRL PR #867); keeping the f32 result, and adding
    it to an existing gradient buffer, is the accumulation a training step does
    across micro-batches.  Returns float64: ``out_prior + x^T y`` per local
    group (``out_prior`` = 0 when absent); a group without rows leaves its
    prior block unchanged.
    """
    d = trans_ragged_dot(x, y, group_sizes, group_offset, g_local, limit)
    if out_prior is None:
        return d
    prior = np.asarray(out_prior, dtype=np.float64)
    assert prior.shape == d.shape
    return prior + d


def f32_sum_bound(x, y, group_sizes, group_offset: int = 0, g_local: Optional[int] = None,
                  limit: Optional[int] = None) -> np.ndarray:
    """Worst-case error of an f32 accumulation of the exact products, any order.

    Each product of two bf16 values is exact in f32; a sum of kc such terms
    in f32 with any association order errs by at most kc * u * sum|x*y| with
    u = 2^-23 (twice the round-to-nearest unit, so that truncating adders are
    covered as well).
    """
    xa = np.abs(np.asarray(x, dtype=np.float64))
    ya = np.abs(np.asarray(y, dtype=np.float64))
    m, k = xa.shape
    n = ya.shape[1]
    if g_local is None:
        g_local = len(group_sizes) - group_offset
    b, _ = group_bounds(group_sizes, m, limit)
    out = np.zeros((g_local, k, n))
    for j in range(g_local):
        lo, hi = b[group_offset + j], b[group_offset + j + 1]
        if hi > lo:
            out[j] = (hi - lo) * 2.0 ** -23 * (xa[lo:hi].T @ ya[lo:hi])
    return out
