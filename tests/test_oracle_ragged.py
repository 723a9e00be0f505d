"""Pins for the float64 grouped-GEMM oracle (CPU only).

Each pin checks the oracle against something other than itself: a
hand-worked example, a brute-force restatement with per-row group lookup,
a special case that reduces to a dense matmul, the boundary-absorbing
formulation of fast_ragged_dot, linear-algebra identities and finite
differences.  Planted-mistake tests at the end show that the pins catch a
dropped term, a wrong index and a transposed operand.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import ragged

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = json.load(open(os.path.join(HERE, "golden", "hand_examples.json")))


# --------------------------------------------------------------------------
# brute force: scalar loops, group of each row found by a linear scan
# --------------------------------------------------------------------------
def _group_of_row(i, sizes):
    start = 0
    for gi, s in enumerate(sizes):
        s = max(int(s), 0)
        if start <= i < start + s:
            return gi
        start += s
    return None


def brute_fwd(lhs, rhs, sizes, off, limit, glu=False, prior=np.nan):
    m, k = len(lhs), len(lhs[0])
    g_local, n = len(rhs), len(rhs[0][0])
    L = m if limit is None else max(0, min(limit, m))
    n_out = n // 2 if glu else n
    out = [[prior] * n_out for _ in range(m)]
    for i in range(L):
        grp = _group_of_row(i, sizes)
        for c in range(n_out):
            if grp is None or not (off <= grp < off + g_local):
                out[i][c] = 0.0
                continue
            w = rhs[grp - off]
            acc = 0.0
            for kk in range(k):
                acc += float(lhs[i][kk]) * float(w[kk][c])
            if glu:
                up = 0.0
                for kk in range(k):
                    up += float(lhs[i][kk]) * float(w[kk][c + n_out])
                acc = acc * (1.0 / (1.0 + math.exp(-acc))) * up
            out[i][c] = acc
    return np.array(out, dtype=np.float64)


def brute_trans_rhs(lhs, rhs, sizes, off, limit):
    m, n = len(lhs), len(lhs[0])
    g_local, k = len(rhs), len(rhs[0])
    L = m if limit is None else max(0, min(limit, m))
    out = [[np.nan] * k for _ in range(m)]
    for i in range(L):
        grp = _group_of_row(i, sizes)
        for c in range(k):
            if grp is None or not (off <= grp < off + g_local):
                out[i][c] = 0.0
                continue
            acc = 0.0
            for nn in range(n):
                acc += float(lhs[i][nn]) * float(rhs[grp - off][c][nn])
            out[i][c] = acc
    return np.array(out, dtype=np.float64)


def brute_trans_ragged(x, y, sizes, off, g_local, limit):
    m, k, n = len(x), len(x[0]), len(y[0])
    L = m if limit is None else max(0, min(limit, m))
    out = np.zeros((g_local, k, n))
    for j in range(g_local):
        for a in range(k):
            for b in range(n):
                acc = 0.0
                for i in range(L):
                    if _group_of_row(i, sizes) == off + j:
                        acc += float(x[i][a]) * float(y[i][b])
                out[j, a, b] = acc
    return out


def _rand_case(rng, m, k, n, g, n_empty=0):
    sizes = rng.multinomial(m, np.full(g, 1.0 / g)).astype(np.int32)
    if n_empty:
        sizes[rng.choice(g, n_empty, replace=False)] = 0
    lhs = rng.integers(-4, 5, size=(m, k)).astype(np.float64)
    rhs = rng.integers(-4, 5, size=(g, k, n)).astype(np.float64)
    return lhs, rhs, sizes


# --------------------------------------------------------------------------
# hand-worked golden values
# --------------------------------------------------------------------------
def test_hand_forward():
    lhs, rhs, gs = GOLDEN["lhs"], np.array(GOLDEN["rhs"], float), GOLDEN["group_sizes"]
    f = GOLDEN["forward"]
    np.testing.assert_array_equal(oracle.ragged_dot(lhs, rhs, gs), f["offset0"])
    np.testing.assert_array_equal(oracle.ragged_dot(lhs, rhs[2:3], gs, group_offset=2),
                                  f["offset2_glocal1"])
    prior = np.full((5, 2), 7.0)
    np.testing.assert_array_equal(oracle.ragged_dot(lhs, rhs, gs, limit=3, out_prior=prior),
                                  f["offset0_limit3_prior7"])


def test_hand_trans_rhs():
    t = GOLDEN["trans_rhs"]
    np.testing.assert_array_equal(
        oracle.ragged_dot_trans_rhs(t["lhs"], np.array(t["rhs"], float), t["group_sizes"]), t["out"])


def test_hand_trans_ragged_dot():
    t = GOLDEN["trans_ragged_dot"]
    np.testing.assert_array_equal(oracle.trans_ragged_dot(t["x"], t["y"], t["group_sizes"]), t["out"])


# --------------------------------------------------------------------------
# brute force on tiny inputs
# --------------------------------------------------------------------------
CASES = [
    # m, k, n, g, n_empty, off, g_local, limit
    (1, 1, 1, 1, 0, 0, 1, None),
    (9, 3, 4, 3, 1, 0, 3, None),
    (17, 4, 6, 5, 2, 1, 3, None),
    (23, 5, 4, 7, 2, 2, 4, 11),
    (30, 2, 8, 17, 6, 5, 9, 29),
    (12, 3, 2, 4, 0, 3, 1, 0),
    (12, 3, 2, 4, 0, 0, 4, 12),
]


@pytest.mark.parametrize("m,k,n,g,n_empty,off,gl,limit", CASES)
def test_brute_force_forward(m, k, n, g, n_empty, off, gl, limit):
    rng = np.random.default_rng(m * 31 + g)
    lhs, rhs, sizes = _rand_case(rng, m, k, n, g, n_empty)
    rhs_local = rhs[off:off + gl]
    want = brute_fwd(lhs.tolist(), rhs_local.tolist(), sizes.tolist(), off, limit)
    got = oracle.ragged_dot(lhs, rhs_local, sizes, group_offset=off, limit=limit)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(want))
    np.testing.assert_allclose(np.nan_to_num(got), np.nan_to_num(want), rtol=0, atol=1e-12)


@pytest.mark.parametrize("m,k,n,g,n_empty,off,gl,limit", CASES)
def test_brute_force_forward_glu(m, k, n, g, n_empty, off, gl, limit):
    n = 2 * n
    rng = np.random.default_rng(m * 37 + g)
    lhs, rhs, sizes = _rand_case(rng, m, k, n, g, n_empty)
    rhs = rhs * 0.25
    rhs_local = rhs[off:off + gl]
    want = brute_fwd(lhs.tolist(), rhs_local.tolist(), sizes.tolist(), off, limit, glu=True)
    got = oracle.ragged_dot(lhs, rhs_local, sizes, group_offset=off, limit=limit, glu=True)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(want))
    np.testing.assert_allclose(np.nan_to_num(got), np.nan_to_num(want), rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("m,k,n,g,n_empty,off,gl,limit", CASES)
def test_brute_force_trans_rhs(m, k, n, g, n_empty, off, gl, limit):
    rng = np.random.default_rng(m * 41 + g)
    lhs, rhs, sizes = _rand_case(rng, m, n, k, g, n_empty)   # lhs [m, n], rhs [g, n, k]
    rhs = np.ascontiguousarray(np.transpose(rhs, (0, 2, 1)))  # [g, k, n]
    rhs_local = rhs[off:off + gl]
    want = brute_trans_rhs(lhs.tolist(), rhs_local.tolist(), sizes.tolist(), off, limit)
    got = oracle.ragged_dot_trans_rhs(lhs, rhs_local, sizes, group_offset=off, limit=limit)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(want))
    np.testing.assert_allclose(np.nan_to_num(got), np.nan_to_num(want), rtol=0, atol=1e-12)


@pytest.mark.parametrize("m,k,n,g,n_empty,off,gl,limit", CASES)
def test_brute_force_trans_ragged_dot(m, k, n, g, n_empty, off, gl, limit):
    rng = np.random.default_rng(m * 43 + g)
    sizes = rng.multinomial(m, np.full(g, 1.0 / g)).astype(np.int32)
    if n_empty:
        sizes[rng.choice(g, n_empty, replace=False)] = 0
    x = rng.integers(-3, 4, size=(m, k)).astype(float)
    y = rng.integers(-3, 4, size=(m, n)).astype(float)
    want = brute_trans_ragged(x.tolist(), y.tolist(), sizes.tolist(), off, gl, limit)
    got = oracle.trans_ragged_dot(x, y, sizes, group_offset=off, g_local=gl, limit=limit)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_negative_and_overflowing_sizes():
    """Negative sizes count as 0; boundaries past m (or L) are clamped."""
    rng = np.random.default_rng(7)
    lhs = rng.standard_normal((10, 3))
    rhs = rng.standard_normal((4, 3, 2))
    sizes = np.array([3, -2, 5, 9], np.int32)   # sum of positives 17 > m = 10
    want = brute_fwd(lhs.tolist(), rhs.tolist(), sizes.tolist(), 0, 8)
    got = oracle.ragged_dot(lhs, rhs, sizes, limit=8)
    np.testing.assert_allclose(np.nan_to_num(got), np.nan_to_num(want), atol=1e-12)
    b, L = oracle.group_bounds(sizes, 10, 8)
    assert L == 8 and list(b) == [0, 3, 3, 8, 8]


# --------------------------------------------------------------------------
# special cases and invariants
# --------------------------------------------------------------------------
def test_single_group_is_dense_matmul():
    rng = np.random.default_rng(11)
    a, w = rng.standard_normal((40, 16)), rng.standard_normal((1, 16, 24))
    np.testing.assert_allclose(oracle.ragged_dot(a, w, [40]), a @ w[0], rtol=1e-13, atol=1e-13)
    do = rng.standard_normal((40, 24))
    np.testing.assert_allclose(oracle.ragged_dot_trans_rhs(do, w, [40]), do @ w[0].T, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(oracle.trans_ragged_dot(a, do, [40])[0], a.T @ do, rtol=1e-13, atol=1e-13)


def test_empty_groups_contribute_nothing():
    rng = np.random.default_rng(12)
    a, w = rng.standard_normal((50, 8)), rng.standard_normal((3, 8, 6))
    sizes = [20, 10, 20]
    ref = oracle.ragged_dot(a, w, sizes)
    # insert empty groups (with arbitrary weights) before, between and after
    w2 = np.concatenate([rng.standard_normal((1, 8, 6)), w[:1], rng.standard_normal((1, 8, 6)),
                         w[1:], rng.standard_normal((1, 8, 6))])
    sizes2 = [0, 20, 0, 10, 20, 0]
    np.testing.assert_array_equal(oracle.ragged_dot(a, w2, sizes2), ref)
    dw = oracle.trans_ragged_dot(a, a[:, :6], sizes2)
    assert np.all(dw[0] == 0) and np.all(dw[2] == 0) and np.all(dw[5] == 0)


def test_offset_equals_restricted_full_output():
    rng = np.random.default_rng(13)
    m, g = 64, 8
    a, w = rng.standard_normal((m, 8)), rng.standard_normal((g, 8, 4))
    sizes = rng.multinomial(m - 5, np.full(g, 1.0 / g))
    full = oracle.ragged_dot(a, w, sizes)
    b, _ = oracle.group_bounds(sizes, m)
    for off, gl in [(0, 3), (3, 2), (5, 3), (7, 1)]:
        got = oracle.ragged_dot(a, w[off:off + gl], sizes, group_offset=off)
        want = np.zeros_like(full)
        want[b[off]:b[off + gl]] = full[b[off]:b[off + gl]]
        np.testing.assert_array_equal(got, want)


def test_adjusted_sizes_formulation_agrees():
    """The boundary-absorbing fast_ragged_dot formulation gives the same output."""
    rng = np.random.default_rng(14)
    for trial in range(20):
        m, g = int(rng.integers(1, 60)), int(rng.integers(1, 9))
        sizes = rng.multinomial(int(rng.integers(0, m + 1)), np.full(g, 1.0 / g))
        a, w = rng.standard_normal((m, 5)), rng.standard_normal((g, 5, 3))
        off = int(rng.integers(0, g))
        gl = int(rng.integers(1, g - off + 1))
        got = oracle.ragged_dot(a, w[off:off + gl], sizes, group_offset=off)
        want = oracle.ragged_dot_adjusted(a, w[off:off + gl], sizes, group_offset=off)
        np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-13)


def test_expert_parallel_shards_sum_to_full():
    rng = np.random.default_rng(15)
    m, g, shards = 96, 8, 4
    a, w = rng.standard_normal((m, 6)), rng.standard_normal((g, 6, 5))
    sizes = rng.multinomial(m, np.full(g, 1.0 / g))
    gl = g // shards
    full = oracle.ragged_dot(a, w, sizes)
    parts = [oracle.ragged_dot(a, w[r * gl:(r + 1) * gl], sizes, group_offset=r * gl) for r in range(shards)]
    np.testing.assert_allclose(sum(parts), full, rtol=1e-13, atol=1e-13)
    dw = oracle.trans_ragged_dot(a, full, sizes)
    dws = [oracle.trans_ragged_dot(a, full, sizes, group_offset=r * gl, g_local=gl) for r in range(shards)]
    np.testing.assert_array_equal(np.concatenate(dws), dw)


def test_rows_at_or_above_limit_keep_prior():
    rng = np.random.default_rng(16)
    a, w = rng.standard_normal((30, 4)), rng.standard_normal((2, 4, 3))
    prior = rng.standard_normal((30, 3))
    for limit in [0, 1, 17, 29, 30, 45]:
        got = oracle.ragged_dot(a, w, [12, 18], limit=limit, out_prior=prior)
        L = min(limit, 30)
        np.testing.assert_array_equal(got[L:], prior[L:])
        # rows >= L of the input do not matter
        a2 = a.copy()
        a2[L:] = np.nan
        got2 = oracle.ragged_dot(a2, w, [12, 18], limit=limit, out_prior=prior)
        np.testing.assert_array_equal(got2, got)


def test_adjoint_identity():
    """<fwd(x, w), do> = <x, dx(do, w)> = <w, dw(x, do)> on local rows."""
    rng = np.random.default_rng(17)
    m, k, n, g = 70, 9, 7, 6
    sizes = rng.multinomial(m - 4, np.full(g, 1.0 / g))
    x, w, do = rng.standard_normal((m, k)), rng.standard_normal((g, k, n)), rng.standard_normal((m, n))
    for off, gl, limit in [(0, g, None), (2, 3, None), (1, 4, 40)]:
        wl = w[off:off + gl]
        out = oracle.ragged_dot(x, wl, sizes, group_offset=off, limit=limit)
        L = m if limit is None else limit
        lhs_ip = np.sum(out[:L] * do[:L])
        dx = oracle.ragged_dot_trans_rhs(do, wl, sizes, group_offset=off, limit=limit)
        dw = oracle.trans_ragged_dot(x, do, sizes, group_offset=off, g_local=gl, limit=limit)
        assert math.isclose(lhs_ip, np.sum(x[:L] * dx[:L]), rel_tol=1e-12, abs_tol=1e-12)
        assert math.isclose(lhs_ip, np.sum(wl * dw), rel_tol=1e-12, abs_tol=1e-12)


def test_finite_differences_dx_dw():
    """Central differences of f(x, w) = <fwd(x, w), do> match dx and dw."""
    rng = np.random.default_rng(18)
    m, k, n, g = 20, 4, 3, 3
    sizes = [7, 0, 11]
    x, w, do = rng.standard_normal((m, k)), rng.standard_normal((g, k, n)), rng.standard_normal((m, n))

    def f(xx, ww):
        return float(np.sum(oracle.ragged_dot(xx, ww, sizes)[:m] * do))

    dx = oracle.ragged_dot_trans_rhs(do, w, sizes)
    dw = oracle.trans_ragged_dot(x, do, sizes)
    h = 1e-3
    for _ in range(10):
        i, a = int(rng.integers(m)), int(rng.integers(k))
        xp, xm = x.copy(), x.copy()
        xp[i, a] += h
        xm[i, a] -= h
        assert math.isclose((f(xp, w) - f(xm, w)) / (2 * h), dx[i, a], rel_tol=1e-7, abs_tol=1e-9)
        j, b = int(rng.integers(g)), int(rng.integers(n))
        wp, wm = w.copy(), w.copy()
        wp[j, a, b] += h
        wm[j, a, b] -= h
        assert math.isclose((f(x, wp) - f(x, wm)) / (2 * h), dw[j, a, b], rel_tol=1e-7, abs_tol=1e-9)


def test_glu_epilogue_is_glu_of_plain_forward():
    rng = np.random.default_rng(19)
    a, w = rng.standard_normal((33, 8)), 0.3 * rng.standard_normal((3, 8, 10))
    sizes = [10, 13, 5]
    plain = oracle.ragged_dot(a, w, sizes, limit=30)
    fused = oracle.ragged_dot(a, w, sizes, limit=30, glu=True)
    g, u = plain[:30, :5], plain[:30, 5:]
    np.testing.assert_allclose(fused[:30], g * (1 / (1 + np.exp(-g))) * u, rtol=1e-14, atol=1e-15)
    assert np.all(fused[:30][28:] == 0)   # rows beyond the groups (28, 29) are zero


# --------------------------------------------------------------------------
# planted mistakes: the pins above must catch each of these
# --------------------------------------------------------------------------
def _wrong_bounds_forward(lhs, rhs, sizes, group_offset=0, limit=None):
    """A plausible bug: inclusive cumulative sum used as the group start."""
    a, w = np.asarray(lhs, float), np.asarray(rhs, float)
    m = a.shape[0]
    cum = np.cumsum(np.maximum(sizes, 0))
    out = np.zeros((m, w.shape[2]))
    for j in range(w.shape[0]):
        lo, hi = cum[group_offset + j], cum[group_offset + j] + sizes[group_offset + j]
        out[lo:min(hi, m)] = a[lo:min(hi, m)] @ w[j]
    return out


def test_planted_wrong_index_is_caught():
    lhs, rhs, gs = GOLDEN["lhs"], np.array(GOLDEN["rhs"], float), GOLDEN["group_sizes"]
    assert not np.array_equal(_wrong_bounds_forward(lhs, rhs, gs), GOLDEN["forward"]["offset0"])


def test_planted_transposed_operand_is_caught():
    t = GOLDEN["trans_rhs"]
    w = np.array(t["rhs"], float)
    wrong = oracle.ragged_dot(t["lhs"], w, t["group_sizes"])     # forgot the transpose
    assert not np.array_equal(wrong, t["out"])


def test_planted_dropped_term_is_caught():
    rng = np.random.default_rng(20)
    lhs, rhs, sizes = _rand_case(rng, 12, 3, 2, 3)
    good = brute_fwd(lhs.tolist(), rhs.tolist(), sizes.tolist(), 0, None)
    dropped = oracle.ragged_dot(lhs[:, :2], rhs[:, :2], sizes)   # last k term dropped
    assert not np.allclose(good, dropped)


# --------------------------------------------------------------------------
# the GLU backward through the down projection
# --------------------------------------------------------------------------
def _ffn_loss(fused, w_down, d_out, sizes, off, limit):
    """<ragged_dot(glu(gate, up), w_down), d_out> over the local rows below L."""
    m, f2 = fused.shape
    f = f2 // 2
    h = oracle.glu_fwd_f64(fused[:, :f], fused[:, f:])
    out = oracle.ragged_dot(h, w_down, sizes, group_offset=off, limit=limit)
    b, L = oracle.group_bounds(sizes, m, limit)
    rows = slice(b[off], b[off + w_down.shape[0]])
    return float(np.sum(out[rows] * d_out[rows]))


def test_glu_bwd_through_down_projection_matches_finite_differences():
    rng = np.random.default_rng(21)
    m, f, n, g = 24, 4, 5, 3
    sizes = [7, 9, 8]
    fused = rng.standard_normal((m, 2 * f))
    w_down = rng.standard_normal((g, f, n))        # forward: h [m, f] @ w_down[j] [f, n]
    d_out = rng.standard_normal((m, n))
    for off, gl, limit in [(0, 3, None), (1, 2, 20)]:
        wl = w_down[off:off + gl]
        grad = oracle.ragged_dot_trans_rhs_glu_bwd(d_out, wl, fused, sizes, off, limit)
        b, L = oracle.group_bounds(sizes, m, limit)
        h = 1e-6
        for _ in range(12):
            i, c = int(rng.integers(0, m)), int(rng.integers(0, 2 * f))
            fp, fm = fused.copy(), fused.copy()
            fp[i, c] += h
            fm[i, c] -= h
            fd = (_ffn_loss(fp, wl, d_out, sizes, off, limit) - _ffn_loss(fm, wl, d_out, sizes, off, limit)) / (2 * h)
            if i < L:
                assert math.isclose(grad[i, c], fd, rel_tol=1e-6, abs_tol=1e-8), (i, c)
            else:
                assert np.isnan(grad[i, c]) and fd == 0.0



def test_dw_f32_accumulate_is_sum_of_microbatches():
    """Accumulating two micro-batches equals one pass over their concatenation."""
    rng = np.random.default_rng(22)
    k, n, g = 5, 4, 3
    x1, y1 = rng.standard_normal((20, k)), rng.standard_normal((20, n))
    x2, y2 = rng.standard_normal((16, k)), rng.standard_normal((16, n))
    s1, s2 = [7, 0, 13], [4, 6, 6]
    acc = oracle.trans_ragged_dot_f32(x1, y1, s1)
    acc = oracle.trans_ragged_dot_f32(x2, y2, s2, out_prior=acc)
    # rows of group j from both micro-batches, stacked
    b1, _ = oracle.group_bounds(s1, 20)
    b2, _ = oracle.group_bounds(s2, 16)
    xs = np.concatenate([np.concatenate([x1[b1[j]:b1[j + 1]], x2[b2[j]:b2[j + 1]]]) for j in range(g)])
    ys = np.concatenate([np.concatenate([y1[b1[j]:b1[j + 1]], y2[b2[j]:b2[j + 1]]]) for j in range(g)])
    sizes = [s1[j] + s2[j] for j in range(g)]
    np.testing.assert_allclose(acc, oracle.trans_ragged_dot(xs, ys, sizes), rtol=1e-13, atol=1e-13)
    prior = rng.standard_normal((g, k, n))
    empty = oracle.trans_ragged_dot_f32(x1, y1, [0, 20, 0], out_prior=prior)
    np.testing.assert_array_equal(empty[0], prior[0])       # no rows: the prior stays
    np.testing.assert_array_equal(empty[2], prior[2])


def test_f32_sum_bound_covers_a_sequential_f32_sum():
    rng = np.random.default_rng(23)
    from oracle import bf16 as obf
    x = obf.round_to_bf16(rng.standard_normal((3000, 4)).astype(np.float32))
    y = obf.round_to_bf16(rng.standard_normal((3000, 3)).astype(np.float32))
    sizes = [1000, 2000]
    ref = oracle.trans_ragged_dot(x, y, sizes)
    bound = ragged.f32_sum_bound(x, y, sizes)
    b, _ = oracle.group_bounds(sizes, 3000)
    for j in range(2):
        s = np.zeros((4, 3), np.float32)
        for i in range(b[j], b[j + 1]):
            s += np.outer(x[i], y[i]).astype(np.float32)
        assert np.all(np.abs(s.astype(np.float64) - ref[j]) <= bound[j])
