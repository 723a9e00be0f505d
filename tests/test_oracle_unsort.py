"""Pins for the unsort-backward oracle (CPU only)."""
import numpy as np

from oracle import bf16 as obf
from oracle import unsort


def _bf16(rng, shape, scale=1.0):
    return obf.round_to_bf16((rng.standard_normal(shape) * scale).astype(np.float32))


def test_brute_force():
    rng = np.random.default_rng(0)
    g, y = _bf16(rng, (9, 16)), _bf16(rng, (9, 16))
    w = rng.uniform(-1, 1, 9).astype(np.float32)
    bits, grad, dot = unsort.unsort_bwd_rows(g, y, w, limit=7)
    assert grad.shape == (7, 16) and dot.shape == (7,)
    for r in range(7):
        acc = 0.0
        for c in range(16):
            want = obf.round_to_bf16(np.float32(g[r, c]) * np.float32(w[r]))
            assert grad[r, c] == want
            acc += float(g[r, c]) * float(y[r, c])
        assert abs(dot[r] - acc) < 1e-12


def test_closed_forms():
    rng = np.random.default_rng(1)
    g = _bf16(rng, (5, 32))
    ones = np.ones(5, np.float32)
    _, grad, dot = unsort.unsort_bwd_rows(g, g, ones)
    np.testing.assert_array_equal(grad, g)                       # w = 1 keeps g exactly
    np.testing.assert_allclose(dot, (g.astype(np.float64) ** 2).sum(1), rtol=1e-15)
    _, grad, _ = unsort.unsort_bwd_rows(g, g, np.full(5, 0.5, np.float32))
    np.testing.assert_array_equal(grad, g * np.float32(0.5))   # a power of two is exact
    _, grad, dot = unsort.unsort_bwd_rows(g, g, ones, limit=0)
    assert grad.shape == (0, 32) and dot.shape == (0,)


def test_rounding_is_a_single_f32_product_then_bf16():
    # g = 1 + 2^-7 (bf16), w chosen so that the f32 product lands on a bf16 tie
    g = np.array([[1.0 + 2.0 ** -7]], np.float32)
    w = np.array([1.0 + 2.0 ** -9], np.float32)
    bits, grad, _ = unsort.unsort_bwd_rows(g, g, w)
    exact = (1.0 + 2.0 ** -7) * (1.0 + 2.0 ** -9)       # representable in f32
    assert grad[0, 0] == obf.round_to_bf16(np.float32(exact))


def test_dot_tolerance_covers_f32_summation():
    rng = np.random.default_rng(2)
    g, y = _bf16(rng, (64, 4096)), _bf16(rng, (64, 4096))
    _, _, dot = unsort.unsort_bwd_rows(g, y, np.ones(64, np.float32))
    tol = unsort.dot_tolerance(g, y)
    s32 = np.zeros(64, np.float32)
    for c in range(4096):                      # a sequential f32 summation
        s32 += g[:, c] * y[:, c]
    assert np.all(np.abs(s32.astype(np.float64) - dot) <= tol)


def test_planted_weight_on_wrong_row_is_caught():
    rng = np.random.default_rng(3)
    g, y = _bf16(rng, (4, 8)), _bf16(rng, (4, 8))
    w = np.array([1.0, 2.0, 3.0, 4.0], np.float32)
    _, grad, _ = unsort.unsort_bwd_rows(g, y, w)
    wrong = obf.round_to_bf16(g * w[::-1, None])
    assert not np.array_equal(grad, wrong)
