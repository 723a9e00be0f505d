"""Pins for the SiLU-GLU oracle and the bf16 helpers (CPU only)."""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import bf16

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = json.load(open(os.path.join(HERE, "golden", "hand_examples.json")))

ALL_BF16 = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)


def test_bf16_rounding_matches_torch():
    """Round-to-nearest-even to bf16 agrees with torch's conversion on random and edge values."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(100000).astype(np.float32) * np.float32(1e3),
        np.array([0.0, -0.0, np.inf, -np.inf, 1e-40, -1e-40, 3.4e38, -3.4e38, 1.0 + 2 ** -8,
                  1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9], np.float32),
        (np.arange(1 << 16, dtype=np.uint32) << 16 | 0x8000).view(np.float32),   # exact ties
    ])
    x = x[~np.isnan(x)]
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(bf16.round_f32_to_bf16_bits(x), want)


def test_ulp_closed_forms():
    assert bf16.ulp(1.0) == 2.0 ** -7
    assert bf16.ulp(1.5) == 2.0 ** -7
    assert bf16.ulp(2.0) == 2.0 ** -6
    assert bf16.ulp(-0.75) == 2.0 ** -8
    assert bf16.ulp(0.0) == 2.0 ** -133
    assert bf16.ulp(1e-40) == 2.0 ** -133


def test_silu_table_values():
    s = GOLDEN["silu"]
    got = oracle.glu_fwd_f64(np.array(s["g"]), np.ones(len(s["g"])))
    np.testing.assert_allclose(got, s["silu"], rtol=1e-15, atol=1e-16)


def test_silu_identities():
    """silu(x) - silu(-x) = x, silu(x)/x -> 1 for large x, glu(g, 0) = 0."""
    x = np.linspace(-30, 30, 2001)
    sp, sm = oracle.glu_fwd_f64(x, 1.0), oracle.glu_fwd_f64(-x, 1.0)
    np.testing.assert_allclose(sp - sm, x, rtol=0, atol=1e-12)
    assert abs(oracle.glu_fwd_f64(40.0, 1.0) - 40.0) < 1e-14
    assert np.all(oracle.glu_fwd_f64(x, 0.0) == 0)


def test_glu_bwd_closed_forms():
    d_gate, d_up = oracle.glu_bwd_f64(0.0, 3.0, 2.0)
    assert d_gate == pytest.approx(3.0 * 2.0 / 2.0, abs=1e-15)   # d * u * sig(0) = d*u/2
    assert d_up == 0.0                                             # silu(0) = 0
    # derivative of silu at large positive g tends to 1, at large negative to 0
    d_gate, _ = oracle.glu_bwd_f64(40.0, 1.0, 1.0)
    assert d_gate == pytest.approx(1.0, abs=1e-12)
    d_gate, _ = oracle.glu_bwd_f64(-40.0, 1.0, 1.0)
    assert abs(d_gate) < 1e-12


def test_glu_bwd_matches_finite_differences():
    rng = np.random.default_rng(1)
    g, u, d = rng.standard_normal(200) * 4, rng.standard_normal(200), rng.standard_normal(200)
    h = 1e-6
    fd_gate = (oracle.glu_fwd_f64(g + h, u) - oracle.glu_fwd_f64(g - h, u)) / (2 * h) * d
    fd_up = (oracle.glu_fwd_f64(g, u + h) - oracle.glu_fwd_f64(g, u - h)) / (2 * h) * d
    d_gate, d_up = oracle.glu_bwd_f64(g, u, d)
    np.testing.assert_allclose(d_gate, fd_gate, rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(d_up, fd_up, rtol=1e-6, atol=1e-8)


def _exp_overflows_f32(g):
    """Where exp(-g) overflows binary32 the op sequence pins the result to a signed zero."""
    with np.errstate(over="ignore"):
        return np.isinf(np.exp(-np.asarray(g, np.float64)).astype(np.float32))


def _finite_within_one_ulp(got_f32, ref64, g):
    fin = np.isfinite(ref64) & np.isfinite(got_f32) & ~_exp_overflows_f32(g)
    err = np.abs(got_f32[fin].astype(np.float64) - ref64[fin])
    return np.all(err <= bf16.ulp(ref64[fin]))


def test_glu_fwd_f32_sequence_within_one_ulp_of_f64_all_gates():
    """Every bf16 gate pattern x random up: the f32 sequence is within 1 bf16 ulp of float64."""
    rng = np.random.default_rng(2)
    g = bf16.bits_to_f32(ALL_BF16)
    for _ in range(4):
        u = bf16.round_to_bf16(rng.standard_normal(g.size).astype(np.float32))
        _, got = oracle.glu_fwd_f32(g, u)
        ref = oracle.glu_fwd_f64(g, u)
        assert _finite_within_one_ulp(got, ref, g)
        # in the overflow regime the sequence gives a signed zero (true value < 1e-35)
        ov = _exp_overflows_f32(g) & np.isfinite(g) & np.isfinite(u)
        assert np.all(got[ov] == 0) and np.all(np.abs(ref[ov]) < 1e-35)
        # where float64 is finite and not NaN, the f32 sequence is not NaN either
        fin = np.isfinite(ref) & np.isfinite(g)
        assert not np.any(np.isnan(got[fin]))


def test_glu_fwd_f32_special_values():
    inf, nan = np.float32(np.inf), np.float32(np.nan)
    g = np.array([-inf, inf, inf, nan, 0.0, -0.0, -100.0, 100.0, 1e-40], np.float32)
    u = np.array([1.0, 1.0, 0.0, 1.0, 5.0, 5.0, 2.0, -1.0, 1.0], np.float32)
    _, r = oracle.glu_fwd_f32(g, u)
    assert np.isnan(r[0])                 # -inf / (1 + inf) = NaN
    assert r[1] == np.inf                 # inf / 1 * 1
    assert np.isnan(r[2])                 # inf * 0
    assert np.isnan(r[3])
    assert r[4] == 0 and not np.signbit(r[4])
    assert r[5] == 0 and np.signbit(r[5])   # -0 / 2 * 5 = -0 (the forward keeps -0)
    assert r[6] == 0 and np.signbit(r[6])   # -100 / (1 + e^100 = inf) = -0; * 2
    assert r[7] == -100.0
    assert r[8] == bf16.round_to_bf16(np.float32(0.5e-40))[()]


def test_glu_bwd_f32_within_tolerance_of_f64_all_gates():
    rng = np.random.default_rng(3)
    g = bf16.bits_to_f32(ALL_BF16)
    for _ in range(2):
        u = bf16.round_to_bf16(rng.standard_normal(g.size).astype(np.float32))
        d = bf16.round_to_bf16(rng.standard_normal(g.size).astype(np.float32))
        (bg, bu), (rg, ru) = oracle.glu_bwd_f32(g, u, d)
        want_g, want_u = oracle.glu_bwd_f64(g, u, d)
        assert _finite_within_one_ulp(ru, want_u, g)
        assert _finite_within_one_ulp(rg, want_g, g)
        assert not np.any(bg == 0x8000) and not np.any(bu == 0x8000)   # the -0 -> +0 fix


def test_glu_bwd_f32_special_values():
    inf = np.float32(np.inf)
    g = np.array([0.0, -0.0, -inf, inf, -200.0], np.float32)
    u = np.array([1.0, -1.0, 1.0, 1.0, 1.0], np.float32)
    d = np.array([-1.0, 1.0, 1.0, 1.0, 1.0], np.float32)
    (bg, bu), (rg, ru) = oracle.glu_bwd_f32(g, u, d)
    assert bu[0] == 0 and bu[1] == 0           # -1 * 0 = -0 -> +0; 1 * -0 = -0 -> +0
    assert rg[0] == -0.5 and rg[1] == -0.5
    assert np.isnan(rg[2]) and np.isnan(ru[2])  # -inf: silu = -inf/inf = NaN
    assert np.isnan(rg[3]) and ru[3] == inf     # +inf: 1 + inf * 0 = NaN in the derivative
    assert bg[4] == 0 and bu[4] == 0           # tiny negative results become +0
