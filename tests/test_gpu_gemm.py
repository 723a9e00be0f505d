"""GPU parity of the grouped GEMMs against the float64 oracle, through the C ABI.

Small shapes that span several 128x256 / 256x256 tiles and ragged edges in every
dimension: group sizes 0, 1, BM-1, BM, BM+1, k and n not multiples of the
tile, group offsets, valid-row limits, NaN-poisoned input rows past the
limit, sentinel-filled output rows past the limit and canary rows after the
output buffer.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import bf16 as obf
from parity_util import assert_close, gemm_tol, glu_epilogue_tol

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda"
SENT = 0x3C3C          # sentinel bf16 pattern for rows that must stay untouched
CANARY_ROWS = 4
EDGE_SIZES = [0, 1, 127, 128, 129, 0, 255, 3]   # sum 643


@pytest.fixture(params=["pair", "single"], autouse=True)
def gemm_variant(request, rd_lib):
    """Every test runs on both the CTA-pair (256-row) and the single-CTA (128-row) kernels."""
    v = rd_lib.VARIANT_PAIR if request.param == "pair" else rd_lib.VARIANT_SINGLE
    with rd_lib.tuning(variant=v):
        yield request.param


def _normal(rng, shape, var=1.0):
    from workloads import normal_bf16_np
    return normal_bf16_np(rng, shape, var)


def _i32(vals):
    return torch.tensor(vals, dtype=torch.int32, device=DEV)


def _sentinel_buffer(rows, cols, lead=()):
    buf = torch.empty(lead + (rows + CANARY_ROWS, cols), dtype=torch.bfloat16, device=DEV)
    buf.view(torch.int16).fill_(SENT)
    return buf


def _f64(t):
    return obf.torch_bf16_to_f64(t)


def _check_rows(bits, m, L, local_mask):
    """rows >= L and canaries keep the sentinel; rows < L outside the groups are +0."""
    assert np.all(bits[L:] == SENT), "a row at or past the limit (or a canary row) was written"
    zero_rows = ~local_mask[:m]
    zero_rows[L:] = False
    assert np.all(bits[:m][zero_rows] == 0), "rows outside the local groups are not +0"


def run_fwd(rd, m, k, n, sizes, off=0, gl=None, limit=None, glu=False, seed=0, poison=True):
    rng = np.random.default_rng(seed)
    g_total = len(sizes)
    gl = g_total - off if gl is None else gl
    lhs = _normal(rng, (m, k))
    rhs = _normal(rng, (gl, k, n), 1.0 / max(k, 1))
    b, L = oracle.group_bounds(sizes, m, limit)
    lhs_dev = lhs.clone()
    if poison:
        lhs_dev[L:] = float("nan")
    n_out = n // 2 if glu else n
    buf = _sentinel_buffer(m, n_out)
    status = _i32([0])
    rd.ragged_dot(lhs_dev.to(DEV), rhs.to(DEV), _i32(sizes), group_offset=off,
                  limit=None if limit is None else _i32([limit]),
                  epilogue=rd.EPI_SILU_GLU if glu else rd.EPI_NONE, out=buf[:m], status=status)
    torch.cuda.synchronize()
    bits = obf.torch_bf16_bits(buf)
    got = _f64(buf[:m])
    a64, w64 = _f64(lhs), _f64(rhs)
    local = np.zeros(m, bool)
    local[b[off]:b[off + gl]] = True
    _check_rows(bits, m, L, local)
    amax = np.abs(a64[:L]).max() if L else 0.0
    bmax = np.abs(w64).max() if w64.size else 0.0
    if glu:
        plain = oracle.ragged_dot(a64, w64, sizes, off, limit)
        F = n_out
        E = 1e-3 * math.sqrt(max(k, 1)) * amax * bmax
        ref, tol = glu_epilogue_tol(plain[:, :F], plain[:, F:], E)
        ref_o = oracle.ragged_dot(a64, w64, sizes, off, limit, glu=True)
        np.testing.assert_allclose(ref[local], ref_o[local], rtol=1e-12, atol=1e-300)
    else:
        ref = oracle.ragged_dot(a64, w64, sizes, off, limit)
        tol = gemm_tol(ref, k, amax, bmax)
    assert_close(got[local], ref[local], tol[local], "forward")
    assert int(status.item()) == 0
    return got


def run_dx(rd, m, k, n, sizes, off=0, gl=None, limit=None, seed=0):
    rng = np.random.default_rng(seed)
    gl = len(sizes) - off if gl is None else gl
    do = _normal(rng, (m, n))
    w = _normal(rng, (gl, k, n), 1.0 / max(k, 1))
    b, L = oracle.group_bounds(sizes, m, limit)
    do_dev = do.clone()
    do_dev[L:] = float("nan")
    buf = _sentinel_buffer(m, k)
    rd.ragged_dot_trans_rhs(do_dev.to(DEV), w.to(DEV), _i32(sizes), group_offset=off,
                            limit=None if limit is None else _i32([limit]), out=buf[:m])
    torch.cuda.synchronize()
    bits = obf.torch_bf16_bits(buf)
    got = _f64(buf[:m])
    a64, w64 = _f64(do), _f64(w)
    local = np.zeros(m, bool)
    local[b[off]:b[off + gl]] = True
    _check_rows(bits, m, L, local)
    ref = oracle.ragged_dot_trans_rhs(a64, w64, sizes, off, limit)
    amax = np.abs(a64[:L]).max() if L else 0.0
    tol = gemm_tol(ref, n, amax, np.abs(w64).max())
    assert_close(got[local], ref[local], tol[local], "dx")


def run_dw(rd, m, k, n, sizes, off=0, gl=None, limit=None, seed=0):
    """dw through both forms: per-group maps (a workspace) and in-smem edge zeroing (none)."""
    for ws in ("auto", None):
        _run_dw(rd, m, k, n, sizes, off, gl, limit, seed, ws)


def _run_dw(rd, m, k, n, sizes, off, gl, limit, seed, ws):
    rng = np.random.default_rng(seed)
    gl = len(sizes) - off if gl is None else gl
    x = _normal(rng, (m, k))
    y = _normal(rng, (m, n))
    b, L = oracle.group_bounds(sizes, m, limit)
    x_dev, y_dev = x.clone(), y.clone()
    # rows past the limit and rows outside the local groups must not enter any sum
    x_dev[L:] = float("nan")
    y_dev[L:] = float("nan")
    if b[off] > 0:
        x_dev[: b[off]] = float("nan")
        y_dev[: b[off]] = float("nan")
    buf = torch.empty((gl + 1, k, n), dtype=torch.bfloat16, device=DEV)   # one guard block after
    buf.view(torch.int16).fill_(SENT)
    out = buf[:gl]
    rd.trans_ragged_dot(x_dev.to(DEV), y_dev.to(DEV), _i32(sizes), group_offset=off, g_local=gl,
                        limit=None if limit is None else _i32([limit]), out=out, workspace=ws)
    torch.cuda.synchronize()
    assert np.all(obf.torch_bf16_bits(buf[gl]) == SENT), "the guard block after dw was written"
    got = _f64(out)
    x64, y64 = _f64(x), _f64(y)
    ref = oracle.trans_ragged_dot(x64, y64, sizes, off, gl, limit)
    for j in range(gl):
        cnt = int(b[off + j + 1] - b[off + j])
        if cnt == 0:
            assert np.all(obf.torch_bf16_bits(out[j]) == 0), f"empty group {j} not +0"
            continue
        rows = slice(b[off + j], b[off + j + 1])
        tol = gemm_tol(ref[j], cnt, np.abs(x64[rows]).max(), np.abs(y64[rows]).max())
        assert_close(got[j], ref[j], tol, f"dw group {j} ({cnt} rows, workspace {ws})")


# ------------------------------------------------------------------ forward
def test_tiny_workload(rd_lib):
    from workloads import tiny_fwd
    w = tiny_fwd()
    run_fwd(rd_lib, w.m, w.k, w.n, w.group_sizes.tolist(), seed=w.seed)


@pytest.mark.parametrize("m,k,n", [(700, 136, 264), (700, 64, 512), (643, 520, 256)])
def test_forward_ragged_edges(rd_lib, m, k, n):
    run_fwd(rd_lib, m, k, n, EDGE_SIZES, seed=m + k + n)


PAIR_EDGE_SIZES = [256, 257, 511, 1, 0, 513, 255]   # sum 1793: edges of 256-row tiles


@pytest.mark.parametrize("limit", [None, 1500, 255])
def test_forward_pair_tile_edges(rd_lib, limit):
    run_fwd(rd_lib, 1800, 128, 512, PAIR_EDGE_SIZES, limit=limit, seed=11)
    run_fwd(rd_lib, 1800, 64, 256, PAIR_EDGE_SIZES, off=1, gl=5, limit=limit, glu=True, seed=12)
    run_dx(rd_lib, 1800, 512, 128, PAIR_EDGE_SIZES, off=2, gl=4, limit=limit, seed=13)


@pytest.mark.parametrize("off,gl,limit", [(2, 4, None), (2, 4, 500), (0, 8, 300), (7, 1, None),
                                          (4, 3, 640)])
def test_forward_offset_and_limit(rd_lib, off, gl, limit):
    run_fwd(rd_lib, 700, 136, 264, EDGE_SIZES, off=off, gl=gl, limit=limit, seed=off * 7 + gl)


@pytest.mark.parametrize("limit", [0, 1, 127, 128, 699, 700, 900])
def test_forward_limit_sweep(rd_lib, limit):
    run_fwd(rd_lib, 700, 72, 256, EDGE_SIZES, limit=limit, seed=limit)


def test_forward_many_groups(rd_lib):
    rng = np.random.default_rng(3)
    sizes = rng.multinomial(1900, np.full(17, 1 / 17)).tolist()
    run_fwd(rd_lib, 2048, 256, 512, sizes, off=3, gl=9, limit=1700, seed=3)


@pytest.mark.parametrize("m,k,n,sizes", [(5, 64, 256, [5]), (1, 8, 8, [1]), (130, 8, 24, [64, 66]),
                                         (300, 64, 256, [300])])
def test_forward_small_and_single_group(rd_lib, m, k, n, sizes):
    run_fwd(rd_lib, m, k, n, sizes, seed=m)


@pytest.mark.parametrize("m,k,F,off,gl,limit", [(700, 136, 136, 0, 8, 650), (700, 64, 128, 2, 4, None),
                                                (300, 256, 256, 0, 1, None), (700, 64, 8, 1, 5, 600)])
def test_forward_glu_epilogue(rd_lib, m, k, F, off, gl, limit):
    sizes = EDGE_SIZES if gl > 1 else [300]
    run_fwd(rd_lib, m, k, 2 * F, sizes, off=off, gl=gl, limit=limit, glu=True, seed=F + off)


def test_forward_k_zero_writes_zeros(rd_lib):
    m, n = 300, 256
    buf = _sentinel_buffer(m, n)
    rd_lib.ragged_dot(torch.empty((m, 0), dtype=torch.bfloat16, device=DEV),
                      torch.empty((2, 0, n), dtype=torch.bfloat16, device=DEV),
                      _i32([100, 150]), out=buf[:m], limit=_i32([280]))
    torch.cuda.synchronize()
    bits = obf.torch_bf16_bits(buf)
    assert np.all(bits[:280] == 0) and np.all(bits[280:] == SENT)


def test_status_bits(rd_lib):
    m, k, n = 256, 64, 256
    lhs = torch.randn(m, k, device=DEV).to(torch.bfloat16)
    rhs = torch.randn(3, k, n, device=DEV).to(torch.bfloat16)
    status = _i32([0])
    rd_lib.ragged_dot(lhs, rhs, _i32([100, -5, 200]), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == (rd_lib.STATUS_NEG_SIZE | rd_lib.STATUS_OVERFLOW)
    names = rd_lib.status_bits(status)
    assert len(names) == 2 and names[0].startswith("STATUS_NEG_SIZE") and names[1].startswith("STATUS_OVERFLOW")
    assert rd_lib.check_status(status) == 3            # the size bits alone do not raise
    with pytest.raises(rd_lib.RdError, match="STATUS_NEG_SIZE"):
        rd_lib.check_status(status, allow=0)


# ------------------------------------------------------------------ tile-order bands
# The forward / dx tile order walks each group in bands of band_tiles m-tiles
# (the last band of a group partial), sweeping every column block inside a
# band.  With the default 6144-row band only groups above 6144 rows span
# several bands, so these tests shrink the band to 1, 2 and 3 tiles: groups of
# 600 to 2000 rows then hold up to 16 bands, most of them with a partial last
# band, over several column tiles, and every output element is compared.
BAND_SIZES = [1500, 0, 700, 2000, 613, 1, 1100]     # sum 5914


@pytest.mark.parametrize("band_tiles", [1, 2, 3])
def test_band_order_forward(rd_lib, gemm_variant, band_tiles):
    tile = 256 if gemm_variant == "pair" else 128
    with rd_lib.tuning(band_rows=band_tiles * tile):
        run_fwd(rd_lib, 6000, 64, 776, BAND_SIZES, seed=band_tiles)
        run_fwd(rd_lib, 6000, 64, 776, BAND_SIZES, off=2, gl=4, limit=5000, seed=band_tiles + 10)


@pytest.mark.parametrize("band_tiles", [1, 3])
def test_band_order_forward_glu(rd_lib, gemm_variant, band_tiles):
    tile = 256 if gemm_variant == "pair" else 128
    with rd_lib.tuning(band_rows=band_tiles * tile):
        run_fwd(rd_lib, 6000, 64, 1040, BAND_SIZES, glu=True, seed=band_tiles + 20)


@pytest.mark.parametrize("band_tiles", [1, 2, 3])
def test_band_order_dx(rd_lib, gemm_variant, band_tiles):
    tile = 256 if gemm_variant == "pair" else 128
    with rd_lib.tuning(band_rows=band_tiles * tile):
        run_dx(rd_lib, 6000, 776, 64, BAND_SIZES, seed=band_tiles + 30)
        run_dx(rd_lib, 6000, 520, 64, BAND_SIZES, off=1, gl=5, limit=4500, seed=band_tiles + 40)


@pytest.mark.parametrize("band_tiles", [1, 3])
def test_band_order_dx_glu_bwd(rd_lib, gemm_variant, band_tiles):
    tile = 256 if gemm_variant == "pair" else 128
    with rd_lib.tuning(band_rows=band_tiles * tile):
        run_dx_glu_bwd(rd_lib, 6000, 520, 64, BAND_SIZES, limit=5500, seed=band_tiles + 50)


def test_tuning_round_trip(rd_lib):
    """rd_set_tuning / rd_get_tuning: values read back, bad ones rejected, defaults restored."""
    before = rd_lib.get_tuning()
    with rd_lib.tuning(band_rows=768, wait_timeout_ns=123456789):
        t = rd_lib.get_tuning()
        assert t["band_rows"] == 768 and t["wait_timeout_ns"] == 123456789
        with pytest.raises(rd_lib.RdError):
            rd_lib.set_tuning(variant=7)
        with pytest.raises(rd_lib.RdError):
            rd_lib.set_tuning(band_rows=-1)
        assert rd_lib.get_tuning()["band_rows"] == 768
    assert rd_lib.get_tuning() == before


# ------------------------------------------------------------------ dx
@pytest.mark.parametrize("m,k,n,off,gl,limit", [(700, 264, 136, 0, 8, None), (700, 264, 136, 2, 4, 500),
                                                (643, 512, 72, 0, 8, 600), (700, 256, 520, 5, 3, None)])
def test_dx(rd_lib, m, k, n, off, gl, limit):
    run_dx(rd_lib, m, k, n, EDGE_SIZES, off=off, gl=gl, limit=limit, seed=k + n + off)


# ------------------------------------------------------------------ dx + fused GLU backward
def run_dx_glu_bwd(rd, m, f, n, sizes, off=0, gl=None, limit=None, seed=0):
    rng = np.random.default_rng(seed)
    gl = len(sizes) - off if gl is None else gl
    d_out = _normal(rng, (m, n))
    w = _normal(rng, (gl, f, n), 1.0 / n)
    fused = _normal(rng, (m, 2 * f), 4.0)
    b, L = oracle.group_bounds(sizes, m, limit)
    d_dev, f_dev = d_out.clone(), fused.clone()
    d_dev[L:] = float("nan")
    f_dev[L:] = float("nan")
    buf = _sentinel_buffer(m, 2 * f)
    rd.ragged_dot_trans_rhs_glu_bwd(d_dev.to(DEV), w.to(DEV), f_dev.to(DEV), _i32(sizes),
                                    group_offset=off,
                                    limit=None if limit is None else _i32([limit]), out=buf[:m])
    torch.cuda.synchronize()
    bits = obf.torch_bf16_bits(buf)
    got = _f64(buf[:m])
    d64, w64, f64 = _f64(d_out), _f64(w), _f64(fused)
    local = np.zeros(m, bool)
    local[b[off]:b[off + gl]] = True
    _check_rows(bits, m, L, local)
    assert not np.any(bits[:m][local] == 0x8000), "a -0 survived the -0 -> +0 fix"
    ref = oracle.ragged_dot_trans_rhs_glu_bwd(d64, w64, f64, sizes, off, limit)
    # dh carries the GEMM error E; it enters d_gate with |u * dsilu| and d_up with |silu|
    E = 1e-3 * math.sqrt(n) * (np.abs(d64[:L]).max() if L else 0.0) * np.abs(w64).max()
    from oracle import glu as oglu
    dg1, du1 = oglu.glu_bwd_f64(f64[:, :f], f64[:, f:], 1.0)
    tol = obf.ulp(ref) + np.concatenate([np.abs(dg1), np.abs(du1)], axis=1) * E
    assert_close(got[local], ref[local], tol[local], "dx + GLU backward")


@pytest.mark.parametrize("m,f,n,off,gl,limit", [(700, 136, 264, 0, 8, None), (700, 256, 128, 2, 4, 500),
                                                (643, 64, 520, 0, 8, 600), (1800, 512, 128, 1, 5, 1500)])
def test_dx_glu_bwd(rd_lib, m, f, n, off, gl, limit):
    sizes = EDGE_SIZES if m < 1800 else PAIR_EDGE_SIZES
    run_dx_glu_bwd(rd_lib, m, f, n, sizes, off=off, gl=gl, limit=limit, seed=f + n + off)


# Gates at and past the ends of binary32's exp range (exp(-g) overflows below
# -88.72 and exp(-|g|) goes subnormal below -87.34 and to zero below -103.28),
# large magnitudes and the special values.  The GEMM in front of the GLU is
# made exact (one-hot rows against the chosen values) so the epilogue alone is
# measured: within 1 bf16 ulp of float64, NaN for NaN, equal infinities.
SPECIAL_GATES = [float("-inf"), float("inf"), float("nan"), -0.0, 0.0, -1e4, -110.0, -103.0,
                 -100.0, -95.0, -91.0, -89.0, -88.5, -88.0, -87.5, -87.0, -60.0, -20.0, -5.0,
                 -1.0, -1e-30, 1e-30, 0.5, 1.0, 5.0, 20.0, 60.0, 88.0, 89.0, 100.0, 1e4, 1e30]
SPECIAL_UPS = [0.5, -1.25, 1.0, -0.0, 0.75, -0.5, 0.0, 1.0]


def _special_table(rows, cols, seed):
    """rows x cols bf16 gates / ups: every special gate in every row, shuffled per row."""
    rng = np.random.default_rng(seed)
    g = np.array([rng.permutation(np.resize(SPECIAL_GATES, cols)) for _ in range(rows)], np.float32)
    u = np.array([rng.permutation(np.resize(SPECIAL_UPS, cols)) for _ in range(rows)], np.float32)
    return torch.from_numpy(g).to(torch.bfloat16), torch.from_numpy(u).to(torch.bfloat16)


def test_fused_glu_forward_special_gates(rd_lib):
    """The fused forward GLU on gates across exp's range edges and special values.

    Group j's weight block holds table row j in its row 0 and zeros elsewhere,
    and every lhs row is the unit vector e_0, so each accumulator is exactly one
    table value (no 0 * inf products).
    """
    k, F, groups, per = 16, 64, 16, 6
    m = groups * per
    g, u = _special_table(groups, F, 11)
    rhs = torch.zeros((groups, k, 2 * F), dtype=torch.bfloat16)
    rhs[:, 0, :F] = g
    rhs[:, 0, F:] = u
    lhs = torch.zeros((m, k), dtype=torch.bfloat16)
    lhs[:, 0] = 1.0
    out = torch.empty((m, F), dtype=torch.bfloat16, device=DEV)
    rd_lib.ragged_dot(lhs.to(DEV), rhs.to(DEV), _i32([per] * groups), epilogue=rd_lib.EPI_SILU_GLU,
                      out=out)
    torch.cuda.synchronize()
    from oracle import glu as oglu
    sel = np.arange(m) // per
    ref = oglu.glu_fwd_f64(_f64(g)[sel], _f64(u)[sel])
    assert_close(_f64(out.cpu()), ref, obf.ulp(ref), "fused GLU forward, special gates")


def test_fused_glu_backward_special_gates(rd_lib):
    """The fused GLU backward (dx of the down projection) on the same gates."""
    n, f, m = 16, 64, 96
    g, u = _special_table(m, f, 12)
    fused = torch.cat([g, u], dim=1)
    rng = np.random.default_rng(13)
    dvals = torch.from_numpy(rng.choice([1.5, -0.75, 2.0, -0.5], size=(f, n)).astype(np.float32))
    w = dvals.to(torch.bfloat16).reshape(1, f, n)           # dh[i, c] = w[c, i % n]
    d_out = torch.zeros((m, n), dtype=torch.bfloat16)
    d_out[torch.arange(m), torch.arange(m) % n] = 1.0
    out = torch.empty((m, 2 * f), dtype=torch.bfloat16, device=DEV)
    rd_lib.ragged_dot_trans_rhs_glu_bwd(d_out.to(DEV), w.to(DEV), fused.to(DEV), _i32([m]), out=out)
    torch.cuda.synchronize()
    bits = obf.torch_bf16_bits(out)
    assert not np.any(bits == 0x8000), "a -0 survived the -0 -> +0 fix"
    from oracle import glu as oglu
    dh = _f64(w[0]).T[np.arange(m) % n]                     # [m, f]
    dg, du = oglu.glu_bwd_f64(_f64(g), _f64(u), dh)
    ref = np.concatenate([dg, du], axis=1)
    assert_close(_f64(out.cpu()), ref, obf.ulp(ref), "fused GLU backward, special gates")


# ------------------------------------------------------------------ dw
DW_SIZES = [0, 1, 63, 64, 65, 200, 0, 130]   # sum 523


def test_dw_group_sizes_around_16_and_64(rd_lib):
    """Group sizes at and around multiples of 16 and 64 (the K step and K block), both forms."""
    sizes = [15, 16, 17, 47, 48, 49, 79, 80, 81, 127, 128, 129, 1, 2, 190, 191, 192, 193]
    run_dw(rd_lib, sum(sizes) + 5, 128, 256, sizes, seed=77)


def test_dw_workspace_checks(rd_lib):
    """A workspace that is too small, misaligned or overlapping an operand is refused."""
    x = torch.zeros((64, 128), dtype=torch.bfloat16, device=DEV)
    y = torch.zeros((64, 256), dtype=torch.bfloat16, device=DEV)
    need = rd_lib.dw_workspace_bytes()
    assert need > 0 and need % 128 == 0
    small = torch.empty(need - 128, dtype=torch.uint8, device=DEV)
    with pytest.raises(rd_lib.RdError):
        rd_lib.trans_ragged_dot(x, y, _i32([30, 34]), workspace=small)
    big = torch.empty(need + 256, dtype=torch.uint8, device=DEV)
    with pytest.raises(rd_lib.RdError):
        rd_lib.trans_ragged_dot(x, y, _i32([30, 34]), workspace=big[64:64 + need])
    with pytest.raises(rd_lib.RdError):   # the workspace overlaps the output
        out = big[:2 * 128 * 256 * 2].view(torch.bfloat16).view(2, 128, 256)
        rd_lib.trans_ragged_dot(x, y, _i32([30, 34]), out=out, workspace=big)


@pytest.mark.parametrize("m,k,n,off,gl,limit", [(600, 136, 264, 0, 8, None), (600, 128, 256, 2, 5, 400),
                                                (523, 264, 72, 0, 8, 523), (600, 64, 520, 3, 4, 130)])
def test_dw(rd_lib, m, k, n, off, gl, limit):
    run_dw(rd_lib, m, k, n, DW_SIZES, off=off, gl=gl, limit=limit, seed=k + n + off)


def run_dw_f32(rd, m, k, n, sizes, off=0, gl=None, limit=None, seed=0, accumulate=False):
    for ws in ("auto", None):
        _run_dw_f32(rd, m, k, n, sizes, off, gl, limit, seed, accumulate, ws)


def _run_dw_f32(rd, m, k, n, sizes, off, gl, limit, seed, accumulate, ws):
    from oracle import ragged
    rng = np.random.default_rng(seed)
    gl = len(sizes) - off if gl is None else gl
    x = _normal(rng, (m, k))
    y = _normal(rng, (m, n))
    b, L = oracle.group_bounds(sizes, m, limit)
    x_dev, y_dev = x.clone(), y.clone()
    x_dev[L:] = float("nan")
    y_dev[L:] = float("nan")
    if b[off] > 0:
        x_dev[: b[off]] = float("nan")
        y_dev[: b[off]] = float("nan")
    prior = torch.from_numpy(rng.standard_normal((gl, k, n)).astype(np.float32))
    buf = torch.full((gl + 1, k, n), 5.5, device=DEV)          # one guard block after the output
    out = buf[:gl]
    if accumulate:
        out.copy_(prior.to(DEV))
    else:
        out.fill_(float("nan"))
    rd.trans_ragged_dot_f32(x_dev.to(DEV), y_dev.to(DEV), _i32(sizes), group_offset=off, g_local=gl,
                            limit=None if limit is None else _i32([limit]), out=out,
                            accumulate=accumulate, workspace=ws)
    torch.cuda.synchronize()
    assert bool((buf[gl] == 5.5).all()), "the guard block after dw was written"
    got = out.cpu().numpy().astype(np.float64)
    x64, y64 = _f64(x), _f64(y)
    p64 = prior.numpy().astype(np.float64)
    ref = oracle.trans_ragged_dot_f32(x64, y64, sizes, off, gl, limit,
                                      out_prior=p64 if accumulate else None)
    bound = ragged.f32_sum_bound(x64, y64, sizes, off, gl, limit)
    # the accumulating form also rounds its final f32 add
    tol = bound + (np.abs(np.spacing(ref.astype(np.float32))).astype(np.float64) if accumulate else 0.0)
    for j in range(gl):
        if b[off + j + 1] == b[off + j]:
            want = p64[j] if accumulate else np.zeros_like(p64[j])
            np.testing.assert_array_equal(got[j], want)
            continue
        assert_close(got[j], ref[j], tol[j], f"dw f32 group {j}")


@pytest.mark.parametrize("accumulate", [False, True])
@pytest.mark.parametrize("m,k,n,off,gl,limit", [(600, 136, 264, 0, 8, None), (600, 128, 256, 2, 5, 400),
                                                (523, 264, 72, 0, 8, 523)])
def test_dw_f32(rd_lib, m, k, n, off, gl, limit, accumulate):
    run_dw_f32(rd_lib, m, k, n, DW_SIZES, off=off, gl=gl, limit=limit, seed=k + n + off,
               accumulate=accumulate)


def test_dw_f32_accumulates_microbatches(rd_lib):
    """Two accumulating calls equal one call over both micro-batches' rows."""
    rng = np.random.default_rng(31)
    k, n = 128, 256
    s1, s2 = [300, 0, 212], [100, 250, 162]
    x1, y1 = _normal(rng, (512, k)).to(DEV), _normal(rng, (512, n)).to(DEV)
    x2, y2 = _normal(rng, (512, k)).to(DEV), _normal(rng, (512, n)).to(DEV)
    acc = torch.zeros((3, k, n), dtype=torch.float32, device=DEV)
    rd_lib.trans_ragged_dot_f32(x1, y1, _i32(s1), out=acc, accumulate=True)
    rd_lib.trans_ragged_dot_f32(x2, y2, _i32(s2), out=acc, accumulate=True)
    torch.cuda.synchronize()
    b1, _ = oracle.group_bounds(s1, 512)
    b2, _ = oracle.group_bounds(s2, 512)
    xs = torch.cat([torch.cat([x1[b1[j]:b1[j + 1]], x2[b2[j]:b2[j + 1]]]) for j in range(3)])
    ys = torch.cat([torch.cat([y1[b1[j]:b1[j + 1]], y2[b2[j]:b2[j + 1]]]) for j in range(3)])
    sizes = [s1[j] + s2[j] for j in range(3)]
    from oracle import ragged
    ref = oracle.trans_ragged_dot(_f64(xs), _f64(ys), sizes)
    bound = ragged.f32_sum_bound(_f64(xs), _f64(ys), sizes) * 2 + np.abs(np.spacing(ref.astype(np.float32)))
    assert_close(acc.cpu().numpy(), ref, bound, "two accumulated micro-batches")


def test_dw_all_groups_empty(rd_lib):
    out = torch.empty((3, 128, 256), dtype=torch.bfloat16, device=DEV)
    out.view(torch.int16).fill_(SENT)
    x = torch.randn(64, 128, device=DEV).to(torch.bfloat16)
    y = torch.randn(64, 256, device=DEV).to(torch.bfloat16)
    rd_lib.trans_ragged_dot(x, y, _i32([10, 20, 34]), limit=_i32([0]), out=out)
    torch.cuda.synchronize()
    assert np.all(obf.torch_bf16_bits(out) == 0)


# ------------------------------------------------------------------ structure
def test_expert_parallel_shards_sum_to_full(rd_lib):
    """Running each expert shard with its group_offset and summing gives the full forward."""
    rng = np.random.default_rng(9)
    m, k, n, g, shards = 1024, 128, 256, 8, 4
    sizes = rng.multinomial(1000, np.full(g, 1 / g)).tolist()
    lhs = _normal(rng, (m, k)).to(DEV)
    rhs = _normal(rng, (g, k, n), 1 / k).to(DEV)
    gs = _i32(sizes)
    full = rd_lib.ragged_dot(lhs, rhs, gs)
    gl = g // shards
    parts = [rd_lib.ragged_dot(lhs, rhs[r * gl:(r + 1) * gl].contiguous(), gs, group_offset=r * gl)
             for r in range(shards)]
    total = sum(p.float() for p in parts)
    torch.cuda.synchronize()
    # every row belongs to exactly one shard, the others write +0 there: the sum is exact
    assert torch.equal(total[:1000].to(torch.bfloat16), full[:1000])
    dw = rd_lib.trans_ragged_dot(lhs, full, gs)
    dws = torch.cat([rd_lib.trans_ragged_dot(lhs, full, gs, group_offset=r * gl, g_local=gl)
                     for r in range(shards)])
    torch.cuda.synchronize()
    assert torch.equal(dw, dws)


def test_cuda_graph_follows_device_group_sizes(rd_lib):
    """Two calls sharing group_sizes captured in one graph; replays see new sizes."""
    rng = np.random.default_rng(10)
    m, k, n, g = 512, 128, 256, 4
    lhs = _normal(rng, (m, k)).to(DEV)
    up = _normal(rng, (g, k, 2 * n), 1 / k).to(DEV)
    down = _normal(rng, (g, n, k), 1 / n).to(DEV)
    gs = _i32([100, 0, 200, 212])
    h = torch.empty((m, n), dtype=torch.bfloat16, device=DEV)
    o = torch.empty((m, k), dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        rd_lib.ragged_dot(lhs, up, gs, epilogue=rd_lib.EPI_SILU_GLU, out=h)   # first calls outside capture
        rd_lib.ragged_dot(h, down, gs, out=o)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        rd_lib.ragged_dot(lhs, up, gs, epilogue=rd_lib.EPI_SILU_GLU, out=h)
        rd_lib.ragged_dot(h, down, gs, out=o)
    for sizes in ([100, 0, 200, 212], [0, 512, 0, 0], [3, 1, 0, 508]):
        gs.copy_(_i32(sizes))
        graph.replay()
        torch.cuda.synchronize()
        ref_h = rd_lib.ragged_dot(lhs, up, gs, epilogue=rd_lib.EPI_SILU_GLU)
        ref_o = rd_lib.ragged_dot(ref_h, down, gs)
        torch.cuda.synchronize()
        assert torch.equal(h, ref_h) and torch.equal(o, ref_o)
        b, _ = oracle.group_bounds(sizes, m)
        a64, w64 = _f64(lhs), _f64(up)
        ref = oracle.ragged_dot(a64, w64, sizes, glu=True)
        plain = oracle.ragged_dot(a64, w64, sizes)
        E = 1e-3 * math.sqrt(k) * np.abs(a64).max() * np.abs(w64).max()
        ref, tol = glu_epilogue_tol(plain[:, :n], plain[:, n:], E)
        assert_close(_f64(h), ref, tol, f"graph replay sizes {sizes}")


def test_cuda_graph_backward_follows_device_group_sizes(rd_lib):
    """The backward of an expert FFN captured in one graph: the fused dx + GLU backward
    through the down projection, dx of the up projection and both weight gradients (dw
    with a preallocated workspace, so each replay rebuilds its per-group tensor maps on
    the device); replays with new sizes equal the same calls made eagerly, bit for bit."""
    rng = np.random.default_rng(11)
    m, d, f, g = 1024, 256, 128, 5
    x = _normal(rng, (m, d)).to(DEV)
    up = _normal(rng, (g, d, 2 * f), 1 / d).to(DEV)
    down = _normal(rng, (g, f, d), 1 / f).to(DEV)
    fused = _normal(rng, (m, 2 * f), 4.0).to(DEV)
    h = _normal(rng, (m, f)).to(DEV)
    d_out = _normal(rng, (m, d)).to(DEV)
    gs = _i32([200, 0, 300, 1, 500])
    ws = torch.empty(rd_lib.dw_workspace_bytes(), dtype=torch.uint8, device=DEV)
    d_fused = torch.empty((m, 2 * f), dtype=torch.bfloat16, device=DEV)
    dx = torch.empty((m, d), dtype=torch.bfloat16, device=DEV)
    dw_down = torch.empty((g, f, d), dtype=torch.bfloat16, device=DEV)
    dw_up = torch.empty((g, d, 2 * f), dtype=torch.bfloat16, device=DEV)

    def step():
        rd_lib.ragged_dot_trans_rhs_glu_bwd(d_out, down, fused, gs, out=d_fused)
        rd_lib.ragged_dot_trans_rhs(d_fused, up, gs, out=dx)
        rd_lib.trans_ragged_dot(h, d_out, gs, out=dw_down, workspace=ws)
        rd_lib.trans_ragged_dot(x, d_fused, gs, out=dw_up, workspace=ws)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step()                               # first calls outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    for sizes in ([200, 0, 300, 1, 500], [0, 1024, 0, 0, 0], [17, 333, 0, 601, 73]):
        gs.copy_(_i32(sizes))
        graph.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in (d_fused, dx, dw_down, dw_up)]
        with torch.cuda.stream(s):
            step()
        torch.cuda.synchronize()
        for a, b in zip(got, (d_fused, dx, dw_down, dw_up)):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), f"replay with sizes {sizes}"
        # and the replayed dx of the up projection matches the oracle
        ref = oracle.ragged_dot_trans_rhs(_f64(got[0].cpu()), _f64(up.cpu()), sizes)
        tol = gemm_tol(ref, 2 * f, np.abs(_f64(got[0].cpu())).max(), np.abs(_f64(up.cpu())).max())
        assert_close(_f64(got[1].cpu()), ref, tol, f"graph replay dx, sizes {sizes}")


# ------------------------------------------------------------------ extremes
def test_maximum_group_count(rd_lib):
    """g_total = RD_MAX_GROUPS (1024), most groups empty, an offset shard of 300 groups."""
    rng = np.random.default_rng(40)
    g = rd_lib.MAX_GROUPS
    sizes = np.zeros(g, np.int64)
    live = rng.choice(g, 96, replace=False)
    sizes[live] = rng.integers(1, 40, 96)
    sizes = sizes.tolist()
    m = int(sum(sizes)) + 17
    run_fwd(rd_lib, m, 64, 256, sizes, off=400, gl=300, seed=40)
    run_dx(rd_lib, m, 256, 64, sizes, off=100, gl=600, seed=41)
    run_dw(rd_lib, m, 64, 256, sizes, off=500, gl=200, seed=42)


def test_empty_inputs_are_no_ops(rd_lib):
    """m = 0 enqueues nothing for the row outputs; dw of zero rows is all zeros."""
    gs = _i32([0, 0])
    e = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    rd_lib.ragged_dot(e, torch.zeros((2, 64, 64), dtype=torch.bfloat16, device=DEV), gs)
    rd_lib.ragged_dot_trans_rhs(e, torch.zeros((2, 64, 64), dtype=torch.bfloat16, device=DEV), gs)
    out = torch.full((2, 64, 64), 3.0, dtype=torch.bfloat16, device=DEV)
    rd_lib.trans_ragged_dot(e, e, gs, out=out)
    f32 = torch.full((2, 64, 64), 3.0, dtype=torch.float32, device=DEV)
    rd_lib.trans_ragged_dot_f32(e, e, gs, out=f32, accumulate=True)
    torch.cuda.synchronize()
    assert bool((out == 0).all())                 # no rows: zeros
    assert bool((f32 == 3.0).all())               # accumulating nothing leaves the buffer


def test_limit_zero_writes_nothing_anywhere(rd_lib):
    m, k, n = 512, 64, 256
    rng = np.random.default_rng(43)
    lhs = _normal(rng, (m, k)).to(DEV)
    w = _normal(rng, (4, k, n), 1 / k).to(DEV)
    fused = _normal(rng, (m, 2 * k)).to(DEV)
    gs = _i32([100, 200, 100, 112])
    zero = _i32([0])
    outs = [_sentinel_buffer(m, n), _sentinel_buffer(m, n // 2), _sentinel_buffer(m, k),
            _sentinel_buffer(m, 2 * k), _sentinel_buffer(m, k)]
    rd_lib.ragged_dot(lhs, w, gs, limit=zero, out=outs[0][:m])
    rd_lib.ragged_dot(lhs, w, gs, limit=zero, epilogue=rd_lib.EPI_SILU_GLU, out=outs[1][:m])
    d_out = _normal(rng, (m, n)).to(DEV)
    rd_lib.ragged_dot_trans_rhs(d_out, w, gs, limit=zero, out=outs[2][:m])
    rd_lib.ragged_dot_trans_rhs_glu_bwd(d_out, w, fused, gs, limit=zero, out=outs[3][:m])
    rd_lib.glu_fwd(fused, limit=zero, out=outs[4][:m])
    torch.cuda.synchronize()
    for o in outs:
        assert bool((o.view(torch.int16) == SENT).all())


def test_binding_rejects_mismatched_buffers(rd_lib):
    """The C ABI sees only pointers and sizes, so the binding checks caller-supplied outputs."""
    lhs = torch.zeros((64, 32), dtype=torch.bfloat16, device=DEV)
    rhs = torch.zeros((2, 32, 64), dtype=torch.bfloat16, device=DEV)
    gs = _i32([32, 32])
    bad = [
        lambda: rd_lib.ragged_dot(lhs, rhs, gs, out=torch.empty((63, 64), dtype=torch.bfloat16, device=DEV)),
        lambda: rd_lib.ragged_dot(lhs, rhs, gs, epilogue=rd_lib.EPI_SILU_GLU,
                                  out=torch.empty((64, 64), dtype=torch.bfloat16, device=DEV)),
        lambda: rd_lib.ragged_dot(lhs, rhs, gs, out=torch.empty((64, 64), dtype=torch.float32, device=DEV)),
        lambda: rd_lib.ragged_dot(lhs, rhs, gs, out=torch.empty((64, 128), dtype=torch.bfloat16,
                                                                 device=DEV)[:, ::2]),
        lambda: rd_lib.ragged_dot(lhs, rhs.cpu(), gs),
        lambda: rd_lib.ragged_dot_trans_rhs(lhs[:, :32], rhs.transpose(1, 2).contiguous(), gs,
                                            out=torch.empty((64, 63), dtype=torch.bfloat16, device=DEV)),
        lambda: rd_lib.trans_ragged_dot(lhs, lhs, gs, out=torch.empty((2, 32, 31), dtype=torch.bfloat16,
                                                                        device=DEV)),
        lambda: rd_lib.glu_fwd(lhs, out=torch.empty((64, 32), dtype=torch.bfloat16, device=DEV)),
        lambda: rd_lib.glu_fwd(lhs, limit=_i32([1, 2])),
    ]
    for i, call in enumerate(bad):
        try:
            call()
        except ValueError:
            continue
        raise AssertionError(f"case {i} was accepted")
