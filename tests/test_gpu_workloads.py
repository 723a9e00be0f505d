"""Parity at the full workload sizes, in the launch configuration the bench times.

The oracle computes sampled outputs one by one (sampled rows x sampled
columns, every group, both edges of every group); properties that hold at any
size are checked on the whole output on the device: rows past the limit keep
their sentinel, rows outside the local groups are exactly +0.
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
SENT = 0x3C3C


def _f64(t):
    return obf.torch_bf16_to_f64(t)


def _sample_rows(b, lo_group, hi_group, rng, per_group=6):
    rows = []
    for j in range(lo_group, hi_group):
        lo, hi = int(b[j]), int(b[j + 1])
        if hi > lo:
            rows += [lo, hi - 1] + rng.integers(lo, hi, per_group).tolist()
    return np.unique(np.array(rows, dtype=np.int64))


def _sample_cols(n, rng, count=192, tile=256):
    cols = np.r_[0:8, n - 8:n, tile - 4:tile + 4, rng.integers(0, n, count)]
    return np.unique(cols[(cols >= 0) & (cols < n)])


def _group_of(rows, b):
    return np.searchsorted(b, rows, side="right") - 1


def test_mixtral_forward_full_size(rd_lib):
    from workloads import mixtral_fwd, normal_bf16

    w = mixtral_fwd()
    lhs = normal_bf16((w.m, w.k), w.lhs_var, 20, DEV)
    rhs = normal_bf16((w.g_total, w.k, w.n), w.rhs_var, 21, DEV)
    gs = torch.tensor(w.group_sizes, dtype=torch.int32, device=DEV)
    out = rd_lib.ragged_dot(lhs, rhs, gs)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    b, _ = oracle.group_bounds(w.group_sizes, w.m)
    rows = _sample_rows(b, 0, w.g_total, rng)
    cols = _sample_cols(w.n, rng)
    a64 = _f64(lhs[torch.from_numpy(rows).to(DEV)])
    got = _f64(out[torch.from_numpy(rows).to(DEV)][:, torch.from_numpy(cols).to(DEV)])
    amax = float(lhs.float().abs().max())
    bmax = float(rhs.float().abs().max())
    grp = _group_of(rows, b)
    for j in range(w.g_total):
        sel = grp == j
        if not sel.any():
            continue
        wj = _f64(rhs[j][:, torch.from_numpy(cols).to(DEV)])
        ref = a64[sel] @ wj
        assert_close(got[sel], ref, gemm_tol(ref, w.k, amax, bmax), f"mixtral group {j}")


def test_packed_glu_forward_full_size(rd_lib):
    from workloads import normal_bf16, packed_glu_fwd

    w = packed_glu_fwd()
    F = w.n // 2
    lhs = normal_bf16((w.m, w.k), 1.0, 30, DEV)
    lhs[w.limit:] = float("nan")             # rows past the limit must not be read
    rhs = normal_bf16((w.g_local, w.k, w.n), w.rhs_var, 31, DEV)
    gs = torch.tensor(w.group_sizes, dtype=torch.int32, device=DEV)
    lim = torch.tensor([w.limit], dtype=torch.int32, device=DEV)
    out = torch.empty((w.m, F), dtype=torch.bfloat16, device=DEV)
    out.view(torch.int16).fill_(SENT)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    rd_lib.ragged_dot(lhs, rhs, gs, w.group_offset, lim, rd_lib.EPI_SILU_GLU, out, status)
    torch.cuda.synchronize()
    b, L = oracle.group_bounds(w.group_sizes, w.m, w.limit)
    s0, s1 = int(b[w.group_offset]), int(b[w.group_offset + w.g_local])
    o16 = out.view(torch.int16)
    assert bool((o16[L:] == SENT).all()), "rows past the limit were written"
    assert bool((o16[:s0] == 0).all()) and bool((o16[s1:L] == 0).all()), "non-local rows not +0"
    assert int(status.item()) == 0
    rng = np.random.default_rng(1)
    rows = _sample_rows(b, w.group_offset, w.group_offset + w.g_local, rng)
    cols = _sample_cols(F, rng, tile=128)
    ridx = torch.from_numpy(rows).to(DEV)
    a64 = _f64(lhs[ridx])
    got = _f64(out[ridx][:, torch.from_numpy(cols).to(DEV)])
    amax = float(lhs[:L].float().abs().max())
    bmax = float(rhs.float().abs().max())
    E = 1e-3 * math.sqrt(w.k) * amax * bmax
    grp = _group_of(rows, b) - w.group_offset
    for j in range(w.g_local):
        sel = grp == j
        wg = _f64(rhs[j][:, torch.from_numpy(cols).to(DEV)])
        wu = _f64(rhs[j][:, torch.from_numpy(cols + F).to(DEV)])
        ref, tol = glu_epilogue_tol(a64[sel] @ wg, a64[sel] @ wu, E)
        assert_close(got[sel], ref, tol, f"packed glu group {j}")


def test_backward_pair_full_size(rd_lib):
    from workloads import backward_pair, normal_bf16

    w = backward_pair()
    x = normal_bf16((w.m, w.k), 1.0, 40, DEV)
    do = normal_bf16((w.m, w.n), 1.0, 41, DEV)
    wt = normal_bf16((w.g_total, w.k, w.n), w.rhs_var, 42, DEV)
    gs = torch.tensor(w.group_sizes, dtype=torch.int32, device=DEV)
    dx = rd_lib.ragged_dot_trans_rhs(do, wt, gs)
    dw = rd_lib.trans_ragged_dot(x, do, gs)
    torch.cuda.synchronize()
    rng = np.random.default_rng(2)
    b, _ = oracle.group_bounds(w.group_sizes, w.m)
    # dx: sampled rows x sampled columns of [m, k]
    rows = _sample_rows(b, 0, w.g_total, rng, per_group=2)
    cols = _sample_cols(w.k, rng)
    ridx, cidx = torch.from_numpy(rows).to(DEV), torch.from_numpy(cols).to(DEV)
    d64 = _f64(do[ridx])
    got = _f64(dx[ridx][:, cidx])
    amax, bmax = float(do.float().abs().max()), float(wt.float().abs().max())
    grp = _group_of(rows, b)
    for j in range(w.g_total):
        sel = grp == j
        if sel.any():
            ref = d64[sel] @ _f64(wt[j][cidx]).T
            assert_close(got[sel], ref, gemm_tol(ref, w.n, amax, bmax), f"dx group {j}")
    # dw: every group, sampled (k, n) entries; empty groups exactly zero
    kk = _sample_cols(w.k, rng, 48, tile=128)
    nn = _sample_cols(w.n, rng, 48)
    for j in range(w.g_total):
        lo, hi = int(b[j]), int(b[j + 1])
        blk = dw[j][torch.from_numpy(kk).to(DEV)][:, torch.from_numpy(nn).to(DEV)]
        if hi == lo:
            assert bool((dw[j].view(torch.int16) == 0).all()), f"empty group {j} not +0"
            continue
        xs = _f64(x[lo:hi][:, torch.from_numpy(kk).to(DEV)])
        ys = _f64(do[lo:hi][:, torch.from_numpy(nn).to(DEV)])
        ref = xs.T @ ys
        tol = gemm_tol(ref, hi - lo, float(x[lo:hi].float().abs().max()),
                       float(do[lo:hi].float().abs().max()))
        assert_close(_f64(blk), ref, tol, f"dw group {j}")


@pytest.mark.parametrize("skewed", [True, False])
def test_decode_pair_in_one_graph(rd_lib, skewed):
    """Up (GLU epilogue) and down projections sharing group_sizes inside one CUDA graph."""
    from workloads import decode_fwd, normal_bf16

    w = decode_fwd(skewed)
    F = w.n // 2
    lhs = normal_bf16((w.m, w.k), 1.0, 50, DEV)
    up = normal_bf16((w.g_total, w.k, w.n), w.rhs_var, 51, DEV)
    down = normal_bf16((w.g_total, F, w.k), 1.0 / F, 52, DEV)
    h_in = normal_bf16((w.m, F), 1.0, 53, DEV)     # independent input of the down call
    gs = torch.tensor(w.group_sizes, dtype=torch.int32, device=DEV)
    h = torch.empty((w.m, F), dtype=torch.bfloat16, device=DEV)
    o = torch.empty((w.m, w.k), dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        rd_lib.ragged_dot(lhs, up, gs, epilogue=rd_lib.EPI_SILU_GLU, out=h)
        rd_lib.ragged_dot(h_in, down, gs, out=o)
    torch.cuda.synchronize()
    h.zero_()
    o.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        rd_lib.ragged_dot(lhs, up, gs, epilogue=rd_lib.EPI_SILU_GLU, out=h)
        rd_lib.ragged_dot(h_in, down, gs, out=o)
    g.replay()
    torch.cuda.synchronize()
    b, _ = oracle.group_bounds(w.group_sizes, w.m)
    rng = np.random.default_rng(3)
    cols = _sample_cols(F, rng, 96, tile=128)
    cidx = torch.from_numpy(cols).to(DEV)
    a64 = _f64(lhs)
    E = 1e-3 * math.sqrt(w.k) * float(lhs.float().abs().max()) * float(up.float().abs().max())
    got_h = _f64(h[:, cidx])
    ocols = _sample_cols(w.k, rng, 96)
    ocidx = torch.from_numpy(ocols).to(DEV)
    got_o = _f64(o[:, ocidx])
    h64 = _f64(h_in)
    Eo_amax, Eo_bmax = float(h_in.float().abs().max()), float(down.float().abs().max())
    for j in range(w.g_total):
        lo, hi = int(b[j]), int(b[j + 1])
        if hi == lo:
            continue
        ref, tol = glu_epilogue_tol(a64[lo:hi] @ _f64(up[j][:, cidx]),
                                    a64[lo:hi] @ _f64(up[j][:, cidx + F]), E)
        assert_close(got_h[lo:hi], ref, tol, f"decode up group {j}")
        ref = h64[lo:hi] @ _f64(down[j][:, ocidx])
        assert_close(got_o[lo:hi], ref, gemm_tol(ref, F, Eo_amax, Eo_bmax), f"decode down group {j}")


@pytest.mark.parametrize("tokens", [4096, 16384])
def test_expert_ffn_chain_in_one_graph(rd_lib, tokens):
    """Up projection with the GLU epilogue feeding the down projection, one CUDA graph.

    The expert FFN forward at batches between weight-bound and compute-bound
    (4096 and 16384 tokens, top-8 of 128 experts).  The down call consumes the
    h the up call wrote inside the same graph; both outputs are checked on
    sampled rows and columns of every live group (h against the float64 GLU of
    the up GEMM, the output against the float64 down GEMM of that h), and on
    the device every row of both must have been written.
    """
    from workloads import expert_ffn, normal_bf16

    w = expert_ffn(tokens)
    F = w.n // 2
    lhs = normal_bf16((w.m, w.k), w.lhs_var, 63, DEV)
    up = normal_bf16((w.g_total, w.k, w.n), w.rhs_var, 61, DEV)
    down = normal_bf16((w.g_total, F, w.k), 1.0 / F, 62, DEV)
    gs = torch.tensor(w.group_sizes, dtype=torch.int32, device=DEV)
    h = torch.empty((w.m, F), dtype=torch.bfloat16, device=DEV)
    o = torch.empty((w.m, w.k), dtype=torch.bfloat16, device=DEV)

    def chain():
        rd_lib.ragged_dot(lhs, up, gs, epilogue=rd_lib.EPI_SILU_GLU, out=h)
        rd_lib.ragged_dot(h, down, gs, out=o)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        chain()
    torch.cuda.synchronize()
    h.fill_(float("nan"))
    o.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        chain()
    g.replay()
    torch.cuda.synchronize()
    # every row is in a group (the sizes sum to m): nothing may keep the NaN fill
    assert not bool(torch.isnan(h).any()), "h rows left unwritten"
    assert not bool(torch.isnan(o).any()), "output rows left unwritten"

    b, _ = oracle.group_bounds(w.group_sizes, w.m)
    rng = np.random.default_rng(tokens)
    rows = _sample_rows(b, 0, w.g_total, rng, per_group=4)
    ridx = torch.from_numpy(rows).to(DEV)
    cols = _sample_cols(F, rng, 96, tile=128)
    cidx = torch.from_numpy(cols).to(DEV)
    ocols = _sample_cols(w.k, rng, 96)
    ocidx = torch.from_numpy(ocols).to(DEV)
    a64 = _f64(lhs[ridx])
    h_rows = h[ridx]
    h64 = _f64(h_rows)
    got_h = _f64(h_rows[:, cidx])
    got_o = _f64(o[ridx][:, ocidx])
    E = 1e-3 * math.sqrt(w.k) * float(lhs.float().abs().max()) * float(up.float().abs().max())
    h_amax, d_amax = float(h.float().abs().max()), float(down.float().abs().max())
    grp = _group_of(rows, b)
    for j in np.unique(grp):
        sel = np.nonzero(grp == j)[0]
        ref, tol = glu_epilogue_tol(a64[sel] @ _f64(up[j][:, cidx]),
                                    a64[sel] @ _f64(up[j][:, cidx + F]), E)
        assert_close(got_h[sel], ref, tol, f"ffn {tokens} up group {j}")
        ref = h64[sel] @ _f64(down[j][:, ocidx])
        assert_close(got_o[sel], ref, gemm_tol(ref, F, h_amax, d_amax),
                     f"ffn {tokens} down group {j}")


def test_backward_pair_dw_f32_full_size(rd_lib):
    """dw kept in f32 at the backward-pair size: stored, and accumulated into a prior buffer.

    Sampled (k, n) entries of every group against float64, within the worst-case
    error of an f32 sum of the exact products (plus one f32 rounding for the
    accumulating add); groups without rows are zero when stored and keep their
    prior block when accumulated.
    """
    from workloads import backward_pair, normal_bf16

    w = backward_pair()
    x = normal_bf16((w.m, w.k), 1.0, 40, DEV)
    do = normal_bf16((w.m, w.n), 1.0, 41, DEV)
    gs = torch.tensor(w.group_sizes, dtype=torch.int32, device=DEV)
    gen = torch.Generator(device=DEV).manual_seed(44)
    prior = torch.randn((w.g_total, w.k, w.n), generator=gen, device=DEV)
    stored = rd_lib.trans_ragged_dot_f32(x, do, gs)
    acc = prior.clone()
    rd_lib.trans_ragged_dot_f32(x, do, gs, out=acc, accumulate=True)
    torch.cuda.synchronize()
    b, _ = oracle.group_bounds(w.group_sizes, w.m)
    rng = np.random.default_rng(5)
    kk = torch.from_numpy(_sample_cols(w.k, rng, 40, tile=128)).to(DEV)
    nn = torch.from_numpy(_sample_cols(w.n, rng, 40)).to(DEV)
    for j in range(w.g_total):
        lo, hi = int(b[j]), int(b[j + 1])
        if hi == lo:
            assert bool((stored[j] == 0).all()), f"empty group {j} not zero"
            assert torch.equal(acc[j], prior[j]), f"empty group {j} changed its prior block"
            continue
        xs, ys = _f64(x[lo:hi][:, kk]), _f64(do[lo:hi][:, nn])
        ref = xs.T @ ys
        bound = (hi - lo) * 2.0 ** -23 * (np.abs(xs).T @ np.abs(ys))
        got = stored[j][kk][:, nn].cpu().numpy().astype(np.float64)
        assert_close(got, ref, bound, f"dw f32 group {j}")
        p64 = prior[j][kk][:, nn].cpu().numpy().astype(np.float64)
        want = p64 + ref
        tol = bound + np.abs(np.spacing(want.astype(np.float32))).astype(np.float64)
        got = acc[j][kk][:, nn].cpu().numpy().astype(np.float64)
        assert_close(got, want, tol, f"dw f32 accumulated group {j}")


def test_packed_dx_glu_bwd_full_size(rd_lib):
    """dx of the down projection with the GLU backward fused, on the packed buffer.

    [225280, 4096] output gradient, experts 16..31 of 64 with down weights
    [16, 1024, 4096], the saved [gate | up] rows, limit 126156 -- the launch the
    bench times.  Rows past the limit keep their sentinel, rows below it outside
    the local groups are +0 (both checked on the device), and sampled rows x
    columns of every local group match float64 within the fused-epilogue bound.
    """
    from oracle import glu as oglu
    from workloads import normal_bf16, packed_glu_fwd

    w = packed_glu_fwd()
    f, n = 1024, 4096
    gs = torch.tensor(w.group_sizes, dtype=torch.int32, device=DEV)
    lim = torch.tensor([w.limit], dtype=torch.int32, device=DEV)
    d_out = normal_bf16((w.m, n), 1.0, 35, DEV)
    w_down = normal_bf16((w.g_local, f, n), 1.0 / n, 36, DEV)
    fused = normal_bf16((w.m, 2 * f), 1.0, 37, DEV)
    out = torch.empty((w.m, 2 * f), dtype=torch.bfloat16, device=DEV)
    out.view(torch.int16).fill_(SENT)
    rd_lib.ragged_dot_trans_rhs_glu_bwd(d_out, w_down, fused, gs, w.group_offset, lim, out)
    torch.cuda.synchronize()
    b, L = oracle.group_bounds(w.group_sizes, w.m, w.limit)
    lo_all, hi_all = int(b[w.group_offset]), int(b[w.group_offset + w.g_local])
    assert bool((out[L:].view(torch.int16) == SENT).all()), "a row past the limit was written"
    assert bool((out[:lo_all].view(torch.int16) == 0).all()), "rows before the shard are not +0"
    assert bool((out[hi_all:L].view(torch.int16) == 0).all()), "rows after the shard are not +0"
    rng = np.random.default_rng(6)
    rows = _sample_rows(b, w.group_offset, w.group_offset + w.g_local, rng, per_group=3)
    ridx = torch.from_numpy(rows).to(DEV)
    cols = _sample_cols(f, rng, 64, tile=128)
    cidx = torch.from_numpy(cols).to(DEV)
    d64 = _f64(d_out[ridx])
    g64, u64 = _f64(fused[ridx][:, cidx]), _f64(fused[ridx][:, cidx + f])
    got_g, got_u = _f64(out[ridx][:, cidx]), _f64(out[ridx][:, cidx + f])
    E = 1e-3 * math.sqrt(n) * float(d_out[lo_all:hi_all].float().abs().max()) * \
        float(w_down.float().abs().max())
    grp = _group_of(rows, b) - w.group_offset
    for j in np.unique(grp):
        sel = np.nonzero(grp == j)[0]
        dh = d64[sel] @ _f64(w_down[j][cidx]).T
        ref_g, ref_u = oglu.glu_bwd_f64(g64[sel], u64[sel], dh)
        dg1, du1 = oglu.glu_bwd_f64(g64[sel], u64[sel], 1.0)
        assert_close(got_g[sel], ref_g, obf.ulp(ref_g) + np.abs(dg1) * E, f"d_gate group {j}")
        assert_close(got_u[sel], ref_u, obf.ulp(ref_u) + np.abs(du1) * E, f"d_up group {j}")
