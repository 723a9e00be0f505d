"""Parity at the full workload sizes, in the launch configuration the bench times.

Every output element is compared with the oracle: the oracle's own functions
run group by group on row chunks of a few thousand rows (float64 on the host
cores), so the whole output of each full-size call is checked, not a sample.
Properties that hold at any size are checked on the whole output on the
device as well: rows past the limit keep their sentinel, rows outside the
local groups are exactly +0.
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
CHUNK = 4096     # rows per oracle call


def _f64(t):
    return obf.torch_bf16_to_f64(t)


def _chunks(lo, hi, ch=CHUNK):
    for r0 in range(int(lo), int(hi), ch):
        yield r0, min(r0 + ch, int(hi))


def _amax(t):
    return float(t.float().abs().max()) if t.numel() else 0.0


def check_forward_full(out, lhs, rhs, sizes, off, L, what, glu=False):
    """Every row of every local group of a forward (optionally GLU) output vs the oracle."""
    m, k = lhs.shape
    g_local = rhs.shape[0]
    b, _ = oracle.group_bounds(sizes, m, L)
    amax, bmax = _amax(lhs[:L]), _amax(rhs)
    E = 1e-3 * math.sqrt(k) * amax * bmax
    for jl in range(g_local):
        lo, hi = b[off + jl], b[off + jl + 1]
        if hi <= lo:
            continue
        w64 = _f64(rhs[jl])[None]
        for r0, r1 in _chunks(lo, hi):
            plain = oracle.ragged_dot(_f64(lhs[r0:r1]), w64, [r1 - r0])
            if glu:
                F = plain.shape[1] // 2
                ref, tol = glu_epilogue_tol(plain[:, :F], plain[:, F:], E)
            else:
                ref, tol = plain, gemm_tol(plain, k, amax, bmax)
            assert_close(_f64(out[r0:r1]), ref, tol, f"{what} group {off + jl} rows [{r0}, {r1})")


def check_dx_full(out, d_out, w, sizes, off, L, what):
    """Every row of every local group of a trans_rhs output vs the oracle."""
    m, n = d_out.shape
    b, _ = oracle.group_bounds(sizes, m, L)
    amax, bmax = _amax(d_out[:L]), _amax(w)
    for jl in range(w.shape[0]):
        lo, hi = b[off + jl], b[off + jl + 1]
        if hi <= lo:
            continue
        w64 = _f64(w[jl])[None]
        for r0, r1 in _chunks(lo, hi):
            ref = oracle.ragged_dot_trans_rhs(_f64(d_out[r0:r1]), w64, [r1 - r0])
            assert_close(_f64(out[r0:r1]), ref, gemm_tol(ref, n, amax, bmax),
                         f"{what} group {off + jl} rows [{r0}, {r1})")


def test_mixtral_forward_full_size(rd_lib):
    from workloads import mixtral_fwd, normal_bf16

    w = mixtral_fwd()
    lhs = normal_bf16((w.m, w.k), w.lhs_var, 20, DEV)
    rhs = normal_bf16((w.g_total, w.k, w.n), w.rhs_var, 21, DEV)
    gs = torch.tensor(w.group_sizes, dtype=torch.int32, device=DEV)
    out = torch.empty((w.m, w.n), dtype=torch.bfloat16, device=DEV)
    out.fill_(float("nan"))
    rd_lib.ragged_dot(lhs, rhs, gs, out=out)
    torch.cuda.synchronize()
    # every row is in a group (the sizes sum to m): nothing may keep the NaN fill
    assert not bool(torch.isnan(out).any()), "output rows left unwritten"
    check_forward_full(out, lhs, rhs, w.group_sizes, 0, w.m, "mixtral")


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
    check_forward_full(out, lhs, rhs, w.group_sizes, w.group_offset, L, "packed glu", glu=True)


def test_backward_pair_full_size(rd_lib):
    from workloads import backward_pair, normal_bf16

    w = backward_pair()
    x = normal_bf16((w.m, w.k), 1.0, 40, DEV)
    do = normal_bf16((w.m, w.n), 1.0, 41, DEV)
    wt = normal_bf16((w.g_total, w.k, w.n), w.rhs_var, 42, DEV)
    gs = torch.tensor(w.group_sizes, dtype=torch.int32, device=DEV)
    dx = torch.full((w.m, w.k), float("nan"), dtype=torch.bfloat16, device=DEV)
    dw = torch.full((w.g_total, w.k, w.n), float("nan"), dtype=torch.bfloat16, device=DEV)
    rd_lib.ragged_dot_trans_rhs(do, wt, gs, out=dx)
    rd_lib.trans_ragged_dot(x, do, gs, out=dw)
    torch.cuda.synchronize()
    assert not bool(torch.isnan(dx).any()), "dx rows left unwritten"
    assert not bool(torch.isnan(dw).any()), "dw blocks left unwritten"
    check_dx_full(dx, do, wt, w.group_sizes, 0, w.m, "dx")
    b, _ = oracle.group_bounds(w.group_sizes, w.m)
    for j in range(w.g_total):
        lo, hi = int(b[j]), int(b[j + 1])
        if hi == lo:
            assert bool((dw[j].view(torch.int16) == 0).all()), f"empty group {j} not +0"
            continue
        xs, ys = _f64(x[lo:hi]), _f64(do[lo:hi])
        ref = oracle.trans_ragged_dot(xs, ys, [hi - lo])[0]
        tol = gemm_tol(ref, hi - lo, np.abs(xs).max(), np.abs(ys).max())
        assert_close(_f64(dw[j]), ref, tol, f"dw group {j}")


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
    h.fill_(float("nan"))
    o.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        rd_lib.ragged_dot(lhs, up, gs, epilogue=rd_lib.EPI_SILU_GLU, out=h)
        rd_lib.ragged_dot(h_in, down, gs, out=o)
    g.replay()
    torch.cuda.synchronize()
    assert not bool(torch.isnan(h).any()) and not bool(torch.isnan(o).any()), "rows left unwritten"
    check_forward_full(h, lhs, up, w.group_sizes, 0, w.m, "decode up", glu=True)
    check_forward_full(o, h_in, down, w.group_sizes, 0, w.m, "decode down")


@pytest.mark.parametrize("tokens", [4096, 16384])
def test_expert_ffn_chain_in_one_graph(rd_lib, tokens):
    """Up projection with the GLU epilogue feeding the down projection, one CUDA graph.

    The expert FFN forward at batches between weight-bound and compute-bound
    (4096 and 16384 tokens, top-8 of 128 experts).  The down call consumes the
    h the up call wrote inside the same graph; every element of both outputs is
    checked (h against the float64 GLU of the up GEMM, the output against the
    float64 down GEMM of that h), and on the device every row of both must have
    been written.
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
    check_forward_full(h, lhs, up, w.group_sizes, 0, w.m, f"ffn {tokens} up", glu=True)
    check_forward_full(o, h, down, w.group_sizes, 0, w.m, f"ffn {tokens} down")


def test_backward_pair_dw_f32_full_size(rd_lib):
    """dw kept in f32 at the backward-pair size: stored, and accumulated into a prior buffer.

    Every entry of every group against float64, within the worst-case error of
    an f32 sum of the exact products (plus one f32 rounding for the
    accumulating add); groups without rows are zero when stored and keep their
    prior block when accumulated.
    """
    from oracle import ragged
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
    for j in range(w.g_total):
        lo, hi = int(b[j]), int(b[j + 1])
        if hi == lo:
            assert bool((stored[j] == 0).all()), f"empty group {j} not zero"
            assert torch.equal(acc[j], prior[j]), f"empty group {j} changed its prior block"
            continue
        xs, ys = _f64(x[lo:hi]), _f64(do[lo:hi])
        p64 = prior[j].cpu().numpy().astype(np.float64)
        ref = oracle.trans_ragged_dot_f32(xs, ys, [hi - lo])[0]
        bound = ragged.f32_sum_bound(xs, ys, [hi - lo])[0]
        assert_close(stored[j].cpu().numpy(), ref, bound, f"dw f32 group {j}")
        want = oracle.trans_ragged_dot_f32(xs, ys, [hi - lo], out_prior=p64[None])[0]
        tol = bound + np.abs(np.spacing(want.astype(np.float32))).astype(np.float64)
        assert_close(acc[j].cpu().numpy(), want, tol, f"dw f32 accumulated group {j}")


def test_packed_dx_glu_bwd_full_size(rd_lib):
    """dx of the down projection with the GLU backward fused, on the packed buffer.

    [225280, 4096] output gradient, experts 16..31 of 64 with down weights
    [16, 1024, 4096], the saved [gate | up] rows, limit 126156 -- the launch the
    bench times.  Rows past the limit keep their sentinel, rows below it outside
    the local groups are +0 (both checked on the device), and every element of
    every local row matches float64 within the fused-epilogue bound.
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
    E = 1e-3 * math.sqrt(n) * _amax(d_out[lo_all:hi_all]) * _amax(w_down)
    for jl in range(w.g_local):
        lo, hi = int(b[w.group_offset + jl]), int(b[w.group_offset + jl + 1])
        if hi <= lo:
            continue
        w64 = _f64(w_down[jl])[None]
        for r0, r1 in _chunks(lo, hi):
            fz = _f64(fused[r0:r1])
            ref = oracle.ragged_dot_trans_rhs_glu_bwd(_f64(d_out[r0:r1]), w64, fz, [r1 - r0])
            dg1, du1 = oglu.glu_bwd_f64(fz[:, :f], fz[:, f:], 1.0)
            tol = obf.ulp(ref) + np.concatenate([np.abs(dg1), np.abs(du1)], axis=1) * E
            got = _f64(out[r0:r1])
            assert not np.any(obf.torch_bf16_bits(out[r0:r1]) == 0x8000), "a -0 survived"
            assert_close(got, ref, tol, f"dx+glu bwd group {w.group_offset + jl} rows [{r0}, {r1})")
