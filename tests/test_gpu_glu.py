"""GPU parity of the standalone SiLU-GLU kernels against the oracle.

Every bf16 bit pattern appears as a gate, with random up / d values and the
special values +-0, +-inf, NaN and subnormals as up / d (the sweep design of
MaxText PR #5760's glu_rows checks), at full and partial valid-row counts.
"""
import numpy as np
import pytest

import oracle
from oracle import bf16 as obf
from parity_util import exp_overflows_f32

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda"
SENT = 0x3C3C
CANARY_ROWS = 4     # rows after each output buffer that no call may touch
SPECIAL = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0x0001, 0x8001, 0x007F, 0x3F80,
                    0xBF80], np.uint16)


def _bits_tensor(bits_np):
    return torch.from_numpy(bits_np.astype(np.uint16).view(np.int16).copy()).view(torch.bfloat16)


def _sweep_inputs(rows, f, seed):
    """fused [rows, 2f] with every bf16 pattern as a gate, d [rows, f]."""
    rng = np.random.default_rng(seed)
    n = rows * f
    gate = np.resize(np.arange(1 << 16, dtype=np.uint32).astype(np.uint16), n)
    up = obf.round_f32_to_bf16_bits(rng.standard_normal(n).astype(np.float32))
    d = obf.round_f32_to_bf16_bits(rng.standard_normal(n).astype(np.float32))
    # sprinkle special values into up and d
    idx = rng.choice(n, size=n // 16, replace=False)
    up[idx] = rng.choice(SPECIAL, size=idx.size)
    idx = rng.choice(n, size=n // 16, replace=False)
    d[idx] = rng.choice(SPECIAL, size=idx.size)
    fused = np.concatenate([gate.reshape(rows, f), up.reshape(rows, f)], axis=1)
    return fused, d.reshape(rows, f)


def _compare(got_bits, g, ref64, ref32_bits, what):
    """1 bf16 ulp of float64 where both are finite and exp(-g) is finite in f32; else bits."""
    got = obf.bits_to_f32(got_bits).astype(np.float64)
    ref32 = obf.bits_to_f32(ref32_bits).astype(np.float64)
    regular = np.isfinite(ref64) & np.isfinite(ref32) & ~exp_overflows_f32(g)
    err = np.abs(got[regular] - ref64[regular])
    bad = err > obf.ulp(ref64[regular])
    assert not np.any(bad), f"{what}: {int(bad.sum())} regular values beyond 1 bf16 ulp"
    special = ~regular
    gs, rs = got_bits[special], ref32_bits[special]
    both_nan = np.isnan(obf.bits_to_f32(gs)) & np.isnan(obf.bits_to_f32(rs))
    mism = (gs != rs) & ~both_nan
    assert not np.any(mism), f"{what}: {int(mism.sum())} special values differ from the f32 sequence"


@pytest.mark.parametrize("rows,f,limit", [(512, 128, None), (520, 128, 517), (1024, 64, 1000)])
def test_glu_fwd_exhaustive_gates(rd_lib, rows, f, limit):
    fused, _ = _sweep_inputs(rows, f, seed=rows + f)
    L = rows if limit is None else limit
    fused_dev = _bits_tensor(fused).to(DEV)
    if L < rows:
        fused_dev[L:] = float("nan")
    buf = torch.empty((rows + CANARY_ROWS, f), dtype=torch.bfloat16, device=DEV)
    buf.view(torch.int16).fill_(SENT)
    rd_lib.glu_fwd(fused_dev, limit=None if limit is None else torch.tensor([limit], dtype=torch.int32,
                                                                             device=DEV), out=buf[:rows])
    torch.cuda.synchronize()
    got = obf.torch_bf16_bits(buf)
    assert np.all(got[L:] == SENT), "a row past the limit or a canary row after the output was written"
    g = obf.bits_to_f32(fused[:L, :f])
    u = obf.bits_to_f32(fused[:L, f:])
    ref64 = oracle.glu_fwd_f64(g, u)
    ref32_bits, _ = oracle.glu_fwd_f32(g, u)
    _compare(got[:L], g, ref64, ref32_bits, "glu_fwd")


@pytest.mark.parametrize("rows,f,limit", [(512, 128, None), (520, 128, 3), (1024, 64, 1000)])
def test_glu_bwd_exhaustive_gates(rd_lib, rows, f, limit):
    fused, d = _sweep_inputs(rows, f, seed=rows * 3 + f)
    L = rows if limit is None else limit
    fused_dev = _bits_tensor(fused).to(DEV)
    d_dev = _bits_tensor(d).to(DEV)
    if L < rows:
        fused_dev[L:] = float("nan")
        d_dev[L:] = float("nan")
    buf = torch.empty((rows + CANARY_ROWS, 2 * f), dtype=torch.bfloat16, device=DEV)
    buf.view(torch.int16).fill_(SENT)
    rd_lib.glu_bwd(fused_dev, d_dev, limit=None if limit is None else torch.tensor([limit], dtype=torch.int32,
                                                                                     device=DEV), out=buf[:rows])
    torch.cuda.synchronize()
    got = obf.torch_bf16_bits(buf)
    assert np.all(got[L:] == SENT), "a row past the limit or a canary row after the output was written"
    g = obf.bits_to_f32(fused[:L, :f])
    u = obf.bits_to_f32(fused[:L, f:])
    dd = obf.bits_to_f32(d[:L])
    want_g64, want_u64 = oracle.glu_bwd_f64(g, u, dd)
    (bg, bu), _ = oracle.glu_bwd_f32(g, u, dd)
    _compare(got[:L, :f], g, want_g64, bg, "glu_bwd d_gate")
    _compare(got[:L, f:], g, want_u64, bu, "glu_bwd d_up")
    assert not np.any(got[:L] == 0x8000), "a -0 survived the -0 -> +0 fix"


@pytest.mark.parametrize("limit", [0, 1, 1023, 125952, 126156, 225280])
def test_glu_limits_packed_buffer_rows(rd_lib, limit):
    """The page's limit list on a [225280, 2*256] buffer: rows >= limit untouched.

    Every valid row of both outputs is compared with the oracle (forward and
    backward, each against its float64 value and the f32 op sequence's special
    bits), and canary rows after both buffers must keep their sentinel.
    """
    rows, f = 225280, 256
    gen = torch.Generator(device=DEV).manual_seed(limit + 1)
    fused = torch.randn((rows, 2 * f), generator=gen, device=DEV).to(torch.bfloat16)
    obuf = torch.empty((rows + CANARY_ROWS, f), dtype=torch.bfloat16, device=DEV)
    obuf.view(torch.int16).fill_(SENT)
    out = obuf[:rows]
    lim = torch.tensor([limit], dtype=torch.int32, device=DEV)
    rd_lib.glu_fwd(fused, limit=lim, out=out)
    dbuf = torch.empty((rows + CANARY_ROWS, 2 * f), dtype=torch.bfloat16, device=DEV)
    dbuf.view(torch.int16).fill_(SENT)
    rd_lib.glu_bwd(fused, out, limit=lim, out=dbuf[:rows])
    torch.cuda.synchronize()
    sent = torch.tensor(SENT, dtype=torch.int16, device=DEV)
    assert bool((obuf[limit:].view(torch.int16) == sent).all())
    assert bool((dbuf[limit:].view(torch.int16) == sent).all())
    for r0 in range(0, limit, 32768):
        r1 = min(r0 + 32768, limit)
        fb = obf.torch_bf16_bits(fused[r0:r1])
        g, u = obf.bits_to_f32(fb[:, :f]), obf.bits_to_f32(fb[:, f:])
        bits, _ = oracle.glu_fwd_f32(g, u)
        got = obf.torch_bf16_bits(out[r0:r1])
        _compare(got, g, oracle.glu_fwd_f64(g, u), bits, f"glu_fwd rows [{r0}, {r1})")
        dd = obf.bits_to_f32(got)        # the backward's d is the forward's output
        want_g64, want_u64 = oracle.glu_bwd_f64(g, u, dd)
        (bg, bu), _ = oracle.glu_bwd_f32(g, u, dd)
        gotd = obf.torch_bf16_bits(dbuf[r0:r1])
        _compare(gotd[:, :f], g, want_g64, bg, f"glu_bwd d_gate rows [{r0}, {r1})")
        _compare(gotd[:, f:], g, want_u64, bu, f"glu_bwd d_up rows [{r0}, {r1})")
