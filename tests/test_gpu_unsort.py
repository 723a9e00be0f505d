"""GPU parity of the valid-rows unsort backward against the oracle.

The weighted gradient is compared bit for bit (one f32 multiply and one bf16
rounding on both sides); the row dot within the worst-case bound of an f32
summation; rows at or past the limit must keep their sentinel.  The limit list
and the two widths (one and several 2048-column blocks) follow the test design
of MaxText PR #5760's unsort_bwd_rows review.
"""
import numpy as np
import pytest

from oracle import bf16 as obf
from oracle import unsort

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda"
SENT = 0x3C3C
CANARY_ROWS = 4     # rows after each output buffer that no call may touch


def _run(rd, rows, hidden, limit, seed):
    from workloads import normal_bf16_np
    rng = np.random.default_rng(seed)
    g = normal_bf16_np(rng, (rows, hidden))
    y = normal_bf16_np(rng, (rows, hidden))
    w = torch.from_numpy(rng.uniform(-1.0, 1.0, rows).astype(np.float32))
    L = rows if limit is None else max(0, min(limit, rows))
    gd, yd, wd = g.to(DEV), y.to(DEV), w.to(DEV)
    gd[L:] = float("nan")
    yd[L:] = float("nan")
    wd[L:] = float("nan")
    gbuf = torch.empty((rows + CANARY_ROWS, hidden), dtype=torch.bfloat16, device=DEV)
    gbuf.view(torch.int16).fill_(SENT)
    dbuf = torch.full((rows + CANARY_ROWS,), 7.0, dtype=torch.float32, device=DEV)
    grad, dot = gbuf[:rows], dbuf[:rows]
    rd.unsort_bwd_rows(gd, yd, wd, limit=None if limit is None else torch.tensor([limit], dtype=torch.int32, device=DEV),
                       grad=grad, dot=dot)
    torch.cuda.synchronize()
    gb = obf.torch_bf16_bits(gbuf)
    assert np.all(gb[L:] == SENT), "gradient rows past the limit (or canary rows) were written"
    assert bool((dbuf[L:] == 7.0).all()), "dot entries past the limit (or canaries) were written"
    gb = gb[:rows]
    g32, y32 = g.float().numpy(), y.float().numpy()
    bits, _, ref = unsort.unsort_bwd_rows(g32, y32, w.numpy(), limit)
    np.testing.assert_array_equal(gb[:L], bits)
    tol = unsort.dot_tolerance(g32, y32, limit)
    err = np.abs(dot[:L].cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= tol), f"dot error {err.max()} beyond the f32 bound"


@pytest.mark.parametrize("hidden", [256, 4096])
@pytest.mark.parametrize("limit", [0, 1, 1000, 1700, 2048, None])
def test_unsort_bwd_rows(rd_lib, hidden, limit):
    _run(rd_lib, 2048, hidden, limit, seed=hidden + (limit or 0))


def test_unsort_bwd_rows_packed_buffer(rd_lib):
    """The page's bench shape: [225280, 4096] with 126156 valid rows, every valid row checked."""
    rows, hidden, limit = 225280, 4096, 126156
    gen = torch.Generator(device=DEV).manual_seed(7)
    g = torch.randn((rows, hidden), generator=gen, device=DEV).to(torch.bfloat16)
    y = torch.randn((rows, hidden), generator=gen, device=DEV).to(torch.bfloat16)
    w = torch.rand((rows,), generator=gen, device=DEV) * 2 - 1
    gbuf = torch.empty((rows + CANARY_ROWS, hidden), dtype=torch.bfloat16, device=DEV)
    gbuf.view(torch.int16).fill_(SENT)
    dbuf = torch.full((rows + CANARY_ROWS,), 7.0, dtype=torch.float32, device=DEV)
    grad, dot = gbuf[:rows], dbuf[:rows]
    rd_lib.unsort_bwd_rows(g, y, w, limit=torch.tensor([limit], dtype=torch.int32, device=DEV), grad=grad, dot=dot)
    torch.cuda.synchronize()
    assert bool((gbuf[limit:].view(torch.int16) == SENT).all())
    assert bool((dbuf[limit:] == 7.0).all())
    for r0 in range(0, limit, 16384):
        r1 = min(r0 + 16384, limit)
        g32, y32 = g[r0:r1].float().cpu().numpy(), y[r0:r1].float().cpu().numpy()
        bits, _, ref = unsort.unsort_bwd_rows(g32, y32, w[r0:r1].cpu().numpy())
        np.testing.assert_array_equal(obf.torch_bf16_bits(grad[r0:r1]), bits)
        err = np.abs(dot[r0:r1].cpu().numpy().astype(np.float64) - ref)
        assert np.all(err <= unsort.dot_tolerance(g32, y32)), f"row dot rows [{r0}, {r1})"
