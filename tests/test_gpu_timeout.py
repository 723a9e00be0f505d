"""Failure detection on the GPU without a fault: every bounded wait runs out.

With the wait bound set to 1 ns (rd_set_tuning) each wait inside the
grouped-GEMM kernel gives up at once.  The kernel must then unwind (let its copies and MMAs in flight finish,
free its tensor memory), return, and report RD_STATUS_TIMEOUT through the
status word; the next call on the same context must be correct again.
"""
import numpy as np
import pytest

import oracle
from oracle import bf16 as obf
from parity_util import assert_close, gemm_tol

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda"


def _inputs(op, seed):
    """Shapes whose waits last tens of microseconds (long contractions), so that
    a 1 ns bound certainly runs out whatever the resolution of the global timer."""
    from workloads import normal_bf16_np
    rng = np.random.default_rng(seed)
    if op.startswith("dw"):
        m, k, n, sizes = 16384, 256, 512, [4096, 4100, 4000, 4188]
    else:
        m, k, n, sizes = 1024, 8192, 512, [256, 300, 200, 268]
    if op == "dx":
        k, n = n, k      # dx contracts over n: do [m, 8192], w [g, 512, 8192]
    a = normal_bf16_np(rng, (m, k)).to(DEV)
    w = normal_bf16_np(rng, (len(sizes), k, n), 1.0 / k).to(DEV)
    do = normal_bf16_np(rng, (m, n)).to(DEV)
    return a, w, do, sizes


def _call(rd, op, a, w, do, gs, status):
    if op == "fwd":
        return rd.ragged_dot(a, w, gs, status=status)
    if op == "dx":
        return rd.ragged_dot_trans_rhs(do, w, gs, status=status)
    if op == "dw_nows":
        return rd.trans_ragged_dot(a, do, gs, status=status, workspace=None)
    return rd.trans_ragged_dot(a, do, gs, status=status)


@pytest.mark.parametrize("variant,op", [("single", "fwd"), ("pair", "fwd"), ("single", "dx"),
                                        ("pair", "dx"), ("single", "dw"), ("pair", "dw"),
                                        ("single", "dw_nows"), ("pair", "dw_nows")])
def test_timeout_unwinds_and_reports(rd_lib, variant, op):
    v = rd_lib.VARIANT_PAIR if variant == "pair" else rd_lib.VARIANT_SINGLE
    a, w, do, sizes = _inputs(op, 1)
    gs = torch.tensor(sizes, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    with rd_lib.tuning(variant=v, wait_timeout_ns=1):
        _call(rd_lib, op, a, w, do, gs, status)
    torch.cuda.synchronize()
    assert int(status.item()) & rd_lib.STATUS_TIMEOUT
    with pytest.raises(rd_lib.RdError, match="STATUS_TIMEOUT"):
        rd_lib.check_status(status)
    # the context, the tensor memory and the library are usable again
    status.zero_()
    with rd_lib.tuning(variant=v):
        out = _call(rd_lib, op, a, w, do, gs, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    a64, w64, d64 = obf.torch_bf16_to_f64(a), obf.torch_bf16_to_f64(w), obf.torch_bf16_to_f64(do)
    got = obf.torch_bf16_to_f64(out)
    if op == "fwd":
        ref = oracle.ragged_dot(a64, w64, sizes)
        tol = gemm_tol(ref, a64.shape[1], np.abs(a64).max(), np.abs(w64).max())
    elif op == "dx":
        ref = oracle.ragged_dot_trans_rhs(d64, w64, sizes)
        tol = gemm_tol(ref, d64.shape[1], np.abs(d64).max(), np.abs(w64).max())
    else:
        ref = oracle.trans_ragged_dot(a64, d64, sizes)
        tol = gemm_tol(ref, max(sizes), np.abs(a64).max(), np.abs(d64).max())
    assert_close(got, ref, tol, f"{op} after a timed-out call")
