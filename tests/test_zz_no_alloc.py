"""The allocation-free weight gradient, rd_trans_ragged_dot_no_alloc, through the C ABI.

It is meant for callers that cannot allocate device memory where they run the
weight gradient (inside an allocator's own callbacks, under a runtime that owns
every allocation, or after a set-up that fixed the process's footprint).  It
runs the same per-group-descriptor dw as rd_trans_ragged_dot with a workspace,
but takes its scratch from an array inside the library.  The array keeps the
last call's contents, so the check covers two calls in a row with different
group sizes: stale descriptors from the first call would show in the second.
Each output is compared with rd_trans_ragged_dot's on the same inputs, within
the GEMM tolerance the other tests use.

This file is named to run after every other test file.
"""
import ctypes

import numpy as np
import pytest

from oracle import bf16 as obf
from parity_util import assert_close, gemm_tol

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda"


def _no_alloc_call(lib, x, y, gs, out):
    """rd_trans_ragged_dot_no_alloc on the current stream, straight through ctypes."""
    f = lib.rd_trans_ragged_dot_no_alloc
    f.restype = ctypes.c_int
    v, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    f.argtypes = [v, v, v, i64, i64, i64, v, i32, i32, i32, v, v, v]
    m, k = x.shape
    n = y.shape[1]
    g = gs.numel()
    code = f(x.data_ptr(), y.data_ptr(), out.data_ptr(), m, k, n, gs.data_ptr(), g, 0, g, None,
             None, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0, lib.rd_status_string(code)


@pytest.mark.parametrize("variant", ["pair", "single"])
def test_no_alloc_dw_matches_the_workspace_form(rd_lib, variant):
    lib = rd_lib.load()
    rng = np.random.default_rng(2024)
    k, n = 256, 384
    cases = [[300, 0, 129, 17, 64, 1, 431], [5, 700, 0, 250, 63, 65, 9]]   # two calls in a row
    m = max(sum(c) for c in cases) + 11
    v = rd_lib.VARIANT_PAIR if variant == "pair" else rd_lib.VARIANT_SINGLE
    with rd_lib.tuning(variant=v):
        for call, sizes in enumerate(cases):
            x = torch.from_numpy(rng.standard_normal((m, k)).astype(np.float32)).to(torch.bfloat16).to(DEV)
            y = torch.from_numpy(rng.standard_normal((m, n)).astype(np.float32)).to(torch.bfloat16).to(DEV)
            gs = torch.tensor(sizes, dtype=torch.int32, device=DEV)
            got = torch.full((len(sizes), k, n), float("nan"), dtype=torch.bfloat16, device=DEV)
            _no_alloc_call(lib, x, y, gs, got)
            want = rd_lib.trans_ragged_dot(x, y, gs, workspace="auto")
            torch.cuda.synchronize()
            b = np.concatenate([[0], np.cumsum(sizes)])
            x64, y64 = obf.torch_bf16_to_f64(x), obf.torch_bf16_to_f64(y)
            g64, w64 = obf.torch_bf16_to_f64(got), obf.torch_bf16_to_f64(want)
            for j, cnt in enumerate(sizes):
                if cnt == 0:
                    assert np.all(obf.torch_bf16_bits(got[j]) == 0), f"call {call}: empty group {j}"
                    continue
                rows = slice(b[j], b[j + 1])
                tol = gemm_tol(w64[j], cnt, np.abs(x64[rows]).max(), np.abs(y64[rows]).max())
                assert_close(g64[j], w64[j], tol, f"call {call} group {j} ({cnt} rows)")
