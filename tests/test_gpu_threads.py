"""Calls from several host threads at once, each on its own stream.

The C entry points keep per-process host state (the per-device SM count and
kernel attributes behind a mutex or atomics, the tensor-map encode cache per
thread) and release the interpreter lock while they run, so two threads can
be inside the library at the same time.  Each thread here runs a mix of
forward, forward + GLU, dx and dw calls with shapes of its own; every output
must equal, bit for bit, the output of the same call made alone (the kernels
add in a fixed order, so a repeat is bitwise identical).
"""
import threading

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda"


def _inputs(seed, m, k, n, sizes):
    from workloads import normal_bf16_np
    rng = np.random.default_rng(seed)
    g = len(sizes)
    lhs = normal_bf16_np(rng, (m, k)).to(DEV)
    rhs = normal_bf16_np(rng, (g, k, n), 1.0 / k).to(DEV)
    do = normal_bf16_np(rng, (m, n)).to(DEV)
    gs = torch.tensor(sizes, dtype=torch.int32, device=DEV)
    return lhs, rhs, do, gs


def _calls(rd, lhs, rhs, do, gs):
    """The thread's calls, each returning a fresh output tensor."""
    return [
        lambda: rd.ragged_dot(lhs, rhs, gs),
        lambda: rd.ragged_dot(lhs, rhs, gs, epilogue=rd.EPI_SILU_GLU),
        lambda: rd.ragged_dot_trans_rhs(do, rhs, gs),
        lambda: rd.trans_ragged_dot(lhs, do, gs),
    ]


def test_concurrent_calls_from_threads(rd_lib):
    cases = [(1, 700, 136, 272, [0, 1, 127, 128, 129, 0, 255, 3, 57]),
             (2, 1793, 264, 512, [256, 257, 511, 1, 0, 513, 255]),
             (3, 900, 64, 1040, [300, 0, 600]),
             (4, 643, 520, 256, [0, 1, 127, 128, 129, 0, 255, 3])]
    work = []
    for seed, m, k, n, sizes in cases:
        ins = _inputs(seed, m, k, n, sizes)
        calls = _calls(rd_lib, *ins)
        ref = [c() for c in calls]
        torch.cuda.synchronize()
        work.append((calls, [r.clone() for r in ref]))

    reps = 12
    results = [[None] * (reps * 4) for _ in work]
    errors = []

    def run(t):
        try:
            calls, _ = work[t]
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                for i in range(reps * 4):
                    results[t][i] = calls[i % 4]()
            stream.synchronize()
        except Exception as e:  # reported below, on the main thread
            errors.append(e)

    threads = [threading.Thread(target=run, args=(t,)) for t in range(len(work))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for t, (_, ref) in enumerate(work):
        for i, got in enumerate(results[t]):
            want = ref[i % 4]
            assert torch.equal(got.view(torch.int16), want.view(torch.int16)), \
                f"thread {t}, call {i}: differs from the same call made alone"
