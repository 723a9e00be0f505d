"""The bench line on the host: the ops summary keeps every row and stays short.

A log that keeps only the last 1500 characters of the bench's output must
still hold every row of the hot path, so the `ops` summary (the last key of
the line) has to fit well inside that.  Built here from a result dict shaped
like run_ops' output, with long floats everywhere, so no GPU is needed.
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _fake_ops():
    f = 123.456789012345
    gemm = {"us": f, "tflops": f, "bound": "tensor", "frac": 0.7891234, "p10_us": f, "p90_us": f,
            "mhz": 1863.5, "power_cap": True, "frac_sustained": 0.8712345}
    hbm = {"us": f, "gbs": f, "bound": "hbm", "frac": 0.9456789, "p10_us": f, "p90_us": f}
    res = {"packed_glu_fwd": dict(gemm), "dx": dict(gemm), "dw": dict(gemm), "dw_f32": dict(gemm),
           "dw_f32_accumulate": dict(hbm), "glu_fwd": dict(hbm), "glu_bwd": dict(hbm),
           "unsort_bwd_rows": dict(hbm),
           "packed_dx_glu_bwd": dict(hbm, unfused_us=f)}
    for tag in ("decode_skewed", "decode_uniform"):
        res[tag] = {"graph_pair_us": f, "up_us": f, "down_us": f, "bound": "hbm", "pair_frac": 0.9654321,
                    "graph_pair_p10_us": f, "graph_pair_p90_us": f}
    res["tiny"] = {"us": 6.1234, "call_us": 15.2961, "call_p10_us": 14.1, "call_p90_us": 17.5,
                   "bound": "latency"}
    res["ffn_sweep"] = [{"tokens": t, "us": f * 10, "frac": 0.7127053, "bound": "hbm"}
                        for t in (256, 1024, 4096, 16384)]
    return res


def test_compact_ops_keeps_every_row_and_fits_the_tail():
    sys.path.insert(0, ROOT)
    import bench

    ops = bench.compact_ops(_fake_ops())
    for key in ("c1_tiny", "c3_glu_fwd", "c4_dx", "c4_dw", "c4_dw_f32", "c4_dw_f32_acc", "c5_skew",
                "c5_unif", "glu_fwd", "glu_bwd", "dx_glu_bwd", "unsort", "ffn"):
        assert key in ops, key
    for key in ("c3_glu_fwd", "c4_dx", "c4_dw", "c4_dw_f32"):
        assert {"mhz", "fs", "cap"} <= set(ops[key]), key
    text = json.dumps({"ops": ops})
    assert len(text) < 1300, len(text)
