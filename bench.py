#!/usr/bin/env python
"""Benchmark of the ragged_dot (MoE grouped GEMM) hot path on GB300.

Headline step: one rd_ragged_dot forward over the Mixtral-shaped workload
(16384 tokens routed top-2 over 8 experts -> lhs [32768, 4096] bf16,
rhs [8, 4096, 14336] bf16, out [32768, 14336] bf16, f32 accumulation).
The metric is TFLOP/s over the valid rows (2 * rows * k * n per step); the
inputs (2.15 GB moved per step) are larger than the 129 MB L2, so no flush
is needed between steps.

Also reported on the same line:
  roofline      the kernel's achieved TFLOP/s (CUDA events on its stream)
                against the measured bf16 dense peak;
  e2e           the same metric through the C ABI with pinned host buffers,
                host->device copies of the inputs and device->host copy of
                the output inside the timed region;
  cpu_baseline  the float64 oracle timed on a bounded sample of the same
                workload on this host's cores;
  ops           the other rows of the hot path at their own workloads
                (packed GLU forward, dx, dw in bf16, f32 and accumulating
                f32, decode pair in one CUDA graph, standalone GLU
                forward/backward, unsort backward, the fused GLU backward
                through the down projection, the tiny workload's latency, and
                the expert FFN forward graph from 256 to 16384 tokens), each as
                time per call in us (50 calls back to back between two events
                after 10 warm-up calls, the total divided by the calls, as for
                the headline), fraction
                of its roofline and the bound ("t" tensor, "h" HBM, "l"
                latency), with p10 / p90 of events around each call for the
                five configs; short keys and 3-4 significant digits keep the
                whole line short.  --ops-json FILE writes the full figures.

--profile NAME runs a few launches of one workload for ncu (mixtral,
mixtral_small, packed_glu, dx, dw, dw_f32acc, packed_dx_glu_bwd, glu_fwd,
glu_bwd, unsort, decode, ffn4096_up).

--impl reference times the oracle itself as the reference arm.
Under torchrun (--gpus N) every rank runs an independent replica (no
data-path collective); times are max-reduced across ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------- helpers
class ClockSampler:
    """nvidia-smi clock / throttle sampling around the timed region.

    Samples carry nvidia-smi's own timestamps; ``mark_start`` / ``mark_end``
    bracket the timed region on the host clock and only the samples inside it
    are summarised (all samples when the region is shorter than one period).
    """

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.proc = None
        self.gpu = gpu_index
        self.period = period_ms
        self.t_start = self.t_end = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def mark_start(self):
        self.t_start = time.time()

    def mark_end(self):
        self.t_end = time.time()

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        import datetime

        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                sm, mx = float(parts[2]), float(parts[3])
            except ValueError:
                continue
            active = {n for n, v in zip(names, parts[6:10]) if v.lower() == "active"}
            rows.append((ts, sm, mx, active))
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        inside = [r for r in rows if self.t_start is not None and self.t_end is not None
                  and self.t_start <= r[0] <= self.t_end]
        use = inside if inside else rows
        reasons = sorted(set().union(*[r[3] for r in use]))
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": use[0][2],
                "reasons": reasons, "samples": len(use),
                "window": "timed region" if inside else "whole sampling window"}


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "expert_ffn_ragged_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes from the committed ncu summary, if still current."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    e = rec.get(kernel, {}).get(workload)
    if not e or e.get("kernel_source_sha") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


def blas_threads():
    try:
        from threadpoolctl import threadpool_info

        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(n[0])
    except Exception:
        pass
    return os.cpu_count()


# ----------------------------------------------------------------- workloads
def mixtral_inputs(device):
    import torch

    from workloads import mixtral_fwd, normal_bf16

    w = mixtral_fwd()
    lhs = normal_bf16((w.m, w.k), w.lhs_var, 20, device)
    rhs = normal_bf16((w.g_total, w.k, w.n), w.rhs_var, 21, device)
    gs = torch.tensor(w.group_sizes, dtype=torch.int32, device=device)
    return w, lhs, rhs, gs


def fwd_flops(w, rows=None):
    rows = int(w.group_sizes.sum()) if rows is None else rows
    return 2.0 * rows * w.k * w.n


def time_launches(fn, steps, warmup, stream):
    """Per-launch CUDA-event durations (ms) on `stream`, plus the total (ms)."""
    import torch

    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        starts[i].record(stream)
        fn()
        ends[i].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return per, t0.elapsed_time(t1)


# ----------------------------------------------------------------- oracle timing
def oracle_sample_run(w, lhs, rhs, target_s: float, max_cols=None):
    """Time the float64 oracle on a bounded sample of the Mixtral workload.

    The sample keeps every row, every group and the full contraction length
    and takes the first `cols` output columns; `cols` is grown until one run
    takes about `target_s` seconds.  Returns (TFLOP/s, seconds, description).
    """
    import numpy as np
    import torch

    import oracle

    a64 = lhs.float().cpu().numpy().astype(np.float64)
    cols = 128
    max_cols = w.n if max_cols is None else max_cols
    while True:
        w64 = rhs[:, :, :cols].float().cpu().numpy().astype(np.float64)
        t = time.perf_counter()
        oracle.ragged_dot(a64, w64, w.group_sizes)
        dt = time.perf_counter() - t
        if dt >= target_s / 4 or cols >= max_cols:
            break
        cols = min(max_cols, cols * 4)
    # final measured run at the size that reaches about target_s
    if dt < target_s and cols < max_cols:
        cols = min(max_cols, max(8, int(cols * target_s / max(dt, 1e-3)) // 8 * 8))
        w64 = rhs[:, :, :cols].float().cpu().numpy().astype(np.float64)
        t = time.perf_counter()
        oracle.ragged_dot(a64, w64, w.group_sizes)
        dt = time.perf_counter() - t
    flops = 2.0 * int(w.group_sizes.sum()) * w.k * cols
    desc = (f"all {int(w.group_sizes.sum())} rows, all 8 groups, k={w.k}, first {cols} of "
            f"{w.n} output columns ({flops / 1e12:.3f} TFLOP)")
    return flops / dt / 1e12, dt, desc, cols


# ----------------------------------------------------------------- other ops
def run_ops(rd, device, stream, peaks):
    """Each remaining hot-path row at its own workload: time per call and roofline fraction."""
    import numpy as np
    import torch

    from workloads import backward_pair, decode_fwd, normal_bf16, packed_glu_fwd, tiny_fwd

    P = peaks["bf16_tflops"] * 1e12
    PS = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * 1e12
    BW = peaks["hbm_gbs"] * 1e9
    res = {}

    spread = []  # (entry, key prefix, p10 us, p90 us) of each timed call

    def clock_probe(fn, entry, flops, seconds=0.25):
        """The SM clock while the call runs back to back (sampled by nvidia-smi), and the
        fraction of the sustained bf16 peak (the cuBLAS figure under the power cap).

        The timed calls run first, on a GPU that is already warm; this loop runs the
        same call for a quarter of a second right after, long enough for several
        clock samples, and only reports the clock it ran at.
        """
        with ClockSampler(device.index if device.index is not None else 0, period_ms=10) as clk:
            clk.mark_start()
            t0 = time.time()
            while time.time() - t0 < seconds:
                for _ in range(5):
                    fn()
                torch.cuda.synchronize()
            clk.mark_end()
        c = clk.summary()
        r = res[entry]
        r["mhz"] = c["sm_mhz"]
        r["power_cap"] = "sw_power_cap" in c["reasons"]
        r["frac_sustained"] = flops / PS / (r["us"] * 1e-6)

    def med(fn, steps=50, warmup=10, entry=None, prefix="", per_call=False):
        """Seconds per call: `steps` calls back to back between two events, divided by
        `steps` (as the headline's value), or with per_call the median of events around
        each call (a single call's latency); the p10 / p90 spread comes from the loop
        with events around every call.  50 calls of these kernels last 5 to 25 ms, the
        burst regime the burst peak is measured in (loops of 0.2 s and more run ~10 %
        slower once the power cap acts)."""
        per, _ = time_launches(fn, steps, warmup, stream)
        if entry is not None:
            q = statistics.quantiles(per, n=10)
            spread.append((entry, prefix, q[0] * 1e3, q[-1] * 1e3))
        if per_call:
            return statistics.median(per) * 1e-3
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(steps):
            fn()
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / steps * 1e-3

    with torch.cuda.stream(stream):
        # packed buffer forward + fused GLU, group_offset 16 of 64, limit 126156
        w = packed_glu_fwd()
        lhs = normal_bf16((w.m, w.k), 1.0, 30, device)
        rhs = normal_bf16((w.g_local, w.k, w.n), w.rhs_var, 31, device)
        gs = torch.tensor(w.group_sizes, dtype=torch.int32, device=device)
        lim = torch.tensor([w.limit], dtype=torch.int32, device=device)
        out = torch.empty((w.m, w.n // 2), dtype=torch.bfloat16, device=device)
        b = np.concatenate([[0], np.cumsum(w.group_sizes)])
        rows = int(b[w.group_offset + w.g_local] - b[w.group_offset])
        F = 2.0 * rows * w.k * w.n
        zero_rows = w.limit - rows
        B = rows * w.k * 2 + w.g_local * w.k * w.n * 2 + w.limit * (w.n // 2) * 2 + 4 * w.g_total
        glu_call = lambda: rd.ragged_dot(lhs, rhs, gs, w.group_offset, lim, rd.EPI_SILU_GLU, out)
        t = med(glu_call, entry="packed_glu_fwd")
        res["packed_glu_fwd"] = {"us": t * 1e6, "tflops": F / t / 1e12, "gbs": B / t / 1e9,
                                 "bound": "hbm" if B / BW > F / P else "tensor",
                                 "frac": max(F / P, B / BW) / t,
                                 "local_rows": rows, "zero_rows": zero_rows}
        clock_probe(glu_call, "packed_glu_fwd", F)
        # standalone GLU on the same packed buffer shape
        fused = normal_bf16((w.m, 2 * 1024), 1.0, 32, device)
        gout = torch.empty((w.m, 1024), dtype=torch.bfloat16, device=device)
        t = med(lambda: rd.glu_fwd(fused, lim, gout), entry="glu_fwd")
        Bg = w.limit * 1024 * 2 * 3
        res["glu_fwd"] = {"us": t * 1e6, "gbs": Bg / t / 1e9, "bound": "hbm", "frac": Bg / BW / t}
        dfused = torch.empty_like(fused)
        t = med(lambda: rd.glu_bwd(fused, gout, lim, dfused), entry="glu_bwd")
        Bb = w.limit * 1024 * 2 * 5
        res["glu_bwd"] = {"us": t * 1e6, "gbs": Bb / t / 1e9, "bound": "hbm", "frac": Bb / BW / t}
        del lhs, rhs, out, fused, gout, dfused
        torch.cuda.empty_cache()

        # packed buffer backward through the down projection: dx (D = 4096 -> F = 1024)
        # with the GLU backward fused, against dx followed by the standalone GLU backward
        d_out = normal_bf16((w.m, 4096), 1.0, 35, device)
        w_down = normal_bf16((w.g_local, 1024, 4096), 1.0 / 4096, 36, device)
        fused2 = normal_bf16((w.m, 2048), 1.0, 37, device)
        dfused2 = torch.empty_like(fused2)
        dh = torch.empty((w.m, 1024), dtype=torch.bfloat16, device=device)
        t_fused = med(lambda: rd.ragged_dot_trans_rhs_glu_bwd(d_out, w_down, fused2, gs, w.group_offset,
                                                              lim, dfused2), entry="packed_dx_glu_bwd")

        def unfused():
            rd.ragged_dot_trans_rhs(d_out, w_down, gs, w.group_offset, lim, dh)
            rd.glu_bwd(fused2, dh, lim, dfused2)

        t_unfused = med(unfused, entry="packed_dx_glu_bwd", prefix="unfused_")
        F2 = 2.0 * rows * 1024 * 4096
        B2 = (rows * 4096 * 2 + w.g_local * 1024 * 4096 * 2 + rows * 2048 * 2
              + w.limit * 2048 * 2 + 4 * w.g_total)
        res["packed_dx_glu_bwd"] = {"us": t_fused * 1e6, "unfused_us": t_unfused * 1e6,
                                    "bound": "hbm" if B2 / BW > F2 / P else "tensor",
                                    "frac": max(F2 / P, B2 / BW) / t_fused}
        del d_out, w_down, fused2, dfused2, dh
        torch.cuda.empty_cache()

        # valid-rows unsort backward at the packed buffer's shape [225280, 4096]
        g = normal_bf16((w.m, 4096), 1.0, 33, device)
        y = normal_bf16((w.m, 4096), 1.0, 34, device)
        wt = torch.rand((w.m,), device=device)
        grad = torch.empty_like(g)
        dot = torch.empty((w.m,), dtype=torch.float32, device=device)
        t = med(lambda: rd.unsort_bwd_rows(g, y, wt, lim, grad, dot), entry="unsort_bwd_rows")
        Bu = w.limit * 4096 * 2 * 3 + w.limit * 8
        res["unsort_bwd_rows"] = {"us": t * 1e6, "gbs": Bu / t / 1e9, "bound": "hbm",
                                  "frac": Bu / BW / t}
        del g, y, wt, grad, dot
        torch.cuda.empty_cache()

        # backward pair: dx and dw
        w = backward_pair()
        x = normal_bf16((w.m, w.k), 1.0, 40, device)
        do = normal_bf16((w.m, w.n), 1.0, 41, device)
        wt = normal_bf16((w.g_total, w.k, w.n), w.rhs_var, 42, device)
        gs = torch.tensor(w.group_sizes, dtype=torch.int32, device=device)
        dx = torch.empty((w.m, w.k), dtype=torch.bfloat16, device=device)
        dw = torch.empty((w.g_total, w.k, w.n), dtype=torch.bfloat16, device=device)
        F = 2.0 * w.m * w.k * w.n
        live = int((w.group_sizes > 0).sum())
        dx_call = lambda: rd.ragged_dot_trans_rhs(do, wt, gs, out=dx)
        t = med(dx_call, entry="dx")
        B = w.m * w.n * 2 + live * w.k * w.n * 2 + w.m * w.k * 2
        res["dx"] = {"us": t * 1e6, "tflops": F / t / 1e12,
                     "bound": "hbm" if B / BW > F / P else "tensor",
                     "frac": max(F / P, B / BW) / t}
        clock_probe(dx_call, "dx", F)
        # dw through per-group tensor maps, in a workspace allocated once
        ws = torch.empty(rd.dw_workspace_bytes(device), dtype=torch.uint8, device=device)
        dw_call = lambda: rd.trans_ragged_dot(x, do, gs, out=dw, workspace=ws)
        t = med(dw_call, entry="dw")
        B = w.m * w.k * 2 + w.m * w.n * 2 + w.g_total * w.k * w.n * 2
        res["dw"] = {"us": t * 1e6, "tflops": F / t / 1e12,
                     "bound": "hbm" if B / BW > F / P else "tensor",
                     "frac": max(F / P, B / BW) / t}
        clock_probe(dw_call, "dw", F)
        del dx, dw
        torch.cuda.empty_cache()
        # dw kept in f32 (stored, then added into an existing gradient buffer)
        dw32 = torch.zeros((w.g_total, w.k, w.n), dtype=torch.float32, device=device)
        for key, acc in (("dw_f32", False), ("dw_f32_accumulate", True)):
            t = med(lambda: rd.trans_ragged_dot_f32(x, do, gs, out=dw32, accumulate=acc, workspace=ws),
                    entry=key)
            # storing writes every block (empty groups' as zeros); accumulating reads
            # and writes only the blocks of groups with rows
            B = w.m * w.k * 2 + w.m * w.n * 2 + (live * w.k * w.n * 4 * 2 if acc
                                                 else w.g_total * w.k * w.n * 4)
            res[key] = {"us": t * 1e6, "tflops": F / t / 1e12,
                        "bound": "tensor" if F / P >= B / BW else "hbm",
                        "frac": max(F / P, B / BW) / t}
            if not acc:
                clock_probe(lambda: rd.trans_ragged_dot_f32(x, do, gs, out=dw32, workspace=ws), key, F)
        del x, do, wt, dw32, ws
        torch.cuda.empty_cache()

        # decode pair (up with GLU, down) sharing group_sizes inside one CUDA graph
        for skew in (True, False):
            w = decode_fwd(skewed=skew)
            lhs = normal_bf16((w.m, w.k), 1.0, 50, device)
            up = normal_bf16((w.g_total, w.k, w.n), w.rhs_var, 51, device)
            down = normal_bf16((w.g_total, w.n // 2, w.k), 1.0 / (w.n // 2), 52, device)
            gs = torch.tensor(w.group_sizes, dtype=torch.int32, device=device)
            h = torch.empty((w.m, w.n // 2), dtype=torch.bfloat16, device=device)
            o = torch.empty((w.m, w.k), dtype=torch.bfloat16, device=device)

            def pair():
                rd.ragged_dot(lhs, up, gs, epilogue=rd.EPI_SILU_GLU, out=h)
                rd.ragged_dot(h, down, gs, out=o)

            pair()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                pair()
            tag = "decode_skewed" if skew else "decode_uniform"
            t_pair = med(g.replay, entry=tag, prefix="graph_pair_")
            t_up = med(lambda: rd.ragged_dot(lhs, up, gs, epilogue=rd.EPI_SILU_GLU, out=h),
                       entry=tag, prefix="up_")
            t_down = med(lambda: rd.ragged_dot(h, down, gs, out=o), entry=tag, prefix="down_")
            live = int((w.group_sizes > 0).sum())
            B_up = w.m * w.k * 2 + live * w.k * w.n * 2 + w.m * (w.n // 2) * 2
            B_dn = w.m * (w.n // 2) * 2 + live * (w.n // 2) * w.k * 2 + w.m * w.k * 2
            res[tag] = {"graph_pair_us": t_pair * 1e6, "up_us": t_up * 1e6, "down_us": t_down * 1e6,
                        "bound": "hbm", "live_groups": live,
                        "up_frac": B_up / BW / t_up, "down_frac": B_dn / BW / t_down,
                        "pair_frac": (B_up + B_dn) / BW / t_pair}
            del lhs, up, down, h, o, g
            torch.cuda.empty_cache()
        # the tiny workload (L2-resident, launch-latency bound): time per call
        w = tiny_fwd()
        lhs = normal_bf16((w.m, w.k), w.lhs_var, 60, device)
        rhs = normal_bf16((w.g_total, w.k, w.n), w.rhs_var, 61, device)
        gs = torch.tensor(w.group_sizes, dtype=torch.int32, device=device)
        out = torch.empty((w.m, w.n), dtype=torch.bfloat16, device=device)
        # on an idle GPU the events around one call also hold the call's host work
        # (argument checks, tensor-map encoding); 20 launches replayed from a CUDA
        # graph give the device time of a launch alone
        t_call = med(lambda: rd.ragged_dot(lhs, rhs, gs, out=out), steps=100, warmup=10, per_call=True,
                     entry="tiny", prefix="call_")
        rd.ragged_dot(lhs, rhs, gs, out=out)
        torch.cuda.synchronize()
        g20 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g20, stream=stream):
            for _ in range(20):
                rd.ragged_dot(lhs, rhs, gs, out=out)
        t20 = med(g20.replay)
        res["tiny"] = {"us": t20 / 20 * 1e6, "call_us": t_call * 1e6, "bound": "latency",
                       "workload": w.name,
                       "note": "us: device time per launch (20 launches in one CUDA graph); "
                               "call_us: events around one call, host work included"}
        del lhs, rhs, out, g20
        # the expert FFN forward (up with GLU, then down) as one CUDA graph, from decode
        # to prefill batch sizes: where the weight stream stops bounding the time
        res["ffn_sweep"] = ffn_sweep(rd, device, stream, peaks)
    for entry, prefix, p10, p90 in spread:
        if entry in res:
            res[entry][prefix + "p10_us"] = p10
            res[entry][prefix + "p90_us"] = p90
    return res


def _sig(x, digits=4):
    """x rounded to `digits` significant digits (keeps the JSON line short)."""
    if x is None or x == 0:
        return x
    return float(f"{x:.{digits}g}")


def compact_ops(res):
    """The ops as a short dict: time (us), roofline fraction and bound of every row.

    Keys name the row and its workload: c1 tiny, c3 packed GLU forward, c4 the
    backward pair (dx, dw, dw in f32, accumulated f32), c5 the decode pair in one
    graph (skewed / uniform routing), the standalone GLU and unsort passes on the
    packed buffer, the fused dx + GLU backward, and the expert-FFN graph by token
    count ([us, frac, bound]).  p10 / p90 are given for the five configs; the
    tensor-bound GEMM rows add the SM clock under their own sustained load (mhz),
    their fraction of the sustained bf16 peak (fs) and the power-cap flag (cap).
    """
    b = {"tensor": "t", "hbm": "h", "latency": "l"}
    out = {}

    def row(key, src, us_key="us", frac_key="frac", spread_prefix="", extra=()):
        if src not in res:
            return
        r = res[src]
        e = {"us": _sig(r[us_key]), "frac": _sig(r.get(frac_key), 3)}
        if "bound" in r:
            e["b"] = b.get(r["bound"], r["bound"])
        p10, p90 = r.get(spread_prefix + "p10_us"), r.get(spread_prefix + "p90_us")
        if key.startswith("c") and p10 is not None:
            e["p10"], e["p90"] = _sig(p10, 3), _sig(p90, 3)
        for k_out, k_in in extra:
            e[k_out] = _sig(r[k_in])
        if r.get("mhz") is not None:
            # the SM clock under this call's sustained load, the fraction of the
            # sustained peak, and whether the power cap was holding the clock down
            e["mhz"] = int(round(r["mhz"]))
            e["fs"] = _sig(r["frac_sustained"], 3)
            e["cap"] = int(bool(r.get("power_cap")))
        out[key] = e

    if "tiny" in res:
        t = res["tiny"]
        out["c1_tiny"] = {"us": _sig(t["us"], 3), "call_us": _sig(t["call_us"], 3),
                          "p10": _sig(t.get("call_p10_us"), 3), "p90": _sig(t.get("call_p90_us"), 3),
                          "b": "l"}
    row("c3_glu_fwd", "packed_glu_fwd")
    row("c4_dx", "dx")
    row("c4_dw", "dw")
    row("c4_dw_f32", "dw_f32")
    row("c4_dw_f32_acc", "dw_f32_accumulate")
    for key, src in (("c5_skew", "decode_skewed"), ("c5_unif", "decode_uniform")):
        row(key, src, us_key="graph_pair_us", frac_key="pair_frac", spread_prefix="graph_pair_",
            extra=(("up_us", "up_us"), ("down_us", "down_us")))
    row("glu_fwd", "glu_fwd")
    row("glu_bwd", "glu_bwd")
    row("dx_glu_bwd", "packed_dx_glu_bwd", extra=(("unfused_us", "unfused_us"),))
    row("unsort", "unsort_bwd_rows")
    if "ffn_sweep" in res:
        out["ffn"] = {str(r["tokens"]): [_sig(r["us"]), _sig(r["frac"], 3), b[r["bound"]]]
                      for r in res["ffn_sweep"]}
    return out


def ffn_sweep(rd, device, stream, peaks, tokens=(256, 1024, 4096, 16384)):
    """Up (GLU) + down projections of 128 experts (4096 -> 1536 -> 4096), top-8 routing."""
    import torch

    from workloads import expert_ffn, normal_bf16

    P = peaks["bf16_tflops"] * 1e12
    BW = peaks["hbm_gbs"] * 1e9
    g, k, n = 128, 4096, 1536
    up = normal_bf16((g, k, n), 1.0 / k, 61, device)
    down = normal_bf16((g, n // 2, k), 1.0 / (n // 2), 62, device)
    rows_out = []
    for t in tokens:
        w = expert_ffn(t)
        assert (w.g_total, w.k, w.n) == (g, k, n)
        sizes = w.group_sizes
        m = w.m
        lhs = normal_bf16((m, k), 1.0, 63, device)
        gs = torch.tensor(sizes, dtype=torch.int32, device=device)
        h = torch.empty((m, n // 2), dtype=torch.bfloat16, device=device)
        o = torch.empty((m, k), dtype=torch.bfloat16, device=device)

        def pair():
            rd.ragged_dot(lhs, up, gs, epilogue=rd.EPI_SILU_GLU, out=h)
            rd.ragged_dot(h, down, gs, out=o)

        with torch.cuda.stream(stream):
            pair()
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                pair()
            per, _ = time_launches(graph.replay, 20, 3, stream)
        tsec = statistics.median(per) * 1e-3
        live = int((sizes > 0).sum())
        flops = 2.0 * m * k * n + 2.0 * m * (n // 2) * k
        byts = (m * k * 2 + live * k * n * 2 + m * (n // 2) * 2) + \
               (m * (n // 2) * 2 + live * (n // 2) * k * 2 + m * k * 2)
        rows_out.append({"tokens": t, "rows": m, "live_groups": live, "us": tsec * 1e6,
                         "tflops": flops / tsec / 1e12, "gbs": byts / tsec / 1e9,
                         "bound": "tensor" if flops / P > byts / BW else "hbm",
                         "frac": max(flops / P, byts / BW) / tsec})
        del lhs, gs, h, o, graph
    del up, down
    torch.cuda.empty_cache()
    return rows_out


# ----------------------------------------------------------------- arms
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if args.impl == "rd" else "gloo"
        dist.init_process_group(backend)
        pg = dist
    return world, rank, local, pg


def max_over_ranks(pg, value, device):
    if pg is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def run_reference(args):
    world, rank, local, pg = dist_setup(args)
    if rank != 0:
        return 0
    import torch

    w, lhs, rhs, gs = mixtral_inputs("cpu") if not torch.cuda.is_available() else \
        mixtral_inputs(f"cuda:{local}")
    # each step: the oracle on a bounded sample of the workload, sized so that
    # the whole run (warm-up + timed steps) takes about two minutes
    per_step = max(0.2, min(3.0, 120.0 / max(1, args.steps + args.warmup)))
    _, _, desc, cols = oracle_sample_run(w, lhs, rhs, target_s=per_step)
    import numpy as np

    import oracle

    a64 = lhs.float().cpu().numpy().astype(np.float64)
    w64 = rhs[:, :, :cols].float().cpu().numpy().astype(np.float64)
    flops = 2.0 * int(w.group_sizes.sum()) * w.k * cols
    for _ in range(args.warmup):
        oracle.ragged_dot(a64, w64, w.group_sizes)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle.ragged_dot(a64, w64, w.group_sizes)
    dt = (time.perf_counter() - t) / args.steps
    value = flops / dt / 1e12
    line = {
        "impl": "reference", "metric": "grouped-GEMM TFLOP/s (valid rows)", "value": value,
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "sample": desc},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
                         "host_cores": os.cpu_count(),
                         "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def run_rd(args):
    import torch

    world, rank, local, pg = dist_setup(args)
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import expert_ffn_ragged_gb300 as rd

    rd.load()
    peaks, peak_src = load_peaks()
    stream = torch.cuda.Stream(device)
    w, lhs, rhs, gs = mixtral_inputs(device)
    out = torch.empty((w.m, w.n), dtype=torch.bfloat16, device=device)
    flops = fwd_flops(w)
    rows = int(w.group_sizes.sum())
    alg_bytes = rows * w.k * 2 + w.g_total * w.k * w.n * 2 + rows * w.n * 2 + 4 * w.g_total

    def step():
        rd.ragged_dot(lhs, rhs, gs, out=out, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        if pg is not None:
            pg.barrier()
        with ClockSampler(local) as clk:
            clk.mark_start()
            per, total_ms = time_launches(step, args.steps, 0, stream)
            clk.mark_end()
        if pg is not None:
            pg.barrier()
    total_ms = max_over_ranks(pg, total_ms, device)
    ms_per_step = total_ms / args.steps
    value = world * flops / (ms_per_step * 1e-3) / 1e12
    mean_launch = statistics.mean(per) * 1e-3
    achieved = flops / mean_launch / 1e12
    peak = peaks["bf16_tflops"]
    traffic = recorded_traffic("grouped_gemm_fwd", w.name)

    # End to end through the C ABI with pinned host buffers: every step copies its
    # inputs (lhs, rhs, group_sizes) host -> device, runs the forward, and copies
    # the output back.  Steps are pipelined over three streams with two device
    # buffer sets: the upload of step i+1 and the download of step i-1 overlap
    # the forward of step i.
    h_lhs = lhs.cpu().pin_memory()
    h_rhs = rhs.cpu().pin_memory()
    h_gs = gs.cpu().pin_memory()
    h_out = [torch.empty((w.m, w.n), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    del lhs, rhs, out
    torch.cuda.empty_cache()
    bufs = [(torch.empty((w.m, w.k), dtype=torch.bfloat16, device=device),
             torch.empty((w.g_total, w.k, w.n), dtype=torch.bfloat16, device=device),
             torch.empty((w.g_total,), dtype=torch.int32, device=device),
             torch.empty((w.m, w.n), dtype=torch.bfloat16, device=device)) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    e2e_steps = max(3, min(args.steps, 20))

    def run_e2e(nsteps):
        loaded = [torch.cuda.Event() for _ in range(nsteps)]
        computed = [torch.cuda.Event() for _ in range(nsteps)]
        stored = [torch.cuda.Event() for _ in range(nsteps)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(s_in)
        for i in range(nsteps):
            d_lhs, d_rhs, d_gs, d_out = bufs[i % 2]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(computed[i - 2])      # buffer set free again
                d_lhs.copy_(h_lhs, non_blocking=True)
                d_rhs.copy_(h_rhs, non_blocking=True)
                d_gs.copy_(h_gs, non_blocking=True)
                loaded[i].record(s_in)
            stream.wait_event(loaded[i])
            if i >= 2:
                stream.wait_event(stored[i - 2])          # output buffer downloaded
            rd.ragged_dot(d_lhs, d_rhs, d_gs, out=d_out, stream=stream)
            computed[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(computed[i])
                h_out[i % 2].copy_(d_out, non_blocking=True)
                stored[i].record(s_out)
        s_out.wait_event(stored[nsteps - 1])
        t1.record(s_out)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    run_e2e(2)  # warm-up
    e2e_ms = max_over_ranks(pg, run_e2e(e2e_steps), device)
    e2e_value = world * flops / (e2e_ms / e2e_steps * 1e-3) / 1e12
    h2d = h_lhs.numel() * 2 + h_rhs.numel() * 2 + h_gs.numel() * 4
    d2h = h_out[0].numel() * 2

    # What bounds the end-to-end step: the host link.  The step's own upload and
    # download run concurrently on the two copy streams (as in the pipeline),
    # each timed on its stream; the step can be no faster than the slower
    # direction or the forward itself.
    def link_gbs(reps=3):
        d_lhs, d_rhs, d_gs, d_out = bufs[0]
        ti = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        to = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        torch.cuda.synchronize()
        ti[0].record(s_in)
        to[0].record(s_out)
        for _ in range(reps):
            with torch.cuda.stream(s_in):
                d_lhs.copy_(h_lhs, non_blocking=True)
                d_rhs.copy_(h_rhs, non_blocking=True)
                d_gs.copy_(h_gs, non_blocking=True)
            with torch.cuda.stream(s_out):
                h_out[0].copy_(d_out, non_blocking=True)
        ti[1].record(s_in)
        to[1].record(s_out)
        torch.cuda.synchronize()
        return (reps * h2d / (ti[0].elapsed_time(ti[1]) * 1e-3) / 1e9,
                reps * d2h / (to[0].elapsed_time(to[1]) * 1e-3) / 1e9)

    # the best of three short measurements: the host link is shared with the rest of the
    # machine, and one slow moment would otherwise set the bound
    trials = [link_gbs() for _ in range(3)]
    h2d_gbs, d2h_gbs = max(t[0] for t in trials), max(t[1] for t in trials)
    step_floor_s = max(h2d / (h2d_gbs * 1e9), d2h / (d2h_gbs * 1e9), ms_per_step * 1e-3)
    e2e_limit = world * flops / step_floor_s / 1e12
    del bufs
    torch.cuda.empty_cache()

    ops = None
    if not args.no_ops and rank == 0:
        detail = run_ops(rd, device, stream, peaks)
        if args.ops_json:
            with open(args.ops_json, "w") as f:
                json.dump(detail, f, indent=1)
        ops = compact_ops(detail)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, dt, desc, _ = oracle_sample_run(w, h_lhs, h_rhs, target_s=10.0)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
               "host_cores": os.cpu_count(), "sample": desc, "seconds": round(dt, 2)}

    if rank == 0:
        line = {
            "metric": "grouped-GEMM TFLOP/s (valid rows)",
            "value": value,
            "unit": "TFLOP/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": ms_per_step,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": w.name, "m": w.m, "k": w.k, "n": w.n, "g": w.g_total,
                       "valid_rows": rows, "group_sizes": w.group_sizes.tolist(),
                       "l2": "inputs larger than L2 (2.15 GB per step), no flush",
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "tensor", "achieved": _sig(achieved, 5), "peak": peak,
                         "unit": "TFLOP/s", "frac": _sig(achieved / peak, 4), "traffic": traffic,
                         "peak_source": f"{peak_src} bf16_tflops (burst)",
                         "algorithmic_bytes": alg_bytes,
                         "kernel": "grouped_gemm_kernel<fwd>"},
            "e2e": {"value": _sig(e2e_value, 5), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "pipelined": "upload i+1 / forward i / download i-1 on three streams",
                    "bound": {"h2d_gbs": _sig(h2d_gbs), "d2h_gbs": _sig(d2h_gbs),
                              "limit": _sig(e2e_limit), "frac": _sig(e2e_value / e2e_limit, 3)}},
            "gpu_launches": args.steps,
            "launch_ms": {"median": _sig(statistics.median(per), 5),
                          "p10": _sig(statistics.quantiles(per, n=10)[0] if len(per) > 1 else per[0], 5),
                          "p90": _sig(statistics.quantiles(per, n=10)[-1] if len(per) > 1 else per[0], 5)},
            "clocks": clk.summary(),
            "cpu_baseline": cpu,
            "ops": ops,
        }
        print(json.dumps(line))
    if pg is not None:
        pg.destroy_process_group()
    return 0


def run_profile(args):
    """A few launches of one workload, for ncu (no extras, no host copies)."""
    import numpy as np
    import torch

    import expert_ffn_ragged_gb300 as rd
    import workloads
    from workloads import normal_bf16

    rd.load()
    device = torch.device("cuda", 0)
    name = args.profile
    if name in ("mixtral", "mixtral_small"):
        w = workloads.mixtral_fwd()
        # mixtral_small: the same forward with a quarter of the tokens (8189 rows, 1.2 GB)
        sizes = w.group_sizes if name == "mixtral" else (w.group_sizes // 4).astype("int32")
        m = int(sizes.sum())
        lhs = normal_bf16((m, w.k), 1.0, 20, device)
        rhs = normal_bf16((w.g_total, w.k, w.n), w.rhs_var, 21, device)
        gs = torch.tensor(sizes, dtype=torch.int32, device=device)
        out = torch.empty((m, w.n), dtype=torch.bfloat16, device=device)
        fn = lambda: rd.ragged_dot(lhs, rhs, gs, out=out)
    elif name == "packed_glu":
        w = workloads.packed_glu_fwd()
        lhs = normal_bf16((w.m, w.k), 1.0, 30, device)
        rhs = normal_bf16((w.g_local, w.k, w.n), w.rhs_var, 31, device)
        gs = torch.tensor(w.group_sizes, dtype=torch.int32, device=device)
        lim = torch.tensor([w.limit], dtype=torch.int32, device=device)
        out = torch.empty((w.m, w.n // 2), dtype=torch.bfloat16, device=device)
        fn = lambda: rd.ragged_dot(lhs, rhs, gs, w.group_offset, lim, rd.EPI_SILU_GLU, out)
    elif name in ("dx", "dw", "dw_f32acc"):
        w = workloads.backward_pair()
        ws = torch.empty(rd.dw_workspace_bytes(device), dtype=torch.uint8, device=device)
        gs = torch.tensor(w.group_sizes, dtype=torch.int32, device=device)
        do = normal_bf16((w.m, w.n), 1.0, 41, device)
        if name == "dw_f32acc":
            x = normal_bf16((w.m, w.k), 1.0, 40, device)
            dw32 = torch.zeros((w.g_total, w.k, w.n), dtype=torch.float32, device=device)
            fn = lambda: rd.trans_ragged_dot_f32(x, do, gs, out=dw32, accumulate=True, workspace=ws)
        elif name == "dx":
            wt = normal_bf16((w.g_total, w.k, w.n), w.rhs_var, 42, device)
            dx = torch.empty((w.m, w.k), dtype=torch.bfloat16, device=device)
            fn = lambda: rd.ragged_dot_trans_rhs(do, wt, gs, out=dx)
        else:
            x = normal_bf16((w.m, w.k), 1.0, 40, device)
            dw = torch.empty((w.g_total, w.k, w.n), dtype=torch.bfloat16, device=device)
            fn = lambda: rd.trans_ragged_dot(x, do, gs, out=dw, workspace=ws)
    elif name == "packed_dx_glu_bwd":
        w = workloads.packed_glu_fwd()
        gs = torch.tensor(w.group_sizes, dtype=torch.int32, device=device)
        lim = torch.tensor([w.limit], dtype=torch.int32, device=device)
        d_out = normal_bf16((w.m, 4096), 1.0, 35, device)
        w_down = normal_bf16((w.g_local, 1024, 4096), 1.0 / 4096, 36, device)
        fused2 = normal_bf16((w.m, 2048), 1.0, 37, device)
        dfused2 = torch.empty_like(fused2)
        fn = lambda: rd.ragged_dot_trans_rhs_glu_bwd(d_out, w_down, fused2, gs, w.group_offset, lim,
                                                     dfused2)
    elif name == "unsort":
        w = workloads.packed_glu_fwd()
        lim = torch.tensor([w.limit], dtype=torch.int32, device=device)
        g = normal_bf16((w.m, 4096), 1.0, 33, device)
        y = normal_bf16((w.m, 4096), 1.0, 34, device)
        wt = torch.rand((w.m,), device=device)
        grad = torch.empty_like(g)
        dot = torch.empty((w.m,), dtype=torch.float32, device=device)
        fn = lambda: rd.unsort_bwd_rows(g, y, wt, lim, grad, dot)
    elif name in ("glu_fwd", "glu_bwd"):
        w = workloads.packed_glu_fwd()
        lim = torch.tensor([w.limit], dtype=torch.int32, device=device)
        fused = normal_bf16((w.m, 2048), 1.0, 32, device)
        gout = torch.empty((w.m, 1024), dtype=torch.bfloat16, device=device)
        dfused = torch.empty_like(fused)
        fn = (lambda: rd.glu_fwd(fused, lim, gout)) if name == "glu_fwd" else \
            (lambda: rd.glu_bwd(fused, gout, lim, dfused))
    elif name == "decode":
        w = workloads.decode_fwd(True)
        lhs = normal_bf16((w.m, w.k), 1.0, 50, device)
        up = normal_bf16((w.g_total, w.k, w.n), w.rhs_var, 51, device)
        down = normal_bf16((w.g_total, w.n // 2, w.k), 1.0 / (w.n // 2), 52, device)
        gs = torch.tensor(w.group_sizes, dtype=torch.int32, device=device)
        h = torch.empty((w.m, w.n // 2), dtype=torch.bfloat16, device=device)
        o = torch.empty((w.m, w.k), dtype=torch.bfloat16, device=device)

        def fn():
            rd.ragged_dot(lhs, up, gs, epilogue=rd.EPI_SILU_GLU, out=h)
            rd.ragged_dot(h, down, gs, out=o)
    elif name == "ffn4096_up":
        # the expert-FFN up projection (GLU) at 4096 tokens: ~256 rows per expert
        w = workloads.expert_ffn(4096)
        lhs = normal_bf16((w.m, w.k), 1.0, 63, device)
        up = normal_bf16((w.g_total, w.k, w.n), 1.0 / w.k, 61, device)
        gs = torch.tensor(w.group_sizes, dtype=torch.int32, device=device)
        h = torch.empty((w.m, w.n // 2), dtype=torch.bfloat16, device=device)
        fn = lambda: rd.ragged_dot(lhs, up, gs, epilogue=rd.EPI_SILU_GLU, out=h)
    else:
        raise SystemExit(f"unknown profile workload {name}")
    for _ in range(args.steps):
        fn()
    torch.cuda.synchronize()
    print(json.dumps({"profile": name, "launches": args.steps}))
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["rd", "reference"], default="rd")
    ap.add_argument("--no-ops", action="store_true", help="skip the other hot-path rows")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", default=None, help="run only a few launches of a workload (for ncu)")
    ap.add_argument("--ops-json", default=None,
                    help="also write the other rows' full timings (p10/p90, GB/s, TFLOP/s) to this file")
    args = ap.parse_args()
    if args.warmup < 3 and args.profile is None:
        args.warmup = 3
    if args.profile:
        return run_profile(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_rd(args)


if __name__ == "__main__":
    sys.exit(main())
