"""Benchmark of the dense GEMM library at M = N = K = 4096.

One step is one pass of the whole path: an FP32 SGEMM (alpha 1, beta 3, C
reset to its seeded values first) followed by an FP16-input / FP32-accumulate
GEMM (alpha 1, beta 0), both 4096^3, inputs resident in HBM.  L2 is flushed
(a 256 MB write) before each GEMM; resets and flushes are outside the
per-GEMM CUDA-event intervals that give ms_per_step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (fp64 triple loop) on the host cores,
on a bounded row sample of the same workload.  Under torchrun (N > 1) every
rank runs the same workload on its own GPU (replicas: the product shards by
output rows with no exchange), rank 0 prints the JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "TFLOPS at 4096³ (FP32 SGEMM; FP16-in/FP32-acc) and % of GB300 roofline"
SIZE = 4096
FLOPS_ONE = 2 * SIZE ** 3
FLOPS_STEP = 2 * FLOPS_ONE
WORKLOAD = ("square 4096^3 x2 per step: FP32 SGEMM (alpha 1, beta 3, C reset to seeded U[-1,1] before each "
            "run, A/B U[-1,1]) then FP16-in/FP32-acc GEMM (alpha 1, beta 0, A/B N(0,1/sqrt(K)) in fp16)")


L2_NOTE = "flushed (256 MB write) before every GEMM, outside the timed intervals"


def bench_config(world: int) -> dict:
    """The workload description both arms print (identical dicts)."""
    return {"workload": WORKLOAD, "M": SIZE, "N": SIZE, "K": SIZE, "l2": L2_NOTE, "parallelism": f"replicas x{world}"}


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms while running.
    Each sample carries nvidia-smi's timestamp; window(t0, t1) limits the
    summary to the samples taken inside a wall-clock interval (the timed
    region), falling back to all samples when none falls inside it."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = os.path.join("/tmp", f"gemm11_clocks_{os.getpid()}.csv")
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=open(self.out, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def window(self, t0: float, t1: float):
        """Restrict the summary to samples between the wall-clock times t0 and t1."""
        self.t0, self.t1 = t0, t1

    @staticmethod
    def _stamp(text: str):
        import datetime
        try:
            return datetime.datetime.strptime(text.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except Exception:
            return None

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        try:
            for line in open(self.out):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10 and parts[2].replace(".", "").isdigit():
                    rows.append(parts)
        except Exception:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        inside = rows
        if self.t0 is not None:
            inside = [r for r in rows if (t := self._stamp(r[0])) is not None and self.t0 <= t <= self.t1]
        scope = "timed region" if inside and self.t0 is not None else "whole run"
        use = inside or rows
        sm = [float(r[2]) for r in use]
        smax = max(float(r[3]) for r in use)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i in range(4) if r[6 + i].lower() == "active"})
        power = [float(r[4]) for r in use if r[4].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": reasons, "samples": len(use),
                "samples_scope": scope, "sampling_ms": 20, "power_w_max": max(power) if power else None}


def max_over_ranks(values, dist=None, device=None):
    """Element-wise max of per-rank timings (every rank gets the result)."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if dist is not None and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def replica_throughput(flops_per_rank_step: float, world: int, ms_per_step_max: float) -> float:
    """Whole-job TFLOP/s of `world` independent replicas timed by the slowest rank."""
    return world * flops_per_rank_step / (ms_per_step_max * 1e-3) / 1e12


def _oracle_inputs():
    import oracle
    from dense_gemm_11_gb300 import inputs
    w32, w16 = inputs.WORKLOADS["f32_sq4096"], inputs.WORKLOADS["f16_4096"]
    return oracle, inputs.make_workload(w32), inputs.make_workload(w16)


def _oracle_rows_for(seconds: float, oracle, d32, threads: int) -> int:
    """Rows of each 4096^3 GEMM (both together) that the oracle evaluates in
    about `seconds` on `threads` host threads (a multiple of threads, 1..4096)."""
    import numpy as np
    rows = np.arange(4 * threads, dtype=np.int64)
    oracle.gemm(d32["A"], d32["B"], d32["C"], alpha=1.0, beta=3.0, rows=rows[:threads], threads=threads)  # warm
    t0 = time.perf_counter()
    oracle.gemm(d32["A"], d32["B"], d32["C"], alpha=1.0, beta=3.0, rows=rows, threads=threads)
    per_row = (time.perf_counter() - t0) / len(rows)
    n = int(min(SIZE, seconds / 2 / max(per_row, 1e-6)))
    return min(SIZE, max(threads, (n // threads) * threads))


def _oracle_step(oracle, d32, d16, rows, threads):
    """One step of the bench workload on the listed output rows of both GEMMs;
    returns (seconds, fp32 seconds, fp16 seconds)."""
    t0 = time.perf_counter()
    oracle.gemm(d32["A"], d32["B"], d32["C"], alpha=1.0, beta=3.0, rows=rows, threads=threads)
    t1 = time.perf_counter()
    oracle.gemm(d16["A"], d16["B"], None, alpha=1.0, beta=0.0, rows=rows, threads=threads)
    t2 = time.perf_counter()
    return t2 - t0, t1 - t0, t2 - t1


def cpu_oracle_sample(target_s: float = 12.0):
    """Time the oracle (as it stands) on rows of both 4096^3 GEMMs; about target_s seconds."""
    import numpy as np
    oracle, d32, d16 = _oracle_inputs()
    threads = oracle.default_threads()
    n = _oracle_rows_for(target_s, oracle, d32, threads)
    rows = np.linspace(0, SIZE - 1, n).astype(np.int64)
    secs, s32, s16 = _oracle_step(oracle, d32, d16, rows, threads)
    flops = 2 * (2 * n * SIZE * SIZE)
    return {
        "value": flops / secs / 1e12,
        "unit": "TFLOPS",
        "cores": threads,
        "kind": "oracle",
        "sample": f"{n} of 4096 output rows of each 4096^3 GEMM (fp32 and fp16-in), fp64 accumulation; "
                  f"{secs:.1f} s on {threads} host threads ({s32:.1f} s fp32 + {s16:.1f} s fp16)",
    }


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm.  Every step (warm-up and timed)
    evaluates the same bounded sample of the workload -- n output rows of
    each 4096^3 GEMM, n sized so that all warm-up and timed steps take about
    --ref-budget-s seconds (100) -- and ms_per_step is the measured wall time
    of those steps."""
    if rank != 0:
        return
    import numpy as np
    oracle, d32, d16 = _oracle_inputs()
    threads = oracle.default_threads()
    n = _oracle_rows_for(args.ref_budget_s / (args.steps + args.warmup), oracle, d32, threads)
    rows = np.linspace(0, SIZE - 1, n).astype(np.int64)
    for _ in range(args.warmup):
        _oracle_step(oracle, d32, d16, rows, threads)
    secs = [_oracle_step(oracle, d32, d16, rows, threads)[0] for _ in range(args.steps)]
    ms = statistics.mean(secs) * 1e3
    flops_step = 2 * (2 * n * SIZE * SIZE)
    value = flops_step / (ms * 1e-3) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "ms_per_step_median":
        statistics.median(secs) * 1e3, "ms_per_step_min": min(secs) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(args.gpus),
        "step_sample": f"each step evaluates {n} of the 4096 output rows of both GEMMs "
                       f"({flops_step / 1e9:.1f} of {FLOPS_STEP / 1e9:.1f} GFLOP)",
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": threads, "kind": "oracle",
                         "sample": f"{n} of 4096 output rows of each 4096^3 GEMM (fp32 and fp16-in) per step, "
                                   f"fp64 accumulation, {threads} host threads; {args.steps} timed steps"},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch

    import dense_gemm_11_gb300 as g
    from dense_gemm_11_gb300 import inputs, roofline

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    hbm_gbs, tc_peak, tc_sustained, peak_src = _peaks()
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    # the tensor core's dense rate per SM, measured (untimed; see gemm_tc_rate_probe)
    try:
        tc_rate = g.tc_rate_probe()
    except g.GemmError:
        tc_rate = None
    # the FP32 FMA units' rate for the packed form gemm_f32 uses and for scalar
    # FMAs (untimed; see gemm_fma_rate_probe)
    try:
        fma_rates = {"packed_ffma2": g.fma_rate_probe(True), "scalar_ffma": g.fma_rate_probe(False)}
    except g.GemmError:
        fma_rates = None

    w32, w16 = inputs.WORKLOADS["f32_sq4096"], inputs.WORKLOADS["f16_4096"]
    d32, d16 = inputs.make_workload(w32), inputs.make_workload(w16)
    A32 = torch.from_numpy(d32["A"]).to(dev)
    B32 = torch.from_numpy(d32["B"]).to(dev)
    C32_0 = torch.from_numpy(d32["C"]).to(dev)
    C32 = C32_0.clone()
    A16 = torch.from_numpy(d16["A"]).to(dev)
    B16 = torch.from_numpy(d16["B"]).to(dev)
    C16 = torch.empty(SIZE, SIZE, device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, device=dev)
    stream = torch.cuda.current_stream(dev)

    launches = [0]
    plans = {}

    def gemm32():
        g.gemm_f32(A32, B32, C32, alpha=1.0, beta=3.0, stream=stream)
        launches[0] += g.last_launch_count()
        plans["sgemm_f32"] = g.last_plan()

    def gemm16():
        g.gemm_f16_f32acc_epilogue(A16, B16, C16, alpha=1.0, beta=0.0, stream=stream)
        launches[0] += g.last_launch_count()
        plans["gemm_f16"] = g.last_plan()

    def step(ev):
        C32.copy_(C32_0)
        flush.fill_(1.0)
        ev[0].record(stream)
        gemm32()
        ev[1].record(stream)
        flush.fill_(2.0)
        ev[2].record(stream)
        gemm16()
        ev[3].record(stream)

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    # Clocks are sampled from the warm-up through the end of the timed region.
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        for _ in range(args.warmup):
            step([torch.cuda.Event(enable_timing=True) for _ in range(4)])
        torch.cuda.synchronize(dev)
        assert g.check(stream) == g.GEMM_OK
        launches[0] = 0
        if dist:
            dist.barrier()
        torch.cuda.synchronize(dev)
        t_wall0 = time.perf_counter()
        t_epoch0 = time.time()
        for s in range(args.steps):
            step(events[s])
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall0
        clk.window(t_epoch0, time.time())
        if dist:
            dist.barrier()
    st = g.check(stream)
    if st != g.GEMM_OK:
        raise RuntimeError(f"watchdog: {g.status_string(st)}")
    t32 = [e[0].elapsed_time(e[1]) for e in events]
    t16 = [e[2].elapsed_time(e[3]) for e in events]
    t_step = [a + b for a, b in zip(t32, t16)]
    ms_step = statistics.mean(t_step)
    gpu_launches = launches[0]

    # e2e through the public API: every step copies its inputs from pinned host
    # memory to the device, runs both GEMMs and reads both results back to
    # pinned host memory.  Steps are pipelined over three device buffer sets
    # and three streams (inputs of step i+1 travel while step i computes;
    # results of step i travel back while step i+1 computes), as a serving
    # loop would.  With three sets the inputs of step i+1 wait only for the
    # results of step i-2, which left while step i-1 ran, so neither copy
    # direction is chained to the other.
    hA32 = torch.from_numpy(d32["A"]).pin_memory()
    hB32 = torch.from_numpy(d32["B"]).pin_memory()
    hC32 = torch.from_numpy(d32["C"]).pin_memory()
    hA16 = torch.from_numpy(d16["A"]).pin_memory()
    hB16 = torch.from_numpy(d16["B"]).pin_memory()
    oC32 = torch.empty(SIZE, SIZE).pin_memory()
    oC16 = torch.empty(SIZE, SIZE).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hA32, hB32, hC32, hA16, hB16))
    d2h = sum(t.numel() * t.element_size() for t in (oC32, oC16))
    NSETS = 3
    bufs = [dict(A32=A32, B32=B32, C32=C32, A16=A16, B16=B16, C16=C16)] + [
        dict(A32=torch.empty_like(A32), B32=torch.empty_like(B32), C32=torch.empty_like(C32),
             A16=torch.empty_like(A16), B16=torch.empty_like(B16), C16=torch.empty_like(C16))
        for _ in range(NSETS - 1)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(NSETS)]
    ev_comp = [torch.cuda.Event() for _ in range(NSETS)]
    ev_out = [torch.cuda.Event() for _ in range(NSETS)]

    def copy_gbs(dst, src, st, reps=5):
        """Best-of-reps GB/s of one pinned-host <-> device copy on its own stream."""
        best = None
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st)
            with torch.cuda.stream(st):
                dst.copy_(src, non_blocking=True)
            b.record(st)
            b.synchronize()
            ms = a.elapsed_time(b)
            best = ms if best is None else min(best, ms)
        return src.numel() * src.element_size() / (best * 1e-3) / 1e9

    h2d_gbs = copy_gbs(bufs[1]["A32"], hA32, s_in)
    d2h_gbs = copy_gbs(oC32, bufs[1]["A32"], s_out)

    def e2e_run(n):
        """n pipelined steps; returns (start, end) events spanning all of them."""
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        stream.wait_event(e0)
        s_out.wait_event(e0)
        out_pending = [False] * NSETS

        def load(i):
            b = bufs[i % NSETS]
            if out_pending[i % NSETS]:
                s_in.wait_event(ev_out[i % NSETS])  # this set's previous results have left
            with torch.cuda.stream(s_in):
                for k, h in (("A32", hA32), ("B32", hB32), ("C32", hC32), ("A16", hA16), ("B16", hB16)):
                    b[k].copy_(h, non_blocking=True)
            ev_in[i % NSETS].record(s_in)

        load(0)
        for i in range(n):
            if i + 1 < n:
                load(i + 1)
            b = bufs[i % NSETS]
            stream.wait_event(ev_in[i % NSETS])
            g.gemm_f32(b["A32"], b["B32"], b["C32"], alpha=1.0, beta=3.0, stream=stream)
            g.gemm_f16_f32acc_epilogue(b["A16"], b["B16"], b["C16"], alpha=1.0, beta=0.0, stream=stream)
            ev_comp[i % NSETS].record(stream)
            s_out.wait_event(ev_comp[i % NSETS])
            with torch.cuda.stream(s_out):
                oC32.copy_(b["C32"], non_blocking=True)
                oC16.copy_(b["C16"], non_blocking=True)
            ev_out[i % NSETS].record(s_out)
            out_pending[i % NSETS] = True
        s_out.wait_stream(s_in)
        s_out.wait_stream(stream)
        e1.record(s_out)
        return e0, e1

    e2e_run(2)
    torch.cuda.synchronize(dev)
    n_e2e = max(3, args.steps)
    e0, e1 = e2e_run(n_e2e)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / n_e2e
    # the results that came back are the GEMMs' own (spot check of one step)
    torch.cuda.synchronize(dev)
    if not (torch.equal(oC16, bufs[(n_e2e - 1) % NSETS]["C16"].cpu()) and torch.isfinite(oC32[:4]).all()):
        raise RuntimeError("e2e: results read back do not match the device results")

    # max over ranks
    stats = [ms_step, e2e_ms, statistics.mean(t32), statistics.mean(t16), statistics.median(t_step), min(t_step),
             statistics.median(t32), min(t32), statistics.median(t16), min(t16)]
    (ms_step, e2e_ms, ms32, ms16, med_step, min_step, med32, min32, med16, min16) = max_over_ranks(stats, dist, dev)
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    clocks = clk.summary()
    f32_peak_max = roofline.fp32_fma_peak_tflops(sms, clocks.get("sm_max_mhz") or 2070.0)
    f32_peak_obs = roofline.fp32_fma_peak_tflops(sms, clocks["sm_mhz"]) if clocks.get("sm_mhz") else None
    ach32 = FLOPS_ONE / (ms32 * 1e-3) / 1e12
    ach16 = FLOPS_ONE / (ms16 * 1e-3) / 1e12
    traffic = _traffic_from_profiles()
    value = replica_throughput(FLOPS_STEP, world, ms_step)
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "ms_per_step_median": med_step,
        "ms_per_step_min": min_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "dtypes": {"sgemm": "f32 (FFMA)", "tensor_core": "f16 in, f32 accumulate"},
        "data": "synthetic",
        "config": bench_config(world),
        "plans": plans,
        "paths": {
            "sgemm_f32": {"ms": ms32, "ms_median": med32, "ms_min": min32, "tflops": ach32,
                          "tflops_at_median": FLOPS_ONE / (med32 * 1e-3) / 1e12,
                          "frac_of_fp32_peak_at_max_clock": ach32 / f32_peak_max,
                          "frac_of_fp32_peak_at_observed_clock": (ach32 / f32_peak_obs) if f32_peak_obs else None},
            "gemm_f16_f32acc": {"ms": ms16, "ms_median": med16, "ms_min": min16, "tflops": ach16,
                                "tflops_at_median": FLOPS_ONE / (med16 * 1e-3) / 1e12,
                                "frac_of_measured_bf16_peak": ach16 / tc_peak},
        },
        "roofline": {"bound": "alu", "achieved": ach32, "peak": f32_peak_max, "unit": "TFLOP/s",
                     "frac": ach32 / f32_peak_max, "traffic": traffic.get("sgemm"),
                     "kernel": "sgemm_tiled_kernel (FP32 FFMA)",
                     "peak_source": f"{sms} SMs x 128 FP32 lanes x 2 x {clocks.get('sm_max_mhz') or 2070.0} MHz",
                     **_fma_ceiling(fma_rates, ach32, sms, clocks.get("sm_mhz") or clocks.get("sm_max_mhz") or 2070.0)},
        "roofline_tensor": {"bound": "tensor", "achieved": ach16, "peak": tc_peak, "unit": "TFLOP/s",
                            "frac": ach16 / tc_peak, "traffic": traffic.get("hgemm"),
                            "kernel": f"tcgen05 f16 GEMM, plan {plans.get('gemm_f16')}",
                            "peak_source": f"{peak_src} bf16 burst (fp16 runs at the bf16 rate)",
                            **_nominal_tensor_peak(tc_rate, sms, clocks.get("sm_max_mhz") or 2070.0, ach16)},
        "e2e": {"value": replica_throughput(FLOPS_STEP, world, e2e_ms), "unit": "TFLOPS",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "h2d_gbs": h2d_gbs, "d2h_gbs": d2h_gbs,
                "copy_bound_ms": max(h2d / (h2d_gbs * 1e9), d2h / (d2h_gbs * 1e9)) * 1e3,
                "copy_streams": "inputs on one stream, results on another, GEMMs on a third",
                "pipelining": "three device buffer sets: inputs of step i+1 and results of step i-1 travel "
                              "while step i computes"},
        "gpu_launches": gpu_launches,
        "clocks": clocks,
        "wall_s_timed_region": t_wall,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_sample()
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def _fma_ceiling(rates, achieved_tflops, sms, mhz):
    """The SGEMM's FMAs per clock per SM (at the observed clock) against the
    measured rates of the packed and scalar FMA forms (gemm_fma_rate_probe)."""
    if not rates:
        return {"fma_rate_probe": None}
    per_clk = achieved_tflops * 1e12 / 2 / (sms * mhz * 1e6)
    return {"fma_rate_probe": {**{k: round(v, 2) for k, v in rates.items()}, "unit": "FMA/clock/SM",
                               "nominal": 128, "sgemm_fma_per_clock_per_sm": round(per_clk, 2),
                               "sgemm_frac_of_packed_rate": per_clk / rates["packed_ffma2"]}}


def _nominal_tensor_peak(rate, sms, mhz, achieved):
    """#SM x the measured dense FLOP per clock per SM x the maximum SM clock."""
    if not rate:
        return {"nominal_peak": None}
    nominal = rate * sms * mhz * 1e6 / 1e12
    return {"nominal_peak": nominal, "frac_of_nominal": achieved / nominal,
            "nominal_source": f"{sms} SMs x {rate:.0f} FLOP/clock/SM (tcgen05 rate probe) x {mhz:.0f} MHz"}


def _traffic_from_profiles():
    """DRAM bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum) from
    profiles/traffic.json; an entry counts only while its kernel sources (the
    .cu file and the shared PTX header) are unchanged."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    out = {}
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return out
    for key, r in rec.items():
        try:
            out[key] = r["bytes"] if source_sha(r["sources"]) == r["sha"] else None
        except Exception:
            out[key] = None
    return out


def source_sha(sources):
    """First 16 hex digits of the SHA-256 of the listed source files, concatenated."""
    import hashlib
    h = hashlib.sha256()
    for src in sources:
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _workload_call(w, d, dev, nsets):
    """Device copies (nsets sets of A, B, C) of a named workload's arrays and
    call(t, stream=None), the library call the workload names."""
    import torch

    import dense_gemm_11_gb300 as g
    in_t = torch.bfloat16 if w.kind == "bf16" else None
    out_t = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[w.out]
    general = w.kind != "f32" and (w.batch > 1 or w.b_trans or w.out != "f32")
    sets = []
    for _ in range(nsets):
        t = {k: torch.from_numpy(d[k]).to(dev) for k in ("A", "B", "C")}
        if in_t is not None:  # bf16 values travel as float32 arrays
            t["A"], t["B"] = t["A"].to(in_t), t["B"].to(in_t)
        t["C"] = t["C"].to(out_t)
        if general and w.batch == 1 and not w.b_trans:
            t = {k: v.unsqueeze(0) for k, v in t.items()}
        sets.append(t)
    bias = torch.from_numpy(d["bias"]).to(dev) if "bias" in d else None

    def call(t, st=None):
        st = torch.cuda.current_stream(dev) if st is None else st
        if general:
            g.gemm_tc_batched(t["A"], t["B"], t["C"], alpha=w.alpha, beta=w.beta, bias=bias, act=w.act,
                              b_trans=w.b_trans, stream=st)
        elif w.kind == "f32":
            g.gemm_f32(t["A"], t["B"], t["C"], alpha=w.alpha, beta=w.beta, stream=st)
        elif w.kind == "f32x3":
            g.gemm_f32_3xtf32(t["A"], t["B"], t["C"], alpha=w.alpha, beta=w.beta, stream=st)
        elif w.kind == "bf16":
            g.gemm_bf16_f32acc_epilogue(t["A"], t["B"], t["C"], alpha=w.alpha, beta=w.beta, bias=bias,
                                        act=w.act, stream=st)
        else:
            g.gemm_f16_f32acc_epilogue(t["A"], t["B"], t["C"], alpha=w.alpha, beta=w.beta, bias=bias,
                                       act=w.act, stream=st)

    return sets, call


def run_profile_case(case: str, repeats: int):
    """One GEMM launched `repeats` times, for ncu captures: the bench's FP32
    SGEMM ("sgemm"), its FP16 GEMM ("hgemm"), FP32 through 3 x TF32 at
    4096^3 ("tf32x3"), or any named workload of inputs.WORKLOADS."""
    import torch

    import dense_gemm_11_gb300 as g
    from dense_gemm_11_gb300 import inputs
    dev = torch.device("cuda", 0)
    if case in inputs.WORKLOADS:
        sets, call = _workload_call(inputs.WORKLOADS[case], inputs.make_workload(inputs.WORKLOADS[case]), dev, 1)
        for _ in range(repeats):
            call(sets[0])
    elif case in ("sgemm", "tf32x3"):
        d = inputs.make_workload(inputs.WORKLOADS["f32_sq4096"])
        A, B, C = (torch.from_numpy(d[k]).to(dev) for k in ("A", "B", "C"))
        fn = g.gemm_f32 if case == "sgemm" else g.gemm_f32_3xtf32
        for _ in range(repeats):
            fn(A, B, C, alpha=1.0, beta=3.0)
    else:
        d = inputs.make_workload(inputs.WORKLOADS["f16_4096"])
        A, B = (torch.from_numpy(d[k]).to(dev) for k in ("A", "B"))
        C = torch.empty(SIZE, SIZE, device=dev)
        for _ in range(repeats):
            g.gemm_f16_f32acc_epilogue(A, B, C, alpha=1.0, beta=0.0)
    torch.cuda.synchronize()
    assert g.check() == g.GEMM_OK
    print(f"{case}: {repeats} launches of plan {g.last_plan()}")


def run_sweep(reps: int, only=None):
    """Time every named workload (one JSON line each).

    Two figures per workload: `ms` is the median of single calls, each after
    a C reset and an L2 flush (cold L2, GPU briefly idle before the call);
    `ms_steady` is the mean over back-to-back calls that cycle through enough
    copies of A, B and C (> 2x L2) that no call finds its inputs in L2 --
    the steady-state throughput of a stream of such GEMMs.  `frac` uses the
    steady figure against min(compute peak, HBM bandwidth x intensity)."""
    import torch

    import dense_gemm_11_gb300 as g
    from dense_gemm_11_gb300 import inputs, roofline
    dev = torch.device("cuda", 0)
    hbm_gbs, tc_peak, _, _ = _peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    f32_peak = roofline.fp32_fma_peak_tflops(sms, 2070.0)
    flush = torch.empty(256 * 1024 * 1024 // 4, device=dev)
    stream = torch.cuda.current_stream(dev)
    l2_bytes = 129 * 1024 * 1024
    for name, w in inputs.WORKLOADS.items():
        if only and name not in only:
            continue
        d = inputs.make_workload(w)
        set_bytes = sum(d[k].nbytes for k in ("A", "B", "C"))
        nbuf = max(1, min(16, -(-3 * l2_bytes // set_bytes)))
        sets, call = _workload_call(w, d, dev, nbuf)
        C0 = sets[0]["C"].clone()

        times = []
        for r in range(reps + 3):
            sets[0]["C"].copy_(C0)
            flush.fill_(float(r))
            torch.cuda._sleep(2_000_000)  # GPU busy while the host enqueues the call
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            call(sets[0])
            e1.record(stream)
            torch.cuda.synchronize(dev)
            if r >= 3:
                times.append(e0.elapsed_time(e1))
        plan = g.last_plan()
        # steady state: back-to-back calls over rotating input sets (C is
        # overwritten with beta = 0 or keeps growing with beta != 0: same work),
        # captured in a CUDA graph so that host-side argument handling is not
        # between the kernels
        n_steady = max(2 * nbuf, 20)
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            for i in range(nbuf):
                call(sets[i])  # split-K scratch is per stream: allocate it outside the capture
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            for i in range(n_steady):
                call(sets[i % nbuf], cap)
        graph.replay()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        assert g.check(stream) == g.GEMM_OK
        ms_steady = e0.elapsed_time(e1) / n_steady
        del graph
        ms = statistics.median(times)
        flops = roofline.gemm_flops(w.M, w.N, w.K, w.batch)
        nbytes = roofline.gemm_bytes(w.M, w.N, w.K, in_bytes=4 if w.kind in ("f32", "f32x3") else 2,
                                     beta_nonzero=w.beta != 0.0, bias=w.bias, out_bytes=4 if w.out == "f32" else 2,
                                     batch=w.batch)
        # 3 x TF32: the FP32 product's flops against the tensor core's TF32 rate
        # (half the measured bf16 rate) divided by the three products it takes.
        peak = f32_peak if w.kind == "f32" else (tc_peak / 2 / 3 if w.kind == "f32x3" else tc_peak)
        roof, bound = roofline.roofline_tflops(flops, nbytes, peak, hbm_gbs)
        tflops = flops / (ms_steady * 1e-3) / 1e12
        print(json.dumps({"workload": name, "batch": w.batch, "M": w.M, "N": w.N, "K": w.K, "plan": plan, "ms": ms,
                          "ms_steady": ms_steady, "input_sets": nbuf, "tflops": tflops,
                          "gbs": nbytes / (ms_steady * 1e-3) / 1e9, "bound": bound, "roofline_tflops": roof,
                          "frac": tflops / roof,
                          "peak_note": {"f32": "fp32 FFMA at 2070 MHz",
                                        "f32x3": "measured bf16 burst / 2 (TF32) / 3 products"}.get(
                                            w.kind, "measured bf16 burst")}),
              flush=True)
        del sets
        torch.cuda.empty_cache()


def run_tma_probe_table(kblocks):
    """The TMA read probe (gemm_tma_read_probe) over own-copy and multicast loads,
    an L2-resident (24 MB) and an HBM (2048 MB) region, 1 to 76 clusters of two
    CTAs and 2 to 6 stages in flight: one JSON line per case."""
    import torch
    import dense_gemm_11_gb300 as g
    torch.cuda.set_device(0)
    for mc in (False, True):
        for region in (24, 2048):
            for cl in (1, 8, 38, 76):
                for st in (2, 4, 6):
                    r = g.tma_read_probe(cl, multicast=mc, stages=st, kblocks=kblocks, region_mb=region)
                    print(json.dumps(dict(clusters=cl, multicast=int(mc), stages=st, region_mb=region, **r)),
                          flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-budget-s", type=float, default=100.0,
                    help="--impl reference: wall-time budget of all its warm-up and timed steps together")
    ap.add_argument("--profile-case", default=None,
                    help="launch one GEMM a few times (for ncu) and exit: sgemm, hgemm or tf32x3 (the 4096^3 "
                         "bench GEMMs) or a workload name of inputs.WORKLOADS")
    ap.add_argument("--repeats", type=int, default=2)
    ap.add_argument("--sweep", action="store_true", help="time every named workload, one JSON line each")
    ap.add_argument("--workloads", default="", help="comma-separated workload names for --sweep (default: all)")
    ap.add_argument("--tma-probe", action="store_true",
                    help="run the TMA read probe over loads, regions, clusters and stages, one JSON line each")
    args = ap.parse_args()
    if args.tma_probe:
        run_tma_probe_table(1024)
        return
    if args.sweep:
        run_sweep(max(3, args.steps // 10), [w for w in args.workloads.split(",") if w])
        return
    if args.profile_case:
        run_profile_case(args.profile_case, args.repeats)
        return
    if args.warmup < 3:
        args.warmup = 3
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
