"""Offline autotuner: times every plan the library can run for a shape and
writes the winners as a tuning table (JSON) for ``load_tuning``.

The planners pick a kernel family, tile width and split-K factor by fixed
rules; this tool measures the alternatives on the GPU at hand, the way the
pages tune per shape and per GPU ("SGEMM优化，从naive到warptiling", kernel 9
and Q10; the DeepGEMM essay "企业官网建设流程全解析", section 1.3).  Every
candidate runs through the library's own C entry points with a one-entry
tuning table installed, so the timings are of exactly what a tuned call runs.

    python -m dense_gemm_11_gb300.autotune --workloads f16_epi1,f32_512 --out table.json
    python -m dense_gemm_11_gb300.autotune --shape tc:128x11008x4096 --shape f32:512x512x512

Timing: for each candidate (and the planner's own choice) R back-to-back
calls over several copies of the inputs (enough to exceed the L2 cache when
memory allows) are captured in a CUDA graph on a stream of its own (so each
graph keeps its own split-K scratch).  Every graph is replayed once to drop
the clear losers, then the planner's graph and the finalists are replayed in
interleaved rounds and each keeps the median: GPU clock and temperature drift
over a tuning run by several percent, and interleaving puts that drift on
every candidate alike.  An entry is written only when the best candidate is a
different plan and beats the planner's own choice by more than ``--min-gain`` (default 3 %: two graphs
of the same plan differ by up to ~4 % on a GB300).
"""
from __future__ import annotations

import argparse
import json
import statistics

from . import GEMM_PATH_F32, GEMM_PATH_TC, last_plan, tune_get, tune_set

SPLITS = (1, 2, 3, 4, 6, 8, 12, 16, 24, 32)
L2_BYTES = 129 * 1024 * 1024


def candidates(path: int, M: int, N: int, K: int):
    """Every (variant, bn, splits) the planner accepts for the shape."""
    out = []
    if path == GEMM_PATH_F32:
        kt = max(1, (K + 31) // 32)
        out.append((1, 0, 0))
        out += [(2, 0, s) for s in SPLITS if s <= max(1, kt // 2)]
        return out
    kb = max(1, (K + 63) // 64)
    out += [(1, bn, 0) for bn in (256, 224, 192)]
    out += [(2, bn, s) for bn in (256, 128) for s in SPLITS if s <= max(1, kb // 2)]
    if M <= 64:
        out += [(3, bn, s) for bn in (32, 64) if M <= bn for s in SPLITS if s <= max(1, kb // 2)]
    # cluster split-K (2..8 CTAs per tile); the library ignores an entry whose
    # CTAs do not all fit on the GPU, so only shapes with few tiles qualify
    tiles_m = (M + 127) // 128
    for bn in (256, 192, 128):
        t = tiles_m * ((N + bn - 1) // bn)
        out += [(4, bn, s) for s in range(2, 9) if s <= kb // 2 and t * s <= sm_count()]
    return out


def sm_count() -> int:
    try:
        import torch
        if torch.cuda.is_available():
            return torch.cuda.get_device_properties(0).multi_processor_count
    except Exception:
        pass
    return 152


class _Timed:
    """A CUDA graph of `reps` calls of one plan, captured on its own stream."""

    def __init__(self, call, nsets: int, reps: int = 12):
        import torch
        self.reps = reps
        self.stream = torch.cuda.Stream()
        with torch.cuda.stream(self.stream):
            for i in range(nsets):
                call(i, self.stream)  # scratch is allocated outside the capture
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            for i in range(reps):
                call(i % nsets, self.stream)
        self.times = []

    def replay(self) -> float:
        import torch
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            e0.record(self.stream)
            self.graph.replay()
            e1.record(self.stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / self.reps
        self.times.append(ms)
        return ms

    @property
    def ms(self) -> float:
        return statistics.median(self.times)


def tune_shape(path: int, M: int, N: int, K: int, *, min_gain: float = 0.03, rounds: int = 7, finalists: int = 4,
               verbose: bool = True):
    """Time the planner's choice and every candidate; returns (entry or None, report)."""
    import torch

    from . import gemm_f16_f32acc_epilogue, gemm_f32
    dev = torch.device("cuda")
    if path == GEMM_PATH_F32:
        set_bytes = 4 * (M * K + K * N + M * N)
    else:
        set_bytes = 2 * (M * K + K * N) + 4 * M * N
    free, _ = torch.cuda.mem_get_info()
    nsets = max(1, min(4, -(-3 * L2_BYTES // set_bytes), int(0.5 * free // max(1, set_bytes))))
    sets = []
    for _ in range(nsets):
        if path == GEMM_PATH_F32:
            sets.append((torch.rand(M, K, device=dev) - 0.5, torch.rand(K, N, device=dev) - 0.5,
                         torch.empty(M, N, device=dev)))
        else:
            sets.append((torch.randn(M, K, device=dev).div_(K ** 0.5).half(),
                         torch.randn(K, N, device=dev).div_(K ** 0.5).half(), torch.empty(M, N, device=dev)))

    def call(i, stream):
        a, b, c = sets[i]
        if path == GEMM_PATH_F32:
            gemm_f32(a, b, c, stream=stream)
        else:
            gemm_f16_f32acc_epilogue(a, b, c, stream=stream)

    saved = tune_get()
    report = {"path": path, "M": M, "N": N, "K": K, "candidates": []}
    try:
        # capture: the plan is chosen when the call is enqueued, so each graph
        # keeps the plan of the table installed at capture time
        tune_set([])
        planner = _Timed(call, nsets)
        call(0, torch.cuda.current_stream())
        planner_plan = last_plan()
        cands = []
        for variant, bn, splits in candidates(path, M, N, K):
            entry = dict(path=path, M=M, N=N, K=K, variant=variant, bn=bn, splits=splits)
            tune_set([entry])
            timed = _Timed(call, nsets)
            call(0, torch.cuda.current_stream())
            cands.append((entry, last_plan(), timed))
    finally:
        tune_set(saved)
    planner.replay()
    for _, _, t in cands:
        t.replay()
    cands.sort(key=lambda c: c[2].ms)
    final = cands[:finalists]
    for r in range(rounds):
        order = [planner] + [t for _, _, t in final]
        for t in (order if r % 2 == 0 else order[::-1]):
            t.replay()
    torch.cuda.synchronize()
    report["planner"] = {"plan": planner_plan, "ms": planner.ms}
    for entry, plan, t in cands:
        report["candidates"].append({**entry, "plan": plan, "ms": t.ms, "replays": len(t.times)})
    best_entry, best_plan, best_t = min(final, key=lambda c: c[2].ms)
    gain = planner.ms / best_t.ms - 1.0
    report["best"] = {**best_entry, "plan": best_plan, "ms": best_t.ms, "gain": gain}
    if verbose:
        print(f"path {path} {M}x{N}x{K}: planner {planner_plan} {planner.ms * 1e3:.1f} us, "
              f"best {best_plan} {best_t.ms * 1e3:.1f} us ({gain * 100:+.1f} %)", flush=True)
    # the planner's own plan under a table entry only measures graph-to-graph
    # drift (a negative min_gain writes the best candidate whatever it is)
    same_plan = min_gain >= 0 and best_plan.replace("+tuned", "") == planner_plan
    return (best_entry if gain > min_gain and not same_plan else None), report


def _parse_shape(text: str):
    kind, dims = text.split(":")
    M, N, K = (int(x) for x in dims.lower().split("x"))
    return (GEMM_PATH_F32 if kind == "f32" else GEMM_PATH_TC), M, N, K


def main(argv=None):
    import torch

    from . import inputs
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--workloads", default="", help="comma-separated names from inputs.WORKLOADS (single matrices)")
    ap.add_argument("--shape", action="append", default=[], help="f32:MxNxK or tc:MxNxK (repeatable)")
    ap.add_argument("--min-gain", type=float, default=0.03)
    ap.add_argument("--out", default="", help="write the table (JSON) here")
    args = ap.parse_args(argv)
    shapes = []
    for name in [w for w in args.workloads.split(",") if w]:
        w = inputs.WORKLOADS[name]
        if w.batch != 1 or w.b_trans or w.kind == "f32x3" or (w.kind == "f32" and (w.M == 1 or w.N == 1)):
            continue
        shapes.append((GEMM_PATH_F32 if w.kind == "f32" else GEMM_PATH_TC, w.M, w.N, w.K))
    shapes += [_parse_shape(s) for s in args.shape]
    shapes = list(dict.fromkeys(shapes))
    entries, reports = [], []
    for path, M, N, K in shapes:
        entry, report = tune_shape(path, M, N, K, min_gain=args.min_gain)
        reports.append(report)
        if entry is not None:
            entries.append(entry)
    doc = {"device": torch.cuda.get_device_name(), "sm_count": torch.cuda.get_device_properties(0).multi_processor_count,
           "min_gain": args.min_gain, "entries": entries, "reports": reports}
    if args.out:
        with open(args.out, "w") as f:
            json.dump(doc, f, indent=1)
    return doc


if __name__ == "__main__":
    main()
