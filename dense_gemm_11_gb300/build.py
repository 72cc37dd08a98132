"""Build libgemm11.so in-tree with nvcc for sm_103a (no cmake, no torch build).

Two variants of the same sources: the release library (``_build/libgemm11.so``)
and the debug library (``_build_debug/libgemm11_debug.so``, compiled with
GEMM11_DEBUG=1: one operand stage in flight, device-side index checks,
guarded scratch, a synchronising check at the end of every call)."""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libgemm11.so")
DEBUG_BUILD_DIR = os.path.join(HERE, "_build_debug")
DEBUG_LIB_PATH = os.path.join(DEBUG_BUILD_DIR, "libgemm11_debug.so")
SOURCES = ["api.cu", "sgemm.cu", "hgemm.cu", "probe.cu"]
HEADERS = ["internal.h", "ptx.cuh", os.path.join("..", "..", "include", "gemm11.h")]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "--expt-relaxed-constexpr",
    "-Xptxas", "-v",
]


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    deps = [src] + [os.path.join(CSRC, h) for h in HEADERS]
    return any(os.path.getmtime(d) > t for d in deps if os.path.exists(d))


def _variant(debug: bool):
    return (DEBUG_BUILD_DIR, DEBUG_LIB_PATH, ["-DGEMM11_DEBUG=1"]) if debug else (BUILD_DIR, LIB_PATH, [])


def build(force: bool = False, verbose: bool = False, debug: bool = False, both: bool = False) -> str:
    """Compile the release library (or the debug one with debug=True; both at
    once with both=True, translation units compiled in parallel); returns the
    path of the requested library."""
    nvcc = _nvcc()
    variants = [False, True] if both else [debug]
    jobs = []
    objs = {}
    for dbg in variants:
        bdir, _, extra = _variant(dbg)
        os.makedirs(bdir, exist_ok=True)
        objs[dbg] = []
        for s in SOURCES:
            src = os.path.join(CSRC, s)
            obj = os.path.join(bdir, s.replace(".cu", ".o"))
            objs[dbg].append(obj)
            if force or _stale(obj, src):
                jobs.append((src, obj, extra))

    def compile_one(job):
        src, obj, extra = job
        cmd = [nvcc, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with ThreadPoolExecutor(max_workers=max(1, len(jobs))) as ex:
        results = list(ex.map(compile_one, jobs))
    for src, obj, r in results:
        log = os.path.join(os.path.dirname(obj), os.path.basename(src) + ".log")
        with open(log, "w") as f:
            f.write(r.stdout + r.stderr)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError(f"nvcc failed for {src}")
        if verbose:
            sys.stderr.write(r.stderr)
    rebuilt = {os.path.dirname(o) for _, o, _ in jobs}
    for dbg in variants:
        bdir, lib, _ = _variant(dbg)
        if force or bdir in rebuilt or not os.path.exists(lib):
            tmp = lib + f".tmp{os.getpid()}"
            cmd = [nvcc, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-o", tmp, *objs[dbg]]
            subprocess.run(cmd, check=True)
            os.replace(tmp, lib)
    return _variant(debug)[1]


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv, both="--both" in sys.argv))
