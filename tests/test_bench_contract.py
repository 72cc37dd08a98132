"""The benchmark's JSON line as the harness reads it, on CPU: the reference
arm (the CPU oracle on a bounded row sample) prints one line with every key
of the contract, and under torchrun only rank 0 prints."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args, env=None):
    e = dict(os.environ)
    e.update(env or {})
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       timeout=600, env=e, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    return [json.loads(line) for line in r.stdout.splitlines() if line.startswith("{")]


@pytest.fixture(scope="module")
def reference_line():
    lines = run_bench("--impl", "reference", "--steps", "2", "--warmup", "0", "--ref-budget-s", "4")
    assert len(lines) == 1
    return lines[0]


def test_reference_line_has_the_contract_keys(reference_line):
    r = reference_line
    assert r["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in r, key
    assert r["value"] > 0 and r["ms_per_step"] > 0
    assert r["unit"] == "TFLOPS" and r["higher_is_better"] is True and r["n_gpus"] == 1
    assert r["warmup"] >= 3  # the timing rules' minimum, applied even when asked for fewer
    assert r["vs_baseline"] is None and r["data"] == "synthetic" and r["scaling"] == "weak"
    assert "workload" in r["config"]
    assert r["steps"] == 2 and r["ms_per_step_min"] <= r["ms_per_step_median"]


def test_both_arms_print_the_same_config():
    sys.path.insert(0, ROOT)
    import bench
    cfg = bench.bench_config(1)
    assert cfg == json.loads(json.dumps(cfg))  # plain JSON, no plan names or other per-arm keys
    assert set(cfg) == {"workload", "M", "N", "K", "l2", "parallelism"}


def test_reference_line_describes_its_cpu_baseline(reference_line):
    cb = reference_line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["unit"] == "TFLOPS"
    assert cb["value"] == reference_line["value"] and isinstance(cb["sample"], str) and cb["sample"]
    e2e = reference_line["e2e"]
    assert e2e == {"value": reference_line["value"], "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}


def test_reference_arm_prints_on_rank_zero_only():
    assert run_bench("--impl", "reference", "--steps", "1", "--ref-budget-s", "2",
                     env={"RANK": "1", "WORLD_SIZE": "2"}) == []


@pytest.mark.gpu
def test_our_line_has_roofline_e2e_launches_and_clocks():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    lines = run_bench("--steps", "3", "--warmup", "3", "--no-cpu-baseline")
    assert len(lines) == 1
    r = lines[0]
    assert r["value"] > 0 and r["n_gpus"] == 1 and r["steps"] == 3
    rf = r["roofline"]
    assert rf["bound"] in ("alu", "tensor", "hbm") and rf["unit"] in ("TFLOP/s", "GB/s")
    assert rf["peak"] > 0 and abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    assert rf["traffic"] is None or rf["traffic"] > 0
    e2e = r["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert r["gpu_launches"] >= 2 * r["steps"]  # at least one launch per GEMM of every timed step
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(r["clocks"])


def test_nominal_tensor_peak_arithmetic():
    sys.path.insert(0, ROOT)
    import bench
    r = bench._nominal_tensor_peak(8192.0, 152, 2070.0, 1500.0)
    assert abs(r["nominal_peak"] - 8192 * 152 * 2070e6 / 1e12) < 1e-9
    assert abs(r["frac_of_nominal"] - 1500.0 / r["nominal_peak"]) < 1e-12
    assert "152 SMs" in r["nominal_source"]
    assert bench._nominal_tensor_peak(None, 152, 2070.0, 1500.0) == {"nominal_peak": None}


def test_profile_summaries_name_commands_the_bench_accepts():
    # every ncu summary gives the command that made it; its bench.py flags and
    # profile cases must still exist, so the capture can be repeated
    import re
    sys.path.insert(0, ROOT)
    from dense_gemm_11_gb300 import inputs
    src = open(os.path.join(ROOT, "bench.py")).read()
    flags = set(re.findall(r'add_argument\("(--[\w-]+)"', src))
    cases = set(inputs.WORKLOADS) | {"sgemm", "hgemm", "tf32x3"}
    pdir = os.path.join(ROOT, "profiles")
    for f in sorted(os.listdir(pdir)):
        if not f.endswith(".md"):
            continue
        text = open(os.path.join(pdir, f), encoding="utf-8").read()
        cmds = re.findall(r"python bench\.py([^\n>&|]*)", text)
        assert cmds, f"{f} names no bench.py command"
        for c in cmds:
            for flag in re.findall(r"(--[\w-]+)", c):
                assert flag in flags, (f, flag)
            for case in re.findall(r"--profile-case\s+(\S+)", c):
                assert case in cases, (f, case)


def test_fma_ceiling_arithmetic():
    sys.path.insert(0, ROOT)
    import bench
    r = bench._fma_ceiling({"packed_ffma2": 96.0, "scalar_ffma": 120.0}, 61.9, 152, 2070.0)["fma_rate_probe"]
    per_clk = 61.9e12 / 2 / (152 * 2070e6)
    assert abs(r["sgemm_fma_per_clock_per_sm"] - round(per_clk, 2)) < 1e-9
    assert abs(r["sgemm_frac_of_packed_rate"] - per_clk / 96.0) < 1e-12
    assert bench._fma_ceiling(None, 61.9, 152, 2070.0) == {"fma_rate_probe": None}


def test_clock_sampler_summarises_the_timed_window(tmp_path):
    sys.path.insert(0, ROOT)
    import bench
    cs = bench.ClockSampler(0)
    cs.out = str(tmp_path / "clk.csv")
    cs.proc = object()  # a sampler that ran
    lines = ["2026/12/02 10:00:00.000, 0, 1500, 2070, 300.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "2026/12/02 10:00:01.000, 0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Active",
             "2026/12/02 10:00:01.020, 0, 2060, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "2026/12/02 10:00:05.000, 0, 1200, 2070, 100.0, 0x0, Active, Not Active, Not Active, Not Active"]
    open(cs.out, "w").write("\n".join(lines) + "\n")
    t0 = cs._stamp("2026/12/02 10:00:00.900")
    t1 = cs._stamp("2026/12/02 10:00:01.100")
    cs.window(t0, t1)
    r = cs.summary()
    assert r["samples"] == 2 and r["samples_scope"] == "timed region"
    assert r["sm_mhz"] == 2065.0 and r["reasons"] == ["sw_power_cap"] and r["power_w_max"] == 950.0
    cs.window(t1 + 10, t1 + 11)  # nothing inside: every sample is used
    assert cs.summary()["samples_scope"] == "whole run" and cs.summary()["samples"] == 4
