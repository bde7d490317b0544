"""The benchmark's JSON contract on a machine without a GPU: the reference
arm (the fp64 oracle on the host cores) prints one line with the keys the
contract asks for, and the source digest that keys the recorded DRAM capture
ignores comments but not code."""

import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "1",
                          "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "impl"):
        assert key in d, key
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "tokens/s"
    assert d["value"] > 0 and d["config"]["workload"] == "tiny" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["uname_m"] and d["cpu_baseline"]["cpu_model"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_source_digest_ignores_comments_only(tmp_path, monkeypatch):
    csrc = tmp_path / "lm_head_loss_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("// a comment\n__global__ void k() { int a = 1; }  /* note */\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    base = bench.kernel_sources_sha256()
    (csrc / "k.cu").write_text("// another comment\n\n__global__  void k() {\n  int a = 1;\n}\n")
    assert bench.kernel_sources_sha256() == base
    (csrc / "k.cu").write_text("__global__ void k() { int a = 2; }\n")
    assert bench.kernel_sources_sha256() != base


def test_phase_fractions_split_the_gemm_time():
    # 2NVD over the forward GEMM, 6NVD over the recompute and grouped launches,
    # each as a fraction of the given peak; with the filter on, the backward
    # counts the lower bound of the FLOPs it executed.
    n, d, v, steps = 8192, 2048, 151552, 10
    per_kind = {"gemm_lse": {"ms": 26.0, "launches": 10}, "gemm_dz": {"ms": 1.6, "launches": 10},
                "gemm_bwd": {"ms": 86.0, "launches": 180}, "combine": {"ms": 0.2, "launches": 10}}
    out = bench.phase_fractions(per_kind, steps, n, d, v, peak=2000.0, skipped=None)
    fwd_tf = 2.0 * n * v * d / 2.6e-3 / 1e12
    bwd_tf = 6.0 * n * v * d / 8.76e-3 / 1e12
    assert abs(out["forward"]["tflops"] - fwd_tf) < 1e-6 * fwd_tf
    assert abs(out["backward"]["tflops"] - bwd_tf) < 1e-6 * bwd_tf
    assert abs(out["forward"]["frac"] - fwd_tf / 2000.0) < 1e-9
    half = bench.phase_fractions(per_kind, steps, n, d, v, peak=2000.0, skipped=0.5)
    assert abs(half["backward"]["tflops"] - bwd_tf * 4.0 / 6.0) < 1e-6 * bwd_tf
    assert bench.phase_fractions({}, steps, n, d, v, 2000.0, None)["forward"]["frac"] is None


def test_host_cpu_names_architecture_and_model():
    info = bench.host_cpu()
    assert info["uname_m"] and isinstance(info["cpu_model"], str) and info["cpu_model"]


def test_clock_summary_keeps_the_timed_region_and_decodes_reasons(tmp_path):
    # Rows as nvidia-smi prints them for ClockSampler.FIELDS: idle samples before
    # and after the timed region, three loaded ones inside it.
    rows = [
        "2026/12/03 09:00:00.000, 0, 1980, 2070, 180.10, 0x0000000000000001, Not Active, Not Active, Not Active, Not Active",
        "2026/12/03 09:00:01.050, 0, 1530, 2070, 950.20, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "2026/12/03 09:00:01.100, 0, 1545, 2070, 960.00, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "2026/12/03 09:00:01.150, 0, 1500, 2070, 955.00, 0x0000000000000006, Not Active, Not Active, Not Active, Active",
        "2026/12/03 09:00:03.000, 0, 2070, 2070, 200.00, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
    ]
    path = tmp_path / "clocks.csv"
    path.write_text("\n".join(rows) + "\n")
    c = bench.ClockSampler(0)
    c.proc, c.path = object(), str(path)
    c.t0 = bench.ClockSampler._stamp("2026/12/03 09:00:01.000")
    c.t1 = bench.ClockSampler._stamp("2026/12/03 09:00:01.200")
    s = c.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 1530.0 and s["sm_mhz_min"] == 1500.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"] and s["other_active"] == ["applications_clocks_setting"]
    assert s["selection"].startswith("timestamps")

    # A region shorter than the sampling period keeps the first sample after it started.
    path.write_text("\n".join(rows) + "\n")
    c.path = str(path)
    c.t0 = bench.ClockSampler._stamp("2026/12/03 09:00:01.010")
    c.t1 = bench.ClockSampler._stamp("2026/12/03 09:00:01.020")
    s = c.summary()
    assert s["samples"] == 1 and s["sm_mhz"] == 1530.0 and s["reasons"] == ["sw_power_cap"]

    # A thermal reason set only in the bitmask is still reported.
    path.write_text(rows[1].replace("0x0000000000000004", "0x0000000000000044") + "\n")
    c.path = str(path)
    c.t0, c.t1 = bench.ClockSampler._stamp("2026/12/03 09:00:01.000"), bench.ClockSampler._stamp("2026/12/03 09:00:02")
    assert bench.ClockSampler(0).summary()["reasons"] == ["nvidia-smi unavailable"]
    assert c.summary()["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
