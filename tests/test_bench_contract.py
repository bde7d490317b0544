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
