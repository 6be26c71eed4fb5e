"""bench.py's reference arm (the FP64 oracle on the host) runs without a GPU
and prints one JSON line with the contract's keys."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    return json.loads(lines[0])


def test_reference_arm_json_line():
    d = _run("--impl", "reference", "--config", "tiny", "--steps", "2", "--warmup", "1")
    for k in ("metric", "value", "unit", "impl", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["higher_is_better"] is False and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert "workload" in d["config"]


def test_reference_arm_e4m3_output_and_nvfp4():
    d = _run("--impl", "reference", "--config", "table1_small_nvfp4", "--steps", "1", "--warmup", "0",
             "--out-dtype", "e4m3")
    assert d["value"] > 0 and "output" in d["config"]
