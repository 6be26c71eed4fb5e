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
    assert d["cpu_baseline"]["cpu_model"] and d["cpu_baseline"]["median"] > 0
    assert "workload" in d["config"]
    # the oracle runs on the host: its line claims no GPU-side timing conditions, and keeps the given warm-up
    assert "l2" not in d["config"] and "parallelism" not in d["config"] and "host" in d["config"]
    assert d["warmup"] == 1 and d["steps"] == 2


def test_reference_arm_e4m3_output_and_nvfp4():
    d = _run("--impl", "reference", "--config", "table1_small_nvfp4", "--steps", "1", "--warmup", "0",
             "--out-dtype", "e4m3")
    assert d["value"] > 0 and "output" in d["config"]


def test_forward_source_hash_ignores_comments_only(tmp_path, monkeypatch):
    """The ncu traffic records stay valid across comment edits of the forward
    sources and lapse on any code change."""
    import shutil
    import importlib.util

    csrc = os.path.join(ROOT, "depth_weighted_scatter_gb300", "csrc")
    fake_root = tmp_path
    dst = fake_root / "depth_weighted_scatter_gb300" / "csrc"
    dst.mkdir(parents=True)
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    for f in bench.FORWARD_SOURCES:
        shutil.copy(os.path.join(csrc, f), dst / f)
    monkeypatch.setattr(bench, "ROOT", str(fake_root))
    h0 = bench.forward_source_hash()
    impl = dst / "forward_impl.cuh"
    text = impl.read_text()
    impl.write_text(text.replace("// forward_impl.cuh --", "// forward_impl.cuh (edited comment) --", 1)
                    + "\n/* a block comment */\n")
    assert bench.forward_source_hash() == h0
    impl.write_text(text.replace("constexpr int kFillCellsMin = 256;", "constexpr int kFillCellsMin = 512;", 1))
    assert bench.forward_source_hash() != h0


def test_bytes_model_matches_the_stated_formula():
    """Footprint and gather bytes of the canonical workload: 12 B per point of ranks, 8 B per interval,
    the depth and feature tensors, the output (footprint); the per-point depth and row reads (gather)."""
    import importlib.util

    spec = importlib.util.spec_from_file_location("bench_under_test2", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    from depth_weighted_scatter_gb300 import workloads

    wl = workloads.make("canonical")
    import oracle

    m = oracle.build_map(wl.cell_ids, *wl.dims(), wl.n_cells)
    bm = bench.bytes_model(wl, m["n_points"], m["n_intervals"])
    assert bm["footprint"] == 30_394_964
    assert bm["gather"] == 57_574_622
