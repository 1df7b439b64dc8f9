"""bench.py's contract without a GPU: the reference arm (the oracle on the host cores)
prints one JSON line with the keys the harness reads, only rank 0 prints under a
multi-rank launch, and the roofline's dominant kernel follows the launch plan."""
import json
import os
import subprocess
import sys

import pytest

import bench
import inputgen

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, env=None):
    e = dict(os.environ)
    e.update(env or {})
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, capture_output=True, text=True,
                       env=e, cwd=ROOT, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    return [json.loads(line) for line in r.stdout.splitlines() if line.startswith("{")]


def test_reference_arm_line():
    lines = _run(["--impl", "reference", "--workload", "dense_small", "--steps", "2", "--warmup", "1"])
    assert len(lines) == 1
    d = lines[0]
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 2
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1 and d["cpu_baseline"]["sample"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["config"]["name"] == "dense_small"


def test_reference_arm_prints_on_rank_zero_only():
    assert _run(["--impl", "reference", "--workload", "dense_small", "--steps", "1", "--warmup", "1"],
                env={"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}) == []


@pytest.mark.parametrize("make,expect", [
    (lambda: inputgen.dense_tall(m=1000, variant="b"), "dense_tile_kernel"),
    (lambda: inputgen.dense_tall(m=1000, variant="b", x_store="bf16"), "dense_tile_kernel"),
    (lambda: inputgen.dense_wide(m=64, n=20_000), "dense_wide_f64_kernel"),
    (lambda: inputgen.dense_multi(m=1000, k=8), "dense_multi_tc_kernel"),
    (lambda: inputgen.dense_multi(m=1000, k=4), "dense_multi_kernel"),
    (lambda: inputgen.csr_uniform(m=20_000), "csr_group_kernel"),
    (lambda: inputgen.csr_powerlaw(m=20_000), "csr_long_kernel"),
])
def test_dominant_kernel_follows_the_plan(make, expect):
    assert bench.dominant_kernel(make()) == expect


def test_model_estimate_is_reported():
    m = bench.model_estimate(inputgen.dense_tall(m=1_000_000, variant="b"))
    assert "kind=tile_tma" in m["plan"] and m["est_us"] > 4.0
    m = bench.model_estimate(inputgen.dense_multi(m=1000, k=8))
    assert m["plan"].startswith("multi ok=1") and m["est_us"] > 0


@pytest.mark.parametrize("content,expect", [
    ('{"hbm_gbs": 7012.5}', (7012.5, "measured")),
    ('{"hbm_gbs": {"value": 7012.5, "unit": "GB/s"}}', (7012.5, "measured")),
    ('{"hbm_copy_gbs": "6950"}', (6950.0, "measured")),
    ('{"hbm_stream_copy_GBps": 7100}', (7100.0, "measured")),
    ('{"bf16_tflops": 1900}', (bench.FALLBACK_HBM_GBS, "fallback")),
    ('{"hbm_gbs": null}', (bench.FALLBACK_HBM_GBS, "fallback")),
    ('not json', (bench.FALLBACK_HBM_GBS, "fallback")),
])
def test_measured_peaks_file(tmp_path, content, expect):
    f = tmp_path / "peaks.json"
    f.write_text(content)
    peak, kind, _ = bench.measured_peaks(str(f))
    assert (peak, kind) == expect


def test_fp64_peak_from_file():
    assert bench.fp64_peak_tflops({}) == bench.FP64_PEAK_TFLOPS
    assert bench.fp64_peak_tflops({"fp64_tflops": {"value": 1.3}}) == 1.3
    assert bench.fp64_peak_tflops({"fp64_tflops": "n/a"}) == bench.FP64_PEAK_TFLOPS
