"""The JSON line bench.py prints: every key of the contract, with values that
agree with each other (the roofline's achieved bytes over the launch time, its
fraction of the peak, the whole-job value over the step time). The reference
arm (the f64 oracle on the host cores) runs here on the CPU; our arm needs the
GPU."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BASE_KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
             "scaling", "vs_baseline", "dtype", "data", "config", "e2e", "cpu_baseline"}


def run_bench(*args, timeout=600):
    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        env.pop(k, None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-3000:]
    return json.loads(lines[0])


def check_common(d, steps, warmup):
    assert BASE_KEYS <= set(d), BASE_KEYS - set(d)
    assert d["unit"] == "GB/s" and d["n_gpus"] == 1 and d["scaling"] == "weak"
    assert d["steps"] == steps and d["warmup"] == warmup
    assert d["higher_is_better"] is True and d["data"] == "synthetic"
    assert d["vs_baseline"] is None  # the pages publish no number for this metric and workload
    assert d["config"]["workload"] == "ce_8192x128256"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    e = d["e2e"]
    assert {"value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"} <= set(e)
    assert e["unit"] == d["unit"] and e["value"] > 0
    c = d["cpu_baseline"]
    assert {"value", "unit", "cores", "kind", "sample"} <= set(c) and c["kind"] == "oracle" and c["cores"] >= 1


def test_reference_arm_line():
    d = run_bench("--impl", "reference", "--steps", "2", "--warmup", "1")
    check_common(d, 2, 1)
    assert d["impl"] == "reference" and d["dtype"] == "f64"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["e2e"]["value"] == d["value"] == d["cpu_baseline"]["value"]


@pytest.mark.gpu
def test_our_arm_line():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = run_bench("--steps", "5", "--warmup", "3", "--cpu-rows", "256")
    check_common(d, 5, 3)
    assert "impl" not in d or d["impl"] != "reference"
    assert d["dtype"] == "f32"
    R, V = d["config"]["rows"], d["config"]["vocab"]
    # whole-job GB/s: the step's algorithmic bytes (gradient written, logits read once, labels,
    # loss rows and tokens) over the step time
    assert d["value"] == pytest.approx((8 * R * V + 16 * R) / (d["ms_per_step"] * 1e-3) / 1e9, rel=2e-3)
    r = d["roofline"]
    assert {"bound", "achieved", "peak", "unit", "frac", "traffic"} <= set(r)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["algorithmic_bytes"] == 8 * R * V + 16 * R
    assert r["achieved"] == pytest.approx(r["algorithmic_bytes"] / (r["ms_per_launch"] * 1e-3) / 1e9, rel=2e-3)
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=2e-3)
    assert 0.5 < r["frac"] < 1.2, "a fraction far above 1 would mean the timed kernel skips work"
    assert r["ms_per_launch"] <= d["ms_per_step"] * 1.05  # the kernel alone is not slower than the step
    assert r["traffic"] is None or 0.9 < r["traffic"] / r["algorithmic_bytes"] < 1.1
    e = d["e2e"]
    assert e["h2d_bytes_per_step"] >= 8 * R * V // 2 and e["d2h_bytes_per_step"] >= 8 + 4 * R
    assert e["ms_per_step"] >= d["ms_per_step"]
    assert d["gpu_launches"] == 2 * d["steps"]
    a = d["argmax"]
    assert a["rows_per_s"] == pytest.approx(256 / (a["ms"] * 1e-3), rel=2e-3)
    assert a["plain_read"]["argmax_over_read"] == pytest.approx(a["ms"] / a["plain_read"]["ms"], rel=2e-3)
    k = d["clocks"]
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(k)
