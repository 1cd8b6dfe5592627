"""The measurement tools beside the bench run on the GPU and report sane
figures: the bench line itself, the cuBLAS comparison (the two arms agree on
the contraction) and the copy-engine measurement."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_compare_with_cublas_on_1024():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "compare.py"),
                        "--workload", "c1", "--rounds", "2"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    shape, summary = lines[0], lines[-1]["summary"]
    assert shape["shape"] == "1024x1024x1024"
    assert shape["ours_us"] > 0 and shape["cublas_us"] > 0
    # Both arms accumulate in fp32 over K = 1024: far inside the parity bound.
    assert shape["max_rel_diff_vs_abs_product"] < 1e-5
    assert summary["shapes"] == 1 and summary["geomean_speedup"] > 0


def test_compare_energy_per_call():
    """Back-to-back blocks with the NVML energy counter: the library, cuBLAS
    and one forced configuration each report positive joules and time per
    call at 2048³."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "compare.py"), "--shape",
                        "2048x2048x2048", "--energy", "--rounds", "1",
                        "--configs", "g1_128x256_s4_a2_direct"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    rows, summary = lines[:-1], lines[-1]["summary"]
    assert [x["arm"] for x in rows] == ["library", "cublas", "g1_128x256_s4_a2_direct"]
    for x in rows:
        assert x["us_per_call"] > 0 and x["joules_per_call"] > 0 and x["watts"] > 0, x
    assert summary["idle_watts"] > 0


def test_copy_engine_rates():
    from dense_fp16_gemm_02_gb300 import peak
    rows = peak.copy_rates(sizes_mib=(8,), reps=2)
    assert len(rows) == 1
    assert rows[0]["h2d_gbs"] > 1.0 and rows[0]["d2h_gbs"] > 1.0
    assert rows[0]["both_directions_gbs"] > 1.0
    assert rows[0]["h2d_two_streams_gbs"] > 1.0 and rows[0]["d2h_two_streams_gbs"] > 1.0


def test_bench_line_has_every_key():
    """A short bench run prints one JSON line with the keys the driver reads:
    throughput, CUDA-event and CUPTI times per shape, the roofline, the
    clocks, the end-to-end figure and the launch count."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "c1",
                        "--steps", "3", "--warmup", "3", "--calls", "2", "--no-cpu-baseline"],
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks", "shapes"):
        assert key in line, key
    assert line["n_gpus"] == 1 and line["value"] > 0 and line["gpu_launches"] == 3 * 2
    s = line["shapes"][0]
    assert s["shape"] == "1024x1024x1024" and s["calls"] == 6 and s["us_median"] > 0
    kt = s.get("us_kernel_median")  # absent only when CUPTI is unavailable
    assert kt is None or 0 < kt <= s["us_median"] * 2
    assert line["roofline"]["bound"] == "tensor" and 0 < line["roofline"]["frac"] < 1.5
    assert line["e2e"]["h2d_bytes_per_step"] == 2 * (2 * 1024 * 1024)

