"""The bench's host-side logic on CPU (no GPU): it runs on one GPU only, both
arms describe the workload with the same config, the reference arm prints
its line, and the helpers behave."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


@pytest.mark.parametrize("argv,env", [(["--gpus", "2"], {}),
                                      (["--gpus", "1"], {"WORLD_SIZE": "2", "RANK": "1"}),
                                      (["--gpus", "8", "--impl", "reference"], {})])
def test_more_than_one_gpu_is_an_argument_error(argv, env):
    """The cluster kernels multicast TMA loads within a cluster; that stays a
    one-GPU feature, so the bench refuses any multi-GPU launch before it
    touches a GPU."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *argv],
                       env=dict(os.environ, **env), capture_output=True, text=True, timeout=120)
    assert r.returncode == 2 and r.stdout.strip() == ""
    assert "one GPU only" in r.stderr


def test_job_value():
    assert bench.job_value(2e12, 1.0) == pytest.approx(2000.0)


def test_default_workload_is_the_eleven_shapes():
    shapes = bench.WORKLOADS["all"]
    assert len(shapes) == len(set(shapes)) == 11
    assert (8192, 8192, 8192) in shapes and (16384, 16384, 16384) in shapes
    assert (2048, 2048, 16384) in shapes and (1024, 1024, 65536) in shapes
    reps = {s: bench.calls_per_step(*s) for s in shapes}
    # Small shapes are called most often, the largest least (the pages' 400 /
    # 200 / 40 / 12 calls, scaled).
    assert reps[(1024, 1024, 1024)] == 60 and reps[(4096, 4096, 4096)] == 30
    assert reps[(8192, 8192, 8192)] == 6 and reps[(16384, 16384, 16384)] == 2


def test_both_arms_share_the_config():
    class A:
        workload, types, values, epilogue = "all", "f16f32", "uniform", "plain"
    cfg = bench.workload_config(A, bench.WORKLOADS["all"])
    assert cfg["parallelism"] == "single GPU" and cfg["workload"].startswith("all: 1024x1024x1024")


def test_reference_arm_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3", "--workload", "c1"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0

    class A:
        workload, types, values, epilogue = "c1", "f16f32", "uniform", "plain"
    assert line["config"] == bench.workload_config(A, bench.WORKLOADS["c1"])


def test_kernel_digest_ignores_comments_and_whitespace():
    code = 'int f(int x) {\n  return x + 1;  // one more\n}\nconst char* s = "a // b";\n'
    same = '/* header */ int f(int x)\n{ return x+1; }\n  const char* s = "a // b";'
    other = 'int f(int x) { return x + 2; }\nconst char* s = "a // b";'
    assert bench._code_only(code) == bench._code_only(same)
    assert bench._code_only(code) != bench._code_only(other)
    assert '"a // b"' in bench._code_only(code)  # string literals are kept whole
    assert len(bench.kernel_source_digest()) == 16


def test_peaks_and_pipe_ceiling():
    """The roofline's tensor peak is the measured burst figure (each call is
    timed alone); the sustained figure and the tcgen05 pipe ceiling are
    reported beside it."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    t, ts, hbm, src = bench.peaks()
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        assert (t, ts, hbm) == (d["bf16_tflops"], d["bf16_tflops_sustained"], d["hbm_gbs"])
        assert "burst" in src
    ceiling, what = bench.pipe_ceiling()
    assert ceiling == pytest.approx(2333.6) and "N224" in what


def test_traffic_table_matches_the_kernel_sources():
    """The bench reports the dominant kernel's DRAM bytes per launch from the
    committed one-launch captures only when they were taken on the current
    kernel sources. The table holds a row for every one of the eleven shapes
    with the default configuration, on these sources."""
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rows = json.load(f)
    digest = bench.kernel_source_digest()
    shapes = {bench.shape_name(s) for s in bench.WORKLOADS["all"]}
    assert {r["shape"] for r in rows if r["kernel_src"] == digest} == shapes
    dominant = [r for r in rows if r["shape"] == "16384x16384x16384"][0]
    assert bench.committed_traffic(dominant["config"], (16384, 16384, 16384)) == \
        dominant["dram_bytes"] > 0


@pytest.mark.parametrize("argv", [["--energy", "--warm"], ["--configs", "x"],
                                  ["--cupti"]])
def test_compare_argument_errors(argv):
    """compare.py refuses inconsistent options before it touches a GPU."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "compare.py"), *argv],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 2 and "error" in r.stderr


@pytest.mark.parametrize("argv", [["--rounds", "0"], ["--steps", "0"],
                                  ["--workload", "nosuch"]])
def test_e2e_variants_argument_errors(argv):
    """e2e_variants.py refuses bad options before it touches a GPU."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "e2e_variants.py"), *argv],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 2 and "error" in r.stderr
