"""The bench's multi-rank logic on CPU with gloo, world size 2 (no GPU).

With N GPUs the bench runs one replica per rank, brackets the timed steps
with barriers and reports every rank's work over the slowest rank's time;
the reference arm runs on rank 0 only.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # Rank r took (r + 1) ms for a step and 3 − r ms end to end.
        got = bench.max_over_ranks([1.0 + rank, 3.0 - rank])
        out.put((rank, got, bench.job_value(2e12, world, got[0])))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, value in res:
        assert got == [2.0, 3.0]  # the slowest rank's times, on every rank
        assert value == pytest.approx(2 * 2e12 / 2e-3 / 1e12)  # both ranks' work / slowest time


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    assert bench.job_value(2e12, 1, 1.0) == pytest.approx(2000.0)


def test_reference_arm_only_on_rank0():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3", "--workload", "c1"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_line():
    import json
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3", "--workload", "c1"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


def test_kernel_digest_ignores_comments_and_whitespace():
    import bench
    code = 'int f(int x) {\n  return x + 1;  // one more\n}\nconst char* s = "a // b";\n'
    same = '/* header */ int f(int x)\n{ return x+1; }\n  const char* s = "a // b";'
    other = 'int f(int x) { return x + 2; }\nconst char* s = "a // b";'
    assert bench._code_only(code) == bench._code_only(same)
    assert bench._code_only(code) != bench._code_only(other)
    assert '"a // b"' in bench._code_only(code)  # string literals are kept whole
    assert len(bench.kernel_source_digest()) == 16


def test_peak_follows_the_power_cap():
    """The roofline's tensor peak is the measured burst figure unless the
    timed region ran under the power cap, then the sustained one."""
    sys.path.insert(0, ROOT)
    import json
    import bench
    with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
        d = json.load(f)
    t, hbm, src = bench.peaks()
    assert (t, hbm) == (d["bf16_tflops"], d["hbm_gbs"]) and "burst" in src
    t, hbm, src = bench.peaks(power_capped=True)
    assert (t, hbm) == (d["bf16_tflops_sustained"], d["hbm_gbs"]) and "sustained" in src
