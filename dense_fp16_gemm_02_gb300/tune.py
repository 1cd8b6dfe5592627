"""Per-shape configuration sweep: times every compiled configuration and
K-decomposition on this GPU and records the fastest for each shape.

    python -m dense_fp16_gemm_02_gb300.tune --out tune.json [--shapes all]
    python -m dense_fp16_gemm_02_gb300.tune --emit tune.json   # writes csrc/wgemm_tuned.inc
    python -m dense_fp16_gemm_02_gb300.tune --rates rates.json # per-configuration cost model
    python -m dense_fp16_gemm_02_gb300.tune --emit-rates rates.json   # writes csrc/wgemm_rates.inc
    python -m dense_fp16_gemm_02_gb300.tune --validate validate.json  # the rule on off-table shapes

Each candidate call runs alone (L2 flushed with a 256 MiB write before it)
and is timed with CUDA events on the launching stream; the median of the
timed calls is kept. Split-K is tried only when the data-parallel tiles leave
most workers idle, stream-K (with either fix-up) when they fill less than two
waves. The emitted
table is compiled into the library, which consults it before its shape rule.

Calls of half a millisecond or more, back to back, run the GB300 into its power
cap, and then the energy a call takes, not its time alone, sets the clock:
a configuration that reads more from DRAM runs slower once the cap holds,
though it ties in a lone call. For such shapes the finalists are also timed
in blocks of consecutive flushed calls (`--sustained`, on by default), and
that time decides. At the other end, calls under 40 µs whose finalists tie
within a timer tick are ranked by their warm-L2 kernel time from CUPTI.
"""
from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
TUNED_INC = os.path.join(HERE, "csrc", "wgemm_tuned.inc")
RATES_INC = os.path.join(HERE, "csrc", "wgemm_rates.inc")
# Shapes outside the table, for checking the rule against an exhaustive sweep.
OFF_TABLE = [(3000, 5000, 3000), (6144, 6144, 2048), (1000, 8000, 4096), (5000, 700, 12000),
             (2304, 4608, 1536), (12288, 3072, 1024), (777, 1999, 5003), (4096, 1024, 8192)]
# Shapes no constant of the rule was chosen against (checked only).
HELD_OUT = [(2500, 7000, 2500), (6000, 4000, 3000), (1536, 6144, 6144), (10000, 10000, 2000),
            (512, 12288, 4096), (9000, 1500, 5000)]

SHAPES = {
    "all": [(1024, 1024, 1024), (1536, 1536, 1536), (2048, 2048, 2048), (3072, 1280, 2048),
            (4096, 4096, 1024), (4096, 4096, 4096), (8192, 2048, 4096), (8192, 8192, 8192),
            (16384, 16384, 16384), (2048, 2048, 16384), (1024, 1024, 65536)],
    "ksplit": [(2048, 2048, 16384), (1024, 1024, 65536)],
    "large": [(8192, 8192, 8192), (16384, 16384, 16384)],
    "small": [(1024, 1024, 1024), (1536, 1536, 1536), (2048, 2048, 2048), (3072, 1280, 2048)],
}


def candidates(M, N, K, names, workers_pair, workers_single):
    kb = -(-K // 64)
    out = []
    for cid, name in enumerate(names):
        if name.endswith("_h") or "_ab" in name:  # 16-bit C or fused: not a plain fp32 call
            continue
        cg = 2 if name.startswith("g2") else 1
        cols, rows = (int(v) for v in name.split("_")[1].split("x"))
        tiles = -(-M // rows) * -(-N // cols)
        workers = workers_pair if cg == 2 else workers_single
        if re.match(r"g\d[mr]2_", name):  # clusters of two MMA groups: half the workers
            workers //= 2
        out.append((cid, 0, 1))
        if not name.endswith("_tma") or kb < 8 or re.match(r"g\dm2_", name):
            continue
        if tiles < 2 * workers:
            out.append((cid, 2, 1))
        if tiles < 2 * workers:
            out.append((cid, 4, 1))  # stream-K with zeroing first
        if tiles >= workers and tiles % workers:
            # whole waves data parallel, the partial wave (and one more) by stream-K
            out.append((cid, 3, 1))
            if tiles >= 2 * workers:
                out.append((cid, 3, 2))
        if tiles * 2 <= workers:
            for s in sorted({2, 3, 4, 6, 8, 9, 12, 16, workers // max(1, tiles)}):
                if 2 <= s <= kb // 4 and tiles * s <= workers:
                    out.append((cid, 1, s))
    return out


def time_candidate(wgemm, torch, bufs, M, N, K, cid, mode, splits, flush, reps=10, warm=3):
    dA, dB, C = bufs
    stream = torch.cuda.current_stream()
    h = stream.cuda_stream
    times = []
    for r in range(warm + reps):
        flush.fill_(float(r))
        torch.cuda._sleep(400_000)  # GPU busy while the call is enqueued
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        rc = wgemm.wgemm_f16f32_config(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K, K, K,
                                       N, cid, mode, splits, h)
        e1.record(stream)
        if rc != 0:
            return None
        if r >= warm:
            times.append((e0, e1))
    torch.cuda.synchronize()
    if wgemm.wgemm_check(h) != 0:
        raise RuntimeError(f"device error in config {cid} mode {mode}: "
                           f"{wgemm.wgemm_last_device_error()}")
    return statistics.median(e0.elapsed_time(e1) * 1e3 for e0, e1 in times)


TICK_US = 1.1        # the event timer's step seen at small sizes, with margin


def finalists(rows, lo=4, hi=8):
    """The screened candidates re-timed in alternating rounds: every one
    within 3 % plus one timer tick of the best (the screen cannot order
    them), at least `lo` and at most `hi`. rows are sorted by time."""
    best = rows[0]["us"]
    n = sum(1 for r in rows if r["us"] <= best * 1.03 + TICK_US)
    return max(min(n, hi), min(lo, len(rows)))


def final_rounds(us):
    """Rounds for the finalists: enough calls that the tick averages out at
    small sizes (about 20 ms of GEMM time per candidate), 20 to 200."""
    return max(20, min(200, int(20000.0 / max(us, 1.0))))


# Calls at least this long run under the power cap when issued back to back
# (8192³ and up: about 0.6 ms and more at full rate).
SUSTAINED_US = 500.0
SUSTAINED_BLOCK_US = 500_000.0  # GEMM time per block of consecutive calls
SUSTAINED_ROUNDS = 3


def time_block(wgemm, torch, bufs, M, N, K, cid, mode, splits, flush, calls):
    """Median per-call time of `calls` consecutive flushed calls, no gate
    between them (the GPU stays busy, as in a long run of large GEMMs); the
    first third are left out while the clock settles."""
    dA, dB, C = bufs
    stream = torch.cuda.current_stream()
    h = stream.cuda_stream
    evs = []
    for r in range(calls):
        flush.fill_(float(r))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        rc = wgemm.wgemm_f16f32_config(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K, K, K,
                                       N, cid, mode, splits, h)
        e1.record(stream)
        if rc != 0:
            return None
        evs.append((e0, e1))
    torch.cuda.synchronize()
    if wgemm.wgemm_check(h) != 0:
        raise RuntimeError(f"device error in config {cid} mode {mode}: "
                           f"{wgemm.wgemm_last_device_error()}")
    return statistics.median(e0.elapsed_time(e1) * 1e3 for e0, e1 in evs[calls // 3:])


# Calls shorter than this whose finalists tie within a timer tick (flushed
# L2, CUDA events) are told apart by their warm-L2 kernel time from CUPTI,
# the measure of "SASS-Level Kernel Generation for Blackwell" ("How we
# measured"): the event time then carries launch costs the kernels share.
WARM_TIEBREAK_US = 40.0


def time_warm_kernels(wgemm, torch, rec, bufs, M, N, K, finals, ids, rounds=4, calls=20):
    """Median CUPTI kernel time (µs) of each finalist with a warm L2: blocks
    of synchronised calls, the finalists' blocks alternating."""
    dA, dB, C = bufs
    h = torch.cuda.current_stream().cuda_stream
    per = {j: [] for j in range(len(finals))}
    for rnd in range(rounds):
        order = list(range(len(finals)))
        if rnd % 2:
            order.reverse()
        for j in order:
            f = finals[j]
            call = lambda: wgemm.wgemm_f16f32_config(dA.data_ptr(), dB.data_ptr(), C.data_ptr(),
                                                     M, N, K, K, K, N, ids[f["config"]],
                                                     f["mode"], f["splits"], h)
            for _ in range(3):
                if call() != 0:
                    return None
            torch.cuda.synchronize()
            rec.start()
            for _ in range(calls):
                call()
                torch.cuda.synchronize()
            rec.stop()
            per[j] += [(e - s0) / 1e3 for n, s0, e, _ in rec.records() if "wgemm_kernel" in n]
    if wgemm.wgemm_check(h) != 0:
        raise RuntimeError(f"device error: {wgemm.wgemm_last_device_error()}")
    return [statistics.median(per[j]) if per[j] else None for j in range(len(finals))]


def block_calls(us):
    """Calls per sustained block: about SUSTAINED_BLOCK_US of GEMM time."""
    return max(30, int(SUSTAINED_BLOCK_US / max(us, 1.0)))


def _mid_mean(xs):
    """Mean of the middle half of xs (a quarter trimmed from each end)."""
    xs = sorted(xs)
    q = len(xs) // 4
    mid = xs[q:len(xs) - q]
    return sum(mid) / len(mid)


def sweep(shapes, out_path, sustained=True):
    import torch

    sys.path.insert(0, ROOT)
    from dense_fp16_gemm_02_gb300 import build, inputs, wgemm
    build.build()
    names = wgemm.config_names()
    torch.cuda.set_device(0)
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    flush = torch.empty((256 << 20) // 4, dtype=torch.float32, device="cuda")
    from dense_fp16_gemm_02_gb300 import ktime
    try:
        rec = ktime.KernelTimes()
    except ktime.KernelTimesUnavailable as e:  # no tie-break by kernel time
        print(f"# CUPTI unavailable: {e}", file=sys.stderr, flush=True)
        rec = None
    results = []
    for (M, N, K) in shapes:
        A, B = inputs.gemm_operands(M, N, K, seed=1000, kind="uniform")
        bufs = (torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(),
                torch.empty((M, N), dtype=torch.float32, device="cuda"))
        del A, B
        rows, failed = [], []
        for cid, mode, s in candidates(M, N, K, names, sm // 2, sm):
            # Progress on stderr first, so a failing candidate is always named.
            print(f"# {M}x{N}x{K} {names[cid]} mode {mode} splits {s}", file=sys.stderr,
                  flush=True)
            us = time_candidate(wgemm, torch, bufs, M, N, K, cid, mode, s, flush)
            if us is not None:
                rows.append({"config": names[cid], "mode": mode, "splits": s, "us": round(us, 3),
                             "tflops": round(2.0 * M * N * K / us / 1e6, 1)})
            else:  # refused by the library for this shape: recorded, never a winner
                failed.append({"config": names[cid], "mode": mode, "splits": s})
        rows.sort(key=lambda r: r["us"])
        # Finalists: the screen times each candidate's calls back to back, so
        # clock and temperature drift over a long sweep can order near-equal
        # candidates wrongly. The best few are timed again in alternating
        # rounds (one call each per round, the order reversed every round),
        # and the mean of the middle half of the rounds decides (the event
        # timer ticks near 1 µs, so a median ties at small sizes; the launch
        # phase against the tick varies, so an average resolves below it).
        long_calls = sustained and rows[0]["us"] >= SUSTAINED_US
        # Under the power cap the lone-call screen orders the candidates
        # loosely, so long calls keep more finalists.
        nf = finalists(rows, hi=16 if long_calls else 8)
        finals = rows[:nf]
        ids = {n: i for i, n in enumerate(names)}
        per = {i: [] for i in range(len(finals))}
        for rnd in range(final_rounds(rows[0]["us"]) + 1):
            order = list(range(len(finals)))
            if rnd % 2:
                order.reverse()
            for j in order:
                f = finals[j]
                us = time_candidate(wgemm, torch, bufs, M, N, K, ids[f["config"]], f["mode"],
                                    f["splits"], flush, reps=1, warm=0)
                if rnd > 0 and us is not None:
                    per[j].append(us)
        for j, f in enumerate(finals):
            f["us_interleaved"] = round(_mid_mean(per[j]), 3)
        finals.sort(key=lambda r: r["us_interleaved"])
        if long_calls:
            # Blocks of consecutive calls, the finalists' blocks alternating
            # (order reversed every round); the mean of a finalist's block
            # medians decides.
            calls = block_calls(rows[0]["us"])
            blk = {j: [] for j in range(len(finals))}
            for rnd in range(SUSTAINED_ROUNDS):
                order = list(range(len(finals)))
                if rnd % 2:
                    order.reverse()
                for j in order:
                    f = finals[j]
                    us = time_block(wgemm, torch, bufs, M, N, K, ids[f["config"]], f["mode"],
                                    f["splits"], flush, calls)
                    if us is not None:
                        blk[j].append(us)
            for j, f in enumerate(finals):
                if len(blk[j]) == SUSTAINED_ROUNDS:
                    f["us_sustained"] = round(sum(blk[j]) / len(blk[j]), 3)
                    f["sustained_blocks_us"] = [round(v, 1) for v in blk[j]]
            finals.sort(key=lambda r: r.get("us_sustained", float("inf")))
        elif finals[0]["us_interleaved"] < WARM_TIEBREAK_US:
            tied = [f for f in finals
                    if f["us_interleaved"] <= finals[0]["us_interleaved"] + TICK_US]
            if len(tied) > 1 and rec is not None:
                warm = time_warm_kernels(wgemm, torch, rec, bufs, M, N, K, tied, ids)
                for f, w in zip(tied, warm or []):
                    if w is not None:
                        f["us_warm_kernel"] = round(w, 3)
                finals.sort(key=lambda r: (0, r["us_warm_kernel"]) if "us_warm_kernel" in r
                            else (1, r["us_interleaved"]))
        rows = finals + rows[nf:]
        results.append({"shape": [M, N, K], "best": rows[0], "candidates": rows,
                        "failed": failed})
        print(json.dumps({"shape": [M, N, K], "best": rows[0], "next": rows[1:4]}), flush=True)
        del bufs
        torch.cuda.empty_cache()
    with open(out_path, "w") as f:
        json.dump({"gpu": torch.cuda.get_device_name(0), "sm_count": sm, "results": results}, f,
                  indent=1)


def _score(c):
    """A candidate's time in one sweep: its sustained time where the sweep
    took one, else its warm-L2 kernel time where ties were broken by it,
    else its interleaved time if it was a finalist, else its screen median."""
    return c.get("us_sustained", c.get("us_warm_kernel", c.get("us_interleaved", c["us"])))


def _sustained(result):
    return any("us_sustained" in c for c in result["candidates"])


def combine(sweeps, known=None):
    """Per shape, the candidate (configuration, mode, splits) with the lowest
    mean time relative to each sweep's best, over the sweeps that timed it.
    Sweeps on different boxes rank near-equal cluster configurations
    differently (each chip groups its SMs differently), so one box's winner
    is not taken on its own; relative times remove the boxes' overall speed.
    Where some sweeps timed a shape's finalists sustained (back to back,
    under the power cap) and others did not, only the sustained ones count
    for that shape: the two regimes rank configurations differently, and
    the sustained one is how long runs of such calls behave. Candidates
    without a sustained time in such a sweep are left out too. Likewise,
    where sweeps broke a short shape's tie by warm-L2 kernel time, only the
    tied finalists count, by that time.
    `known`: the configurations compiled now; candidates of others (removed
    since a sweep) are dropped. Sweeps that tried fewer candidates of a
    shape than the widest sweep of it (made before configurations were
    added) do not count for that shape, so new configurations can win; a
    candidate a sweep tried and the library refused is listed under
    "failed" and still counts as tried.
    Returns {shape: (candidate dict with "us" = mean time, relative score)}."""
    sustained_shapes = {tuple(r["shape"]) for d in sweeps for r in d["results"]
                        if _sustained(r)}
    warm_shapes = {tuple(r["shape"]) for d in sweeps for r in d["results"]
                   if any("us_warm_kernel" in c for c in r["candidates"])}

    def usable(r):
        cands = r["candidates"]
        if known is not None:
            cands = [c for c in cands if c["config"] in known]
        if tuple(r["shape"]) in sustained_shapes:
            cands = [c for c in cands if "us_sustained" in c]
        elif tuple(r["shape"]) in warm_shapes:  # the tied finalists, by kernel time
            cands = [c for c in cands if "us_warm_kernel" in c]
        return cands

    def tried(r):
        keys = {(c["config"], c["mode"], c["splits"]) for c in r["candidates"] + r.get("failed", [])}
        return {k for k in keys if known is None or k[0] in known}

    widest = {}
    for d in sweeps:
        for r in d["results"]:
            shape = tuple(r["shape"])
            widest[shape] = max(widest.get(shape, 0), len(tried(r)))
    per_shape = {}
    for d in sweeps:
        for r in d["results"]:
            shape = tuple(r["shape"])
            cands = usable(r)
            if not cands or len(tried(r)) < widest[shape]:
                continue
            best = min(_score(c) for c in cands)
            acc = per_shape.setdefault(shape, {})
            for c in cands:
                key = (c["config"], c["mode"], c["splits"])
                rel, us = acc.get(key, ([], []))
                rel.append(_score(c) / best)
                us.append(_score(c))
                acc[key] = (rel, us)
    out = {}
    for shape, acc in per_shape.items():
        n = max(len(v[0]) for v in acc.values())
        # Candidates timed in every sweep only (a candidate that failed on a
        # box, or was not compiled there, does not win by absence).
        full = {k: v for k, v in acc.items() if len(v[0]) == n}
        key, (rel, us) = min(full.items(), key=lambda kv: sum(kv[1][0]) / len(kv[1][0]))
        out[shape] = ({"config": key[0], "mode": key[1], "splits": key[2],
                       "us": sum(us) / len(us)}, sum(rel) / len(rel))
    return out


def emit(json_paths, inc_path=TUNED_INC, known=None):
    """Writes the measured winners as a C table the library compiles in, from
    one sweep or several (see combine)."""
    if isinstance(json_paths, str):
        json_paths = [json_paths]
    sweeps = []
    for path in json_paths:
        with open(path) as f:
            sweeps.append(json.load(f))
    d = sweeps[0]
    boxes = f"{len(sweeps)} sweep" + ("s" if len(sweeps) > 1 else "")
    lines = [
        "// Measured per-shape winners (generated by dense_fp16_gemm_02_gb300/tune.py from",
        f"// {boxes} on {d.get('gpu', 'a GB300')} with {d.get('sm_count')} SMs; do not edit by hand).",
        "// {M, N, K, configuration name, mode (0 data parallel, 1 split-K, 2 stream-K,",
        "//  3 data-parallel waves + stream-K tail, 4 stream-K with zeroing first),",
        "//  splits, measured µs per call (mean over the sweeps; back to back where the",
        "//  sweeps timed the shape so; warm-L2 kernel time where it broke a tie)}",
    ]
    chosen = combine(sweeps, known)
    # Every shape any sweep timed, in the order the sweeps list them.
    shapes = []
    for sw in sweeps:
        for r in sw["results"]:
            if tuple(r["shape"]) not in shapes:
                shapes.append(tuple(r["shape"]))
    for (M, N, K) in shapes:
        b, _ = chosen[(M, N, K)]
        lines.append(f'{{{M}, {N}, {K}, "{b["config"]}", {b["mode"]}, {b["splits"]}, '
                     f'{b["us"]:.3f}}},')
    with open(inc_path, "w") as f:
        f.write("\n".join(lines) + "\n")
    return inc_path


def _time_calls(wgemm, torch, bufs, M, N, K, fn, flush, reps=7, warm=2):
    stream = torch.cuda.current_stream()
    times = []
    for r in range(warm + reps):
        flush.fill_(float(r))
        torch.cuda._sleep(400_000)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        rc = fn()
        e1.record(stream)
        if rc != 0:
            return None
        if r >= warm:
            times.append((e0, e1))
    torch.cuda.synchronize()
    if wgemm.wgemm_check(stream.cuda_stream) != 0:
        raise RuntimeError(f"device error: {wgemm.wgemm_last_device_error()}")
    return statistics.median(e0.elapsed_time(e1) * 1e3 for e0, e1 in times)


# (waves, K) points of the rate fit: the K range of most off-table calls.
RATE_POINTS = [(1, 1024), (1, 4096), (2, 1024), (2, 4096), (3, 2048), (4, 3072)]


def rates(out_path, points=RATE_POINTS, only=None):
    """Per data-parallel configuration: time whole waves of tiles (as many
    tiles per wave as co-resident workers) at several K and wave counts and
    fit t = t0 + waves · (a + b · kblocks) by least squares; once with operand
    rows on 32-byte sectors (pitch a multiple of 16 elements) and once with
    rows 16 bytes off them (pitch ≡ 8 mod 16). `only`: a regular expression
    the configuration names must match (default: all)."""
    import numpy as np
    import torch

    sys.path.insert(0, ROOT)
    from dense_fp16_gemm_02_gb300 import build, inputs, wgemm
    build.build()
    lib = wgemm.load()
    names = wgemm.config_names()
    torch.cuda.set_device(0)
    h = torch.cuda.current_stream().cuda_stream
    flush = torch.empty((256 << 20) // 4, dtype=torch.float32, device="cuda")
    max_waves = max(w for w, _ in points)
    Kmax = max(k for _, k in points)
    pitches = {"": Kmax + 16, "u": Kmax + 8}  # the buffers hold Kmax + 16 per row
    out = []
    for cid, name in enumerate(names):
        if only and not re.search(only, name):
            continue
        W = lib.wgemm_debug_max_workers(cid)
        cols, rows = (int(v) for v in name.split("_")[1].split("x"))
        tn = max(d for d in range(1, 9) if W % d == 0)
        tm = W // tn
        M1, N = tm * rows, tn * cols
        A, B = inputs.gemm_operands(max_waves * M1, N, Kmax, seed=11, kind="uniform",
                                    lda=Kmax + 16, ldb=Kmax + 16)
        dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
        # A 16-bit-output configuration ("_h") is timed writing fp16 C.
        c_type = wgemm.WGEMM_F16 if name.endswith("_h") else wgemm.WGEMM_F32
        C = torch.empty((max_waves * M1, N), device="cuda",
                        dtype=torch.float16 if name.endswith("_h") else torch.float32)
        del A, B
        print(f"# rates {name} W={W} tiles {tm}x{tn}", file=sys.stderr, flush=True)
        row = {"config": name, "workers": W}
        for tag, ld in pitches.items():
            X, y = [], []
            for waves, K in points:
                M = waves * M1
                if "_ab" in name:  # fused epilogue: D = 1·A·Bᵀ + 1·D (Cin read in place)
                    call = (lambda M=M, K=K, ld=ld: wgemm.wgemm_gemm_ex_config(
                        dA.data_ptr(), dB.data_ptr(), C.data_ptr(), C.data_ptr(), None, 1.0,
                        1.0, wgemm.WGEMM_F16, c_type, M, N, K, ld, ld, N, N, cid, h))
                else:
                    call = (lambda M=M, K=K, ld=ld: wgemm.wgemm_gemm_config(
                        dA.data_ptr(), dB.data_ptr(), C.data_ptr(), wgemm.WGEMM_F16, c_type, M,
                        N, K, ld, ld, N, cid, 0, 1, h))
                t = _time_calls(wgemm, torch, None, M, N, K, call, flush)
                kb = (K + 63) // 64
                X.append([1.0, waves, waves * kb])
                y.append(t)
            (t0, a, b), *_ = np.linalg.lstsq(np.array(X), np.array(y), rcond=None)
            row.update({f"t0{tag}_us": round(float(t0), 3), f"a{tag}_us": round(float(a), 3),
                        f"b{tag}_us": round(float(b), 5),
                        f"runs{tag}_us": [round(v, 2) for v in y]})
        out.append(row)
        print(json.dumps(row), flush=True)
        del dA, dB, C
        torch.cuda.empty_cache()
    with open(out_path, "w") as f:
        json.dump({"gpu": torch.cuda.get_device_name(0), "points": points, "rates": out}, f,
                  indent=1)


_RATE_KEYS = ("t0_us", "a_us", "b_us", "t0u_us", "au_us", "bu_us")


def read_rates_inc(inc_path=RATES_INC):
    """The rows of a written rates table, as `--rates` rows (by name)."""
    rows = {}
    with open(inc_path) as f:
        for line in f:
            m = re.match(r'\{"([^"]+)",((?:\s*-?[\d.]+,?){6})\},?\s*$', line.strip())
            if m:
                vals = [float(v) for v in m.group(2).split(",") if v.strip()]
                rows[m.group(1)] = {"config": m.group(1), **dict(zip(_RATE_KEYS, vals))}
    return rows


def emit_rates(json_paths, inc_path=RATES_INC, keep=False):
    """Writes the rates table from one or more `--rates` outputs; a
    configuration measured in a later file replaces its earlier row. With
    `keep`, the table's current rows come first (a new measurement of a
    configuration replaces its row, other rows stay)."""
    if isinstance(json_paths, str):
        json_paths = [json_paths]
    merged, d = (read_rates_inc(inc_path) if keep else {}), {}
    for path in json_paths:
        with open(path) as f:
            d = json.load(f)
        for r in d["rates"]:
            merged[r["config"]] = r
    lines = [
        "// Measured per-configuration rates (generated by dense_fp16_gemm_02_gb300/tune.py",
        f"// --rates on {d.get('gpu', 'a GB300')}; do not edit by hand). {{configuration,",
        "// t0 µs, a µs per wave, b µs per wave per k-block: rows on 32-byte sectors; the",
        "// same three with rows 16 bytes off}.",
    ]
    for r in merged.values():
        lines.append(f'{{"{r["config"]}", {r["t0_us"]:.3f}, {r["a_us"]:.3f}, {r["b_us"]:.5f}, '
                     f'{r["t0u_us"]:.3f}, {r["au_us"]:.3f}, {r["bu_us"]:.5f}}},')
    with open(inc_path, "w") as f:
        f.write("\n".join(lines) + "\n")
    return inc_path


def validate(out_path, shapes=OFF_TABLE + HELD_OUT):
    """For shapes outside the table: the rule's own choice against the best of
    an exhaustive sweep of configurations and K-decompositions."""
    import torch

    sys.path.insert(0, ROOT)
    from dense_fp16_gemm_02_gb300 import build, inputs, wgemm
    build.build()
    names = wgemm.config_names()
    torch.cuda.set_device(0)
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    h = torch.cuda.current_stream().cuda_stream
    flush = torch.empty((256 << 20) // 4, dtype=torch.float32, device="cuda")
    res = []
    for (M, N, K) in shapes:
        ld = (K + 7) // 8 * 8
        A, B = inputs.gemm_operands(M, N, K, seed=3, kind="uniform", lda=ld, ldb=ld)
        dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
        C = torch.empty((M, (N + 3) // 4 * 4), dtype=torch.float32, device="cuda")
        ldc = C.shape[1]
        cid, mode, sp = wgemm.wgemm_select(M, N, K, ld, ld)
        t_rule = _time_calls(wgemm, torch, None, M, N, K,
                             lambda: wgemm.wgemm_f16f32(dA.data_ptr(), dB.data_ptr(),
                                                        C.data_ptr(), M, N, K, ld, ld, ldc, h),
                             flush)
        best = None
        lib = wgemm.load()
        timed = []
        for c2, m2, s2 in candidates(M, N, K, names, sm // 2, sm):
            print(f"# validate {M}x{N}x{K} {names[c2]} mode {m2} splits {s2}", file=sys.stderr,
                  flush=True)
            t = _time_calls(wgemm, torch, None, M, N, K,
                            lambda: wgemm.wgemm_f16f32_config(
                                dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K, ld, ld,
                                ldc, c2, m2, s2, h), flush, reps=5)
            if t is not None and (best is None or t < best[0]):
                best = (t, names[c2], m2, s2)
            if t is not None:
                pred = lib.wgemm_debug_predict_us(M, N, K, ld, ld, c2, m2, s2,
                                                  lib.wgemm_debug_max_workers(c2))
                timed.append([names[c2], m2, s2, round(t, 2), round(pred, 2)])
        row = {"shape": [M, N, K], "set": "held out" if (M, N, K) in HELD_OUT else "tuned",
               "rule": [names[cid], mode, sp], "rule_us": round(t_rule, 2),
               "best": [best[1], best[2], best[3]], "best_us": round(best[0], 2),
               "rule_over_best": round(t_rule / best[0], 3),
               "candidates": sorted(timed, key=lambda x: x[3])}
        res.append(row)
        print(json.dumps(row), flush=True)
        del dA, dB, C
        torch.cuda.empty_cache()
    with open(out_path, "w") as f:
        json.dump(res, f, indent=1)


PDL_SHAPES = [(1024, 1024, 1024), (2048, 2048, 2048), (4096, 4096, 1024), (4096, 4096, 4096),
              (8192, 8192, 8192)]


def pdl_report(out_path, shapes=PDL_SHAPES, calls=40, rounds=8):
    """Back-to-back calls of one shape (no L2 flush between them), with
    programmatic dependent launch off and on: time per call. A separate
    report: the per-call metric times every call alone."""
    import torch

    sys.path.insert(0, ROOT)
    from dense_fp16_gemm_02_gb300 import build, inputs, wgemm
    build.build()
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    h = stream.cuda_stream
    flush = torch.empty((256 << 20) // 4, dtype=torch.float32, device="cuda")
    res = []
    for (M, N, K) in shapes:
        A, B = inputs.gemm_operands(M, N, K, seed=5, kind="uniform")
        dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
        C = torch.empty((M, N), dtype=torch.float32, device="cuda")
        row = {"shape": [M, N, K], "calls": calls}
        per = {False: [], True: []}
        # Rounds alternate off, on, off, on ... so that both settings see the
        # same clocks and temperature (long batches settle under the power cap).
        for r in range(rounds + 1):
            for pdl in ((False, True) if r % 2 == 0 else (True, False)):
                wgemm.wgemm_set_pdl(pdl)
                flush.fill_(float(r))
                torch.cuda._sleep(2_000_000)  # the whole batch is enqueued before it starts
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(calls):
                    rc = wgemm.wgemm_f16f32(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K,
                                            K, K, N, h)
                    if rc != 0:
                        raise RuntimeError(f"call failed: {rc}")
                e1.record(stream)
                e1.synchronize()
                if r > 0:
                    per[pdl].append(e0.elapsed_time(e1) * 1e3 / calls)
        wgemm.wgemm_set_pdl(False)
        if wgemm.wgemm_check(h) != 0:
            raise RuntimeError(f"device error: {wgemm.wgemm_last_device_error()}")
        row["pdl_off_us"] = round(statistics.median(per[False]), 3)
        row["pdl_on_us"] = round(statistics.median(per[True]), 3)
        row["saved_us_per_call"] = round(row["pdl_off_us"] - row["pdl_on_us"], 3)
        row["tflops_pdl_on"] = round(2.0 * M * N * K / (row["pdl_on_us"] * 1e-6) / 1e12, 1)
        res.append(row)
        print(json.dumps(row), flush=True)
        del dA, dB, C
        torch.cuda.empty_cache()
    with open(out_path, "w") as f:
        json.dump({"gpu": torch.cuda.get_device_name(0), "rows": res}, f, indent=1)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--out", default="tune.json")
    ap.add_argument("--shapes", default="all", choices=sorted(SHAPES))
    ap.add_argument("--no-sustained", action="store_true",
                    help="skip the back-to-back timing of long calls' finalists")
    ap.add_argument("--emit", metavar="JSON", nargs="+",
                    help="write csrc/wgemm_tuned.inc from one or more sweeps (several boxes)")
    ap.add_argument("--rates", metavar="JSON", help="measure per-configuration rates")
    ap.add_argument("--emit-rates", metavar="JSON", nargs="+",
                    help="write csrc/wgemm_rates.inc (later files override earlier rows)")
    ap.add_argument("--only", metavar="REGEX", help="--rates: configurations matching REGEX")
    ap.add_argument("--keep", action="store_true",
                    help="--emit-rates: keep the table's rows not measured in the given files")
    ap.add_argument("--validate", metavar="JSON", help="check the rule on off-table shapes")
    ap.add_argument("--pdl-report", metavar="JSON",
                    help="back-to-back calls with programmatic dependent launch off and on")
    args = ap.parse_args(argv)
    if args.emit:
        sys.path.insert(0, ROOT)
        from dense_fp16_gemm_02_gb300 import wgemm
        print(emit(args.emit, known=set(wgemm.config_names())))
        return 0
    if args.emit_rates:
        print(emit_rates(args.emit_rates, keep=args.keep))
        return 0
    if args.rates:
        rates(args.rates, only=args.only)
        return 0
    if args.validate:
        validate(args.validate)
        return 0
    if args.pdl_report:
        pdl_report(args.pdl_report)
        return 0
    sweep(SHAPES[args.shapes], args.out, sustained=not args.no_sustained)
    return 0


if __name__ == "__main__":
    sys.exit(main())
