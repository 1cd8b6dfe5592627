"""Summaries of ncu captures for profiles/: the roofline table of the eleven
shapes from one capture per shape (with the DRAM traffic table bench.py
reads), the bench's launch list, and older tables of the sweep shapes.

    python ncu_summary.py dram DRAM_CSV
    python ncu_summary.py roofline ROOFLINE_CSV BENCH_JSON
    python ncu_summary.py launches LAUNCHES_CSV
    python ncu_summary.py warm WARM_CSV COMPARE_JSONL
    python ncu_summary.py shapes CSV_DIR BENCH_JSON
    python ncu_summary.py launches-all LAUNCHES_CSV BENCH_JSON
    python ncu_summary.py bench BENCH_JSON

DRAM_CSV is the `--csv --log-file` output of the dram command in
profiles/dram_sweep.md; ROOFLINE_CSV and BENCH_JSON are those of
profiles/roofline_all_shapes.md; LAUNCHES_CSV that of
profiles/launches_sweep.md (every launch with gpu__time_duration.sum). The files under profiles/ are rewritten
(their prose is kept; the tables and the kernel-source digest are replaced).
`warm` prints the table of profiles/warm_l2_kernel_times.md from the launch
list of `compare --warm` and that command's output. `bench` rewrites the
head of profiles/bench_default_all_shapes.md (result, roofline line and
per-shape table) from the default bench line; its "Reading." stays.
"""
from __future__ import annotations

import csv
import io
import json
import os
import re
import statistics
import sys
from collections import OrderedDict

ROOT = os.path.dirname(os.path.abspath(__file__))
PROFILES = os.path.join(ROOT, "profiles")


def _bench():
    sys.path.insert(0, ROOT)
    import bench
    return bench


def read_ncu_csv(path: str) -> "OrderedDict[str, dict]":
    """Per launch ID: {metric name: value (float), "kernel": name}."""
    with open(path) as f:
        lines = [l for l in f.read().splitlines() if l.startswith('"')]
    by = OrderedDict()
    for r in csv.DictReader(io.StringIO("\n".join(lines))):
        d = by.setdefault(r["ID"], {"kernel": r["Kernel Name"]})
        try:
            d[r["Metric Name"]] = float(r["Metric Value"].replace(",", ""))
        except ValueError:
            d[r["Metric Name"]] = r["Metric Value"]
    return by


def _replace_table(text: str, header: str, rows: list[str]) -> str:
    """Replace the markdown table that starts with `header` by header + rows."""
    start = text.index(header)
    end = start + len(header)
    lines = text[end:].split("\n")
    n = 0
    while n < len(lines) and lines[n].startswith("|"):
        n += 1
    return text[:end] + "\n".join(rows) + "\n" + "\n".join(lines[n:])


def _set_digest(text: str, digest: str) -> str:
    return re.sub(r"digest\s*`[0-9a-f]{16}`", f"digest `{digest}`", text)


def dram(csv_path: str) -> None:
    """The DRAM table of profiles/dram_sweep.md (the six sweep shapes, one
    launch each). profiles/traffic.json comes from `shapes`, which covers all
    eleven shapes."""
    b = _bench()
    shapes = b.WORKLOADS["sweep"]
    by = read_ncu_csv(csv_path)
    if len(by) != len(shapes):
        raise SystemExit(f"{len(by)} launches in {csv_path}, expected {len(shapes)}")
    digest = b.kernel_source_digest()
    rows = []
    for (M, N, K), v in zip(shapes, by.values()):
        cfg = _config_of_kernel(v["kernel"])
        rd, wr = v["dram__bytes_read.sum"], v["dram__bytes_write.sum"]
        t = v["gpu__time_duration.sum"] / 1000.0
        rows.append(f"| {M}x{N}x{K} | {cfg} | {t:.1f} | {rd / 1e6:.1f} | {wr / 1e6:.1f} | "
                    f"{2 * (M * K + N * K) / 1e6:.1f} | {4 * M * N / 1e6:.1f} |")
    p = os.path.join(PROFILES, "dram_sweep.md")
    text = open(p).read()
    header = ("| shape | configuration | µs (ncu) | DRAM read MB | DRAM write MB | "
              "compulsory A+B MB | C MB |\n|---|---|---|---|---|---|---|\n")
    text = _set_digest(_replace_table(text, header, rows), digest)
    open(p, "w").write(text)
    print("\n".join(rows))


def _bench_line(bench_json: str) -> dict:
    with open(bench_json) as f:
        return json.loads([l for l in f.read().splitlines() if l.startswith("{")][-1])


SHAPE_HEADER = ("| M×N×K | configuration | mode | grid (CTAs) | waves | bench µs (events, median) | "
                "kernel µs (CUPTI, flushed) | kernel µs (CUPTI, warm) | bench TFLOP/s | tensor frac "
                "(bench) | ncu µs | SM clock GHz (ncu) | tensor pipe active % (ncu) | SM active % "
                "(ncu) | DRAM read MB | DRAM write MB | DRAM read ÷ compulsory A+B |\n"
                "|---|---|---|---|---|---|---|---|---|---|---|---|---|---|---|---|---|\n")
OLD_SHAPE_HEADER = ("| M×N×K | configuration | mode | grid (CTAs) | waves | bench µs (events, median) | "
                    "kernel µs (CUPTI, flushed) | kernel µs (CUPTI, warm) | bench TFLOP/s | tensor "
                    "frac (bench) | ncu µs | tensor pipe active % (ncu) | SM active % (ncu) | DRAM "
                    "read MB | DRAM write MB | DRAM read ÷ compulsory A+B |\n"
                    "|---|---|---|---|---|---|---|---|---|---|---|---|---|---|---|---|\n")


def shapes(csv_dir: str, bench_json: str) -> None:
    """One ncu capture per shape (CSV_DIR/<M>x<N>x<K>.csv: one launch of the
    shape's default configuration, one pass of seven counters) beside the
    bench line: the table of profiles/roofline_all_shapes.md, and the DRAM
    traffic per launch of every shape's kernel in profiles/traffic.json
    (which the bench reads for its roofline line)."""
    b = _bench()
    d = _bench_line(bench_json)
    digest = b.kernel_source_digest()
    rows, traffic = [], []
    for s in d["shapes"]:
        M, N, K = (int(x) for x in s["shape"].split("x"))
        by = read_ncu_csv(os.path.join(csv_dir, s["shape"] + ".csv"))
        v = [x for x in by.values() if "wgemm_kernel" in x["kernel"]][-1]
        cfg = _config_of_kernel(v["kernel"])
        if cfg != s["config"]:
            raise SystemExit(f"{s['shape']}: captured {cfg}, bench ran {s['config']}")
        t = v["gpu__time_duration.sum"] / 1000.0
        active = 100.0 * v["sm__cycles_active.avg"] / v["gpc__cycles_elapsed.max"]
        ghz = v["gpc__cycles_elapsed.max"] / v["gpu__time_duration.sum"]  # cycles per ns
        grid = int(v.get("launch__grid_size", 0))
        rd, wr = v["dram__bytes_read.sum"], v["dram__bytes_write.sum"]
        ab = 2.0 * (M * K + N * K)
        rows.append(
            f"| {M}×{N}×{K} | {cfg} | {s['mode']} | {grid} | "
            f"{_waves(cfg, M, N, grid, s['mode'], s.get('splits', 1))} | "
            f"{s['us_median']:.3f} | {s.get('us_kernel_median', float('nan')):.3f} | "
            f"{s.get('us_kernel_warm_median', float('nan')):.3f} | {s['tflops']} | "
            f"{s['tensor_frac']} | {t:.1f} | {ghz:.2f} | "
            f"{v['sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_elapsed']:.1f} | "
            f"{active:.1f} | {rd / 1e6:.1f} | {wr / 1e6:.1f} | {rd / ab:.2f} |")
        traffic.append({"kernel_src": digest, "config": cfg, "shape": s["shape"],
                        "dram_bytes": int(rd + wr),
                        "source": (f"profiles/roofline_all_shapes.md (dram__bytes_read.sum "
                                   f"{int(rd):,} B + dram__bytes_write.sum {int(wr):,} B, "
                                   "one launch)")})
    with open(os.path.join(PROFILES, "traffic.json"), "w") as f:
        json.dump(traffic, f, indent=1)
    p = os.path.join(PROFILES, "roofline_all_shapes.md")
    text = open(p).read()
    if SHAPE_HEADER not in text:  # a table written before the clock column
        text = text.replace(OLD_SHAPE_HEADER, SHAPE_HEADER)
    text = _set_digest(_replace_table(text, SHAPE_HEADER, rows), digest)
    open(p, "w").write(text)
    print("\n".join(rows))


def launches_all(csv_path: str, bench_json: str) -> None:
    """The launch list of a bench run (every GEMM launch with
    gpu__time_duration.sum; cold-cache and serialised under ncu) per
    configuration: launches, total µs and share of the GEMM time, beside the
    share of the bench line's own timed steps (CUDA events) for the same
    configuration. Writes the table of profiles/launches_all_shapes.md."""
    b = _bench()
    d = _bench_line(bench_json)
    by = read_ncu_csv(csv_path)
    # Only the launches of the warm-up and timed steps, which come first and
    # have the same calls: the end-to-end passes after them call each shape
    # once, the large ones in row panels.
    per_step = sum(d["timing"]["calls_per_step"].values())
    keep = (d["warmup"] + d["steps"]) * per_step
    launches = [v for _, v in sorted(by.items(), key=lambda kv: int(kv[0]))
                if "wgemm_kernel" in v["kernel"]][:keep]
    agg = OrderedDict()
    for v in launches:
        a = agg.setdefault(_config_of_kernel(v["kernel"]), [0, 0.0])
        a[0] += 1
        a[1] += v["gpu__time_duration.sum"] / 1000.0
    total = sum(a[1] for a in agg.values())
    # The weighted share puts each configuration's mean launch time on the
    # bench's calls per step (the same as the plain share when every launch
    # kept belongs to a step).
    bench_ms, calls = OrderedDict(), OrderedDict()
    for s in d["shapes"]:
        bench_ms[s["config"]] = bench_ms.get(s["config"], 0.0) + s["us_median"] * s["calls"]
        calls[s["config"]] = calls.get(s["config"], 0) + s["calls"]
    btotal = sum(bench_ms.values())
    weighted = {cfg: us / n * calls.get(cfg, 0) for cfg, (n, us) in agg.items()}
    wtotal = sum(weighted.values())
    rows = []
    for cfg, (n, us) in sorted(agg.items(), key=lambda kv: -kv[1][1]):
        shapes_of = ", ".join(s["shape"] for s in d["shapes"] if s["config"] == cfg)
        rows.append(f"| {cfg} | {shapes_of} | {n} | {us:.1f} | {us / n:.1f} | "
                    f"{100.0 * us / total:.1f} % | {100.0 * weighted[cfg] / wtotal:.1f} % | "
                    f"{100.0 * bench_ms.get(cfg, 0.0) / btotal:.1f} % |")
    p = os.path.join(PROFILES, "launches_all_shapes.md")
    text = open(p).read()
    header = ("| configuration | shapes | launches (ncu) | total µs (ncu) | mean µs per launch (ncu) "
              "| share of GEMM time (ncu) | share, weighted by the bench's calls per step (ncu) "
              "| share of the bench's timed steps (events) |\n"
              "|---|---|---|---|---|---|---|---|\n")
    text = _set_digest(_replace_table(text, header, rows), b.kernel_source_digest())
    open(p, "w").write(text)
    print("\n".join(rows))


def roofline(csv_path: str, bench_json: str) -> None:
    b = _bench()
    by = read_ncu_csv(csv_path)
    with open(bench_json) as f:
        line = [l for l in f.read().splitlines() if l.startswith("{")][-1]
    d = json.loads(line)
    if len(by) != len(d["shapes"]):
        raise SystemExit(f"{len(by)} launches, {len(d['shapes'])} shapes")
    rows = []
    for s, v in zip(d["shapes"], by.values()):
        M, N, K = (int(x) for x in s["shape"].split("x"))
        t = v["gpu__time_duration.sum"] / 1000.0
        active = 100.0 * v["sm__cycles_active.avg"] / v["gpc__cycles_elapsed.max"]
        grid = int(v.get("launch__grid_size", 0))
        rows.append(
            f"| {M}×{N}×{K} | {s['config']} | {s['mode']} | {grid} | "
            f"{_waves(s['config'], M, N, grid, s['mode'], s.get('splits', 1))} | "
            f"{s['us_median']:.3f} | {s['tflops']} | "
            f"{s['tensor_frac']} | {t:.1f} | {2 * M * N * K / t / 1e6:.1f} | "
            f"{v['sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_elapsed']:.1f} | "
            f"{active:.1f} | {v['dram__bytes_read.sum'] / 1e6:.1f} | "
            f"{v['dram__bytes_write.sum'] / 1e6:.1f} | {s['hbm_frac']} |")
    p = os.path.join(PROFILES, "roofline_all_shapes.md")
    text = open(p).read()
    header = ("| M×N×K | configuration | mode | grid (CTAs) | waves | bench µs (median) | "
              "bench TFLOP/s | tensor frac (bench) | ncu µs | ncu TFLOP/s | tensor pipe active % "
              "(ncu) | SM active % (ncu) | DRAM read MB | DRAM write MB | HBM frac (bench, "
              "compulsory bytes) |\n"
              "|---|---|---|---|---|---|---|---|---|---|---|---|---|---|---|\n")
    text = _set_digest(_replace_table(text, header, rows), b.kernel_source_digest())
    open(p, "w").write(text)
    print("\n".join(rows))


def launches(csv_path: str) -> None:
    """Per kernel of a launch list: launches, total device time and shares."""
    by = read_ncu_csv(csv_path)
    agg = OrderedDict()
    for v in by.values():
        a = agg.setdefault(v["kernel"], [0, 0.0])
        a[0] += 1
        a[1] += v["gpu__time_duration.sum"] / 1000.0
    total = sum(a[1] for a in agg.values())
    gemm = sum(a[1] for k, a in agg.items() if "wgemm_kernel" in k)
    rows = []
    for k, (n, us) in agg.items():
        name = k if len(k) <= 90 else k[:87] + "..."
        cfg = _config_of_kernel(k) if "wgemm_kernel" in k else "—"
        g = 100.0 * us / gemm if "wgemm_kernel" in k and gemm > 0 else 0.0
        rows.append(f"| `{name}` | {cfg} | {n} | {us:.1f} | {100.0 * us / total:.1f} % | "
                    f"{g:.1f} % |")
    p = os.path.join(PROFILES, "launches_sweep.md")
    text = open(p).read()
    header = ("| kernel | configuration | launches | total µs | share of all | share of wgemm |\n"
              "|---|---|---|---|---|---|\n")
    text = _set_digest(_replace_table(text, header, rows), _bench().kernel_source_digest())
    open(p, "w").write(text)
    print("\n".join(rows))


def warm(csv_path: str, compare_jsonl: str) -> None:
    """Kernel-only times of `compare --warm` from its ncu launch list (taken
    with --cache-control none): per shape, the library's launches come first
    and cuBLAS's after them; a cuBLAS call may launch several kernels, whose
    times are summed per call. Medians of the timed calls (the warm-up calls
    dropped). Prints the table rows."""
    with open(compare_jsonl) as f:
        lines = [json.loads(l) for l in f if l.startswith("{")]
    shapes = [d for d in lines if "shape" in d]
    rounds = [d for d in lines if "summary" in d][0]["summary"]["rounds"]
    calls = 3 + rounds
    by = list(read_ncu_csv(csv_path).values())
    # Runs of consecutive launches, library (wgemm) or not; skip what comes
    # before the first library launch (the start-up probe).
    runs = []
    for v in by:
        ours = "wgemm_kernel" in v["kernel"]
        if not runs and not ours:
            continue
        if runs and runs[-1][0] == ours:
            runs[-1][1].append(v["gpu__time_duration.sum"] / 1000.0)
        else:
            runs.append((ours, [v["gpu__time_duration.sum"] / 1000.0]))
    if len(runs) != 2 * len(shapes):
        raise SystemExit(f"{len(runs)} launch runs for {len(shapes)} shapes")
    out = []
    for i, d in enumerate(shapes):
        M, N, K = (int(x) for x in d["shape"].split("x"))
        (o1, t_ours), (o2, t_ref) = runs[2 * i], runs[2 * i + 1]
        if not (o1 and not o2) or len(t_ours) != calls or len(t_ref) % calls:
            raise SystemExit(f"{d['shape']}: {len(t_ours)} and {len(t_ref)} launches")
        k = len(t_ref) // calls
        ref_calls = [sum(t_ref[j * k:(j + 1) * k]) for j in range(calls)]
        us_o = statistics.median(t_ours[3:])
        us_r = statistics.median(ref_calls[3:])
        fl = 2.0 * M * N * K
        out.append(f"| {M}×{N}×{K} | {us_o:.2f} | {us_r:.2f} | {us_r / us_o:.3f} | "
                   f"{fl / us_o / 1e6:.1f} | {k} | {d['ours_us']:.2f} | {d['cublas_us']:.2f} |")
    print("| M×N×K | wgemm kernel µs | cuBLAS kernel µs (per call) | cuBLAS ÷ wgemm | "
          "wgemm TFLOP/s | cuBLAS kernels per call | wgemm event µs | cuBLAS event µs |")
    print("|---|---|---|---|---|---|---|---|")
    print("\n".join(out))


def _waves(config: str, M: int, N: int, grid: int, mode: str, splits: int) -> str:
    """Worker tiles (units, for split-K) per co-resident worker: the number
    of waves of the launch, from the configuration's tile and cluster."""
    a = _entry_args(config)
    if not a or grid <= 0:
        return "—"
    cg, reps, bn, _, _, _, mc, _, _, _, mr, _ = a
    tile_cols, tile_rows = 128 * reps * cg * mc, bn * mr
    tiles = -(-M // tile_rows) * -(-N // tile_cols)
    cluster = cg * mc * mr
    workers = grid // cluster
    if config.endswith("_clc"):
        # One cluster per tile is launched; the co-resident ones take tiles
        # from the others (GB300: 152 CTAs, 76 pairs, 36 clusters of four).
        workers = min(workers, {1: 152, 2: 76, 4: 36}.get(cluster, workers))
    if mode == "split-K":
        tiles *= splits
    elif mode.startswith("stream-K"):
        return "1 (stream)"
    elif mode == "data-parallel + stream-K tail":
        return f"{tiles / workers:.2f} (stream-K tail)"
    return f"{tiles / workers:.2f}"


def _config_of_kernel(kernel: str) -> str:
    """The configuration name of a launched kernel, from its Cfg<...> arguments."""
    m = re.search(r"Cfg<([0-9, ]+)>", kernel)
    if not m:
        return kernel
    args = tuple(int(x) for x in m.group(1).split(","))
    if len(args) == 10:  # captures from before the MR argument existed
        args += (1,)
    if len(args) == 11:  # captures from before the KPS argument existed
        args += (1,)
    sys.path.insert(0, ROOT)
    from dense_fp16_gemm_02_gb300 import build, wgemm
    build.build()
    for name in wgemm.config_names():
        if _entry_args(name) == args:
            return name
    return kernel


def _entry_args(name: str):
    """The Cfg<CG, REPS, BN, STAGES, ACC, EPI, MC, SCHED, OUT, FUSE, MR, KPS>
    arguments of a configuration, rebuilt from its name (g<CG>[m<MC>|r<MR>]_
    <tile columns>x<tile rows>_s<STAGES>[x<KPS>]_a<ACC>_<epilogue>[_clc][_ab<FUSE>][_h])."""
    m = re.match(r"g(\d)(?:m(\d))?(?:r(\d))?_(\d+)x(\d+)_s(\d+)(?:x(\d))?_a(\d)_(tma|direct)"
                 r"(_clc)?(?:_ab(\d))?(_h)?$", name)
    if not m:
        return None
    cg = int(m.group(1))
    mc = int(m.group(2) or 1)
    mr = int(m.group(3) or 1)
    cols, rows = int(m.group(4)), int(m.group(5))
    reps = cols // (128 * cg * mc)
    return (cg, reps, rows // mr, int(m.group(6)), int(m.group(8)),
            1 if m.group(9) == "tma" else 0, mc, 1 if m.group(10) else 0,
            1 if m.group(12) else 0, int(m.group(11) or 0), mr, int(m.group(7) or 1))


# The pages' B200 kernel times per call (µs; "SASS-Level Kernel Generation for
# Blackwell", section "The numbers", the shape table): context, another chip.
PAGES_B200_US = {
    "1024x1024x1024": "4.64–4.67", "1536x1536x1536": "7.87", "2048x2048x2048": "14.46",
    "3072x1280x2048": "14.08", "4096x4096x1024": "26.11", "4096x4096x4096": "75.78–75.97",
    "8192x2048x4096": "75.84–75.97", "8192x8192x8192": "553.1–554.3",
    "16384x16384x16384": "4132.8–4239.4", "2048x2048x16384": "73.92–74.11",
    "1024x1024x65536": "76.93–77.22",
}

BENCH_HEADER = ("| M×N×K | configuration | mode | calls | event µs median (min–max) | "
                "kernel µs, flushed (CUPTI) | kernel µs, warm (CUPTI) | TFLOP/s (events) | "
                "of measured peak | of pipe ceiling | TFLOP/s (warm kernel) | "
                "pages' B200 kernel µs (context) |\n|---|---|---|---|---|---|---|---|---|---|---|---|\n")


def bench_profile(bench_json: str) -> None:
    """The head of profiles/bench_default_all_shapes.md from a default bench
    line: the command, the result, the roofline line and the per-shape table.
    Everything from the line "Reading." on is kept."""
    b = _bench()
    d = _bench_line(bench_json)
    path = os.path.join(PROFILES, "bench_default_all_shapes.md")
    with open(path) as f:
        old = f.read()
    reading = old[old.index("\nReading.") + 1:] if "\nReading." in old else "Reading.\n"
    ro, ck, e2e, cpu = d["roofline"], d["clocks"], d["e2e"], d["cpu_baseline"]
    launches = d["gpu_launches"]
    reasons = ck.get("reasons") or []
    noted = (" (kept and noted: the power cap during the large shapes)"
             if "sw_power_cap" in reasons else "")
    rows = []
    for r in d["shapes"]:
        M, N, K = (int(x) for x in r["shape"].split("x"))
        mode = r["mode"] + (f" {r['splits']}" if r["mode"] == "split-K" else "")
        rows.append(
            f"| {M}×{N}×{K} | {r['config']} | {mode} | {r['calls']} | "
            f"{r['us_median']:.2f} ({r['us_min']:.2f}–{r['us_max']:.2f}) | "
            f"{r.get('us_kernel_median', float('nan')):.2f} | "
            f"{r.get('us_kernel_warm_median', float('nan')):.2f} | {r['tflops']} | "
            f"{r['tensor_frac']:.3f} | {r['pipe_frac']:.3f} | "
            f"{r.get('tflops_kernel_warm', float('nan'))} | {PAGES_B200_US.get(r['shape'], '')} |")
    head = f"""# The default bench line: all eleven shapes, one GB300

The driver's own command, on the kernel sources of digest `{b.kernel_source_digest()}` (bench.py
`kernel_source_digest`). One step calls every shape several times, each call
alone: an L2 flush (a 256 MiB write), a GPU-side gate, then CUDA events
around the call. After the timed steps, CUPTI records the kernel time of 20
flushed calls per shape and of 20 calls with a warm L2 and a device
synchronisation after each call (the pages' protocol, "How we measured").

    python bench.py                 # --steps 20 --warmup 5 by default; prints one JSON line
    python ncu_summary.py bench bench.json   # writes this head; the reading below is prose

Result: `value` {d['value']} TFLOP/s (Σ flops of a step ÷ its summed event time;
the step is dominated by 16384³), {launches} timed launches, {d['wall_s_timed']} s timed. Clocks in
the timed region: SM {ck['sm_mhz']} MHz median of {ck['sm_max_mhz']} ({ck['samples']} samples), reasons {reasons}{noted}. End to end
({d['timing']['e2e']}): {e2e['value']} TFLOP/s,
{e2e['h2d_bytes_per_step']} B up and {e2e['d2h_bytes_per_step']} B down per step. CPU oracle: {cpu['value']:.4f} TFLOP/s on {cpu['cores']} cores
(row-sampled).

Roofline line: the dominant kernel is `{ro['kernel']}` ({ro['launches']} launches in the timed steps; its
`traffic` is taken at {ro['traffic_shape']}),
{ro['achieved']} TFLOP/s over its event times, {ro['frac']:.3f} of the measured cuBLAS bf16 burst rate
({ro['peak']}), {ro['frac_vs_sustained']:.3f} of the sustained rate ({ro['peak_sustained']}), {ro['frac_vs_pipe_ceiling']:.3f} of the tcgen05 pipe ceiling
({ro['pipe_ceiling']}, `profiles/tensor_pipe_ceiling.md`); {ro['achieved_kernel_time']} TFLOP/s from its CUPTI
kernel times. DRAM bytes per launch (`traffic`): {ro['traffic'] if ro['traffic'] is not None else "none in this line (no capture of this kernel at that shape on these sources when it ran)"}.

"""
    text = head + BENCH_HEADER + "\n".join(rows) + "\n\n" + reading
    with open(path, "w") as f:
        f.write(text)
    print(text[:len(head) + len(BENCH_HEADER)] + "\n".join(rows))


def main(argv=None) -> int:
    argv = sys.argv[1:] if argv is None else argv
    if len(argv) >= 2 and argv[0] == "dram":
        dram(argv[1])
    elif len(argv) >= 3 and argv[0] == "roofline":
        roofline(argv[1], argv[2])
    elif len(argv) >= 2 and argv[0] == "launches":
        launches(argv[1])
    elif len(argv) >= 3 and argv[0] == "warm":
        warm(argv[1], argv[2])
    elif len(argv) >= 3 and argv[0] == "shapes":
        shapes(argv[1], argv[2])
    elif len(argv) >= 3 and argv[0] == "launches-all":
        launches_all(argv[1], argv[2])
    elif len(argv) >= 2 and argv[0] == "bench":
        bench_profile(argv[1])
    else:
        print(__doc__)
        return 2
    return 0


if __name__ == "__main__":
    sys.exit(main())
