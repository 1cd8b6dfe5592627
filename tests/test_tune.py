"""Host logic of the tuner: the table it writes and the statistic that picks
the winner among the finalists (no GPU)."""
import json

from dense_fp16_gemm_02_gb300 import tune


def test_mid_mean_trims_a_quarter_each_end():
    assert tune._mid_mean([5.0] * 8) == 5.0
    # One slow outlier and one fast one do not move it.
    assert tune._mid_mean([1.0, 2.0, 2.0, 2.0, 2.0, 2.0, 2.0, 90.0]) == 2.0
    # Quantised ticks average to a figure between them.
    assert tune._mid_mean([20.5, 21.5] * 10) == 21.0


def _sweep(shape, cands):
    return {"gpu": "test GPU", "sm_count": 152, "results": [
        {"shape": list(shape), "best": cands[0], "candidates": cands}]}


def _c(config, us, inter=None, mode=0, splits=1):
    c = {"config": config, "mode": mode, "splits": splits, "us": us}
    if inter is not None:
        c["us_interleaved"] = inter
    return c


def test_emit_prefers_the_interleaved_time(tmp_path):
    d = _sweep((64, 128, 256), [_c("g1_128x64_s8_a2_direct", 9.0, 8.5),
                                _c("g1_128x128_s6_a2_tma", 8.9, 8.8)])
    d["results"].append({"shape": [1024, 1024, 65536], "candidates": [
        _c("g2_512x256_s4_a1_tma", 96.25, mode=1, splits=9)]})
    js = tmp_path / "t.json"
    js.write_text(json.dumps(d))
    inc = tmp_path / "t.inc"
    tune.emit(str(js), str(inc))
    rows = [l for l in inc.read_text().splitlines() if l.startswith("{")]
    assert rows == ['{64, 128, 256, "g1_128x64_s8_a2_direct", 0, 1, 8.500},',
                    '{1024, 1024, 65536, "g2_512x256_s4_a1_tma", 1, 9, 96.250},']
    assert "do not edit by hand" in inc.read_text()


def test_combine_takes_the_best_mean_over_boxes():
    # X wins box 1 by 2 % but loses box 2 by 10 %; Y is steady. Box 2 is 5 %
    # faster overall, which the relative scores remove.
    shape = (1536, 1536, 1536)
    box1 = _sweep(shape, [_c("X", 15.0, 15.0), _c("Y", 15.3, 15.3)])
    box2 = _sweep(shape, [_c("Y", 14.5, 14.5), _c("X", 15.95, 15.95)])
    got, score = tune.combine([box1, box2])[shape]
    assert got["config"] == "Y" and abs(got["us"] - 14.9) < 1e-9
    assert abs(score - (15.3 / 15.0 + 1.0) / 2) < 1e-12
    # One sweep alone keeps its own winner.
    assert tune.combine([box1])[shape][0]["config"] == "X"
    # A candidate the library refused on one box cannot win by absence.
    box3 = _sweep(shape, [_c("Z", 10.0, 10.0), _c("Y", 15.0, 15.0)])
    box4 = _sweep(shape, [_c("Y", 15.0, 15.0)])
    box4["results"][0]["failed"] = [{"config": "Z", "mode": 0, "splits": 1}]
    assert tune.combine([box3, box4])[shape][0]["config"] == "Y"
    # A sweep made before Z existed tried fewer candidates: it no longer
    # counts for the shape, and Z, timed by every wider sweep, can win.
    old = _sweep(shape, [_c("Y", 14.0, 14.0)])
    assert tune.combine([box3, old])[shape][0]["config"] == "Z"
    # Configurations no longer compiled are dropped before that comparison.
    assert tune.combine([box3, old], known={"Y"})[shape][0]["config"] == "Y"


def _rows(*us):
    return [{"us": u} for u in us]


def test_finalists_take_every_candidate_within_a_tick():
    # Seven candidates within one tick of the best at 20 µs: the screen cannot
    # order them, so all are re-timed.
    assert tune.finalists(_rows(20.5, 20.5, 20.5, 21.5, 21.5, 21.5, 21.5, 24.0, 30.0)) == 7
    # Clearly separated candidates still give four finalists.
    assert tune.finalists(_rows(80.0, 90.0, 95.0, 99.0, 120.0)) == 4
    # Never more than eight, never more than there are.
    assert tune.finalists(_rows(*[20.5] * 12)) == 8
    assert tune.finalists(_rows(10.0, 50.0)) == 2


def test_final_rounds_scale_with_call_time():
    assert tune.final_rounds(20.0) == 200
    assert tune.final_rounds(600.0) == 33
    assert tune.final_rounds(5000.0) == 20


def _sus(c, sustained):
    c = dict(c)
    c["us_sustained"] = sustained
    return c


def test_sustained_time_decides_where_a_sweep_took_it(tmp_path):
    shape = (16384, 16384, 16384)
    # A lone-call sweep prefers X; the sustained sweep prefers Y, and X is
    # 4 % slower back to back.
    lone = _sweep(shape, [_c("X", 5100.0, 5100.0), _c("Y", 5200.0, 5200.0)])
    held = _sweep(shape, [_sus(_c("Y", 5300.0, 5300.0), 5160.0),
                          _sus(_c("X", 5150.0, 5150.0), 5370.0),
                          _c("Z", 5000.0)])  # screened only: no sustained time, left out
    got, score = tune.combine([lone, held])[shape]
    assert got["config"] == "Y" and got["us"] == 5160.0 and score == 1.0
    # Without the sustained sweep the lone-call winner stands.
    assert tune.combine([lone])[shape][0]["config"] == "X"
    # A shape no sweep timed back to back is combined as before.
    other = (1024, 1024, 1024)
    a = _sweep(other, [_c("P", 10.0, 10.0), _c("Q", 10.5, 10.5)])
    assert tune.combine([a, held])[other][0]["config"] == "P"
    # The table lists every shape of every sweep, in the sweeps' order.
    paths = []
    for i, d in enumerate((a, held)):
        js = tmp_path / f"s{i}.json"
        js.write_text(json.dumps(d))
        paths.append(str(js))
    inc = tmp_path / "t.inc"
    tune.emit(paths, str(inc))
    rows = [l for l in inc.read_text().splitlines() if l.startswith("{")]
    assert rows == ['{1024, 1024, 1024, "P", 0, 1, 10.000},',
                    '{16384, 16384, 16384, "Y", 0, 1, 5160.000},']


def test_block_calls_cover_half_a_second():
    assert tune.block_calls(5000.0) == 100
    assert tune.block_calls(600.0) == 833
    assert tune.block_calls(100000.0) == 30


def test_rates_table_keeps_rows_not_measured_again(tmp_path):
    inc = tmp_path / "r.inc"
    inc.write_text('// header\n{"A", 1.000, 2.000, 0.10000, 1.500, 2.500, 0.20000},\n'
                   '{"B", 3.000, -0.500, 0.30000, 3.500, 4.000, 0.40000},\n')
    assert tune.read_rates_inc(str(inc))["B"]["a_us"] == -0.5
    js = tmp_path / "new.json"
    js.write_text(json.dumps({"gpu": "test GPU", "rates": [
        {"config": "B", "t0_us": 5.0, "a_us": 6.0, "b_us": 0.7, "t0u_us": 5.5, "au_us": 6.5,
         "bu_us": 0.8},
        {"config": "C", "t0_us": 9.0, "a_us": 1.0, "b_us": 0.9, "t0u_us": 9.5, "au_us": 1.5,
         "bu_us": 0.95}]}))
    tune.emit_rates([str(js)], str(inc), keep=True)
    rows = [l for l in inc.read_text().splitlines() if l.startswith("{")]
    assert rows == ['{"A", 1.000, 2.000, 0.10000, 1.500, 2.500, 0.20000},',
                    '{"B", 5.000, 6.000, 0.70000, 5.500, 6.500, 0.80000},',
                    '{"C", 9.000, 1.000, 0.90000, 9.500, 1.500, 0.95000},']
    # Without keep, only the measured rows are written.
    tune.emit_rates([str(js)], str(inc))
    assert len([l for l in inc.read_text().splitlines() if l.startswith("{")]) == 2


def _warm(c, us):
    c = dict(c)
    c["us_warm_kernel"] = us
    return c


def test_warm_kernel_time_breaks_short_ties():
    shape = (1024, 1024, 1024)
    # Two finalists tie on flushed events; the warm-L2 kernel time decides.
    tied = _sweep(shape, [_warm(_c("P", 10.2, 10.22), 6.9), _warm(_c("Q", 10.2, 10.221), 6.4),
                          _c("R", 12.3, 12.3)])
    got, _ = tune.combine([tied])[shape]
    assert got["config"] == "Q" and got["us"] == 6.4
    # A sweep without the tie-break does not outvote it.
    plain = _sweep(shape, [_c("P", 10.1, 10.1), _c("Q", 10.3, 10.3), _c("R", 12.0, 12.0)])
    assert tune.combine([tied, plain])[shape][0]["config"] == "Q"
