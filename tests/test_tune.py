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
    # A candidate missing from a sweep cannot win by absence.
    box3 = _sweep(shape, [_c("Z", 10.0, 10.0), _c("Y", 15.0, 15.0)])
    box4 = _sweep(shape, [_c("Y", 15.0, 15.0)])
    assert tune.combine([box3, box4])[shape][0]["config"] == "Y"


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
