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


def test_emit_prefers_the_interleaved_time(tmp_path):
    d = {"gpu": "test GPU", "sm_count": 152, "results": [
        {"shape": [64, 128, 256],
         "best": {"config": "g1_128x64_s8_a2_direct", "mode": 0, "splits": 1, "us": 9.0,
                  "us_interleaved": 8.5}},
        {"shape": [1024, 1024, 65536],
         "best": {"config": "g2_512x256_s4_a1_tma", "mode": 1, "splits": 9, "us": 96.25}},
    ]}
    js = tmp_path / "t.json"
    js.write_text(json.dumps(d))
    inc = tmp_path / "t.inc"
    tune.emit(str(js), str(inc))
    rows = [l for l in inc.read_text().splitlines() if l.startswith("{")]
    assert rows == ['{64, 128, 256, "g1_128x64_s8_a2_direct", 0, 1, 8.500},',
                    '{1024, 1024, 65536, "g2_512x256_s4_a1_tma", 1, 9, 96.250},']
    assert "do not edit by hand" in inc.read_text()


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
