"""Host logic of bench.py that needs no GPU: the split of a traced step into
its stages when the score and top-k run in several windows."""
import pytest

import bench


def test_one_window_is_the_plain_event_differences():
    t = [0.002, 0.010, 0.022, 0.042, 0.051]              # events 1..5 after event 0 (ms)
    st = bench.stage_split(t, [(0.010, 0.022), (-5.0, -4.0)])
    assert st == pytest.approx({"k_append": 0.002, "indexer_score": 0.008, "topk": 0.012,
                                "sparse_attn": 0.020, "attn_combine": 0.009})


def test_windows_sum_and_stale_slots_end_them():
    # three windows: score 1, top-k 2, score 3, top-k 1, score 2, top-k 4 (ms),
    # then a stale slot recorded before event 0 and one never reached
    t = [0.5, 1.5, 13.5, 20.0, 21.0]
    pairs = [(1.5, 3.5), (6.5, 7.5), (9.5, 13.5), (-2.0, -1.0), (14.0, 15.0)]
    st = bench.stage_split(t, pairs)
    assert st["topk"] == pytest.approx(7.0)
    assert st["indexer_score"] == pytest.approx(13.5 - 0.5 - 7.0)
    assert sum(st.values()) == pytest.approx(t[4])


def test_no_recorded_window_falls_back_to_the_first_top_k():
    t = [0.0, 1.0, 3.0, 4.0, 5.0]
    st = bench.stage_split(t, [])
    assert st["topk"] == pytest.approx(2.0) and st["indexer_score"] == pytest.approx(1.0)
