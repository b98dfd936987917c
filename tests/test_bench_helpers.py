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


def test_cpu_baseline_is_bounded_and_reports_one_thread():
    """Whole steps for a small decode batch; for a chunk of more than 64
    tokens a spread sample of single-token decodes (a full prefill step of
    the oracle would take minutes to hours); a single-thread figure."""
    import dsa_synth as S
    for wl in (S.config(1), S.prefill_workload("p", 3, 200, 130, H_I=4, H=8, top_k=64)):
        inp = S.make_inputs(wl)
        cb = bench.run_oracle_sample(wl, inp, 0.05)
        assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1
        assert cb["single_thread"]["cores"] == 1 and cb["single_thread"]["value"] > 0
        if wl.T > 64:
            assert "spread evenly" in cb["sample"]
        else:
            assert "full steps" in cb["sample"]
    subs = bench.token_subs(wl, inp, [0, 129])
    assert [o.q_pos for o, _ in subs] == [[200], [329]]
    assert subs[1][1].k_cache.shape[0] == 330
