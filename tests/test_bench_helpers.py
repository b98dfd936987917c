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


def test_exclusive_spans_split_an_overlapped_step():
    """Kernels that start early (programmatic dependent launch) and wait for
    their predecessor are charged from the predecessor's end; the shares add
    up to the step's span."""
    spans = {"indexer_score": (0.0, 9.26), "topk": (3.46, 17.12), "sparse_attn": (7.5, 30.11),
             "attn_combine": (30.78, 35.6)}
    ex = bench.exclusive_spans(spans)
    assert ex == pytest.approx({"indexer_score": 9.26, "topk": 7.86, "sparse_attn": 12.99, "attn_combine": 4.82})
    assert sum(ex.values()) == pytest.approx(35.6 - 0.67)     # the gap before the combine is nobody's
    # a kernel that starts after its predecessor ends keeps its own span
    assert bench.exclusive_spans({"k_append": (0, 1), "indexer_score": (2, 5)}) == {"k_append": 1, "indexer_score": 3}


def test_kernel_rooflines_follow_the_workload_kind():
    import dsa_synth as S
    pk = dict(hbm_gbs=6000.0, bf16_tflops=2000.0, bf16_tflops_sustained=1800.0)
    dec, pre = S.config(2), S.config(4)
    a_dec, a_pre = bench.algorithmic(dec), bench.algorithmic(pre)
    r = bench.kernel_roofline("sparse_attn", 0.010, dec, a_dec, pk)
    assert r["bound"] == "hbm" and r["achieved"] == pytest.approx(8 * 2048 * 1152 / 1e-5 / 1e9)
    r = bench.kernel_roofline("indexer_score", 0.4, pre, a_pre, pk)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["algorithmic_flops"] == 25167872 * 64 * 256                  # causal pairs x heads x 2*128
    assert r["frac"] == pytest.approx(r["achieved"] / 2000.0)
    r = bench.kernel_roofline("sparse_attn", 3.0, pre, a_pre, pk)
    assert r["bound"] == "tensor" and r["algorithmic_flops"] == 4096 * 2048 * 64 * 2 * 1088


def test_score_windows_from_the_launch_count():
    class Fake:
        def __init__(self, n):
            self.n = n

        def dsa_decode_launches(self, batch, H_I, H, k):
            return self.n

    class B:
        max_q_per_seq = 1
    assert bench.score_windows(Fake(3), B()) == 1              # score, top-k, attention
    B.max_q_per_seq = 16384
    assert bench.score_windows(Fake(18), B()) == 8             # append + 8 x (score, top-k) + attention
