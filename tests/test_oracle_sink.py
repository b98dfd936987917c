"""Pins of the oracle's attention-sink selection (ik_llama_opt commit log,
"GLM-5.2 DSA indexer: per-sequence attention sink" and "UPDATE 6": the first
n_sink positions of the query's own sequence, counted from its first present
position, always survive the top-k).

Each case is checked against a brute-force restatement written here: the
sink positions first (in position order), then the remaining positions by
(score desc, position asc), the first k taken, output ascending.
"""
import numpy as np
import pytest

import oracle


def brute(row, pos, k, lo, hi):
    n = pos + 1
    sinks = [s for s in range(n) if lo <= s < hi]
    rest = sorted((s for s in range(n) if not (lo <= s < hi)), key=lambda s: (-row[s], s))
    chosen = sorted((sinks + rest)[:min(k, n)])
    return chosen + [-1] * (k - len(chosen))


@pytest.mark.parametrize("n_sink", [0, 1, 4, 40])
@pytest.mark.parametrize("k", [1, 8, 33])
def test_sink_selection_matches_brute_force(n_sink, k):
    rng = np.random.default_rng(7 + n_sink * 100 + k)
    pos = [63, 30, 3, 50]
    s = rng.standard_normal((len(pos), 64))
    s[1, 10:20] = 0.25                               # ties among ordinary positions
    got = oracle.topk_sink(s, pos, k, n_sink)
    for r, p in enumerate(pos):
        assert got[r].tolist() == brute(s[r], p, k, 0, n_sink), (r, p)


def test_zero_sink_is_plain_topk():
    rng = np.random.default_rng(3)
    s = rng.standard_normal((3, 200))
    pos = [199, 120, 17]
    assert np.array_equal(oracle.topk_sink(s, pos, 16, 0), oracle.topk(s, pos, 16))


def test_sinks_survive_even_when_scored_lowest():
    s = np.zeros((1, 100))
    s[0, :3] = -1e30                                 # the indexer ranks the sink last
    got = oracle.topk_sink(s, [99], 10, 3)
    assert got[0, :3].tolist() == [0, 1, 2]
    assert oracle.topk(s, [99], 10)[0, :3].tolist() == [3, 4, 5]


def test_more_sinks_than_k_keeps_the_first_k_positions():
    rng = np.random.default_rng(11)
    s = rng.standard_normal((1, 50))
    assert oracle.topk_sink(s, [49], 4, 10)[0].tolist() == [0, 1, 2, 3]


def test_anchor_per_sequence():
    rng = np.random.default_rng(5)
    s = rng.standard_normal((2, 80))
    s[:, 20:24] = -100.0
    got = oracle.topk_sink(s, [79, 79], 6, 4, seq_of_row=[0, 1], anchors=[0, 20])
    assert got[1].tolist() == brute(s[1], 79, 6, 20, 24)
    assert set(range(20, 24)) <= set(got[1].tolist())
    assert got[0].tolist() == brute(s[0], 79, 6, 0, 4)


def test_sink_beyond_visible_range_is_ignored():
    rng = np.random.default_rng(9)
    s = rng.standard_normal((1, 40))
    # anchor past the query's position: no sink is visible
    got = oracle.topk_sink(s, [10], 4, 3, seq_of_row=[0], anchors=[30])
    assert np.array_equal(got, oracle.topk(s, [10], 4))
