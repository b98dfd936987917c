"""Pins of the oracle's top-k: brute force, ties, signed zeros, short rows.

The selection keeps min(top_k, n) keys (ik_llama_opt commit log, "Add
GLM-5.2/DeepSeek-V3.2 DSA lightning indexer": ggml_top_k(min(top_k,
n_tokens))); ties go to the lower position and positions are returned in
ascending order.
"""
import numpy as np
import pytest

import oracle


def brute(row, n, k):
    """Rank by pairwise comparison: s is kept iff fewer than k visible
    positions beat it, where u beats s when score(u) > score(s), or equal
    scores and u < s."""
    keep = []
    for s in range(n):
        beats = sum(1 for u in range(n)
                    if row[u] > row[s] or (row[u] == row[s] and u < s))
        if beats < k:
            keep.append(s)
    return keep + [-1] * (k - len(keep))


@pytest.mark.parametrize("seed", range(12))
def test_matches_pairwise_brute_force(seed):
    rng = np.random.default_rng(seed)
    L = int(rng.integers(1, 60))
    T = 4
    k = int(rng.integers(1, 70))
    # few distinct values so that ties are common
    scores = rng.integers(-3, 4, (T, L)).astype(np.float64) / 2
    pos = rng.integers(0, L, T)
    got = oracle.topk(scores, pos, k)
    for t in range(T):
        assert got[t].tolist() == brute(scores[t], pos[t] + 1, k)


def test_all_equal_row_takes_lowest_positions():
    s = np.full((1, 100), 0.5)
    assert oracle.topk(s, [99], 10)[0].tolist() == list(range(10))


def test_short_row_returns_all_visible_then_pad():
    s = np.random.default_rng(0).standard_normal((1, 10))
    got = oracle.topk(s, [6], 16)[0].tolist()
    assert got == list(range(7)) + [-1] * 9


def test_signed_zeros_tie_by_position():
    s = np.array([[0.0, -0.0, 1.0, -0.0, 0.0, -1.0]])
    assert oracle.topk(s, [5], 3)[0].tolist() == [0, 1, 2]
    assert oracle.topk(s, [5], 4)[0].tolist() == [0, 1, 2, 3]


def test_masked_tail_never_selected():
    s = np.array([[1.0, 2.0, 3.0, 100.0, 200.0]])
    assert oracle.topk(s, [2], 2)[0].tolist() == [1, 2]


def test_neg_inf_visible_scores_rank_last():
    s = np.array([[-np.inf, 1.0, -np.inf, -5.0]])
    assert oracle.topk(s, [3], 3)[0].tolist() == [0, 1, 3]


def test_full_sort_definition_large_random():
    rng = np.random.default_rng(7)
    s = rng.standard_normal((3, 5000)).astype(np.float32).astype(np.float64)
    pos = [4999, 3000, 2047]
    got = oracle.topk(s, pos, 2048)
    for t, p in enumerate(pos):
        n = p + 1
        order = np.lexsort((np.arange(n), -s[t, :n]))   # score desc, position asc
        want = np.sort(order[:2048])
        want = np.concatenate([want, -np.ones(2048 - len(want), np.int64)])
        assert np.array_equal(got[t], want)
