"""Pins of the oracle's kpool indexer (GLM-5.3-Flash, vllm-rdna PR #2
"Glm5Next (GLM-5.3-Flash) on gfx1030": kpool 4, pool compression
softmax(gate+ape), always_select_tail, tail <= 3 -> width 2051; packed rows
k|gate|valid).  The reading is stated in oracle/dsa_oracle.h.

Compression: closed forms (uniform weights give the mean, one dominant gate
gives that row's key, two equal dominant gates their mean), invalid rows
excluded, dims independent, and only gate + ape matters.  Selection: a
brute-force restatement of the rule on the pool scores the oracle reports,
and those scores cross-checked through the (separately pinned) indexer-score
oracle run on a cache of the pooled keys.
"""
import numpy as np
import pytest

import dsa_synth as S
import oracle

D = 128


def _pool_rows(rng, gate=None, valid=(1, 1, 1, 1)):
    k = (rng.standard_normal((4, D)) / np.sqrt(D)).astype(np.float16)
    g = np.zeros((4, D), np.float16) if gate is None else np.asarray(gate, np.float16)
    return S.pack_kpool_rows(k, g, np.asarray(valid, np.float16)), k


def test_uniform_weights_give_the_mean():
    rng = np.random.default_rng(1)
    rows, k = _pool_rows(rng)
    has, key = oracle.kpool_pool_key(rows, 0, np.zeros((4, D), np.float32))
    assert has
    assert np.array_equal(key, k.astype(np.float64).mean(axis=0).astype(np.float16))


@pytest.mark.parametrize("i", [0, 3])
def test_one_dominant_gate_gives_that_key(i):
    rng = np.random.default_rng(2 + i)
    g = rng.standard_normal((4, D)) * 0.5
    g[i] = 30.0                                       # e^-30 of the others: far below an fp16 ulp
    rows, k = _pool_rows(rng, g)
    has, key = oracle.kpool_pool_key(rows, 0, np.zeros((4, D), np.float32))
    assert has and np.array_equal(key, k[i])


def test_two_equal_dominant_gates_give_their_mean():
    """The midpoint of two fp16 values is often an exact rounding tie, so the
    other two weights must be exactly zero: their gates sit at the fp16
    minimum, whose exponentials underflow to 0."""
    rng = np.random.default_rng(4)
    g = np.full((4, D), -65504.0)
    g[1] = g[2] = 30.0
    rows, k = _pool_rows(rng, g)
    has, key = oracle.kpool_pool_key(rows, 0, np.zeros((4, D), np.float32))
    assert np.array_equal(key, ((k[1].astype(np.float64) + k[2]) / 2).astype(np.float16))


def test_invalid_rows_are_left_out():
    rng = np.random.default_rng(5)
    rows, k = _pool_rows(rng, valid=(1, 0, 1, 0))
    has, key = oracle.kpool_pool_key(rows, 0, np.zeros((4, D), np.float32))
    assert has and np.array_equal(key, ((k[0].astype(np.float64) + k[2]) / 2).astype(np.float16))
    rows0, _ = _pool_rows(rng, valid=(0, 0, 0, 0))
    assert not oracle.kpool_pool_key(rows0, 0, np.zeros((4, D), np.float32))[0]


def test_dims_are_independent_and_only_gate_plus_ape_counts():
    rng = np.random.default_rng(6)
    g = rng.integers(-3, 4, (4, D)).astype(np.float64)        # exact in fp16 and float32
    a = rng.integers(-3, 4, (4, D)).astype(np.float32)
    rows, k = _pool_rows(rng, g)
    _, key = oracle.kpool_pool_key(rows, 0, a)
    swapped, _ = _pool_rows(np.random.default_rng(6), a)        # same k draws, gate and ape swapped
    swapped[:, :D] = rows[:, :D]
    _, key2 = oracle.kpool_pool_key(swapped, 0, g.astype(np.float32))
    assert np.array_equal(key, key2)
    a3 = a.copy()
    a3[:, 7] += 5.0                                             # one dim's embedding changes
    _, key3 = oracle.kpool_pool_key(rows, 0, a3)
    changed = np.nonzero(key3 != key)[0]
    assert set(changed.tolist()) <= {7}
    a4 = a + 2.0                                                # a shift common to the pool's 4 slots
    _, key4 = oracle.kpool_pool_key(rows, 0, a4)
    assert np.array_equal(key4, key)


def test_pool_j_reads_its_own_four_rows():
    rng = np.random.default_rng(7)
    k = (rng.standard_normal((12, D)) / np.sqrt(D)).astype(np.float16)
    rows = S.pack_kpool_rows(k, np.zeros((12, D), np.float16))
    _, key = oracle.kpool_pool_key(rows, 2, np.zeros((4, D), np.float32))
    assert np.array_equal(key, k[8:12].astype(np.float64).mean(axis=0).astype(np.float16))


# ----------------------------------------------------------------- selection

def _brute(scores_row, p, top_k, valid):
    n_pools = (p + 1) // 4
    pools = [j for j in range(n_pools) if np.isfinite(scores_row[j])]
    best = sorted(pools, key=lambda j: (-scores_row[j], j))[:top_k // 4]
    pos = [4 * j + r for j in sorted(best) for r in range(4) if valid[4 * j + r]]
    pos += [s for s in range(4 * n_pools, p + 1) if valid[s]]
    width = (top_k // 4) * 4 + 3
    return pos + [-1] * (width - len(pos))


def _kpool_case(lengths, H_I=4, top_k=16, seed=11, invalid=()):
    wl = S.decode_workload("kp", seed, lengths, H_I=H_I, H=8, top_k=top_k)
    inp = S.make_kpool_inputs(wl)
    b = oracle.Batch.of(wl)
    rows = inp.rows.copy()
    oracle.kpool_write_rows(inp.k_new, inp.gate_new, b, rows)
    for r in invalid:
        rows[r, 2 * D] = 0.0
    return wl, inp, b, rows


@pytest.mark.parametrize("top_k", [4, 16, 2048])
def test_selection_follows_the_rule_on_the_reported_pool_scores(top_k):
    lengths = [100, 37, 3, 2, 1, 64, 65]
    wl, inp, b, rows = _kpool_case(lengths, top_k=top_k, invalid=(5, 40, 41, 42, 43, 136))
    idx, sc = oracle.kpool_select(inp.q_idx, inp.w, rows, inp.ape, b, top_k, scores=True)
    assert idx.shape == (wl.T, (top_k // 4) * 4 + 3)
    for t, L in enumerate(lengths):
        off = wl.kv_off[t]
        valid = rows[off:off + L, 2 * D] != 0
        assert idx[t].tolist() == _brute(sc[t], wl.q_pos[t], top_k, valid), t


def test_ties_go_to_the_lower_pool():
    wl, inp, b, rows = _kpool_case([64], H_I=4, top_k=8)
    w0 = np.zeros_like(inp.w)                                  # every pool scores 0
    idx = oracle.kpool_select(inp.q_idx, w0, rows, inp.ape, b, 8)
    assert idx[0].tolist() == [0, 1, 2, 3, 4, 5, 6, 7, -1, -1, -1]


def test_tail_is_always_selected_and_width_is_2051():
    wl, inp, b, rows = _kpool_case([4098], H_I=2, top_k=2048, seed=12)    # 1024 pools, tail {4096, 4097}
    idx = oracle.kpool_select(inp.q_idx, inp.w, rows, inp.ape, b, 2048)
    assert idx.shape == (1, 2051)
    assert idx[0, 2048:].tolist() == [4096, 4097, -1]
    v = idx[0, :2048]
    assert np.all(np.diff(v) > 0) and np.all(v % 4 == np.tile(np.arange(4), 512))


def test_all_pools_selected_when_top_k_covers_them():
    wl, inp, b, rows = _kpool_case([30, 9], top_k=64)
    idx = oracle.kpool_select(inp.q_idx, inp.w, rows, inp.ape, b, 64)
    assert idx[0, :30].tolist() == list(range(30)) and np.all(idx[0, 30:] == -1)
    assert idx[1, :9].tolist() == list(range(9))


def test_pool_scores_match_the_indexer_score_on_pooled_keys():
    """The kpool scores are the indexer formula over the pooled keys: the
    indexer-score oracle (pinned on its own) run on a cache of pooled keys
    with each query seeing its complete pools gives the same numbers."""
    lengths = [90, 41, 8]
    wl, inp, b, rows = _kpool_case(lengths, H_I=6, top_k=16, seed=13)
    _, sc = oracle.kpool_select(inp.q_idx, inp.w, rows, inp.ape, b, 16, scores=True)
    for t, L in enumerate(lengths):
        n_pools = (wl.q_pos[t] + 1) // 4
        off = wl.kv_off[t]
        keys = np.stack([oracle.kpool_pool_key(rows[off:off + L], j, inp.ape)[1] for j in range(n_pools)])
        one = oracle.Batch([0, 1], [n_pools - 1], [0])
        ref = oracle.indexer_score(inp.q_idx[t:t + 1], inp.w[t:t + 1], keys, one, False)
        assert np.array_equal(sc[t, :n_pools], ref[0])
