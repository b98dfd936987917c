"""Pins of the oracle's lightning-indexer score.

I(t,s) = sum_h w[t,h] * ReLU(q[t,h] . k[s]) for s <= pos(t), per ik_llama_opt
commit log, "Add GLM-5.2/DeepSeek-V3.2 DSA lightning indexer" (ReLU of the
dot, scaled per-head weights, sum over heads, causal mask).
"""
import numpy as np
import pytest
import scipy.linalg

import dsa_synth as S
import oracle


def _one_seq(L, p_list):
    return oracle.Batch([0, len(p_list)], p_list, [0])


def _f16(a):
    return np.asarray(a, dtype=np.float16)


def test_hand_worked_example():
    # Two heads, three cached keys, one query at position 2; every value is
    # exact in fp16 so the expected scores are exact rationals.
    k = np.zeros((3, 128))
    k[0, 0], k[0, 1] = 1.0, 0.5       # key 0
    k[1, 0], k[1, 2] = -1.0, 2.0      # key 1
    k[2, 1], k[2, 2] = 0.25, -0.5     # key 2
    q = np.zeros((1, 2, 128))
    q[0, 0, 0], q[0, 0, 1] = 2.0, 1.0      # head 0
    q[0, 1, 2], q[0, 1, 1] = 1.0, -4.0     # head 1
    w = np.array([[0.5, -0.25]], dtype=np.float32)
    # head 0 dots: k0: 2+0.5=2.5; k1: -2; k2: 0.25   -> ReLU 2.5, 0, 0.25
    # head 1 dots: k0: -2; k1: 2; k2: -1-0.5=-1.5    -> ReLU 0, 2, 0
    # I = 0.5*h0 - 0.25*h1: k0 1.25; k1 -0.5; k2 0.125
    got = oracle.indexer_score(_f16(q), w, _f16(k), _one_seq(3, [2]), False)
    assert got.tolist() == [[1.25, -0.5, 0.125]]
    # position 1 sees keys 0..1 only; the rest is masked with -inf
    got = oracle.indexer_score(_f16(q), w, _f16(k), _one_seq(3, [1]), False, ld=3)
    assert got[0, :2].tolist() == [1.25, -0.5] and got[0, 2] == -np.inf


def test_single_head_unit_weight_is_relu_of_dot():
    rng = np.random.default_rng(0)
    k = _f16(rng.standard_normal((50, 128)) / 11)
    q = _f16(rng.standard_normal((1, 1, 128)) / 11)
    got = oracle.indexer_score(q, np.ones((1, 1), np.float32), k, _one_seq(50, [49]), False)[0]
    dots = k.astype(np.float64) @ q[0, 0].astype(np.float64)
    assert np.allclose(got, np.maximum(dots, 0), rtol=1e-14, atol=1e-16)
    neg = oracle.indexer_score(q, -np.ones((1, 1), np.float32), k, _one_seq(50, [49]), False)[0]
    assert np.allclose(neg, -np.maximum(dots, 0), rtol=1e-14, atol=1e-16)
    assert (neg <= 0).all() and (got >= 0).all()


def test_against_dense_numpy_multihead():
    rng = np.random.default_rng(1)
    H_I, L = 6, 70
    k = _f16(rng.standard_normal((L, 128)) / 11)
    q = _f16(rng.standard_normal((3, H_I, 128)) / 11)
    w = (rng.standard_normal((3, H_I)) / 3).astype(np.float32)
    pos = [10, 41, 69]
    got = oracle.indexer_score(q, w, k, _one_seq(L, pos), False, ld=L)
    d = np.einsum("thd,sd->ths", q.astype(np.float64), k.astype(np.float64))
    ref = np.einsum("th,ths->ts", w.astype(np.float64), np.maximum(d, 0))
    for t, p in enumerate(pos):
        assert np.allclose(got[t, :p + 1], ref[t, :p + 1], rtol=1e-13, atol=1e-15)
        assert np.all(got[t, p + 1:] == -np.inf)


def test_weight_scale_scales_scores_and_keeps_selection():
    rng = np.random.default_rng(2)
    k = _f16(rng.standard_normal((300, 128)) / 11)
    q = _f16(rng.standard_normal((1, 4, 128)) / 11)
    w = (rng.standard_normal((1, 4)) / 2).astype(np.float32)
    b = _one_seq(300, [299])
    a = oracle.indexer_score(q, w, k, b, False)
    c = oracle.indexer_score(q, (w * 4).astype(np.float32), k, b, False)
    assert np.allclose(c, 4 * a, rtol=1e-14, atol=0)
    assert np.array_equal(oracle.topk(a, [299], 32), oracle.topk(c, [299], 32))


def test_multi_sequence_uses_own_cache_rows():
    wl = S.decode_workload("t", 3, [20, 33], H_I=4, H=8, top_k=8)
    inp = S.make_inputs(wl, parts=("k_cache", "q_idx", "w"))
    got = oracle.indexer_score(inp.q_idx, inp.w, inp.k_cache, oracle.Batch.of(wl), False, ld=33)
    for t in range(2):
        off, L = wl.kv_off[t], wl.kv_len[t]
        solo = oracle.indexer_score(inp.q_idx[t:t + 1], inp.w[t:t + 1],
                                    inp.k_cache[off:off + L], _one_seq(L, [L - 1]), False, ld=33)
        assert np.array_equal(got[t], solo[0])


def test_rotation_invariance_within_cache_rounding():
    """Scores with rotated q and k (k stored in fp16) equal the unrotated ones
    up to the fp16 re-rounding of the stored keys."""
    wl = S.decode_workload("t", 5, [500], H_I=8, H=8, top_k=32, hadamard=True)
    inp = S.make_inputs(wl, parts=("k_cache", "q_idx", "w"))
    b = oracle.Batch.of(wl)
    H = scipy.linalg.hadamard(128) / np.sqrt(128)
    k_rot = (inp.k_cache.astype(np.float64) @ H.T).astype(np.float16)
    plain = oracle.indexer_score(inp.q_idx, inp.w, inp.k_cache, b, False)
    rot = oracle.indexer_score(inp.q_idx, inp.w, k_rot, b, True)
    # bound: each stored key element moves by at most half an fp16 ulp
    kerr = np.abs(k_rot.astype(np.float64) - inp.k_cache.astype(np.float64) @ H.T)
    qr = np.abs(inp.q_idx[0].astype(np.float64) @ H.T)          # |H q| per head
    bound = np.abs(inp.w[0]).astype(np.float64) @ (qr @ kerr.T)  # per key
    assert np.all(np.abs(rot - plain)[0] <= bound * (1 + 1e-9) + 1e-15)
    assert np.max(np.abs(rot - plain)) > 0        # the rounding really differs
    assert np.allclose(rot, plain, rtol=0, atol=1e-3 * np.abs(plain).max())


def test_rejects_bad_sizes():
    k = np.zeros((4, 128), np.float16)
    w = np.ones((1, 1), np.float32)
    with pytest.raises(ValueError):      # row too short for position 3
        oracle.indexer_score(np.zeros((1, 1, 128), np.float16), w, k, _one_seq(4, [3]), False, ld=3)
    with pytest.raises(ValueError):      # no heads
        oracle.indexer_score(np.zeros((1, 0, 128), np.float16), np.zeros((1, 0), np.float32), k,
                             _one_seq(4, [3]), False)
