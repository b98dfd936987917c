"""Pins of the oracle's sparse MLA attention.

(a) With top_k >= n the sparse path is dense causal attention (ik_llama_opt
    commit log: the indexer is an exact no-op when top_k >= n_tokens).
(c) The absorbed latent form equals the unabsorbed form that expands each
    cached row through kv_b (ds4 PR #523, milestone M3, glm_mla_attention_one:
    per-row 448 = 192 nope-key + 256 value dims per head, rope tail from the
    row's last 64 values, one softmax over the candidates; absorbed wk_b/wv_b
    per ik_llama_opt "MLA tensor parallelism under -sm graph").
"""
import numpy as np
import pytest
import scipy.special

import dsa_synth as S
import oracle


def _bf16(x):
    return S.f64_to_bf16_bits(np.asarray(x, np.float64))


def _deq(b):
    return S.bf16_bits_to_f32(b).astype(np.float64)


def _wl(L, H=4, T_pos=None, seed=11):
    pos = T_pos if T_pos is not None else [L - 1]
    return S.Workload("t", seed, [L], pos, [0, len(pos)], H_I=4, H=H, top_k=8)


def test_matches_scipy_softmax_on_given_rows():
    wl = _wl(90, H=3, T_pos=[89, 40])
    inp = S.make_inputs(wl, parts=("q_lat", "q_rope", "kv_cache"))
    rng = np.random.default_rng(0)
    idx = np.stack([np.sort(rng.choice(90, 20, replace=False)),
                    np.concatenate([np.sort(rng.choice(41, 15, replace=False)), -np.ones(5, int)])])
    out, lse = oracle.sparse_attn(inp.q_lat, inp.q_rope, inp.kv_cache, oracle.Batch.of(wl), idx, 0.3)
    C = _deq(inp.kv_cache)
    for t in range(2):
        rows = idx[t][idx[t] >= 0]
        for h in range(3):
            q = np.concatenate([_deq(inp.q_lat[t, h]), _deq(inp.q_rope[t, h])])
            z = 0.3 * (C[rows] @ q)
            p = scipy.special.softmax(z)
            assert np.allclose(out[t, h], p @ C[rows, :512], rtol=1e-12, atol=1e-15)
            assert abs(lse[t, h] - scipy.special.logsumexp(z)) < 1e-12


def test_dense_equivalence_when_k_covers_all_visible():
    wl = _wl(64, H=4, T_pos=[63, 20, 0])
    inp = S.make_inputs(wl, parts=("q_lat", "q_rope", "kv_cache"))
    b = oracle.Batch.of(wl)
    scores = np.random.default_rng(1).standard_normal((3, 64))
    idx = oracle.topk(scores, wl.q_pos, 64)          # k >= n: every visible position
    ql, qr = _deq(inp.q_lat), _deq(inp.q_rope)
    sp, sl = oracle.sparse_attn_f64(ql, qr, inp.kv_cache, b, idx, 0.1)
    de, dl = oracle.dense_attn_f64(ql, qr, inp.kv_cache, b, 0.1)
    assert np.array_equal(sp, de) and np.array_equal(sl, dl)    # identical, not just close
    # and once the selection bites it is no longer dense
    idx2 = oracle.topk(scores, wl.q_pos, 16)
    sp2, _ = oracle.sparse_attn_f64(ql, qr, inp.kv_cache, b, idx2, 0.1)
    assert not np.allclose(sp2[0], de[0])


def test_single_row_selection_returns_that_row():
    wl = _wl(30, H=2)
    inp = S.make_inputs(wl, parts=("q_lat", "q_rope", "kv_cache"))
    idx = np.array([[-1, 17, -1, -1]], np.int32)
    out, lse = oracle.sparse_attn(inp.q_lat, inp.q_rope, inp.kv_cache, oracle.Batch.of(wl), idx, 0.2)
    C = _deq(inp.kv_cache)
    assert np.array_equal(out[0, 0], C[17, :512]) and np.array_equal(out[0, 1], C[17, :512])
    q = np.concatenate([_deq(inp.q_lat[0, 1]), _deq(inp.q_rope[0, 1])])
    assert abs(lse[0, 1] - 0.2 * C[17] @ q) < 1e-13


def test_identical_rows_return_the_row_and_add_log_n():
    wl = _wl(12, H=2)
    inp = S.make_inputs(wl, parts=("q_lat", "q_rope", "kv_cache"))
    kv = inp.kv_cache.copy()
    kv[:] = kv[5]
    idx = np.array([[0, 3, 7, 11]], np.int32)
    out, lse = oracle.sparse_attn(inp.q_lat, inp.q_rope, kv, oracle.Batch.of(wl), idx, 0.2)
    C = _deq(kv)
    assert np.allclose(out[0, 0], C[5, :512], rtol=1e-15, atol=0)
    _, lse1 = oracle.sparse_attn(inp.q_lat, inp.q_rope, kv, oracle.Batch.of(wl),
                                 np.array([[5, -1, -1, -1]], np.int32), 0.2)
    assert abs(lse[0, 0] - (lse1[0, 0] + np.log(4))) < 1e-12


def test_empty_selection_gives_zero_and_neg_inf():
    wl = _wl(8, H=1)
    inp = S.make_inputs(wl, parts=("q_lat", "q_rope", "kv_cache"))
    out, lse = oracle.sparse_attn(inp.q_lat, inp.q_rope, inp.kv_cache, oracle.Batch.of(wl),
                                  -np.ones((1, 3), np.int32), 0.2)
    assert (out == 0).all() and lse[0, 0] == -np.inf


def test_rejects_non_causal_index():
    wl = _wl(8, H=1, T_pos=[3])
    inp = S.make_inputs(wl, parts=("q_lat", "q_rope", "kv_cache"))
    with pytest.raises(ValueError):
        oracle.sparse_attn(inp.q_lat, inp.q_rope, inp.kv_cache, oracle.Batch.of(wl),
                           np.array([[0, 4]], np.int32), 0.2)


def test_absorbed_equals_unabsorbed():
    """W_UV . o_absorbed == o_unabsorbed with q_lat = W_UK^T q_nope."""
    H, L = 3, 40
    wl = _wl(L, H=H, T_pos=[39, 25])
    inp = S.make_inputs(wl, parts=("q_rope", "kv_cache"))
    W_UK = S.normal(11, S.TID_W_UK, (H, 192, 512), 1 / np.sqrt(512), "f64")
    W_UV = S.normal(11, S.TID_W_UV, (H, 256, 512), 1 / np.sqrt(512), "f64")
    q_nope = S.normal(11, S.TID_Q_NOPE, (2, H, 192), 1 / np.sqrt(192), "f64")
    q_rope = _deq(inp.q_rope)
    rng = np.random.default_rng(3)
    idx = np.stack([np.sort(rng.choice(40, 12, replace=False)), np.sort(rng.choice(26, 12, replace=False))])
    b = oracle.Batch.of(wl)
    un = oracle.unabsorbed_attn(q_nope, q_rope, inp.kv_cache, b, W_UK, W_UV, idx, 1 / np.sqrt(192))
    q_lat = np.einsum("hed,the->thd", W_UK, q_nope)        # absorbed query
    ab, _ = oracle.sparse_attn_f64(q_lat, q_rope, inp.kv_cache, b, idx, 1 / np.sqrt(192))
    lifted = np.einsum("hvd,thd->thv", W_UV, ab)
    assert np.allclose(lifted, un, rtol=0, atol=1e-10)
    assert np.abs(un).max() > 1e-3
    # a transposed up-projection breaks it
    bad = np.einsum("hvd,thd->thv", W_UV[::-1], ab)
    assert not np.allclose(bad, un, atol=1e-6)
