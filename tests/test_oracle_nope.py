"""Pins of the oracle's MLA-NoPE sparse attention.

vllm-rdna PR #2 "Glm5Next (GLM-5.3-Flash) on gfx1030": the DSA layers are
MLA-NoPE -- the 512-d kv latent is cached per token and no RoPE is applied
anywhere, so in the absorbed form a score is sm_scale * q_lat . c[0:512] and
the output is the softmax-weighted sum of the selected latent rows.

(a) It is the rope form (already pinned against scipy, dense attention and
    the unabsorbed form) with a zero rope query: the rope tail then adds
    nothing, whatever the rows' tails hold.
(b) Special cases: one selected row returns that row and its own score as
    the log-sum-exp; rows with equal scores average; a row with no entry
    gives zero and -inf.
"""
import numpy as np
import pytest

import dsa_synth as S
import oracle


def _bf16(x):
    return S.f64_to_bf16_bits(np.asarray(x, np.float64))


def _deq(b):
    return S.bf16_bits_to_f32(b).astype(np.float64)


def _case(L=120, H=5, pos=(119, 60, 7), seed=3):
    wl = S.Workload("n", seed, [L], list(pos), [0, len(pos)], H_I=4, H=H, top_k=8)
    inp = S.make_inputs(wl, parts=("q_lat", "q_rope", "kv_cache"))
    return wl, inp


def test_equals_the_rope_form_with_a_zero_rope_query():
    wl, inp = _case()
    b = oracle.Batch.of(wl)
    rng = np.random.default_rng(5)
    idx = np.full((3, 24), -1, np.int32)
    for t, p in enumerate(wl.q_pos):
        n = min(24, p + 1)
        idx[t, :n] = np.sort(rng.choice(p + 1, n, replace=False))
    ql = _deq(inp.q_lat)
    zero_rope = np.zeros(inp.q_rope.shape, np.float64)
    ro, rl = oracle.sparse_attn_f64(ql, zero_rope, inp.kv_cache, b, idx, 1 / 16)
    latent = np.ascontiguousarray(inp.kv_cache[:, :512])
    no, nl = oracle.sparse_attn_nope_f64(ql, latent, b, idx, 1 / 16)
    assert np.array_equal(no, ro) and np.array_equal(nl, rl)
    # bf16 queries go through the same arithmetic
    bo, bl = oracle.sparse_attn_nope(inp.q_lat, latent, b, idx, 1 / 16)
    assert np.array_equal(bo, no) and np.array_equal(bl, nl)


def test_single_row_equal_scores_and_empty_rows():
    L, H = 40, 2
    wl = S.Workload("n", 0, [L], [39, 39, 39], [0, 3], H_I=4, H=H, top_k=4)
    b = oracle.Batch.of(wl)
    rng = np.random.default_rng(9)
    latent = _bf16(rng.standard_normal((L, 512)) / 8)
    q = _bf16(rng.standard_normal((3, H, 512)) / 8)
    idx = np.array([[17, -1, -1, -1],          # one row
                    [3, 30, -1, -1],           # two rows, scores made equal below
                    [-1, -1, -1, -1]], np.int32)
    ql = _deq(q)
    C = _deq(latent)
    # token 1: a query orthogonal to both rows' latents gives equal (zero) scores
    A = np.stack([C[3], C[30]], axis=1)
    for h in range(H):
        ql[1, h] -= A @ np.linalg.solve(A.T @ A, A.T @ ql[1, h])
    out, lse = oracle.sparse_attn_nope_f64(ql, latent, b, idx, 0.25)
    for h in range(H):
        assert np.allclose(out[0, h], C[17], rtol=0, atol=1e-15)
        assert abs(lse[0, h] - 0.25 * (ql[0, h] @ C[17])) < 1e-12
        z = 0.25 * np.array([ql[1, h] @ C[3], ql[1, h] @ C[30]])
        assert np.all(np.abs(z) < 1e-12)
        assert np.allclose(out[1, h], (C[3] + C[30]) / 2, rtol=0, atol=1e-12)
        assert abs(lse[1, h] - np.log(2.0)) < 1e-12
        assert np.all(out[2, h] == 0) and lse[2, h] == -np.inf


def test_non_causal_index_is_rejected():
    wl, inp = _case(L=50, H=2, pos=(20,))
    idx = np.array([[3, 21, -1]], np.int32)        # 21 > q_pos = 20
    latent = np.ascontiguousarray(inp.kv_cache[:, :512])
    with pytest.raises(ValueError, match="code -2"):
        oracle.sparse_attn_nope(inp.q_lat, latent, oracle.Batch.of(wl), idx, 0.1)
