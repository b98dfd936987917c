"""The comparison rules of the GPU parity tests are sharp enough to catch the
mistakes they are meant to catch.  Each mistake is planted on the CPU, in the
oracle's inputs, and must fail its rule; the arithmetic the kernels actually
use must pass it.

ik_llama_opt commit log, "Add GLM-5.2/DeepSeek-V3.2 DSA lightning indexer":
the Walsh-Hadamard rotation is orthonormal, so rotated and unrotated scores
are equal; the kernel keeps the rotated query in two fp16 parts so that the
rotation does not cost it precision.
"""
import math

import numpy as np
import pytest
import scipy.linalg

import dsa_synth as S
import oracle
from _helpers import check_attention, check_scores, score_bound, score_tolerance


def _rotated_row():
    wl = S.decode_workload("rule", 81, [3000], H_I=64, H=8, top_k=16, hadamard=True)
    inp = S.make_inputs(wl, parts=("k_cache", "q_idx", "w"))
    ob = oracle.Batch.of(wl)
    exact = oracle.indexer_score(inp.q_idx, inp.w, inp.k_cache, ob, True)[0]
    A = score_tolerance(inp.q_idx, inp.w, inp.k_cache, wl, 0, True)
    q_rot = inp.q_idx[0].astype(np.float64) @ (scipy.linalg.hadamard(128) / math.sqrt(128)).T
    return wl, inp, ob, exact, A, q_rot


def test_single_rounded_rotated_query_fails_the_score_rule():
    wl, inp, ob, exact, A, q_rot = _rotated_row()
    # the mistake: rotate, then round the query to fp16 once (no lo part)
    single = oracle.indexer_score(q_rot.astype(np.float16)[None], inp.w, inp.k_cache, ob, False)[0]
    n_bad = int(np.count_nonzero(np.abs(single - exact) > score_bound(exact, A)))
    assert n_bad > 100, n_bad
    with pytest.raises(AssertionError):
        check_scores(single, exact, A, name="rule pin")


def test_hi_lo_rotated_query_passes_the_score_rule():
    wl, inp, ob, exact, A, q_rot = _rotated_row()
    # the kernel's form: the float32 rotation carried as hi + lo fp16 parts
    q32 = q_rot.astype(np.float32)
    hi = q32.astype(np.float16)
    lo = (q32 - hi.astype(np.float32)).astype(np.float16)
    q_eff = hi.astype(np.float64) + lo.astype(np.float64)
    k = inp.k_cache[:3000].astype(np.float64)
    hilo = inp.w[0].astype(np.float64) @ np.maximum(q_eff @ k.T, 0.0)
    check_scores(hilo, exact, A, name="rule pin")


def test_dropping_selected_rows_fails_the_attention_rule():
    """64 of a token's 2048 selected rows left out moves the output by far
    less than 2e-3 (the outputs themselves are a few 1e-3), but not by less
    than 1e-2 of the largest output."""
    wl = S.decode_workload("rule_a", 82, [8192], H_I=4, H=64, top_k=2048)
    inp = S.make_inputs(wl, parts=("q_lat", "q_rope", "kv_cache"))
    rng = np.random.default_rng(82)
    idx = oracle.topk(rng.standard_normal((1, 8192)), wl.q_pos, 2048)
    ob = oracle.Batch.of(wl)
    ref_o, ref_l = oracle.sparse_attn(inp.q_lat, inp.q_rope, inp.kv_cache, ob, idx, wl.sm_scale)
    short = idx.copy()
    short[0, rng.choice(2048, 64, replace=False)] = -1
    bad_o, bad_l = oracle.sparse_attn(inp.q_lat, inp.q_rope, inp.kv_cache, ob, short, wl.sm_scale)
    assert np.abs(bad_o - ref_o).max() < 2e-3             # the absolute bound alone would pass it
    with pytest.raises(AssertionError):
        check_attention(bad_o, None, ref_o, None, name="rule pin")
