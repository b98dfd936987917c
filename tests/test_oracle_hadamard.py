"""Pins of the oracle's Walsh-Hadamard transform and key append.

The transform is orthonormal and score preserving, (Hq).(Hk) = q.k
(ik_llama_opt commit log, "Add GLM-5.2/DeepSeek-V3.2 DSA lightning indexer",
simplifications; and "decode-correct via persistent indexer-K cache").
"""
import numpy as np
import pytest
import scipy.linalg

import dsa_synth as S
import oracle


def test_matches_scipy_sylvester_matrix():
    H = scipy.linalg.hadamard(128).astype(np.float64) / np.sqrt(128)
    rng = np.random.default_rng(0)
    for _ in range(20):
        x = rng.standard_normal(128)
        assert np.allclose(oracle.fwht128(x), H @ x, rtol=0, atol=1e-13)


def test_involution_and_unit_vectors():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(128)
    assert np.allclose(oracle.fwht128(oracle.fwht128(x)), x, rtol=0, atol=1e-13)
    e0 = np.zeros(128)
    e0[0] = 1
    assert np.allclose(oracle.fwht128(e0), np.full(128, 1 / np.sqrt(128)), rtol=0, atol=1e-15)
    # e_j maps to row j of the Sylvester matrix: signs (-1)^popcount(i & j)
    for j in (1, 5, 64, 127):
        ej = np.zeros(128)
        ej[j] = 1
        sign = np.array([(-1) ** bin(i & j).count("1") for i in range(128)])
        assert np.allclose(oracle.fwht128(ej) * np.sqrt(128), sign, rtol=0, atol=1e-13)


def test_inner_products_preserved():
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    assert abs(oracle.fwht128(q) @ oracle.fwht128(k) - q @ k) < 1e-12


@pytest.mark.parametrize("hadamard", [False, True])
@pytest.mark.parametrize("kdt", ["f32", "f16"])
def test_k_append_rows_and_rounding(hadamard, kdt):
    wl = S.decode_workload("t", 7, [40, 9, 130], H_I=4, H=8, top_k=16)
    inp = S.make_inputs(wl, parts=("k_cache", "k_new"))
    kn = inp.k_new if kdt == "f32" else inp.k_new.astype(np.float16)
    kc = inp.k_cache.copy()
    oracle.k_append(kn, oracle.Batch.of(wl), kc, hadamard)
    H = scipy.linalg.hadamard(128) / np.sqrt(128)
    touched = set()
    for t, (off, p) in enumerate(zip(wl.kv_off, wl.q_pos)):
        x = kn[t].astype(np.float64)
        want = (H @ x if hadamard else x).astype(np.float16)
        assert np.array_equal(kc[off + p], want)
        touched.add(off + p)
    others = [r for r in range(wl.cache_rows) if r not in touched]
    assert np.array_equal(kc[others], inp.k_cache[others])
