"""The seeded generator: determinism, per-element regeneration, distribution."""
import math

import numpy as np

import dsa_synth as S


def test_splitmix64_known_values():
    # SplitMix64 seeded with 0: the published first outputs of the sequence
    # x_n = 0x9E3779B97F4A7C15 * n, finalised.
    out = S.splitmix64(np.array([0, 0x9E3779B97F4A7C15], dtype=np.uint64))
    assert int(out[0]) == 0xE220A8397B1DCDAF
    assert int(out[1]) == 0x6E789E6AA1B965F4


def test_whole_tensor_equals_elementwise_regeneration():
    a = S.normal(3, S.TID_Q_IDX, (5, 7, 128), 0.25, "f16")
    e = np.array([0, 17, 4479], dtype=np.uint64)
    z = S.standard_normal_at(3, S.TID_Q_IDX, e) * 0.25
    assert np.array_equal(a.reshape(-1)[e.astype(np.int64)], z.astype(np.float16))


def test_threaded_chunks_match_single_chunk():
    a = S.normal(9, S.TID_KV_CACHE, (3000, 576), 1 / 24, "bf16", chunk=1 << 16)
    b = S.normal(9, S.TID_KV_CACHE, (3000, 576), 1 / 24, "bf16", chunk=1 << 30)
    assert np.array_equal(a, b)


def test_distribution_moments():
    z = S.standard_normal_at(0, 1, np.arange(1 << 20, dtype=np.uint64))
    assert abs(z.mean()) < 5e-3
    assert abs(z.var() - 1) < 5e-3
    assert abs((z ** 4).mean() - 3) < 3e-2       # Gaussian kurtosis


def test_tensors_and_seeds_do_not_overlap():
    a = S.standard_normal_at(1, 3, np.arange(1000, dtype=np.uint64))
    b = S.standard_normal_at(1, 4, np.arange(1000, dtype=np.uint64))
    c = S.standard_normal_at(2, 3, np.arange(1000, dtype=np.uint64))
    assert not np.allclose(a, b) and not np.allclose(a, c)


def test_workloads():
    w = S.config(1)
    assert (w.B, w.T, w.H_I, w.H, w.top_k, w.q_pos) == (1, 1, 4, 8, 64, [255])
    w = S.config(2)
    assert w.cache_rows == 8 * 8192 and w.kv_off[3] == 3 * 8192 and w.max_kv == 8192
    w = S.config(3)
    assert w.B == 32 and w.hadamard and all(4096 <= L <= 65536 for L in w.kv_len)
    assert w.kv_len == S.ragged_lengths(2, 32)
    w = S.config(4)
    assert w.T == 4096 and w.q_pos[0] == 4096 and w.q_pos[-1] == 8191 and w.cache_rows == 8192
    w = S.config(5)
    assert w.T == 16384 and w.q_pos[0] == 114688 and w.cache_rows == 131072
    assert abs(w.sm_scale - 1 / math.sqrt(192)) < 1e-15
