"""GPU parity of each step through the C ABI against the CPU oracle.

Sizes span several 128-key tiles and ragged tails; cases cover the degenerate
inputs of each step (ties, signed zeros, short rows, padding entries).
"""
import math

import numpy as np
import pytest

import dsa_synth as S
import oracle
from _helpers import (assert_sorted_unique, check_attention, check_scores, dev_batch, score_tolerance, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    from dsa_sparse_attention_score_gb300 import build
    build.build()
    import dsa_sparse_attention_score_gb300 as m
    return m


def _status_clean(dsa, ws):
    assert dsa.dsa_read_device_status(ws) == 0


# ----------------------------------------------------------------- k_append

@pytest.mark.parametrize("hadamard", [False, True])
@pytest.mark.parametrize("kdt", ["f32", "f16"])
def test_k_append_bit_exact(dsa, hadamard, kdt):
    import torch
    wl = S.decode_workload("app", 21, [7, 130, 513, 64], H_I=4, H=8, top_k=8)
    inp = S.make_inputs(wl, parts=("k_cache", "k_new"))
    kn = inp.k_new if kdt == "f32" else inp.k_new.astype(np.float16)
    ref = inp.k_cache.copy()
    oracle.k_append(kn, oracle.Batch.of(wl), ref, hadamard)
    kc = to_dev(inp.k_cache)
    b = dev_batch(wl)
    ws = dsa.workspace(dsa.DSA_OP_K_APPEND, b)
    dsa.dsa_indexer_k_append(to_dev(kn), b, kc, hadamard, ws)
    got = kc.cpu().numpy()
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))
    _status_clean(dsa, ws)


def test_k_append_prefill_rows(dsa):
    wl = S.prefill_workload("app2", 22, 100, 77, H_I=4, H=8, top_k=8)
    inp = S.make_inputs(wl, parts=("k_cache", "k_new"))
    ref = inp.k_cache.copy()
    oracle.k_append(inp.k_new, oracle.Batch.of(wl), ref, True)
    kc = to_dev(inp.k_cache)
    b = dev_batch(wl)
    ws = dsa.workspace(dsa.DSA_OP_K_APPEND, b)
    dsa.dsa_indexer_k_append(to_dev(inp.k_new), b, kc, True, ws)
    assert np.array_equal(kc.cpu().numpy().view(np.uint16), ref.view(np.uint16))


# ----------------------------------------------------------------- score

SCORE_CASES = [
    # name, lengths / prefill spec, H_I, hadamard
    ("decode_HI4", dict(lengths=[40, 300, 1000]), 4, False),
    ("decode_HI32", dict(lengths=[129, 2000, 777]), 32, False),
    ("decode_HI64_rot", dict(lengths=[1500, 256, 90]), 64, True),
    ("decode_HI48", dict(lengths=[640, 1025]), 48, False),
    ("prefill_HI64", dict(cached=500, T=70), 64, False),
    # two MMA steps per key tile; each last group takes one (g <= tokens per step)
    ("prefill_HI64_tail2", dict(cached=200, T=10), 64, False),
    ("prefill_HI16", dict(cached=700, T=45), 16, False),
    ("prefill_HI48", dict(cached=333, T=23), 48, False),
    ("prefill_HI16_rot", dict(cached=300, T=37), 16, True),
    ("prefill_HI32_rot", dict(cached=1000, T=9), 32, True),
]


def _score_wl(spec, H_I, hadamard, seed):
    if "lengths" in spec:
        return S.decode_workload("s", seed, spec["lengths"], H_I=H_I, H=8, top_k=16, hadamard=hadamard)
    return S.prefill_workload("s", seed, spec["cached"], spec["T"], H_I=H_I, H=8, top_k=16,
                              hadamard=hadamard)


@pytest.mark.parametrize("name,spec,H_I,hadamard", SCORE_CASES, ids=[c[0] for c in SCORE_CASES])
def test_indexer_score_matches_oracle(dsa, name, spec, H_I, hadamard):
    import torch
    wl = _score_wl(spec, H_I, hadamard, seed=31)
    inp = S.make_inputs(wl, parts=("k_cache", "q_idx", "w"))
    ld = wl.max_kv + 37                      # extra columns must read -inf
    ref = oracle.indexer_score(inp.q_idx, inp.w, inp.k_cache, oracle.Batch.of(wl), hadamard, ld=ld)
    b = dev_batch(wl)
    ws = dsa.workspace(dsa.DSA_OP_INDEXER_SCORE, b)
    scores = torch.full((wl.T, ld), float("nan"), device="cuda")
    dsa.dsa_indexer_score(to_dev(inp.q_idx), to_dev(inp.w), to_dev(inp.k_cache), b, hadamard, scores, ws)
    got = scores.cpu().numpy()
    for t in range(wl.T):
        p = wl.q_pos[t]
        A = score_tolerance(inp.q_idx, inp.w, inp.k_cache, wl, t, hadamard)
        check_scores(got[t, :p + 1], ref[t, :p + 1], A)
        assert np.all(np.isneginf(got[t, p + 1:])), f"row {t}: masked tail not -inf"
    _status_clean(dsa, ws)


# ----------------------------------------------------------------- top-k

def _topk_case(kind, rng):
    if kind == "random":
        L, pos = 5000, [4999, 3001, 2047, 2048, 100]
        s = rng.standard_normal((len(pos), L)).astype(np.float32)
    elif kind == "ties":
        L, pos = 4097, [4096, 4000, 2500]
        s = (rng.integers(-4, 5, (len(pos), L)) * 0.25).astype(np.float32)
    elif kind == "all_equal":
        L, pos = 3000, [2999, 2048]
        s = np.full((len(pos), L), 0.125, np.float32)
    elif kind == "signed_zero":
        L, pos = 3000, [2999, 2500]
        s = np.where(rng.random((len(pos), L)) < 0.5, np.float32(0.0), np.float32(-0.0))
        s[:, ::97] = 1.0
    elif kind == "neg_inf":
        L, pos = 2600, [2599]
        s = rng.standard_normal((1, L)).astype(np.float32)
        s[0, ::2] = -np.inf
    elif kind == "long_row":
        L, pos = 131072, [131071, 70000]
        s = rng.standard_normal((len(pos), L)).astype(np.float32)
    elif kind == "cluster3":                    # aligned rows spread over a 3-CTA cluster
        L, pos = 20000, [19999, 12000, 8191, 8192, 3000, 100]
        s = rng.standard_normal((len(pos), L)).astype(np.float32)
        s[:, 5000:5100] = 0.5                   # a run of ties inside one CTA's share
    elif kind in ("cluster5", "cluster7"):      # cluster sizes that do not divide the histogram
        L = 70000 if kind == "cluster5" else 110000
        pos = [L - 1, L // 2, 16384, 16383, 5000]
        s = (rng.integers(-64, 64, (len(pos), L)) * 2.0 ** -6).astype(np.float32)   # many ties
    elif kind == "beyond_cluster":              # longer than a cluster holds: streaming path
        L, pos = 140000, [139999, 131072]
        s = rng.standard_normal((len(pos), L)).astype(np.float32)
    elif kind == "beyond_cluster_unaligned":    # and not 16-byte aligned: shared-memory path
        L, pos = 140001, [140000, 131072]
        s = rng.standard_normal((len(pos), L)).astype(np.float32)
    elif kind == "unaligned_cluster5":          # a row stride the 16-byte path cannot take: cluster of 5
        L = 70001
        pos = [L - 1, L // 2, 16384, 16383, 5000]
        s = (rng.integers(-64, 64, (len(pos), L)) * 2.0 ** -6).astype(np.float32)
    # at least as many long rows as SMs: the one-pass streaming path
    elif kind == "stream_random":
        L = 30000
        pos = [L - 1 - 97 * i for i in range(152)] + [16384, 16383, 9000, 100]
        s = rng.standard_normal((len(pos), L)).astype(np.float32)
        s[:, 5000:5100] = 0.5                   # a run of ties
    elif kind == "stream_all_equal":            # the pass keeps every key: the general path finishes
        L = 40000
        pos = [L - 1 - 13 * i for i in range(160)]
        s = np.full((len(pos), L), 0.125, np.float32)
    elif kind == "stream_sample_miss":          # the sampled keys are the largest: too few kept
        L = 60000
        pos = [L - 1 - 101 * i for i in range(160)]
        s = rng.standard_normal((len(pos), L)).astype(np.float32)
        for t, p in enumerate(pos):
            n = p + 1
            s[t, (np.arange(0, 4096, 20) * n) // 4096] = 100.0
    # few rows of 4097..8192 keys: the one-CTA 16-bit-digit path
    elif kind == "row16_all_equal":             # every key in one bin: the second 16-bit digit
        L, pos = 6000, [5999, 4500, 4097]
        s = np.full((len(pos), L), -0.375, np.float32)
    elif kind == "row16_mixed":                 # -inf, signed zeros and a run of ties around the threshold
        L, pos = 7000, [6999, 6000, 5000, 4097]
        s = rng.standard_normal((len(pos), L)).astype(np.float32)
        s[:, ::3] = -np.inf
        s[:, 1::7] = np.where(rng.random((len(pos), len(range(1, L, 7)))) < 0.5, np.float32(0.0), np.float32(-0.0))
        s[:, 2000:2040] = 0.6745
    elif kind == "narrow":                      # distinct values that share high bits
        L, pos = 9000, [8999]
        s = (1.0 + rng.integers(0, 1 << 12, (1, L)) * 2.0 ** -23).astype(np.float32)
    else:
        raise ValueError(kind)
    return s, pos


@pytest.mark.parametrize("kind", ["random", "ties", "all_equal", "signed_zero", "neg_inf", "long_row", "narrow",
                                  "cluster3", "cluster5", "cluster7", "beyond_cluster", "beyond_cluster_unaligned",
                                  "unaligned_cluster5", "row16_all_equal", "row16_mixed",
                                  "stream_random", "stream_all_equal", "stream_sample_miss"])
@pytest.mark.parametrize("k", [1, 2048])
def test_topk_bit_exact_on_oracle_scores(dsa, kind, k):
    import torch
    rng = np.random.default_rng(abs(hash((kind, k))) % (1 << 31))
    s, pos = _topk_case(kind, rng)
    T, L = s.shape
    ref = oracle.topk(s.astype(np.float64), pos, k)
    b = dsa.Batch.from_host([0, T], pos, [0], cache_rows=L, max_q_per_seq=T, max_kv=L)
    ws = dsa.workspace(dsa.DSA_OP_TOPK, b, k=k)
    idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    dsa.dsa_topk(to_dev(s), b, k, idx, ws)
    got = idx.cpu().numpy()
    assert np.array_equal(got, ref)
    for t in range(T):
        assert_sorted_unique(got[t], pos[t] + 1)
    _status_clean(dsa, ws)


@pytest.mark.parametrize("kind", ["stream_random", "stream_sample_miss"])
@pytest.mark.parametrize("k", [2049, 4096])
def test_topk_streaming_large_k(dsa, kind, k):
    """k above 2048 takes the streaming kernel's 512-thread configuration."""
    test_topk_bit_exact_on_oracle_scores(dsa, kind, k)


def test_topk_short_rows_and_k_boundaries(dsa):
    import torch
    rng = np.random.default_rng(5)
    L = 3000
    pos = [0, 5, 2046, 2047, 2048, 2999]
    s = rng.standard_normal((len(pos), L)).astype(np.float32)
    b = dsa.Batch.from_host([0, len(pos)], pos, [0], cache_rows=L, max_q_per_seq=len(pos), max_kv=L)
    for k in (2048, 1000, 3000):
        ref = oracle.topk(s.astype(np.float64), pos, k)
        ws = dsa.workspace(dsa.DSA_OP_TOPK, b, k=k)
        idx = torch.empty((len(pos), k), dtype=torch.int32, device="cuda")
        dsa.dsa_topk(to_dev(s), b, k, idx, ws)
        assert np.array_equal(idx.cpu().numpy(), ref), k


# ----------------------------------------------------------------- attention

ATTN_CASES = [
    # name, lengths, H, k, scores-seed
    ("decode_H64_k256", [300, 700], 64, 256),
    ("decode_H8_k64", [256], 8, 64),
    ("decode_H40_k100_partial_tile", [500, 129, 1000], 40, 100),
    ("decode_H64_k2048_padded", [1500, 2600], 64, 2048),
    ("decode_H16_k1", [50, 60], 16, 1),
    # more than 64 heads: two head groups of 64 per token
    ("decode_H128_k2048", [3000, 2500], 128, 2048),
    ("decode_H72_k300_partial_group", [700, 420], 72, 300),
]


@pytest.mark.parametrize("name,lengths,H,k", ATTN_CASES, ids=[c[0] for c in ATTN_CASES])
def test_sparse_attention_matches_oracle(dsa, name, lengths, H, k):
    import torch
    wl = S.decode_workload("a", 41, lengths, H_I=4, H=H, top_k=k)
    inp = S.make_inputs(wl, parts=("q_lat", "q_rope", "kv_cache"))
    rng = np.random.default_rng(7)
    scores = rng.standard_normal((wl.T, wl.max_kv))
    idx = oracle.topk(scores, wl.q_pos, k)
    ob = oracle.Batch.of(wl)
    ref_o, ref_l = oracle.sparse_attn(inp.q_lat, inp.q_rope, inp.kv_cache, ob, idx, wl.sm_scale)
    b = dev_batch(wl)
    ws = dsa.workspace(dsa.DSA_OP_SPARSE_ATTN, b, H=H, k=k)
    out = torch.full((wl.T, H, 512), float("nan"), device="cuda")
    lse = torch.full((wl.T, H), float("nan"), device="cuda")
    dsa.dsa_sparse_mla_attn(to_dev(inp.q_lat), to_dev(inp.q_rope), to_dev(inp.kv_cache), b,
                            to_dev(idx), wl.sm_scale, out, lse, ws)
    go, gl = out.cpu().numpy(), lse.cpu().numpy()
    check_attention(go, gl, ref_o, ref_l)
    _status_clean(dsa, ws)


@pytest.mark.parametrize("H", [16, 96])
def test_sparse_attention_many_tokens_no_split(dsa, H):
    """Enough tokens that each CTA walks all tiles of its token (online softmax)."""
    import torch
    wl = S.prefill_workload("a2", 43, 600, 320, H_I=4, H=H, top_k=400)
    inp = S.make_inputs(wl, parts=("q_lat", "q_rope", "kv_cache"))
    rng = np.random.default_rng(8)
    scores = rng.standard_normal((wl.T, wl.max_kv)) * 3
    idx = oracle.topk(scores, wl.q_pos, wl.top_k)
    ref_o, ref_l = oracle.sparse_attn(inp.q_lat, inp.q_rope, inp.kv_cache, oracle.Batch.of(wl), idx,
                                      wl.sm_scale)
    b = dev_batch(wl)
    ws = dsa.workspace(dsa.DSA_OP_SPARSE_ATTN, b, H=H, k=wl.top_k)
    out = torch.empty((wl.T, H, 512), device="cuda")
    lse = torch.empty((wl.T, H), device="cuda")
    dsa.dsa_sparse_mla_attn(to_dev(inp.q_lat), to_dev(inp.q_rope), to_dev(inp.kv_cache), b,
                            to_dev(idx), wl.sm_scale, out, lse, ws)
    check_attention(out.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l)


def test_sparse_attention_rescale_and_padding_entries(dsa):
    """Large logits force the running maximum to move between tiles; -1
    entries anywhere in the list are skipped; an all -1 row gives zeros."""
    import torch
    wl = S.decode_workload("a3", 44, [900, 900, 900], H_I=4, H=64, top_k=512)
    inp = S.make_inputs(wl, parts=("q_lat", "q_rope", "kv_cache"))
    q_lat = S.f64_to_bf16_bits(S.bf16_bits_to_f32(inp.q_lat).astype(np.float64) * 40)   # sharp softmax
    rng = np.random.default_rng(9)
    idx = np.stack([rng.permutation(900)[:512] for _ in range(3)]).astype(np.int32)
    idx[0, ::3] = -1
    idx[2, :] = -1
    ob = oracle.Batch.of(wl)
    ref_o, ref_l = oracle.sparse_attn(q_lat, inp.q_rope, inp.kv_cache, ob, idx, wl.sm_scale)
    b = dev_batch(wl)
    ws = dsa.workspace(dsa.DSA_OP_SPARSE_ATTN, b, H=64, k=512)
    out = torch.empty((3, 64, 512), device="cuda")
    lse = torch.empty((3, 64), device="cuda")
    dsa.dsa_sparse_mla_attn(to_dev(q_lat), to_dev(inp.q_rope), to_dev(inp.kv_cache), b, to_dev(idx),
                            wl.sm_scale, out, lse, ws)
    go, gl = out.cpu().numpy(), lse.cpu().numpy()
    check_attention(go[:2], gl[:2], ref_o[:2], ref_l[:2], name="attention (sharp)",
                    lse_tol=1e-3 * max(1.0, np.abs(ref_l[:2]).max() / 100))
    assert np.all(go[2] == 0) and np.all(np.isneginf(gl[2]))
    _status_clean(dsa, ws)


def test_sparse_attention_flags_out_of_range_index(dsa):
    import torch
    wl = S.decode_workload("a4", 45, [300], H_I=4, H=8, top_k=16)
    inp = S.make_inputs(wl, parts=("q_lat", "q_rope", "kv_cache"))
    idx = np.arange(16, dtype=np.int32)[None, :].copy()
    idx[0, 3] = 5000                       # beyond the visible range: skipped and flagged
    ok = idx.copy()
    ok[0, 3] = -1
    ref_o, _ = oracle.sparse_attn(inp.q_lat, inp.q_rope, inp.kv_cache, oracle.Batch.of(wl), ok, wl.sm_scale)
    b = dev_batch(wl)
    ws = dsa.workspace(dsa.DSA_OP_SPARSE_ATTN, b, H=8, k=16)
    out = torch.empty((1, 8, 512), device="cuda")
    dsa.dsa_sparse_mla_attn(to_dev(inp.q_lat), to_dev(inp.q_rope), to_dev(inp.kv_cache), b, to_dev(idx),
                            wl.sm_scale, out, None, ws)
    check_attention(out.cpu().numpy(), None, ref_o, None)
    assert dsa.dsa_read_device_status(ws) == dsa.DSA_DEV_BAD_INDEX
    assert dsa.dsa_read_device_status(ws) == 0      # read clears


def test_bad_positions_are_flagged_not_faulted(dsa):
    import torch
    wl = S.decode_workload("bp", 46, [100, 100], H_I=4, H=8, top_k=16)
    inp = S.make_inputs(wl)
    b = dsa.Batch.from_host(wl.cu_q, [99, 150], wl.kv_off, wl.cache_rows, max_q_per_seq=1, max_kv=100)
    ws = dsa.workspace(dsa.DSA_OP_DECODE, b, 4, 8, 16)
    out = torch.empty((2, 8, 512), device="cuda")
    dsa.dsa_decode(to_dev(inp.k_new), to_dev(inp.q_idx), to_dev(inp.w), to_dev(inp.q_lat), to_dev(inp.q_rope),
                   to_dev(inp.k_cache), to_dev(inp.kv_cache), b, 16, wl.sm_scale, False, out, None, None, ws)
    assert dsa.dsa_read_device_status(ws) & dsa.DSA_DEV_BAD_POSITION
    assert np.isfinite(out[0].cpu().numpy()).all()
