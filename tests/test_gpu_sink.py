"""GPU parity of the attention-sink selection (ik_llama_opt commit log,
"GLM-5.2 DSA indexer: per-sequence attention sink" and "UPDATE 6": the first
n_sink positions of each query's own sequence, counted from its first present
position, always survive the top-k).

dsa_topk_sink is checked bit-exact against the oracle on oracle-supplied
scores, over the register (one CTA and cluster), streaming and shared-memory
paths; dsa_decode_sink end to end with the selection rule and attention tolerance of
the other decode tests, plus the exact presence of every sink position.
"""
import numpy as np
import pytest

import dsa_synth as S
import oracle
from _helpers import assert_sorted_unique, check_attention, check_selection, dev_batch, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    from dsa_sparse_attention_score_gb300 import build
    build.build()
    import dsa_sparse_attention_score_gb300 as m
    return m


CASES = [
    # name, row length, positions, sequence boundaries (cu_q), anchors per sequence
    ("one_cta_unaligned", 5000, [4999, 3001, 2048, 2500], [0, 2, 4], [0, 37]),
    ("cluster3_aligned", 20000, [19999, 12000, 8192], [0, 3], [0]),
    ("beyond_cluster", 140000, [139999, 131072], [0, 1, 2], [3, 0]),
    ("shared_memory_path", 140001, [140000, 131072], [0, 1, 2], [3, 0]),
    ("streaming_path", 20000, [19999 - 61 * i for i in range(160)], [0, 80, 160], [0, 5]),
]


@pytest.mark.parametrize("name,L,pos,cu_q,anchors", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("n_sink,k", [(1, 2048), (4, 2048), (100, 64), (3000, 2048)])
def test_topk_sink_bit_exact(dsa, name, L, pos, cu_q, anchors, n_sink, k):
    import torch
    rng = np.random.default_rng(abs(hash((name, n_sink, k))) % (1 << 31))
    T = len(pos)
    s = rng.standard_normal((T, L)).astype(np.float32)
    s[:, :200] -= 50.0                              # the indexer ranks the early keys last
    seq = np.searchsorted(cu_q, np.arange(T), side="right") - 1
    ref = oracle.topk_sink(s.astype(np.float64), pos, k, n_sink, seq_of_row=seq, anchors=anchors)
    B = len(cu_q) - 1
    b = dsa.Batch.from_host(cu_q, pos, [0] * B, cache_rows=L, max_q_per_seq=int(max(np.diff(cu_q))), max_kv=L)
    ws = dsa.workspace(dsa.DSA_OP_TOPK, b, k=k)
    idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    anc = torch.tensor(anchors, dtype=torch.int32, device="cuda")
    dsa.dsa_topk_sink(to_dev(s), b, k, n_sink, anc, idx, ws)
    got = idx.cpu().numpy()
    assert np.array_equal(got, ref)
    for t in range(T):
        assert_sorted_unique(got[t], pos[t] + 1)
    assert dsa.dsa_read_device_status(ws) == 0


def test_topk_sink_zero_is_topk(dsa):
    import torch
    rng = np.random.default_rng(1)
    s = rng.standard_normal((3, 9000)).astype(np.float32)
    pos = [8999, 4000, 100]
    b = dsa.Batch.from_host([0, 3], pos, [0], cache_rows=9000, max_q_per_seq=3, max_kv=9000)
    ws = dsa.workspace(dsa.DSA_OP_TOPK, b, k=512)
    a = torch.full((3, 512), -7, dtype=torch.int32, device="cuda")
    c = torch.full((3, 512), -7, dtype=torch.int32, device="cuda")
    dsa.dsa_topk(to_dev(s), b, 512, a, ws)
    dsa.dsa_topk_sink(to_dev(s), b, 512, 0, None, c, ws)
    assert torch.equal(a, c)


def test_decode_sink_end_to_end(dsa):
    import torch
    wl = S.Workload("decode_sink", 71, kv_len=[3000, 1500, 4000], q_pos=[2999, 1499, 3999], cu_q=[0, 1, 2, 3],
                    H_I=16, H=16, top_k=256, hadamard=True)
    n_sink, anchors = 4, [0, 5, 0]
    inp = S.make_inputs(wl)
    b = dev_batch(wl)
    ws = dsa.workspace(dsa.DSA_OP_DECODE, b, wl.H_I, wl.H, wl.top_k)
    kc = to_dev(inp.k_cache)
    out = torch.full((wl.T, wl.H, 512), float("nan"), device="cuda")
    lse = torch.full((wl.T, wl.H), float("nan"), device="cuda")
    idx = torch.full((wl.T, wl.top_k), -7, dtype=torch.int32, device="cuda")
    dsa.dsa_decode_sink(to_dev(inp.k_new), to_dev(inp.q_idx), to_dev(inp.w), to_dev(inp.q_lat), to_dev(inp.q_rope),
                        kc, to_dev(inp.kv_cache), b, wl.top_k, wl.sm_scale, wl.hadamard, n_sink,
                        torch.tensor(anchors, dtype=torch.int32, device="cuda"), out, lse, idx, ws)
    assert dsa.dsa_read_device_status(ws) == 0
    g_idx, g_out, g_lse = idx.cpu().numpy(), out.cpu().numpy(), lse.cpu().numpy()
    kc_ref = inp.k_cache.copy()
    ob = oracle.Batch.of(wl)
    oracle.k_append(inp.k_new, ob, kc_ref, wl.hadamard)
    scores = oracle.indexer_score(inp.q_idx, inp.w, kc_ref, ob, wl.hadamard, ld=wl.max_kv)
    boosted = scores.copy()
    for t in range(wl.T):
        a = anchors[t]
        boosted[t, a:min(a + n_sink, wl.q_pos[t] + 1)] = np.inf
    ref = oracle.topk_sink(scores, wl.q_pos, wl.top_k, n_sink, seq_of_row=list(range(wl.T)), anchors=anchors)
    for t in range(wl.T):
        n = wl.q_pos[t] + 1
        assert_sorted_unique(g_idx[t], n)
        assert set(range(anchors[t], anchors[t] + n_sink)) <= set(g_idx[t].tolist())
        check_selection(g_idx[t], ref[t], boosted[t, :n], wl.top_k)
    ref_o, ref_l = oracle.sparse_attn(inp.q_lat, inp.q_rope, inp.kv_cache, ob, g_idx, wl.sm_scale)
    check_attention(g_out, g_lse, ref_o, ref_l, name="sink attention")
