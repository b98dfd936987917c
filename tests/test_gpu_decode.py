"""End-to-end parity of dsa_decode on the five workloads.

Small workloads are checked in full; the two prefill workloads run in full
on the GPU and are checked on a deterministic sample of query rows (every
64th row, the first and last rows, and the rows around 128-key tile
boundaries), each recomputed by the oracle from its definition.
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


def run_gpu(dsa, wl, inp):
    import torch
    b = dev_batch(wl)
    ws = dsa.workspace(dsa.DSA_OP_DECODE, b, wl.H_I, wl.H, wl.top_k)
    kc = to_dev(inp.k_cache)
    out = torch.full((wl.T, wl.H, 512), float("nan"), device="cuda")
    lse = torch.full((wl.T, wl.H), float("nan"), device="cuda")
    idx = torch.full((wl.T, wl.top_k), -7, dtype=torch.int32, device="cuda")
    dsa.dsa_decode(to_dev(inp.k_new), to_dev(inp.q_idx), to_dev(inp.w), to_dev(inp.q_lat), to_dev(inp.q_rope),
                   kc, to_dev(inp.kv_cache), b, wl.top_k, wl.sm_scale, wl.hadamard, out, lse, idx, ws)
    status = dsa.dsa_read_device_status(ws)
    return dict(k_cache=kc.cpu().numpy(), idx=idx.cpu().numpy(), out=out.cpu().numpy(),
                lse=lse.cpu().numpy(), status=status)


def sample_rows(T):
    rows = set(range(0, T, 64)) | {0, T - 1}
    for edge in range(128, T, 128 * 7):
        rows |= {edge - 1, edge}
    return sorted(r for r in rows if 0 <= r < T)


def check_rows(wl, inp, g, rows, kc_ref):
    ob = oracle.Batch.of(wl)
    sub = ob.rows(rows)
    ld = max(wl.q_pos[t] for t in rows) + 1
    scores = oracle.indexer_score(inp.q_idx[rows], inp.w[rows], kc_ref, sub, wl.hadamard, ld=ld)
    ref_idx = oracle.topk(scores, sub.q_pos, wl.top_k)
    swaps = 0
    for i, t in enumerate(rows):
        n = wl.q_pos[t] + 1
        assert_sorted_unique(g["idx"][t], n)
        swaps += check_selection(g["idx"][t], ref_idx[i], scores[i, :n], wl.top_k)
    ref_o, ref_l = oracle.sparse_attn(inp.q_lat[rows], inp.q_rope[rows], inp.kv_cache, sub,
                                      g["idx"][rows], wl.sm_scale)
    check_attention(g["out"][rows], g["lse"][rows], ref_o, ref_l, name="decode attention")
    return swaps


def check_workload(dsa, wl, sample=False):
    inp = S.make_inputs(wl)
    g = run_gpu(dsa, wl, inp)
    assert g["status"] == 0
    kc_ref = inp.k_cache.copy()
    oracle.k_append(inp.k_new, oracle.Batch.of(wl), kc_ref, wl.hadamard)
    assert np.array_equal(g["k_cache"].view(np.uint16), kc_ref.view(np.uint16))
    rows = sample_rows(wl.T) if sample else list(range(wl.T))
    return check_rows(wl, inp, g, rows, kc_ref)


def test_tiny_decode_k64(dsa):
    check_workload(dsa, S.config(1))


def test_tiny_decode_dense_equivalence_k256(dsa):
    """top_k >= L: the sparse path must be dense causal attention."""
    wl = S.config(1, top_k=256)
    inp = S.make_inputs(wl)
    g = run_gpu(dsa, wl, inp)
    assert g["idx"][0].tolist() == list(range(256))
    ql = S.bf16_bits_to_f32(inp.q_lat).astype(np.float64)
    qr = S.bf16_bits_to_f32(inp.q_rope).astype(np.float64)
    de, dl = oracle.dense_attn_f64(ql, qr, inp.kv_cache, oracle.Batch.of(wl), wl.sm_scale)
    check_attention(g["out"], g["lse"], de, dl, name="dense equivalence")


def test_tiny_decode_hadamard(dsa):
    check_workload(dsa, S.config(1, hadamard=True))


def test_batched_decode(dsa):
    check_workload(dsa, S.config(2))


def test_ragged_long_context_decode_hadamard(dsa):
    check_workload(dsa, S.config(3))


def test_prefill_chunk_sampled(dsa):
    check_workload(dsa, S.config(4), sample=True)


def test_long_prefill_sampled(dsa):
    check_workload(dsa, S.config(5), sample=True)


def test_deepseek_shaped_decode_128_heads(dsa):
    """128 query heads (DeepSeek-V3.2, the other model of the indexer commit):
    two head groups of 64 per token, split across CTAs and combined."""
    wl = S.decode_workload("ds128", 52, [8192, 5000, 3001, 2048], H_I=64, H=128, top_k=2048)
    check_workload(dsa, wl)


def test_one_token_attends_65536_rows(dsa):
    """k = 65536 for a single token: 1024 row tiles, which would ask for more
    split partials than the combine merges; the split is capped at 128."""
    wl = S.decode_workload("k64k", 53, [70000], H_I=4, H=8, top_k=65536)
    check_workload(dsa, wl)


def test_multi_sequence_prefill_chunks(dsa):
    """Two sequences with several query tokens each (varlen), mixed lengths."""
    wl = S.Workload("mixed", 51, kv_len=[700, 3000], q_pos=[680 + i for i in range(20)] + [2990 + i for i in range(10)],
                    cu_q=[0, 20, 30], H_I=64, H=64, top_k=512, hadamard=True)
    check_workload(dsa, wl)


def _decode_on(dsa, wl, inp, b, ws, kc, kv):
    import torch
    out = torch.full((wl.T, wl.H, 512), float("nan"), device="cuda")
    lse = torch.full((wl.T, wl.H), float("nan"), device="cuda")
    idx = torch.full((wl.T, wl.top_k), -7, dtype=torch.int32, device="cuda")
    dsa.dsa_decode(to_dev(inp.k_new), to_dev(inp.q_idx), to_dev(inp.w), to_dev(inp.q_lat), to_dev(inp.q_rope),
                   kc, kv, b, wl.top_k, wl.sm_scale, wl.hadamard, out, lse, idx, ws)
    status = dsa.dsa_read_device_status(ws)
    return dict(idx=idx.cpu().numpy(), out=out.cpu().numpy(), lse=lse.cpu().numpy(), status=status)


def test_decode_steps_reuse_workspace(dsa):
    """Consecutive single-token steps on one workspace, whose score slab,
    index rows and split partials each step overwrites.  The rows cover
    n < k, n == k, n == k + 1, rows that one top-k CTA holds in registers and
    rows spread over a cluster, and sequences scored by one CTA and by many."""
    kv_len = [40000, 3000, 2049, 70000, 200]
    steps = [[38990, 1000, 2046, 68990, 10],
             [38991, 1001, 2047, 68991, 11],
             [38992, 2999, 2048, 69999, 199]]
    wl0 = S.Workload("decode_steps", 61, kv_len=kv_len, q_pos=steps[0], cu_q=list(range(6)),
                     H_I=32, H=16, top_k=2048)
    inp = S.make_inputs(wl0)
    max_kv = max(kv_len)
    batches = [dsa.Batch.from_host(wl0.cu_q, q, wl0.kv_off, wl0.cache_rows, max_q_per_seq=1, max_kv=max_kv)
               for q in steps]
    ws = dsa.workspace(dsa.DSA_OP_DECODE, batches[0], wl0.H_I, wl0.H, wl0.top_k)
    kc, kv = to_dev(inp.k_cache), to_dev(inp.kv_cache)
    kc_ref = inp.k_cache.copy()
    for q, b in zip(steps, batches):
        wl = S.Workload("decode_steps", 61, kv_len=kv_len, q_pos=q, cu_q=wl0.cu_q, H_I=32, H=16, top_k=2048)
        g = _decode_on(dsa, wl, inp, b, ws, kc, kv)
        assert g["status"] == 0
        oracle.k_append(inp.k_new, oracle.Batch.of(wl), kc_ref, False)
        assert np.array_equal(kc.cpu().numpy().view(np.uint16), kc_ref.view(np.uint16))
        check_rows(wl, inp, g, list(range(wl.T)), kc_ref)


def test_decode_all_scores_tied(dsa):
    """Zero indexer weights make every visible score 0: the selection must be
    the k lowest positions, for rows held in shared memory and for rows so
    long that the threshold bin itself exceeds the shared-memory scratch."""
    wl = S.Workload("decode_ties", 62, kv_len=[70000, 5000, 1000], q_pos=[69999, 4999, 999],
                    cu_q=[0, 1, 2, 3], H_I=16, H=8, top_k=2048)
    inp = S.make_inputs(wl)
    inp.w[:] = 0.0
    b = dev_batch(wl)
    ws = dsa.workspace(dsa.DSA_OP_DECODE, b, wl.H_I, wl.H, wl.top_k)
    g = _decode_on(dsa, wl, inp, b, ws, to_dev(inp.k_cache), to_dev(inp.kv_cache))
    assert g["status"] == 0
    assert g["idx"][0].tolist() == list(range(2048))
    assert g["idx"][1].tolist() == list(range(2048))
    assert g["idx"][2].tolist() == list(range(1000)) + [-1] * 1048


def test_decode_with_tokenless_sequences(dsa):
    """Sequences with no query token this step (cu_q[b + 1] == cu_q[b]) in
    the middle and at the end of a batch of long rows, whose score CTAs are
    shared out by sequence length: the empty sequences get no CTA and raise
    no status."""
    wl = S.Workload("decode_gaps", 63, kv_len=[30000, 9000, 50000, 4000, 20000, 7000],
                    q_pos=[29999, 49000, 19990], cu_q=[0, 1, 1, 2, 2, 3, 3], H_I=16, H=8, top_k=2048)
    check_workload(dsa, wl)


def test_decode_many_ragged_sequences(dsa):
    """120 sequences of 1k-16k keys: the length-proportional shares of the
    score grid range from one CTA to the cap of two tiles per CTA."""
    kv_len = S.ragged_lengths(64, 120, lo=1000, hi=16000)
    kv_len[7], kv_len[50] = 16000, 129
    wl = S.decode_workload("decode_many", 64, kv_len, H_I=16, H=8, top_k=512)
    check_workload(dsa, wl)


def test_results_written_into_mapped_pinned_host_memory(dsa):
    """out and lse may be pinned host memory that the driver maps at the same
    address: the kernels then write the result there directly.  The result
    must equal the device-resident run's bit for bit."""
    import torch
    import bench
    wl = S.config(2)
    inp = S.make_inputs(wl)
    h_out = torch.full((wl.T, wl.H, 512), float("nan")).pin_memory()
    h_lse = torch.full((wl.T, wl.H), float("nan")).pin_memory()
    m_out, m_lse = bench.host_mapped_alias(torch, h_out), bench.host_mapped_alias(torch, h_lse)
    if m_out is None or m_lse is None:
        pytest.skip("pinned host memory is not mapped at the same address on this system")
    b = dev_batch(wl)
    ws = dsa.workspace(dsa.DSA_OP_DECODE, b, wl.H_I, wl.H, wl.top_k)
    args = [to_dev(inp.k_new), to_dev(inp.q_idx), to_dev(inp.w), to_dev(inp.q_lat), to_dev(inp.q_rope),
            to_dev(inp.k_cache), to_dev(inp.kv_cache), b, wl.top_k, wl.sm_scale, wl.hadamard]
    out = torch.empty((wl.T, wl.H, 512), device="cuda")
    lse = torch.empty((wl.T, wl.H), device="cuda")
    idx = torch.empty((wl.T, wl.top_k), dtype=torch.int32, device="cuda")
    dsa.dsa_decode(*args, out, lse, idx, ws)
    dsa.dsa_decode(*args, m_out, m_lse, idx, ws)        # the append rewrites the same keys
    torch.cuda.synchronize()
    assert dsa.dsa_read_device_status(ws) == 0
    assert torch.equal(h_out, out.cpu()) and torch.equal(h_lse, lse.cpu())
