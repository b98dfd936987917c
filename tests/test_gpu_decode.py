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
from _helpers import assert_sorted_unique, check_selection, dev_batch, to_dev

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
    err_o = np.abs(g["out"][rows] - ref_o).max()
    err_l = np.abs(g["lse"][rows] - ref_l).max()
    assert err_o <= 2e-3, err_o
    assert err_l <= 1e-3, err_l
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
    assert np.abs(g["out"] - de).max() <= 2e-3
    assert np.abs(g["lse"] - dl).max() <= 1e-3


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


def test_multi_sequence_prefill_chunks(dsa):
    """Two sequences with several query tokens each (varlen), mixed lengths."""
    wl = S.Workload("mixed", 51, kv_len=[700, 3000], q_pos=[680 + i for i in range(20)] + [2990 + i for i in range(10)],
                    cu_q=[0, 20, 30], H_I=64, H=64, top_k=512, hadamard=True)
    check_workload(dsa, wl)
