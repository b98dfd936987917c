"""The failure path of the bounded device waits, exercised without a GPU
fault.  Every wait in the score and attention kernels gives up after a limit;
the test hook shortens that limit to 2 ms and makes the kernels' producers
issue no copies, so the consumers' waits run out with nothing in flight.
The kernels must then report DSA_DEV_TIMEOUT in the status word, free their
tensor memory and return -- and the next ordinary call on the same context
must be clean and correct."""
import numpy as np
import pytest

import dsa_synth as S
import oracle
from _helpers import check_attention, dev_batch, to_dev

pytestmark = pytest.mark.gpu

LIMIT_NS = 2_000_000


@pytest.fixture(scope="module")
def dsa():
    from dsa_sparse_attention_score_gb300 import build
    build.build()
    import dsa_sparse_attention_score_gb300 as m
    yield m
    m.dsa_set_test_faults(0, False)


def _score(dsa, wl, inp, ws, scores):
    b = dev_batch(wl)
    dsa.dsa_indexer_score(to_dev(inp.q_idx), to_dev(inp.w), to_dev(inp.k_cache), b, wl.hadamard, scores, ws)


def test_score_kernel_wait_runs_out_then_recovers(dsa):
    import torch
    wl = S.decode_workload("to_s", 71, [700, 1500], H_I=32, H=8, top_k=16)
    inp = S.make_inputs(wl, parts=("k_cache", "q_idx", "w"))
    b = dev_batch(wl)
    ws = dsa.workspace(dsa.DSA_OP_INDEXER_SCORE, b)
    scores = torch.zeros((wl.T, wl.max_kv), device="cuda")
    dsa.dsa_set_test_faults(LIMIT_NS, True)
    try:
        _score(dsa, wl, inp, ws, scores)
        flags = dsa.dsa_read_device_status(ws)
    finally:
        dsa.dsa_set_test_faults(0, False)
    assert flags & dsa.DSA_DEV_TIMEOUT, flags
    # the same call again, hooks off: clean status, scores as the oracle's
    _score(dsa, wl, inp, ws, scores)
    assert dsa.dsa_read_device_status(ws) == 0
    ref = oracle.indexer_score(inp.q_idx, inp.w, inp.k_cache, oracle.Batch.of(wl), False, ld=wl.max_kv)
    got = scores.cpu().numpy()
    for t in range(wl.T):
        p = wl.q_pos[t]
        assert np.allclose(got[t, :p + 1], ref[t, :p + 1], rtol=1e-3, atol=1e-5)


def test_attention_kernel_wait_runs_out_then_recovers(dsa):
    import torch
    wl = S.decode_workload("to_a", 72, [900, 2600], H_I=4, H=64, top_k=512)
    inp = S.make_inputs(wl, parts=("q_lat", "q_rope", "kv_cache"))
    rng = np.random.default_rng(72)
    idx = oracle.topk(rng.standard_normal((wl.T, wl.max_kv)), wl.q_pos, wl.top_k)
    b = dev_batch(wl)
    ws = dsa.workspace(dsa.DSA_OP_SPARSE_ATTN, b, H=wl.H, k=wl.top_k)
    out = torch.zeros((wl.T, wl.H, 512), device="cuda")
    lse = torch.zeros((wl.T, wl.H), device="cuda")
    args = (to_dev(inp.q_lat), to_dev(inp.q_rope), to_dev(inp.kv_cache), b, to_dev(idx), wl.sm_scale, out, lse, ws)
    dsa.dsa_set_test_faults(LIMIT_NS, True)
    try:
        dsa.dsa_sparse_mla_attn(*args)
        flags = dsa.dsa_read_device_status(ws)
    finally:
        dsa.dsa_set_test_faults(0, False)
    assert flags & dsa.DSA_DEV_TIMEOUT, flags
    dsa.dsa_sparse_mla_attn(*args)
    assert dsa.dsa_read_device_status(ws) == 0
    ref_o, ref_l = oracle.sparse_attn(inp.q_lat, inp.q_rope, inp.kv_cache, oracle.Batch.of(wl), idx, wl.sm_scale)
    check_attention(out.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l)


def test_fused_decode_wait_runs_out_then_recovers(dsa):
    """The whole chain with the hook on: the score and attention kernels time
    out, the top-k and combine kernels between them run on whatever the
    workspace holds (no fault), the status reports the timeout; the next
    ordinary step is correct."""
    import torch
    wl = S.config(1)
    inp = S.make_inputs(wl)
    b = dev_batch(wl)
    ws = dsa.workspace(dsa.DSA_OP_DECODE, b, wl.H_I, wl.H, wl.top_k)
    kc = to_dev(inp.k_cache)
    out = torch.zeros((wl.T, wl.H, 512), device="cuda")
    lse = torch.zeros((wl.T, wl.H), device="cuda")
    idx = torch.zeros((wl.T, wl.top_k), dtype=torch.int32, device="cuda")
    args = (to_dev(inp.k_new), to_dev(inp.q_idx), to_dev(inp.w), to_dev(inp.q_lat), to_dev(inp.q_rope), kc,
            to_dev(inp.kv_cache), b, wl.top_k, wl.sm_scale, wl.hadamard, out, lse, idx, ws)
    dsa.dsa_set_test_faults(LIMIT_NS, True)
    try:
        dsa.dsa_decode(*args)
        flags = dsa.dsa_read_device_status(ws)
    finally:
        dsa.dsa_set_test_faults(0, False)
    assert flags & dsa.DSA_DEV_TIMEOUT, flags
    dsa.dsa_decode(*args)
    assert dsa.dsa_read_device_status(ws) == 0
    ref = oracle.decode(inp, wl)
    assert np.array_equal(kc.cpu().numpy().view(np.uint16), ref["k_cache"].view(np.uint16))
    g_idx = idx.cpu().numpy()
    ref_o, ref_l = oracle.sparse_attn(inp.q_lat, inp.q_rope, inp.kv_cache, oracle.Batch.of(wl), g_idx, wl.sm_scale)
    check_attention(out.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l)
