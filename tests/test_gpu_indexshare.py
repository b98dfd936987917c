"""IndexShare (ik_llama_opt commit log, "GLM-5.2 DSA: IndexShare (shared
layers reuse full-layer top-k)"): a shared layer attends over the selection
of the most recent full layer.  Through the C ABI: a full layer's dsa_decode
returns its selection, and a shared layer's dsa_sparse_mla_attn on that
selection must match the oracle's attention of the shared layer's own queries
and cache over the same positions.
"""
import numpy as np
import pytest

import dsa_synth as S
import oracle
from _helpers import check_attention, dev_batch, to_dev

pytestmark = pytest.mark.gpu


def full_layer(il):
    # the page's rule: full iff il <= 1 or il % 4 == 2
    return il <= 1 or il % 4 == 2


def test_layer_rule_counts():
    full = [il for il in range(78) if full_layer(il)]
    assert len(full) == 21 and full[:4] == [0, 1, 2, 6]


def test_shared_layer_reuses_full_layer_selection():
    import torch
    from dsa_sparse_attention_score_gb300 import build
    build.build()
    import dsa_sparse_attention_score_gb300 as dsa
    base = S.Workload("indexshare", 81, kv_len=[1500, 2600], q_pos=[1499, 2599], cu_q=[0, 1, 2],
                      H_I=16, H=16, top_k=256)
    b = dev_batch(base)
    ws = dsa.workspace(dsa.DSA_OP_DECODE, b, base.H_I, base.H, base.top_k)
    idx = torch.full((base.T, base.top_k), -7, dtype=torch.int32, device="cuda")
    out = torch.empty((base.T, base.H, 512), device="cuda")
    lse = torch.empty((base.T, base.H), device="cuda")
    last_full = None
    for il in range(4):                              # layers 0, 1, 2 full; 3 shared
        wl = S.Workload("indexshare", 81 + il, kv_len=base.kv_len, q_pos=base.q_pos, cu_q=base.cu_q,
                        H_I=16, H=16, top_k=256)
        inp = S.make_inputs(wl)
        if full_layer(il):
            dsa.dsa_decode(to_dev(inp.k_new), to_dev(inp.q_idx), to_dev(inp.w), to_dev(inp.q_lat),
                           to_dev(inp.q_rope), to_dev(inp.k_cache), to_dev(inp.kv_cache), b, wl.top_k,
                           wl.sm_scale, wl.hadamard, out, lse, idx, ws)
            last_full = idx.cpu().numpy()
        else:
            dsa.dsa_sparse_mla_attn(to_dev(inp.q_lat), to_dev(inp.q_rope), to_dev(inp.kv_cache), b, idx,
                                    wl.sm_scale, out, lse, ws)
            ref_o, ref_l = oracle.sparse_attn(inp.q_lat, inp.q_rope, inp.kv_cache, oracle.Batch.of(wl),
                                              last_full, wl.sm_scale)
            check_attention(out.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, name="indexshare attention")
        assert dsa.dsa_read_device_status(ws) == 0
