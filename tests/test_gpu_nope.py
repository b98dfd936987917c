"""MLA-NoPE sparse attention (512-d latent rows, no rope tail) on the GPU
against the oracle, through dsa_sparse_mla_attn_nope.

vllm-rdna PR #2 "Glm5Next (GLM-5.3-Flash) on gfx1030": the DSA layers cache
the 512-d kv latent per token and apply no RoPE; qk head dim 256, so the
softmax scale is 1/16.
"""
import numpy as np
import pytest

import dsa_synth as S
import oracle
from _helpers import check_attention, dev_batch, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    from dsa_sparse_attention_score_gb300 import build
    build.build()
    import dsa_sparse_attention_score_gb300 as m
    return m


NOPE_CASES = [
    # name, lengths, H, k: split decode, padded heads with a partial tile, many tokens per CTA
    ("decode_H64_k2048", [3000, 2100], 64, 2048),
    ("decode_H40_k100", [500, 129, 1000], 40, 100),
    ("decode_H16_k1", [50, 60], 16, 1),
]


def _run(dsa, wl, H, k, idx, latent, q_lat):
    import torch
    b = dev_batch(wl)
    ws = dsa.workspace(dsa.DSA_OP_SPARSE_ATTN, b, H=H, k=k)
    out = torch.full((wl.T, H, 512), float("nan"), device="cuda")
    lse = torch.full((wl.T, H), float("nan"), device="cuda")
    dsa.dsa_sparse_mla_attn_nope(to_dev(q_lat), to_dev(latent), b, to_dev(idx), 1 / 16, out, lse, ws)
    assert dsa.dsa_read_device_status(ws) == 0
    return out.cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("name,lengths,H,k", NOPE_CASES, ids=[c[0] for c in NOPE_CASES])
def test_nope_attention_matches_oracle(dsa, name, lengths, H, k):
    wl = S.decode_workload("n", 51, lengths, H_I=4, H=H, top_k=k)
    inp = S.make_inputs(wl, parts=("q_lat", "kv_cache"))
    latent = np.ascontiguousarray(inp.kv_cache[:, :512])       # 512-wide rows: no rope tail
    rng = np.random.default_rng(3)
    idx = oracle.topk(rng.standard_normal((wl.T, wl.max_kv)), wl.q_pos, k)
    ref_o, ref_l = oracle.sparse_attn_nope(inp.q_lat, latent, oracle.Batch.of(wl), idx, 1 / 16)
    go, gl = _run(dsa, wl, H, k, idx, latent, inp.q_lat)
    check_attention(go, gl, ref_o, ref_l, name="nope attention")


def test_nope_attention_prefill_tokens_and_padding_entries(dsa):
    """Many tokens (each CTA walks all tiles of its token), a sharp softmax
    that moves the running maximum, -1 entries and an empty row."""
    wl = S.prefill_workload("n2", 52, 700, 300, H_I=4, H=16, top_k=384)
    inp = S.make_inputs(wl, parts=("q_lat", "kv_cache"))
    latent = np.ascontiguousarray(inp.kv_cache[:, :512])
    q_lat = S.f64_to_bf16_bits(S.bf16_bits_to_f32(inp.q_lat).astype(np.float64) * 30)
    rng = np.random.default_rng(4)
    idx = oracle.topk(rng.standard_normal((wl.T, wl.max_kv)) * 3, wl.q_pos, wl.top_k)
    idx[5, ::4] = -1
    idx[7, :] = -1
    ref_o, ref_l = oracle.sparse_attn_nope(q_lat, latent, oracle.Batch.of(wl), idx, 1 / 16)
    go, gl = _run(dsa, wl, 16, wl.top_k, idx, latent, q_lat)
    keep = np.isfinite(ref_l)
    check_attention(go, gl, ref_o, ref_l, name="nope attention (sharp)",
                    lse_tol=1e-3 * max(1.0, np.abs(ref_l[keep]).max() / 100))
    assert np.all(go[7] == 0) and np.all(np.isneginf(gl[7]))
