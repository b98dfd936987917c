"""Paged caches (vllm-rdna PR #2 "Glm5Next (GLM-5.3-Flash) on gfx1030": the
latent and indexer caches are paged attention groups and the DSA backend
gathers latents through the page table).

Each sequence's logical rows are scattered into a pooled cache of shuffled
physical blocks whose unused rows hold large garbage values;
dsa_decode_paged on the pool must match the oracle on the logical,
contiguous arrays: the appended key bit-exact at its physical row, the
selection by the decode tests' rule, attention by the shared attention rule.
"""
import numpy as np
import pytest

import dsa_synth as S
import oracle
from _helpers import assert_sorted_unique, check_attention, check_selection, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    from dsa_sparse_attention_score_gb300 import build
    build.build()
    import dsa_sparse_attention_score_gb300 as m
    return m


def paginate(wl, inp, bs, seed):
    rng = np.random.default_rng(seed)
    nblk = [(L + bs - 1) // bs for L in wl.kv_len]
    n_phys = sum(nblk) + 3                              # spare blocks stay unmapped
    perm = rng.permutation(n_phys)
    max_blocks = max(nblk) + 1
    table = np.full((wl.B, max_blocks), -1, np.int32)
    k_phys = np.full((n_phys * bs, 128), 60000.0, np.float16)
    kv_phys = np.full((n_phys * bs, 576), 0x7F00, np.uint16)  # bf16 ~1.7e38: garbage if ever read
    nxt = 0
    for b in range(wl.B):
        off, L = wl.kv_off[b], wl.kv_len[b]
        for j in range(nblk[b]):
            blk = int(perm[nxt]); nxt += 1
            table[b, j] = blk
            n = min(bs, L - j * bs)
            k_phys[blk * bs: blk * bs + n] = inp.k_cache[off + j * bs: off + j * bs + n]
            kv_phys[blk * bs: blk * bs + n] = inp.kv_cache[off + j * bs: off + j * bs + n]
    return table, k_phys, kv_phys


def logical_rows(table, bs, b, L, phys):
    rows = [table[b, p // bs] * bs + p % bs for p in range(L)]
    return phys[rows]


CASES = [
    ("decode_bs64", 64, S.Workload("paged", 91, kv_len=[700, 3000, 1500], q_pos=[699, 2999, 1499],
                                   cu_q=[0, 1, 2, 3], H_I=16, H=16, top_k=256, hadamard=True)),
    ("decode_bs128", 128, S.Workload("paged", 92, kv_len=[700, 3000, 1500], q_pos=[699, 2999, 1499],
                                     cu_q=[0, 1, 2, 3], H_I=16, H=16, top_k=256)),
    ("decode_bs256", 256, S.Workload("paged", 93, kv_len=[4100, 300], q_pos=[4099, 299], cu_q=[0, 1, 2],
                                     H_I=32, H=64, top_k=2048, hadamard=True)),
    # 40 sequences selecting 2048 of 2100-4000 keys: the attention splits
    # each token over few CTAs of many tiles, which prefetch their next
    # tile's (paged) rows into L2
    ("decode_many_bs64", 64, S.decode_workload("paged_many", 95, S.ragged_lengths(95, 40, lo=2100, hi=4000),
                                              H_I=16, H=16, top_k=2048)),
    ("chunks_bs64", 64, S.Workload("paged", 94, kv_len=[700, 3000],
                                   q_pos=[680 + i for i in range(20)] + [2990 + i for i in range(10)],
                                   cu_q=[0, 20, 30], H_I=64, H=64, top_k=512, hadamard=True)),
]


@pytest.mark.parametrize("name,bs,wl", CASES, ids=[c[0] for c in CASES])
def test_paged_decode_matches_oracle(dsa, name, bs, wl):
    import torch
    inp = S.make_inputs(wl)
    table, k_phys, kv_phys = paginate(wl, inp, bs, seed=bs)
    b = dsa.Batch.from_host(wl.cu_q, wl.q_pos, [0] * wl.B, k_phys.shape[0], max_q_per_seq=wl.max_q_per_seq,
                            max_kv=wl.max_kv)
    ws = dsa.workspace(dsa.DSA_OP_DECODE, b, wl.H_I, wl.H, wl.top_k)
    kc = to_dev(k_phys)
    out = torch.full((wl.T, wl.H, 512), float("nan"), device="cuda")
    lse = torch.full((wl.T, wl.H), float("nan"), device="cuda")
    idx = torch.full((wl.T, wl.top_k), -7, dtype=torch.int32, device="cuda")
    dsa.dsa_decode_paged(to_dev(inp.k_new), to_dev(inp.q_idx), to_dev(inp.w), to_dev(inp.q_lat),
                         to_dev(inp.q_rope), kc, to_dev(kv_phys), b, torch.from_numpy(table).cuda(), bs,
                         wl.top_k, wl.sm_scale, wl.hadamard, out, lse, idx, ws)
    assert dsa.dsa_read_device_status(ws) == 0
    ob = oracle.Batch.of(wl)
    kc_ref = inp.k_cache.copy()
    oracle.k_append(inp.k_new, ob, kc_ref, wl.hadamard)
    k_after = kc.cpu().numpy()
    for bi in range(wl.B):
        off, L = wl.kv_off[bi], wl.kv_len[bi]
        got = logical_rows(table, bs, bi, L, k_after)
        assert np.array_equal(got.view(np.uint16), kc_ref[off:off + L].view(np.uint16)), bi
    g_idx, g_out, g_lse = idx.cpu().numpy(), out.cpu().numpy(), lse.cpu().numpy()
    scores = oracle.indexer_score(inp.q_idx, inp.w, kc_ref, ob, wl.hadamard, ld=wl.max_kv)
    ref_idx = oracle.topk(scores, wl.q_pos, wl.top_k)
    for t in range(wl.T):
        n = wl.q_pos[t] + 1
        assert_sorted_unique(g_idx[t], n)
        check_selection(g_idx[t], ref_idx[t], scores[t, :n], wl.top_k)
    ref_o, ref_l = oracle.sparse_attn(inp.q_lat, inp.q_rope, inp.kv_cache, ob, g_idx, wl.sm_scale)
    check_attention(g_out, g_lse, ref_o, ref_l, name="paged attention")


def test_paged_rejects_bad_block_size(dsa):
    import torch
    wl = CASES[1][2]
    inp = S.make_inputs(wl, parts=("k_new",))
    b = dsa.Batch.from_host(wl.cu_q, wl.q_pos, [0] * wl.B, 1 << 14, max_q_per_seq=1, max_kv=wl.max_kv)
    ws = dsa.workspace(dsa.DSA_OP_DECODE, b, wl.H_I, wl.H, wl.top_k)
    t = torch.zeros((wl.B, 64), dtype=torch.int32, device="cuda")
    z16 = torch.zeros((1 << 14, 128), dtype=torch.float16, device="cuda")
    zb = torch.zeros((1 << 14, 576), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((wl.T, wl.H_I, 128), dtype=torch.float16, device="cuda")
    w = torch.zeros((wl.T, wl.H_I), device="cuda")
    ql = torch.zeros((wl.T, wl.H, 512), dtype=torch.bfloat16, device="cuda")
    qr = torch.zeros((wl.T, wl.H, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((wl.T, wl.H, 512), device="cuda")
    lse = torch.empty((wl.T, wl.H), device="cuda")
    idx = torch.empty((wl.T, wl.top_k), dtype=torch.int32, device="cuda")
    with pytest.raises(dsa.DsaError):
        dsa.dsa_decode_paged(to_dev(inp.k_new), q, w, ql, qr, z16, zb, b, t, 96, wl.top_k, wl.sm_scale, False,
                             out, lse, idx, ws)
