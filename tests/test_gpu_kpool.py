"""GPU parity of the GLM-5.3-Flash kpool indexer (vllm-rdna PR #2 "Glm5Next
(GLM-5.3-Flash) on gfx1030": kpool 4, softmax(gate+ape) pool compression,
always_select_tail, width 2051) through the C ABI, against the oracle.

The caches start from synthetic packed rows; the pool keys of the context are
built by a first dsa_kpool_append over every cached position (with the rows'
own k and gate), then the step under test runs.  Rules: packed rows and
pooled keys bit-exact (both sides compress in float64 and round once to
fp16); selections compared pool by pool with the end-to-end tie band on the
oracle's pool scores, tail positions exact; attention by the shared rule on
the GPU's own selection.
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


def _decode_wl(name, seed, lengths, H_I, H, top_k):
    """One query token per sequence at position L - 1; each sequence's rows
    start at a multiple of 4 (its capacity rounded up), as pools require."""
    cap = [(L + 3) // 4 * 4 for L in lengths]
    return S.Workload(name, seed, kv_len=cap, q_pos=[L - 1 for L in lengths], cu_q=list(range(len(lengths) + 1)),
                      H_I=H_I, H=H, top_k=top_k)


def _context_batch(dsa, wl, holes=()):
    """Every cached position before each sequence's first query token, minus holes."""
    import torch
    q_pos, cu = [], [0]
    for b in range(wl.B):
        first = min(wl.q_pos[wl.cu_q[b]:wl.cu_q[b + 1]])
        q_pos += [s for s in range(first) if wl.kv_off[b] + s not in holes]
        cu.append(len(q_pos))
    return q_pos, cu


def _setup(dsa, wl, inp, holes=()):
    """Device caches with the context's pool keys built by dsa_kpool_append."""
    import torch
    rows = inp.rows.copy()
    for r in holes:
        rows[r, 256] = 0.0                               # absent rows: never appended
    d_rows = to_dev(rows)
    n_pool = (wl.cache_rows + 3) // 4
    d_pool = torch.zeros((n_pool, 128), dtype=torch.float16, device="cuda")
    q_pos, cu = _context_batch(dsa, wl, holes)
    if q_pos:
        tok = [wl.kv_off[b] + s for b in range(wl.B) for s in q_pos[cu[b]:cu[b + 1]]]
        b_ctx = dsa.Batch.from_host(cu, q_pos, wl.kv_off, wl.cache_rows, max_q_per_seq=max(
            cu[i + 1] - cu[i] for i in range(wl.B)) or 1, max_kv=max(q_pos) + 1)
        ws = dsa.workspace(dsa.DSA_OP_K_APPEND, b_ctx)
        k_ctx = to_dev(np.ascontiguousarray(inp.rows[tok, :128]))
        g_ctx = to_dev(np.ascontiguousarray(inp.rows[tok, 128:256]))
        dsa.dsa_kpool_append(k_ctx, g_ctx, to_dev(inp.ape), b_ctx, d_rows, d_pool, ws)
        assert dsa.dsa_read_device_status(ws) == 0
    return rows, d_rows, d_pool


def _oracle_pool_keys(rows, wl, ape, upto):
    """Oracle pooled keys of every complete pool below position `upto[b]`."""
    keys = {}
    for b in range(wl.B):
        off = wl.kv_off[b]
        for j in range(upto[b] // 4):
            has, key = oracle.kpool_pool_key(rows[off:], j, ape)
            if has:
                keys[off // 4 + j] = key
    return keys


def _check_selection(g_idx, o_idx, scores, wl, top_k):
    """Pools compared with the tie band on the oracle's pool scores; tail exact."""
    kp = top_k // 4
    swaps = 0
    for t in range(wl.T):
        p = wl.q_pos[t]
        n_pools = (p + 1) // 4
        g = [int(s) for s in g_idx[t] if s >= 0]
        o = [int(s) for s in o_idx[t] if s >= 0]
        assert g == sorted(g) and len(g) == len(set(g))
        g_tail, o_tail = [s for s in g if s >= 4 * n_pools], [s for s in o if s >= 4 * n_pools]
        assert g_tail == o_tail, (t, g_tail, o_tail)
        gp, op = {s // 4 for s in g if s < 4 * n_pools}, {s // 4 for s in o if s < 4 * n_pools}
        assert len(gp) == len(op), (t, len(gp), len(op))
        if gp != op:
            row = scores[t, :n_pools]
            kth = np.sort(row[np.isfinite(row)])[::-1][min(kp, np.isfinite(row).sum()) - 1]
            for j in gp ^ op:
                assert abs(row[j] - kth) <= 1e-3 * abs(kth), (t, j, row[j], kth)
            swaps += len(gp ^ op)
    return swaps


def _run_decode(dsa, wl, top_k, holes=(), H=None):
    import torch
    H = H or wl.H
    inp = S.make_kpool_inputs(wl)
    rows, d_rows, d_pool = _setup(dsa, wl, inp, holes)
    b = dev_batch(wl)
    ws = dsa.workspace(dsa.DSA_OP_KPOOL, b, wl.H_I, H, top_k)
    width = dsa.kpool_width(top_k)
    out = torch.full((wl.T, H, 512), float("nan"), device="cuda")
    lse = torch.full((wl.T, H), float("nan"), device="cuda")
    idx = torch.full((wl.T, width), -7, dtype=torch.int32, device="cuda")
    dsa.dsa_decode_kpool(to_dev(inp.k_new), to_dev(inp.gate_new), to_dev(inp.ape), to_dev(inp.q_idx), to_dev(inp.w),
                         to_dev(inp.q_lat), d_rows, d_pool, to_dev(inp.kv_latent), b, top_k, wl.sm_scale, out, lse,
                         idx, ws)
    assert dsa.dsa_read_device_status(ws) == 0
    # oracle: the same rows after the step's append
    ob = oracle.Batch.of(wl)
    oracle.kpool_write_rows(inp.k_new, inp.gate_new, ob, rows)
    assert np.array_equal(d_rows.cpu().numpy().view(np.uint16), rows.view(np.uint16)), "packed rows differ"
    upto = [max(wl.q_pos[wl.cu_q[b_]:wl.cu_q[b_ + 1]]) + 1 for b_ in range(wl.B)]
    g_pool = d_pool.cpu().numpy()
    for r, key in _oracle_pool_keys(rows, wl, inp.ape, upto).items():
        assert np.array_equal(g_pool[r].view(np.uint16), key.view(np.uint16)), f"pool key row {r}"
    o_idx, sc = oracle.kpool_select(inp.q_idx, inp.w, rows, inp.ape, ob, top_k, scores=True)
    g_idx = idx.cpu().numpy()
    _check_selection(g_idx, o_idx, sc, wl, top_k)
    latent = np.ascontiguousarray(inp.kv_latent)
    ref_o, ref_l = oracle.sparse_attn_nope(inp.q_lat, latent, ob, g_idx, wl.sm_scale)
    check_attention(out.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l, name="kpool attention")
    return g_idx


def test_kpool_decode_glm53_flash_shape(dsa):
    """GLM-5.3-Flash DSA decode: 32 indexer heads, 64 heads of 512-d latent
    (no rope), top_k 2048 -> 2051 positions; lengths with every residue mod 4,
    so tokens complete a pool, or leave a tail of 1, 2 or 3."""
    wl = _decode_wl("kp_dec", 91, [8192, 9001, 8194, 8195, 3000], H_I=32, H=64, top_k=2048)
    g = _run_decode(dsa, wl, 2048)
    assert g.shape == (5, 2051)


def test_kpool_long_rows_balanced_grid(dsa):
    """Rows of up to 30000 pools: the decode score grid shares its CTAs out
    by sequence length in pool mode; a sequence with no complete pool gets
    no CTA and an empty row (tail only)."""
    wl = _decode_wl("kp_long", 97, [120001, 40002, 3], H_I=32, H=8, top_k=2048)
    g = _run_decode(dsa, wl, 2048)
    assert g[2].tolist()[:3] == [0, 1, 2] and all(x == -1 for x in g[2].tolist()[3:])


def test_kpool_short_sequences_and_small_top_k(dsa):
    """Tokens with no complete pool (tail only), fewer pools than selected,
    and top_k below one pool's worth (tail only)."""
    wl = _decode_wl("kp_short", 92, [1, 3, 4, 7, 40, 300], H_I=8, H=16, top_k=16)
    _run_decode(dsa, wl, 16)
    wl2 = _decode_wl("kp_k3", 93, [50, 9], H_I=8, H=8, top_k=3)
    g = _run_decode(dsa, wl2, 3)
    assert g[0].tolist() == [48, 49, -1] and g[1].tolist() == [8, -1, -1]


def test_kpool_absent_rows(dsa):
    """Rows never appended (valid 0) are left out of their pool's softmax,
    of the expansion of a selected pool, and of the tail."""
    wl = _decode_wl("kp_holes", 94, [64, 66], H_I=8, H=8, top_k=64)
    holes = (1, 2, 9, 64 + 41, 64 + 64)                   # none completes a pool (positions = 3 mod 4)
    g = _run_decode(dsa, wl, 64, holes=holes)
    assert not set(g[0].tolist()) & {1, 2, 9} and 0 in g[0]
    assert 41 not in g[1] and 64 not in g[1] and 65 in g[1]


def test_kpool_prefill_chunk(dsa):
    """A chunk of 70 tokens after 300 cached (several pools complete inside
    the chunk: rows first, then the pooled keys), plus a second sequence."""
    wl = S.Workload("kp_pre", 95, kv_len=[372, 130], q_pos=[302 + i for i in range(70)] + [100 + i for i in range(30)],
                    cu_q=[0, 70, 100], H_I=32, H=16, top_k=128)
    _run_decode(dsa, wl, 128)


def test_kpool_select_matches_oracle(dsa):
    """dsa_kpool_select alone (no append in the call), window of several tokens."""
    import torch
    wl = S.prefill_workload("kp_sel", 96, 2000, 24, H_I=32, H=8, top_k=256)
    inp = S.make_kpool_inputs(wl)
    # every row, the chunk's included, is in the cache already: append them all as context
    ctx = S.Workload("kp_sel", 96, kv_len=[2024], q_pos=[2024], cu_q=[0, 1], H_I=32, H=8, top_k=256)
    rows, d_rows, d_pool = _setup(dsa, ctx, inp)
    b = dev_batch(wl)
    ws = dsa.workspace(dsa.DSA_OP_KPOOL, b, wl.H_I, 64, 256)
    idx = torch.full((wl.T, dsa.kpool_width(256)), -7, dtype=torch.int32, device="cuda")
    dsa.dsa_kpool_select(to_dev(inp.q_idx), to_dev(inp.w), d_rows, d_pool, b, 256, idx, ws)
    assert dsa.dsa_read_device_status(ws) == 0
    o_idx, sc = oracle.kpool_select(inp.q_idx, inp.w, rows, inp.ape, oracle.Batch.of(wl), 256, scores=True)
    _check_selection(idx.cpu().numpy(), o_idx, sc, wl, 256)
