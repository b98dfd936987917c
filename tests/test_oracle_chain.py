"""The oracle's whole step is the composition of its four steps, and with
top_k >= n it reproduces dense causal attention (tiny decode workload)."""
import numpy as np

import dsa_synth as S
import oracle


def test_chain_is_composition_of_steps():
    wl = S.config(1)
    inp = S.make_inputs(wl)
    r = oracle.decode(inp, wl)
    b = oracle.Batch.of(wl)
    kc = inp.k_cache.copy()
    oracle.k_append(inp.k_new, b, kc, wl.hadamard)
    assert np.array_equal(kc, r["k_cache"])
    sc = oracle.indexer_score(inp.q_idx, inp.w, kc, b, wl.hadamard)
    assert np.array_equal(sc, r["scores"])
    idx = oracle.topk(sc, wl.q_pos, wl.top_k)
    assert np.array_equal(idx, r["idx"])
    out, lse = oracle.sparse_attn(inp.q_lat, inp.q_rope, inp.kv_cache, b, idx, wl.sm_scale)
    assert np.array_equal(out, r["out"]) and np.array_equal(lse, r["lse"])
    # the own key (position 255) was appended before scoring
    assert r["scores"][0, 255] == sc[0, 255]
    assert np.array_equal(kc[255], inp.k_new[0].astype(np.float16))


def test_tiny_decode_dense_equivalence_at_k256():
    wl = S.config(1, top_k=256)
    inp = S.make_inputs(wl)
    r = oracle.decode(inp, wl)
    assert r["idx"][0].tolist() == list(range(256))
    b = oracle.Batch.of(wl)
    ql = S.bf16_bits_to_f32(inp.q_lat).astype(np.float64)
    qr = S.bf16_bits_to_f32(inp.q_rope).astype(np.float64)
    de, dl = oracle.dense_attn_f64(ql, qr, inp.kv_cache, b, wl.sm_scale)
    assert np.array_equal(r["out"], de) and np.array_equal(r["lse"], dl)


def test_tiny_decode_selection_bites_at_k64():
    wl = S.config(1)
    r = oracle.decode(S.make_inputs(wl), wl)
    sel = r["idx"][0]
    assert (sel >= 0).all() and len(set(sel.tolist())) == 64 and np.all(np.diff(sel) > 0)
    kth = np.sort(r["scores"][0, :256])[::-1][63]
    assert np.all(r["scores"][0, sel] >= kth)
