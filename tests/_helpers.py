"""Shared pieces of the GPU parity tests: upload of synthetic inputs and the
comparison rules.

Comparison rules (derived from the arithmetic of each path):
  k_append   bit-exact fp16 (both sides round the exact float64 transform once).
  score      |g - o| <= 1e-3 |o| + 1e-5 A, with A = sum_h |w_h| sum_d |q'_hd k_d|:
             the relative bound asked for, plus a floor for cancellation that
             is two orders above the float32 accumulation error over 128
             products; masked positions must be -inf on both sides.
  top-k      bit-exact index set on float32 scores the oracle supplies.
  selection  (end to end) same size; every position in the symmetric
             difference has an oracle score within 1e-3 relative of the
             oracle's k-th score.
  attention  max |g - o| <= 2e-3 on out, 1e-3 on lse, computed on the
             GPU's own selection.
"""
from __future__ import annotations

import numpy as np

import dsa_synth as S


def torch():
    import torch as _t
    return _t


def to_dev(a, dtype=None):
    t = torch()
    if a.dtype == np.uint16:                       # bf16 bit patterns
        x = t.from_numpy(a.view(np.int16).copy()).view(t.bfloat16)
    else:
        x = t.from_numpy(np.ascontiguousarray(a))
    return x.cuda()


def dev_batch(wl):
    import dsa_sparse_attention_score_gb300 as dsa
    return dsa.Batch.from_host(wl.cu_q, wl.q_pos, wl.kv_off, wl.cache_rows,
                               max_q_per_seq=wl.max_q_per_seq, max_kv=wl.max_kv)


def score_tolerance(q_idx, w, k_cache, wl, t, hadamard):
    """Per-position absolute tolerance of row t (float64 array over 0..p_t)."""
    import scipy.linalg
    b = int(np.searchsorted(wl.cu_q, t, side="right") - 1)
    p = wl.q_pos[t]
    off = wl.kv_off[b]
    q = q_idx[t].astype(np.float64)
    if hadamard:
        q = q @ (scipy.linalg.hadamard(128) / np.sqrt(128)).T
    k = np.abs(k_cache[off:off + p + 1].astype(np.float64))
    A = np.abs(w[t].astype(np.float64)) @ (np.abs(q) @ k.T)
    return A


def check_scores(got, ref, A):
    """got/ref over the visible range of one row; A per position."""
    err = np.abs(got.astype(np.float64) - ref)
    tol = 1e-3 * np.abs(ref) + 1e-5 * A
    bad = np.nonzero(err > tol)[0]
    assert bad.size == 0, f"{bad.size} scores out of tolerance, first {bad[:5]}: " \
                          f"got {got[bad[:5]]} ref {ref[bad[:5]]} tol {tol[bad[:5]]}"


def check_selection(gpu_idx, ref_idx, ref_scores, k):
    """Selection rule of the end-to-end comparison (one row)."""
    g = set(int(x) for x in gpu_idx if x >= 0)
    o = set(int(x) for x in ref_idx if x >= 0)
    assert len(g) == len(o), (len(g), len(o))
    if g == o:
        return 0
    n = len(ref_scores)
    kth = np.sort(ref_scores)[::-1][min(k, n) - 1]
    band = 1e-3 * abs(kth)
    diff = g ^ o
    for s in diff:
        assert abs(ref_scores[s] - kth) <= band, (s, ref_scores[s], kth)
    return len(diff)


def assert_sorted_unique(idx_row, n_vis):
    v = idx_row[idx_row >= 0]
    assert np.all(np.diff(v) > 0) and (v.size == 0 or (v[0] >= 0 and v[-1] < n_vis))
    m = v.size
    assert np.all(idx_row[m:] == -1)


def inputs(wl, parts=None):
    return S.make_inputs(wl) if parts is None else S.make_inputs(wl, parts=parts)
