"""Shared pieces of the GPU parity tests: upload of synthetic inputs and the
comparison rules.

Comparison rules (derived from the arithmetic of each path):
  k_append   bit-exact fp16 (both sides round the exact float64 transform once).
  score      |g - o| <= 1e-3 max(|o|, 1e-3 A), with A = sum_h |w_h| ReLU(q'_h . k):
             1e-3 relative, with a floor for scores that cancel towards zero
             across heads of both signs; masked positions must be -inf on
             both sides.  The floor (1e-6 A) sits far above the float32
             accumulation error of the products but below the error of a
             rotated query rounded once to fp16, so it tells the hi + lo
             query of the kernel from a single rounding.
  top-k      bit-exact index set on float32 scores the oracle supplies.
  selection  (end to end) same size; every position in the symmetric
             difference has an oracle score within 1e-3 relative of the
             oracle's k-th score.
  attention  max |g - o| <= 2e-3 and <= 1e-2 max |o| on out (the outputs of
             the workloads are small, so the relative bound is the sharper
             one), max |g - o| <= 1e-3 on lse; computed on the GPU's own
             selection.
The achieved worst errors are recorded (ERRORS) and printed at the end of the
run by conftest.py.
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


# worst achieved error of each rule over the run: name -> (error, bound) at
# the largest error / bound ratio seen
ERRORS = {}


def record(name, err, bound):
    if not bound > 0 or not np.isfinite(bound):
        return
    old = ERRORS.get(name)
    if old is None or err / bound > old[0] / old[1]:
        ERRORS[name] = (float(err), float(bound))


def score_tolerance(q_idx, w, k_cache, wl, t, hadamard):
    """A = sum_h |w_h| ReLU(q'_h . k_s) for each visible position s of row t
    (float64 array over 0..p_t), q' the (rotated) query in float64."""
    import scipy.linalg
    b = int(np.searchsorted(wl.cu_q, t, side="right") - 1)
    p = wl.q_pos[t]
    off = wl.kv_off[b]
    q = q_idx[t].astype(np.float64)
    if hadamard:
        q = q @ (scipy.linalg.hadamard(128) / np.sqrt(128)).T
    k = k_cache[off:off + p + 1].astype(np.float64)
    return np.abs(w[t].astype(np.float64)) @ np.maximum(q @ k.T, 0.0)


def score_bound(ref, A):
    return 1e-3 * np.maximum(np.abs(ref), 1e-3 * A)


def check_scores(got, ref, A, name="score"):
    """got/ref over the visible range of one row; A per position."""
    err = np.abs(got.astype(np.float64) - ref)
    tol = score_bound(ref, A)
    bad = np.nonzero(err > tol)[0]
    assert bad.size == 0, f"{bad.size} scores out of tolerance, first {bad[:5]}: " \
                          f"got {got[bad[:5]]} ref {ref[bad[:5]]} tol {tol[bad[:5]]}"
    pos = tol > 0
    if pos.any():
        i = int(np.argmax(np.where(pos, err / np.where(pos, tol, 1.0), -1.0)))
        record(name, err[i], tol[i])


def check_attention(go, gl, ref_o, ref_l, name="attention", lse_tol=1e-3):
    """Output and lse rule: max |g - o| <= min(2e-3, 1e-2 max |o|) on the
    output, <= lse_tol (1e-3) on the (finite) lse."""
    err_o = float(np.abs(go - ref_o).max()) if go.size else 0.0
    bound_o = min(2e-3, 1e-2 * float(np.abs(ref_o).max())) if go.size else 1.0
    if bound_o == 0.0:                      # all-zero reference (empty selections)
        assert err_o == 0.0, err_o
    else:
        assert err_o <= bound_o, (err_o, bound_o)
        record(name + " out", err_o, bound_o)
    if gl is not None:
        fin = np.isfinite(ref_l)
        assert np.array_equal(np.isfinite(gl), fin)
        if fin.any():
            err_l = float(np.abs(gl[fin] - ref_l[fin]).max())
            assert err_l <= lse_tol, err_l
            record(name + " lse", err_l, lse_tol)
    return err_o


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
