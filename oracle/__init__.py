"""ctypes front end of the CPU oracle (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg use this package.  The CUDA library never imports it and it never imports
the CUDA library.  Every function takes and returns numpy arrays; fp16 inputs
are numpy float16, bf16 inputs are uint16 bit patterns.
"""
from __future__ import annotations

import ctypes as C

import numpy as np

from . import build as _build

_LIB = None

P = C.c_void_p
I32 = C.c_int
I64 = C.c_int64
F64 = C.c_double


def lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = C.CDLL(path)
        sig = {
            "oracle_f16_to_f64": (F64, [C.c_uint16]),
            "oracle_bf16_to_f64": (F64, [C.c_uint16]),
            "oracle_f64_to_f16": (C.c_uint16, [F64]),
            "oracle_fwht128": (None, [P, P]),
            "oracle_k_append": (I32, [P, I32, I32, I32, P, P, P, P, I32]),
            "oracle_indexer_score": (I32, [P, P, P, I32, I32, P, P, P, I32, I32, P, I64]),
            "oracle_topk": (I32, [P, I64, I32, P, I32, P]),
            "oracle_topk_sink": (I32, [P, I64, I32, P, I32, I32, P, P]),
            "oracle_sparse_attn_f64": (I32, [P, P, P, I32, I32, P, P, P, P, I32, I32, F64, P, P]),
            "oracle_sparse_attn": (I32, [P, P, P, I32, I32, P, P, P, P, I32, I32, F64, P, P]),
            "oracle_sparse_attn_nope_f64": (I32, [P, P, I32, I32, P, P, P, P, I32, I32, F64, P, P]),
            "oracle_sparse_attn_nope": (I32, [P, P, I32, I32, P, P, P, P, I32, I32, F64, P, P]),
            "oracle_dense_attn_f64": (I32, [P, P, P, I32, I32, P, P, P, I32, F64, P, P]),
            "oracle_unabsorbed_attn": (I32, [P, P, P, I32, I32, P, P, P, P, P, P, I32, I32, F64, P]),
            "oracle_decode": (I32, [P, I32, P, P, P, P, P, P, I32, I32, P, P, P, I32, I32, I32, F64,
                                    I32, P, I64, P, P, P]),
            "oracle_set_threads": (I32, [I32]),
            "oracle_kpool_write_rows": (I32, [P, P, I32, I32, P, P, P, P]),
            "oracle_kpool_pool_key": (I32, [P, I64, P, P]),
            "oracle_kpool_select": (I32, [P, P, P, P, I32, I32, P, P, P, I32, I32, P, P, I64]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _LIB = L
    return _LIB


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


class Batch:
    """Host batch description: cu_q [B+1], q_pos [T], kv_off [B]."""

    def __init__(self, cu_q, q_pos, kv_off):
        self.cu_q = _c(cu_q, np.int32)
        self.q_pos = _c(q_pos, np.int32)
        self.kv_off = _c(kv_off, np.int64)
        self.B = len(self.cu_q) - 1
        self.T = len(self.q_pos)

    @classmethod
    def of(cls, wl):
        return cls(wl.cu_q, wl.q_pos, wl.kv_off)

    def rows(self, ts):
        """Sub-batch of the given query tokens (each kept in its own sequence)."""
        ts = [int(t) for t in ts]
        seq = np.searchsorted(self.cu_q, ts, side="right") - 1
        return Batch(list(range(len(ts) + 1)), self.q_pos[ts], self.kv_off[seq])

    def args(self):
        return (self.B, self.T, _p(self.cu_q), _p(self.q_pos), _p(self.kv_off))


def set_threads(n: int = 0) -> int:
    return lib().oracle_set_threads(n)


def f16_to_f64(h: int) -> float:
    return lib().oracle_f16_to_f64(h)


def f64_to_f16_bits(x: float) -> int:
    return lib().oracle_f64_to_f16(x)


def fwht128(x) -> np.ndarray:
    x = _c(x, np.float64)
    assert x.shape == (128,)
    y = np.empty(128, np.float64)
    lib().oracle_fwht128(_p(x), _p(y))
    return y


def k_append(k_new, batch: Batch, k_cache: np.ndarray, hadamard: bool) -> None:
    """Writes the new keys into k_cache (float16 [rows,128]) in place."""
    assert k_cache.dtype == np.float16 and k_cache.flags.c_contiguous
    if k_new.dtype == np.float16:
        kn, kd = _c(k_new, np.float16), 1
    else:
        kn, kd = _c(k_new, np.float32), 0
    _check(lib().oracle_k_append(_p(kn), kd, *batch.args(), _p(k_cache), int(hadamard)), "k_append")


def indexer_score(q_idx, w, k_cache, batch: Batch, hadamard_q: bool, ld: int | None = None):
    q = _c(q_idx, np.float16)
    T, H_I, _ = q.shape
    ld = int(ld if ld is not None else (batch.q_pos.max() + 1 if T else 1))
    out = np.empty((T, ld), np.float64)
    _check(lib().oracle_indexer_score(_p(q), _p(_c(w, np.float32)), _p(_c(k_cache, np.float16)),
                                      *batch.args(), H_I, int(hadamard_q), _p(out), ld),
           "indexer_score")
    return out


def topk(scores, q_pos, k: int) -> np.ndarray:
    s = _c(scores, np.float64)
    qp = _c(q_pos, np.int32)
    T = s.shape[0]
    idx = np.empty((T, k), np.int32)
    _check(lib().oracle_topk(_p(s), s.shape[1], T, _p(qp), k, _p(idx)), "topk")
    return idx


def topk_sink(scores, q_pos, k: int, n_sink: int, seq_of_row=None, anchors=None) -> np.ndarray:
    """Top-k with the attention sink forced in.

    ik_llama_opt commit log, "GLM-5.2 DSA indexer: decode-correct via
    persistent indexer-K cache" (attention-sink force-inclusion) and "per-
    sequence attention sink": the first n_sink keys of the query's OWN
    sequence get a +1e20 boost before the argsort, so they always survive;
    "UPDATE 6": the sink is anchored on the sequence's first present position.
    Here the boost is taken as unbounded (+inf, which is what +1e20 becomes
    next to float32 scores: the boosted scores tie with one another), then the
    plain selection runs: ties go to the lower position (oracle_topk_sink in
    dsa_oracle.c).
      seq_of_row [T]: sequence of each row (needed with anchors);
      anchors [B]: first present position of each sequence (default 0).
    """
    s = _c(scores, np.float64)
    qp = _c(q_pos, np.int32)
    T = s.shape[0]
    anchor = None
    if anchors is not None:
        anchor = _c([int(anchors[int(seq_of_row[r])]) for r in range(T)], np.int32)
    idx = np.empty((T, k), np.int32)
    _check(lib().oracle_topk_sink(_p(s), s.shape[1], T, _p(qp), k, int(n_sink), _p(anchor), _p(idx)),
           "topk_sink")
    return idx


def sparse_attn(q_lat, q_rope, kv_cache, batch: Batch, idx, sm_scale: float):
    """bf16-bit queries.  Returns (out [T,H,512], lse [T,H]) in float64."""
    ql = _c(q_lat, np.uint16)
    qr = _c(q_rope, np.uint16)
    T, H, _ = ql.shape
    ix = _c(idx, np.int32)
    out = np.empty((T, H, 512), np.float64)
    lse = np.empty((T, H), np.float64)
    _check(lib().oracle_sparse_attn(_p(ql), _p(qr), _p(_c(kv_cache, np.uint16)), *batch.args(),
                                    _p(ix), ix.shape[1], H, sm_scale, _p(out), _p(lse)),
           "sparse_attn")
    return out, lse


def sparse_attn_f64(q_lat, q_rope, kv_cache, batch: Batch, idx, sm_scale: float):
    ql = _c(q_lat, np.float64)
    qr = _c(q_rope, np.float64)
    T, H, _ = ql.shape
    ix = _c(idx, np.int32)
    out = np.empty((T, H, 512), np.float64)
    lse = np.empty((T, H), np.float64)
    _check(lib().oracle_sparse_attn_f64(_p(ql), _p(qr), _p(_c(kv_cache, np.uint16)), *batch.args(),
                                        _p(ix), ix.shape[1], H, sm_scale, _p(out), _p(lse)),
           "sparse_attn_f64")
    return out, lse


def sparse_attn_nope(q_lat, kv_latent, batch: Batch, idx, sm_scale: float):
    """MLA-NoPE (no rope tail; vllm-rdna PR #2 "Glm5Next (GLM-5.3-Flash) on
    gfx1030"): bf16-bit queries [T,H,512] against bf16-bit latent rows
    [rows,512].  Returns (out [T,H,512], lse [T,H]) in float64."""
    ql = _c(q_lat, np.uint16)
    T, H, _ = ql.shape
    ix = _c(idx, np.int32)
    out = np.empty((T, H, 512), np.float64)
    lse = np.empty((T, H), np.float64)
    _check(lib().oracle_sparse_attn_nope(_p(ql), _p(_c(kv_latent, np.uint16)), *batch.args(),
                                         _p(ix), ix.shape[1], H, sm_scale, _p(out), _p(lse)),
           "sparse_attn_nope")
    return out, lse


def sparse_attn_nope_f64(q_lat, kv_latent, batch: Batch, idx, sm_scale: float):
    ql = _c(q_lat, np.float64)
    T, H, _ = ql.shape
    ix = _c(idx, np.int32)
    out = np.empty((T, H, 512), np.float64)
    lse = np.empty((T, H), np.float64)
    _check(lib().oracle_sparse_attn_nope_f64(_p(ql), _p(_c(kv_latent, np.uint16)), *batch.args(),
                                             _p(ix), ix.shape[1], H, sm_scale, _p(out), _p(lse)),
           "sparse_attn_nope_f64")
    return out, lse


def dense_attn_f64(q_lat, q_rope, kv_cache, batch: Batch, sm_scale: float):
    ql = _c(q_lat, np.float64)
    qr = _c(q_rope, np.float64)
    T, H, _ = ql.shape
    out = np.empty((T, H, 512), np.float64)
    lse = np.empty((T, H), np.float64)
    _check(lib().oracle_dense_attn_f64(_p(ql), _p(qr), _p(_c(kv_cache, np.uint16)), *batch.args(),
                                       H, sm_scale, _p(out), _p(lse)), "dense_attn")
    return out, lse


def unabsorbed_attn(q_nope, q_rope, kv_cache, batch: Batch, W_UK, W_UV, idx, sm_scale: float):
    qn = _c(q_nope, np.float64)
    qr = _c(q_rope, np.float64)
    T, H, _ = qn.shape
    ix = _c(idx, np.int32)
    out = np.empty((T, H, 256), np.float64)
    _check(lib().oracle_unabsorbed_attn(_p(qn), _p(qr), _p(_c(kv_cache, np.uint16)), *batch.args(),
                                        _p(_c(W_UK, np.float64)), _p(_c(W_UV, np.float64)),
                                        _p(ix), ix.shape[1], H, sm_scale, _p(out)),
           "unabsorbed_attn")
    return out


def decode(inp, wl, k_cache=None, ld: int | None = None):
    """The whole chain on host arrays of a synthetic workload.

    Returns dict(k_cache, scores, idx, out, lse).  k_cache is a copy of the
    input cache with the new keys appended.
    """
    b = Batch.of(wl)
    kc = np.array(inp.k_cache if k_cache is None else k_cache, dtype=np.float16, copy=True)
    T = wl.T
    ld = int(ld if ld is not None else wl.max_kv)
    scores = np.empty((T, ld), np.float64)
    idx = np.empty((T, wl.top_k), np.int32)
    out = np.empty((T, wl.H, 512), np.float64)
    lse = np.empty((T, wl.H), np.float64)
    kn = _c(inp.k_new, np.float32)
    _check(lib().oracle_decode(_p(kn), 0, _p(_c(inp.q_idx, np.float16)), _p(_c(inp.w, np.float32)),
                               _p(_c(inp.q_lat, np.uint16)), _p(_c(inp.q_rope, np.uint16)),
                               _p(kc), _p(_c(inp.kv_cache, np.uint16)), *b.args(),
                               wl.H_I, wl.H, wl.top_k, wl.sm_scale, int(wl.hadamard),
                               _p(scores), ld, _p(idx), _p(out), _p(lse)), "decode")
    return dict(k_cache=kc, scores=scores, idx=idx, out=out, lse=lse)


# ---------------------------------------------------------------- kpool indexer
# GLM-5.3-Flash (vllm-rdna PR #2 "Glm5Next (GLM-5.3-Flash) on gfx1030"): the
# reading is stated in dsa_oracle.h.

KPOOL = 4
KPOOL_ROW = 257


def kpool_width(top_k: int) -> int:
    """Index entries per token: floor(top_k / 4) pools of 4 positions plus a
    tail of at most 3 (2051 for top_k = 2048)."""
    return (top_k // KPOOL) * KPOOL + KPOOL - 1


def kpool_write_rows(k_new, gate_new, batch: Batch, rows: np.ndarray) -> None:
    """Packed rows k|gate|1.0 (fp16, [rows, 257]) of the new tokens, in place."""
    assert rows.dtype == np.float16 and rows.flags.c_contiguous and rows.shape[1] == KPOOL_ROW
    _check(lib().oracle_kpool_write_rows(_p(_c(k_new, np.float16)), _p(_c(gate_new, np.float16)), *batch.args(),
                                         _p(rows)), "kpool_write_rows")


def kpool_pool_key(seq_rows, j: int, ape):
    """(has_key, key fp16 [128]) of pool j of a sequence's packed rows."""
    r = _c(seq_rows, np.float16)
    key = np.zeros(128, np.float16)
    has = lib().oracle_kpool_pool_key(_p(r), int(j), _p(_c(ape, np.float32)), _p(key))
    return bool(has), key


def kpool_select(q_idx, w, rows, ape, batch: Batch, top_k: int, scores: bool = False):
    """Token positions [T, kpool_width(top_k)] (and, with scores, the pool
    scores [T, max pools])."""
    q = _c(q_idx, np.float16)
    T, H_I, _ = q.shape
    width = kpool_width(top_k)
    idx = np.empty((T, width), np.int32)
    ld = int(max(1, (int(batch.q_pos.max()) + 1) // KPOOL)) if T else 1
    sc = np.empty((T, ld), np.float64) if scores else None
    _check(lib().oracle_kpool_select(_p(q), _p(_c(w, np.float32)), _p(_c(rows, np.float16)), _p(_c(ape, np.float32)),
                                     *batch.args(), H_I, top_k, _p(idx), _p(sc), ld), "kpool_select")
    return (idx, sc) if scores else idx
