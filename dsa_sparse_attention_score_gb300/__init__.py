"""Python binding of the GB300 DSA hot-path library (libdsa_gb300.so).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current stream.  The
functions carry the C-ABI names and raise DsaError on any non-OK status.
There is no fallback: if the compiled library is missing, loading raises.

Tensor conventions (all CUDA, contiguous):
  fp16 tensors are torch.float16, bf16 tensors torch.bfloat16,
  positions torch.int32, offsets torch.int64, scores/outputs torch.float32.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdsa_gb300.so")

DSA_OK = 0
DSA_ERR_INVALID_ARGUMENT = 1
DSA_ERR_UNSUPPORTED = 2
DSA_ERR_MISALIGNED = 3
DSA_ERR_WORKSPACE_TOO_SMALL = 4
DSA_ERR_CUDA = 5
DSA_ERR_DEVICE = 6

DSA_DEV_BAD_POSITION = 1
DSA_DEV_BAD_INDEX = 2
DSA_DEV_TIMEOUT = 4
DSA_DEV_SMEM_LAYOUT = 8

DSA_KEY_F32 = 0
DSA_KEY_F16 = 1

DSA_OP_K_APPEND = 0
DSA_OP_INDEXER_SCORE = 1
DSA_OP_TOPK = 2
DSA_OP_SPARSE_ATTN = 3
DSA_OP_DECODE = 4
DSA_OP_KPOOL = 5

KPOOL = 4            # positions per pool of the kpool indexer
KPOOL_ROW = 257      # fp16 values per packed indexer row: k | gate | valid

# Every symbol the header declares, with (restype, argtypes).
_P = C.c_void_p
_I = C.c_int
_I64 = C.c_int64
_SZ = C.c_size_t
_F = C.c_float


class dsa_batch_t(C.Structure):
    _fields_ = [("batch", C.c_int32), ("total_q", C.c_int32), ("max_q_per_seq", C.c_int32),
                ("max_kv", C.c_int32), ("cache_rows", C.c_int64), ("cu_q", _P), ("q_pos", _P),
                ("kv_off", _P)]


_BP = C.POINTER(dsa_batch_t)
SIGNATURES = {
    "dsa_indexer_k_append": (_I, [_P, _I, _BP, _P, _I, _P, _SZ, _P]),
    "dsa_indexer_score": (_I, [_P, _P, _P, _BP, _I, _I, _P, _I64, _P, _SZ, _P]),
    "dsa_topk": (_I, [_P, _I64, _BP, _I, _P, _P, _SZ, _P]),
    "dsa_topk_sink": (_I, [_P, _I64, _BP, _I, _I, _P, _P, _P, _SZ, _P]),
    "dsa_sparse_mla_attn": (_I, [_P, _P, _P, _BP, _P, _I, _I, _F, _P, _P, _P, _SZ, _P]),
    "dsa_sparse_mla_attn_nope": (_I, [_P, _P, _BP, _P, _I, _I, _F, _P, _P, _P, _SZ, _P]),
    "dsa_decode": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _BP, _I, _I, _I, _F, _I, _P, _P, _P, _P, _SZ, _P]),
    "dsa_decode_sink": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _BP, _I, _I, _I, _F, _I, _I, _P, _P, _P, _P, _P,
                             _SZ, _P]),
    "dsa_decode_paged": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _BP, C.c_void_p, _I, _I, _I, _F, _I, _P, _P, _P, _P,
                              _SZ, _P]),
    "dsa_decode_noalloc": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _BP, _I, _I, _I, _F, _I, _P, _P, _P, _P]),
    "dsa_workspace_size": (_I, [_I, _BP, _I, _I, _I, C.POINTER(C.c_size_t)]),
    "dsa_workspace_init": (_I, [_P, _SZ, _P]),
    "dsa_decode_launches": (_I, [_BP, _I, _I, _I, C.POINTER(C.c_int)]),
    "dsa_read_device_status": (_I, [_P, _P, C.POINTER(C.c_uint32)]),
    "dsa_status_string": (C.c_char_p, [_I]),
    "dsa_set_trace_events": (_I, [_P, _I]),
    "dsa_set_timeline": (_I, [_P]),
    "dsa_set_test_faults": (_I, [C.c_uint64, _I]),
    "dsa_kpool_append": (_I, [_P, _P, _P, _BP, _P, _P, _I64, _P, _SZ, _P]),
    "dsa_kpool_select": (_I, [_P, _P, _P, _P, _I64, _BP, _I, _I, _P, _P, _SZ, _P]),
    "dsa_decode_kpool": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _P, _BP, _I, _I, _I, _F, _P, _P, _P, _P, _SZ,
                              _P]),
    "dsa_version": (_I, []),
}

_LIB = None


class DsaError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {lib().dsa_status_string(code).decode()} (code {code})")


def lib():
    """The loaded CUDA library.  Raises if it has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: run dsa_sparse_attention_score_gb300.build.build()")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _LIB = L
    return _LIB


def _check(code: int, what: str):
    if code != DSA_OK:
        raise DsaError(code, what)


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


# Fixed innermost extents of the tensors the calls take (include/dsa.h).
_WIDTH = {"k_new": 128, "gate_new": 128, "ape": 128, "q_idx": 128, "k_cache": 128, "q_lat": 512, "q_rope": 64, "kv_cache": 576,
          "kv_latent": 512, "out": 512}


def _req(t, dtype, name):
    if t is None:
        return
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise TypeError(f"{name}: expected a contiguous CUDA {dtype} tensor, got {t.dtype} on {t.device}")
    if name in _WIDTH and (t.dim() < 2 or t.shape[-1] != _WIDTH[name]):
        raise TypeError(f"{name}: expected rows of {_WIDTH[name]} elements, got shape {tuple(t.shape)}")


@dataclass
class Batch:
    """Device batch description plus its host bounds."""
    cu_q: object           # int32 [B+1]
    q_pos: object          # int32 [T]
    kv_off: object         # int64 [B]
    max_q_per_seq: int
    max_kv: int
    cache_rows: int

    @classmethod
    def from_host(cls, cu_q, q_pos, kv_off, cache_rows: int, device="cuda",
                  max_q_per_seq: int | None = None, max_kv: int | None = None):
        import torch
        cu = torch.as_tensor(list(cu_q), dtype=torch.int32)
        qp = torch.as_tensor(list(q_pos), dtype=torch.int32)
        ko = torch.as_tensor(list(kv_off), dtype=torch.int64)
        mq = max_q_per_seq if max_q_per_seq is not None else int((cu[1:] - cu[:-1]).max())
        mk = max_kv if max_kv is not None else int(qp.max()) + 1
        return cls(cu.to(device), qp.to(device), ko.to(device), mq, mk, int(cache_rows))

    @property
    def B(self) -> int:
        return self.cu_q.numel() - 1

    @property
    def T(self) -> int:
        return self.q_pos.numel()

    def desc(self) -> dsa_batch_t:
        import torch
        _req(self.cu_q, torch.int32, "cu_q")
        _req(self.q_pos, torch.int32, "q_pos")
        _req(self.kv_off, torch.int64, "kv_off")
        return dsa_batch_t(self.B, self.T, self.max_q_per_seq, self.max_kv, self.cache_rows,
                           self.cu_q.data_ptr(), self.q_pos.data_ptr(), self.kv_off.data_ptr())


def dsa_workspace_size(op: int, batch: Batch, H_I: int, H: int, k: int) -> int:
    n = C.c_size_t(0)
    d = dsa_batch_t(batch.B, batch.T, batch.max_q_per_seq, batch.max_kv, batch.cache_rows, None, None, None)
    _check(lib().dsa_workspace_size(op, C.byref(d), H_I, H, k, C.byref(n)), "dsa_workspace_size")
    return n.value


def dsa_decode_launches(batch: Batch, H_I: int, H: int, k: int) -> int:
    n = C.c_int(0)
    d = dsa_batch_t(batch.B, batch.T, batch.max_q_per_seq, batch.max_kv, batch.cache_rows, None, None, None)
    _check(lib().dsa_decode_launches(C.byref(d), H_I, H, k, C.byref(n)), "dsa_decode_launches")
    return n.value


def dsa_workspace_init(ws, stream=None):
    _check(lib().dsa_workspace_init(_ptr(ws), ws.numel(), _stream(stream)), "dsa_workspace_init")


def workspace(op: int, batch: Batch, H_I: int = 1, H: int = 1, k: int = 1, device="cuda"):
    """Allocate (with torch) and initialise a workspace for `op`."""
    import torch
    n = dsa_workspace_size(op, batch, H_I, H, k)
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    dsa_workspace_init(ws)
    return ws


def dsa_read_device_status(ws, stream=None) -> int:
    """Synchronises the stream; returns and clears the DSA_DEV_* bits."""
    f = C.c_uint32(0)
    code = lib().dsa_read_device_status(_ptr(ws), _stream(stream), C.byref(f))
    if code not in (DSA_OK, DSA_ERR_DEVICE):
        raise DsaError(code, "dsa_read_device_status")
    return f.value


def dsa_indexer_k_append(k_new, batch: Batch, k_cache, hadamard: bool, ws, stream=None):
    import torch
    kd = DSA_KEY_F16 if k_new.dtype == torch.float16 else DSA_KEY_F32
    _req(k_new, torch.float16 if kd == DSA_KEY_F16 else torch.float32, "k_new")
    _req(k_cache, torch.float16, "k_cache")
    d = batch.desc()
    _check(lib().dsa_indexer_k_append(_ptr(k_new), kd, C.byref(d), _ptr(k_cache), int(hadamard),
                                      _ptr(ws), ws.numel(), _stream(stream)), "dsa_indexer_k_append")


def dsa_indexer_score(q_idx, w, k_cache, batch: Batch, hadamard_q: bool, scores, ws, stream=None):
    import torch
    _req(q_idx, torch.float16, "q_idx")
    _req(w, torch.float32, "w")
    _req(k_cache, torch.float16, "k_cache")
    _req(scores, torch.float32, "scores")
    d = batch.desc()
    _check(lib().dsa_indexer_score(_ptr(q_idx), _ptr(w), _ptr(k_cache), C.byref(d), q_idx.shape[1],
                                   int(hadamard_q), _ptr(scores), scores.shape[1], _ptr(ws), ws.numel(),
                                   _stream(stream)), "dsa_indexer_score")


def dsa_topk(scores, batch: Batch, k: int, idx, ws, stream=None):
    import torch
    _req(scores, torch.float32, "scores")
    _req(idx, torch.int32, "idx")
    d = batch.desc()
    _check(lib().dsa_topk(_ptr(scores), scores.shape[1], C.byref(d), k, _ptr(idx), _ptr(ws), ws.numel(),
                          _stream(stream)), "dsa_topk")


def dsa_topk_sink(scores, batch: Batch, k: int, n_sink: int, sink_pos0, idx, ws, stream=None):
    """dsa_topk with the first n_sink positions of each sequence (from
    sink_pos0[b], an int32 CUDA tensor [B], or 0 when None) forced in."""
    import torch
    _req(scores, torch.float32, "scores")
    _req(idx, torch.int32, "idx")
    _req(sink_pos0, torch.int32, "sink_pos0")
    d = batch.desc()
    _check(lib().dsa_topk_sink(_ptr(scores), scores.shape[1], C.byref(d), k, n_sink, _ptr(sink_pos0), _ptr(idx),
                               _ptr(ws), ws.numel(), _stream(stream)), "dsa_topk_sink")


def dsa_sparse_mla_attn(q_lat, q_rope, kv_cache, batch: Batch, idx, sm_scale: float, out, lse, ws,
                        stream=None):
    import torch
    _req(q_lat, torch.bfloat16, "q_lat")
    _req(q_rope, torch.bfloat16, "q_rope")
    _req(kv_cache, torch.bfloat16, "kv_cache")
    _req(idx, torch.int32, "idx")
    _req(out, torch.float32, "out")
    _req(lse, torch.float32, "lse")
    d = batch.desc()
    _check(lib().dsa_sparse_mla_attn(_ptr(q_lat), _ptr(q_rope), _ptr(kv_cache), C.byref(d), _ptr(idx),
                                     idx.shape[1], q_lat.shape[1], sm_scale, _ptr(out), _ptr(lse),
                                     _ptr(ws), ws.numel(), _stream(stream)), "dsa_sparse_mla_attn")


def dsa_sparse_mla_attn_nope(q_lat, kv_latent, batch: Batch, idx, sm_scale: float, out, lse, ws, stream=None):
    """MLA-NoPE: q_lat [T,H,512] against latent rows kv_latent [rows,512] (no rope tail)."""
    import torch
    _req(q_lat, torch.bfloat16, "q_lat")
    _req(kv_latent, torch.bfloat16, "kv_latent")
    _req(idx, torch.int32, "idx")
    _req(out, torch.float32, "out")
    _req(lse, torch.float32, "lse")
    d = batch.desc()
    _check(lib().dsa_sparse_mla_attn_nope(_ptr(q_lat), _ptr(kv_latent), C.byref(d), _ptr(idx), idx.shape[1],
                                          q_lat.shape[1], sm_scale, _ptr(out), _ptr(lse), _ptr(ws), ws.numel(),
                                          _stream(stream)), "dsa_sparse_mla_attn_nope")


def dsa_decode(k_new, q_idx, w, q_lat, q_rope, k_cache, kv_cache, batch: Batch, k: int, sm_scale: float,
               hadamard: bool, out, lse, idx_out, ws, stream=None):
    import torch
    kd = DSA_KEY_F16 if k_new.dtype == torch.float16 else DSA_KEY_F32
    _req(k_new, torch.float16 if kd == DSA_KEY_F16 else torch.float32, "k_new")
    _req(q_idx, torch.float16, "q_idx")
    _req(w, torch.float32, "w")
    _req(q_lat, torch.bfloat16, "q_lat")
    _req(q_rope, torch.bfloat16, "q_rope")
    _req(k_cache, torch.float16, "k_cache")
    _req(kv_cache, torch.bfloat16, "kv_cache")
    _req(out, torch.float32, "out")
    _req(lse, torch.float32, "lse")
    _req(idx_out, torch.int32, "idx_out")
    d = batch.desc()
    _check(lib().dsa_decode(_ptr(k_new), kd, _ptr(q_idx), _ptr(w), _ptr(q_lat), _ptr(q_rope), _ptr(k_cache),
                            _ptr(kv_cache), C.byref(d), q_idx.shape[1], q_lat.shape[1], k, sm_scale,
                            int(hadamard), _ptr(out), _ptr(lse), _ptr(idx_out), _ptr(ws), ws.numel(),
                            _stream(stream)), "dsa_decode")


class dsa_paging_t(C.Structure):
    _fields_ = [("block_table", C.c_void_p), ("max_blocks", C.c_int32), ("block_size", C.c_int32)]


def dsa_decode_paged(k_new, q_idx, w, q_lat, q_rope, k_cache, kv_cache, batch: Batch, block_table,
                     block_size: int, k: int, sm_scale: float, hadamard: bool, out, lse, idx_out, ws,
                     stream=None):
    """dsa_decode over paged caches: block_table is an int32 CUDA tensor
    [B, max_blocks]; position pos of sequence b lives at cache row
    block_table[b, pos // block_size] * block_size + pos % block_size."""
    import torch
    kd = DSA_KEY_F16 if k_new.dtype == torch.float16 else DSA_KEY_F32
    _req(k_new, torch.float16 if kd == DSA_KEY_F16 else torch.float32, "k_new")
    _req(q_idx, torch.float16, "q_idx")
    _req(w, torch.float32, "w")
    _req(q_lat, torch.bfloat16, "q_lat")
    _req(q_rope, torch.bfloat16, "q_rope")
    _req(k_cache, torch.float16, "k_cache")
    _req(kv_cache, torch.bfloat16, "kv_cache")
    _req(block_table, torch.int32, "block_table")
    _req(out, torch.float32, "out")
    _req(lse, torch.float32, "lse")
    _req(idx_out, torch.int32, "idx_out")
    d = batch.desc()
    pg = dsa_paging_t(block_table.data_ptr(), block_table.shape[1], block_size)
    _check(lib().dsa_decode_paged(_ptr(k_new), kd, _ptr(q_idx), _ptr(w), _ptr(q_lat), _ptr(q_rope), _ptr(k_cache),
                                  _ptr(kv_cache), C.byref(d), C.byref(pg), q_idx.shape[1], q_lat.shape[1], k,
                                  sm_scale, int(hadamard), _ptr(out), _ptr(lse), _ptr(idx_out), _ptr(ws),
                                  ws.numel(), _stream(stream)), "dsa_decode_paged")


def dsa_decode_sink(k_new, q_idx, w, q_lat, q_rope, k_cache, kv_cache, batch: Batch, k: int, sm_scale: float,
                    hadamard: bool, n_sink: int, sink_pos0, out, lse, idx_out, ws, stream=None):
    """dsa_decode with the attention sink forced into every selection (see
    dsa_topk_sink)."""
    import torch
    kd = DSA_KEY_F16 if k_new.dtype == torch.float16 else DSA_KEY_F32
    _req(k_new, torch.float16 if kd == DSA_KEY_F16 else torch.float32, "k_new")
    _req(q_idx, torch.float16, "q_idx")
    _req(w, torch.float32, "w")
    _req(q_lat, torch.bfloat16, "q_lat")
    _req(q_rope, torch.bfloat16, "q_rope")
    _req(k_cache, torch.float16, "k_cache")
    _req(kv_cache, torch.bfloat16, "kv_cache")
    _req(sink_pos0, torch.int32, "sink_pos0")
    _req(out, torch.float32, "out")
    _req(lse, torch.float32, "lse")
    _req(idx_out, torch.int32, "idx_out")
    d = batch.desc()
    _check(lib().dsa_decode_sink(_ptr(k_new), kd, _ptr(q_idx), _ptr(w), _ptr(q_lat), _ptr(q_rope), _ptr(k_cache),
                                 _ptr(kv_cache), C.byref(d), q_idx.shape[1], q_lat.shape[1], k, sm_scale,
                                 int(hadamard), n_sink, _ptr(sink_pos0), _ptr(out), _ptr(lse), _ptr(idx_out),
                                 _ptr(ws), ws.numel(), _stream(stream)), "dsa_decode_sink")


def dsa_decode_noalloc(k_new, q_idx, w, q_lat, q_rope, k_cache, kv_cache, batch: Batch, k: int,
                       sm_scale: float, hadamard: bool, out, lse, idx_out, stream=None):
    """dsa_decode with the library's static scratch instead of a workspace
    (for callers that cannot allocate device memory)."""
    import torch
    kd = DSA_KEY_F16 if k_new.dtype == torch.float16 else DSA_KEY_F32
    _req(k_new, torch.float16 if kd == DSA_KEY_F16 else torch.float32, "k_new")
    _req(q_idx, torch.float16, "q_idx")
    _req(w, torch.float32, "w")
    _req(q_lat, torch.bfloat16, "q_lat")
    _req(q_rope, torch.bfloat16, "q_rope")
    _req(k_cache, torch.float16, "k_cache")
    _req(kv_cache, torch.bfloat16, "kv_cache")
    _req(out, torch.float32, "out")
    _req(lse, torch.float32, "lse")
    _req(idx_out, torch.int32, "idx_out")
    d = batch.desc()
    _check(lib().dsa_decode_noalloc(_ptr(k_new), kd, _ptr(q_idx), _ptr(w), _ptr(q_lat), _ptr(q_rope),
                                    _ptr(k_cache), _ptr(kv_cache), C.byref(d), q_idx.shape[1], q_lat.shape[1], k,
                                    sm_scale, int(hadamard), _ptr(out), _ptr(lse), _ptr(idx_out),
                                    _stream(stream)), "dsa_decode_noalloc")


def kpool_width(top_k: int) -> int:
    """Positions per token of a kpool selection: 4 * floor(top_k / 4) + 3."""
    return (top_k // KPOOL) * KPOOL + KPOOL - 1


def _req_rows(rows):
    import torch
    if not rows.is_cuda or rows.dtype != torch.float16 or not rows.is_contiguous() or rows.dim() != 2 \
            or rows.shape[1] != KPOOL_ROW:
        raise TypeError(f"idx_rows: expected a contiguous CUDA float16 [rows, {KPOOL_ROW}] tensor")


def dsa_kpool_append(k_new, gate_new, ape, batch: Batch, idx_rows, pool_keys, ws, stream=None):
    """Packed rows k|gate|1.0 of the new tokens and the pooled key of every
    pool they complete (GLM-5.3-Flash kpool indexer)."""
    import torch
    _req(k_new, torch.float16, "k_new")
    _req(gate_new, torch.float16, "gate_new")
    _req(ape, torch.float32, "ape")
    _req_rows(idx_rows)
    _req(pool_keys, torch.float16, "k_cache")
    d = batch.desc()
    _check(lib().dsa_kpool_append(_ptr(k_new), _ptr(gate_new), _ptr(ape), C.byref(d), _ptr(idx_rows),
                                  _ptr(pool_keys), pool_keys.shape[0], _ptr(ws), ws.numel(), _stream(stream)),
           "dsa_kpool_append")


def dsa_kpool_select(q_idx, w, idx_rows, pool_keys, batch: Batch, top_k: int, idx, ws, stream=None):
    """Positions [T, kpool_width(top_k)] of the best top_k/4 pools and the tail."""
    import torch
    _req(q_idx, torch.float16, "q_idx")
    _req(w, torch.float32, "w")
    _req_rows(idx_rows)
    _req(pool_keys, torch.float16, "k_cache")
    _req(idx, torch.int32, "idx")
    d = batch.desc()
    _check(lib().dsa_kpool_select(_ptr(q_idx), _ptr(w), _ptr(idx_rows), _ptr(pool_keys), pool_keys.shape[0],
                                  C.byref(d), q_idx.shape[1], top_k, _ptr(idx), _ptr(ws), ws.numel(),
                                  _stream(stream)), "dsa_kpool_select")


def dsa_decode_kpool(k_new, gate_new, ape, q_idx, w, q_lat, idx_rows, pool_keys, kv_latent, batch: Batch, top_k: int,
                     sm_scale: float, out, lse, idx_out, ws, stream=None):
    """The fused GLM-5.3-Flash DSA step: kpool append, selection, MLA-NoPE attention."""
    import torch
    _req(k_new, torch.float16, "k_new")
    _req(gate_new, torch.float16, "gate_new")
    _req(ape, torch.float32, "ape")
    _req(q_idx, torch.float16, "q_idx")
    _req(w, torch.float32, "w")
    _req(q_lat, torch.bfloat16, "q_lat")
    _req_rows(idx_rows)
    _req(pool_keys, torch.float16, "k_cache")
    _req(kv_latent, torch.bfloat16, "kv_latent")
    _req(out, torch.float32, "out")
    _req(lse, torch.float32, "lse")
    _req(idx_out, torch.int32, "idx_out")
    d = batch.desc()
    _check(lib().dsa_decode_kpool(_ptr(k_new), _ptr(gate_new), _ptr(ape), _ptr(q_idx), _ptr(w), _ptr(q_lat),
                                  _ptr(idx_rows), _ptr(pool_keys), pool_keys.shape[0], _ptr(kv_latent), C.byref(d),
                                  q_idx.shape[1], q_lat.shape[1], top_k, sm_scale, _ptr(out), _ptr(lse),
                                  _ptr(idx_out), _ptr(ws), ws.numel(), _stream(stream)), "dsa_decode_kpool")


def dsa_set_trace_events(events):
    """events: list of torch.cuda.Event (enable_timing=True) or None to disable."""
    global _TRACE_KEEP
    if not events:
        _TRACE_KEEP = None
        _check(lib().dsa_set_trace_events(None, 0), "dsa_set_trace_events")
        return
    for e in events:
        e.record()  # makes torch create the underlying event
    arr = (C.c_void_p * len(events))(*[e.cuda_event for e in events])
    _TRACE_KEEP = arr
    _check(lib().dsa_set_trace_events(C.cast(arr, C.c_void_p), len(events)), "dsa_set_trace_events")


_TRACE_KEEP = None


def dsa_set_timeline(buf):
    """buf: CUDA int64/uint64 tensor of 10 slots, or None to disable."""
    _check(lib().dsa_set_timeline(_ptr(buf)), "dsa_set_timeline")


def dsa_set_test_faults(wait_limit_ns: int = 0, skip_copies: bool = False):
    """Failure-path test hook: bound every device wait by wait_limit_ns (0:
    the default second) and, with skip_copies, make the score and attention
    producers issue no copies so that the waits run out (DSA_DEV_TIMEOUT)."""
    _check(lib().dsa_set_test_faults(int(wait_limit_ns), int(bool(skip_copies))), "dsa_set_test_faults")


def dsa_status_string(code: int) -> str:
    return lib().dsa_status_string(code).decode()


def dsa_version() -> int:
    return lib().dsa_version()
