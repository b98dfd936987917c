"""Seeded synthetic inputs for the DSA hot path.

This module is shared by the CPU oracle's tests and by the CUDA path's tests
and benchmark.  It holds only random numbers, storage rounding and workload
shapes -- none of the method's arithmetic (no scores, no selection, no
attention).

Generator.  Every element is drawn from a counter, so any element can be
regenerated alone:

    x      = (seed << 44) | (tensor_id << 36) | 2*e      (e = flat element index)
    h1, h2 = splitmix64(x), splitmix64(x + 1)            (Steele, Lea, Flood 2014)
    u1     = ((h1 >> 11) + 1) * 2**-53                   in (0, 1]
    u2     =  (h2 >> 11)      * 2**-53                   in [0, 1)
    z      = sqrt(-2 ln u1) * cos(2 pi u2)               (Box-Muller, float64)
    value  = round_to_storage_dtype(z * scale)           (RNE from float64)

All values are produced on the host with numpy and copied to the device, so
both sides see identical bits.  fp16 rounding uses numpy's float64->float16
conversion (round-to-nearest-even); bf16 rounding is done directly from the
float64 bits (no float32 double rounding).
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

_M64 = np.uint64(0xFFFFFFFFFFFFFFFF)

# Tensor ids: one per logical input so that draws never overlap.
TID_K_CACHE = 1
TID_K_NEW = 2
TID_Q_IDX = 3
TID_W = 4
TID_Q_LAT = 5
TID_Q_ROPE = 6
TID_KV_CACHE = 7
TID_LENGTHS = 8
TID_W_UK = 9
TID_W_UV = 10
TID_Q_NOPE = 11
TID_SCORES = 12
TID_GATE_CACHE = 13
TID_GATE_NEW = 14
TID_APE = 15


def splitmix64(x: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser on a uint64 array (wrapping arithmetic)."""
    with np.errstate(over="ignore"):
        z = x + np.uint64(0x9E3779B97F4A7C15)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        return z ^ (z >> np.uint64(31))


def _base(seed: int, tensor_id: int) -> np.uint64:
    return np.uint64(((seed & 0xFFFFF) << 44) | ((tensor_id & 0xFF) << 36))


def standard_normal_at(seed: int, tensor_id: int, elems: np.ndarray) -> np.ndarray:
    """Standard normal draws (float64) for the given flat element indices."""
    e = np.asarray(elems, dtype=np.uint64)
    x = _base(seed, tensor_id) | (e << np.uint64(1))
    h1 = splitmix64(x)
    h2 = splitmix64(x + np.uint64(1))
    u1 = ((h1 >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u2 = (h2 >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)


def uniform_u64_at(seed: int, tensor_id: int, elems: np.ndarray) -> np.ndarray:
    """Raw 64-bit draws for the given flat element indices."""
    e = np.asarray(elems, dtype=np.uint64)
    return splitmix64(_base(seed, tensor_id) | (e << np.uint64(1)))


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 to bfloat16 (RNE, directly from the float64 bits).

    Valid for finite inputs whose magnitude is zero or within the normal bf16
    range, which the generator guarantees.  Returns uint16 bit patterns.
    """
    b = np.ascontiguousarray(x, dtype=np.float64).view(np.uint64)
    lsb = (b >> np.uint64(45)) & np.uint64(1)
    with np.errstate(over="ignore"):
        b = b + np.uint64((1 << 44) - 1) + lsb
    b = b & ~np.uint64((1 << 45) - 1)
    f32 = b.view(np.float64).astype(np.float32)  # exact: at most 8 significant bits
    return (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


_POOL: ThreadPoolExecutor | None = None


def _pool() -> ThreadPoolExecutor:
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1)))
    return _POOL


def normal(seed: int, tensor_id: int, shape, scale: float, dtype: str,
           chunk: int = 1 << 22) -> np.ndarray:
    """A whole tensor of scaled normal draws in storage dtype.

    dtype: 'f16' -> np.float16, 'bf16' -> np.uint16 bit patterns,
           'f32' -> np.float32, 'f64' -> np.float64.
    """
    n = int(np.prod(shape)) if len(shape) else 1
    out_dt = {"f16": np.float16, "bf16": np.uint16, "f32": np.float32, "f64": np.float64}[dtype]
    out = np.empty(n, dtype=out_dt)

    def work(lo: int) -> None:
        hi = min(n, lo + chunk)
        z = standard_normal_at(seed, tensor_id, np.arange(lo, hi, dtype=np.uint64)) * scale
        if dtype == "bf16":
            out[lo:hi] = f64_to_bf16_bits(z)
        else:
            out[lo:hi] = z.astype(out_dt)

    if n <= chunk:
        work(0)
    else:
        list(_pool().map(work, range(0, n, chunk)))
    return out.reshape(shape)


# ---------------------------------------------------------------------------
# Workloads
# ---------------------------------------------------------------------------

D_I = 128       # indexer head dim
D_L = 512       # latent width
D_R = 64        # rope tail width
D_ROW = D_L + D_R


@dataclass
class Workload:
    """Shapes and positions of one synthetic batch.

    Sequences are packed back to back in the pooled caches: sequence b owns
    cache rows kv_off[b] .. kv_off[b] + kv_len[b] - 1.  Query token t of
    sequence b sits at absolute position q_pos[t]; its own indexer key is
    appended at that position before scoring.
    """
    name: str
    seed: int
    kv_len: list            # cache length per sequence
    q_pos: list             # absolute position per query token (T)
    cu_q: list              # query offsets per sequence (B+1)
    H_I: int
    H: int
    top_k: int
    hadamard: bool = False
    sm_scale: float = 1.0 / math.sqrt(192.0)
    extra: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return len(self.kv_len)

    @property
    def T(self) -> int:
        return len(self.q_pos)

    @property
    def kv_off(self) -> list:
        off, acc = [], 0
        for L in self.kv_len:
            off.append(acc)
            acc += L
        return off

    @property
    def cache_rows(self) -> int:
        return int(sum(self.kv_len))

    @property
    def max_kv(self) -> int:
        return max(p + 1 for p in self.q_pos)

    @property
    def max_q_per_seq(self) -> int:
        return max(self.cu_q[b + 1] - self.cu_q[b] for b in range(self.B))


def decode_workload(name, seed, lengths, H_I, H, top_k, hadamard=False) -> Workload:
    B = len(lengths)
    return Workload(name=name, seed=seed, kv_len=list(lengths),
                    q_pos=[L - 1 for L in lengths], cu_q=list(range(B + 1)),
                    H_I=H_I, H=H, top_k=top_k, hadamard=hadamard)


def prefill_workload(name, seed, cached, T, H_I, H, top_k, hadamard=False) -> Workload:
    return Workload(name=name, seed=seed, kv_len=[cached + T],
                    q_pos=[cached + i for i in range(T)], cu_q=[0, T],
                    H_I=H_I, H=H, top_k=top_k, hadamard=hadamard)


def ragged_lengths(seed: int, B: int, lo: int = 4096, hi: int = 65536) -> list:
    """Per-sequence lengths uniform on [lo, hi] drawn from the counter."""
    u = uniform_u64_at(seed, TID_LENGTHS, np.arange(B, dtype=np.uint64))
    return [int(lo + int(v) % (hi - lo + 1)) for v in u]


def config(i: int, **over) -> Workload:
    """The five standard workloads (1-based index).

    1 tiny decode; 2 batched decode; 3 ragged long-context decode with the
    Hadamard rotation; 4 prefill chunk; 5 long prefill.
    """
    if i == 1:
        w = decode_workload("tiny_decode_L256", 0, [256], H_I=4, H=8, top_k=64)
    elif i == 2:
        w = decode_workload("batched_decode_B8_L8192", 1, [8192] * 8, H_I=32, H=64, top_k=2048)
    elif i == 3:
        w = decode_workload("ragged_decode_B32_L4k-64k", 2, ragged_lengths(2, 32),
                            H_I=64, H=64, top_k=2048, hadamard=True)
    elif i == 4:
        w = prefill_workload("prefill_T4096_after4096", 3, 4096, 4096, H_I=64, H=64, top_k=2048)
    elif i == 5:
        w = prefill_workload("prefill_T16384_after114688", 4, 114688, 16384, H_I=64, H=64, top_k=2048)
    else:
        raise ValueError(f"no workload {i}")
    for k, v in over.items():
        setattr(w, k, v)
    return w


@dataclass
class Inputs:
    """Host arrays of one workload (storage dtypes as numpy arrays).

    k_cache   float16 [rows, 128]   indexer keys; the rows of the query
                                    tokens' own positions hold stale draws
                                    until the append writes them
    k_new     float32 [T, 128]      new indexer keys (unrotated)
    q_idx     float16 [T, H_I, 128] indexer queries (unrotated)
    w         float32 [T, H_I]      per-head indexer weights
    q_lat     uint16  [T, H, 512]   bf16 bits, absorbed latent queries
    q_rope    uint16  [T, H, 64]    bf16 bits, rope queries
    kv_cache  uint16  [rows, 576]   bf16 bits, latent rows (512 latent + 64 rope)
    """
    k_cache: np.ndarray
    k_new: np.ndarray
    q_idx: np.ndarray
    w: np.ndarray
    q_lat: np.ndarray
    q_rope: np.ndarray
    kv_cache: np.ndarray


def make_inputs(wl: Workload, parts=("k_cache", "k_new", "q_idx", "w", "q_lat", "q_rope", "kv_cache")) -> Inputs:
    s = wl.seed
    rows, T = wl.cache_rows, wl.T
    g = {}
    if "k_cache" in parts:
        g["k_cache"] = normal(s, TID_K_CACHE, (rows, D_I), 1 / math.sqrt(D_I), "f16")
    if "k_new" in parts:
        g["k_new"] = normal(s, TID_K_NEW, (T, D_I), 1 / math.sqrt(D_I), "f32")
    if "q_idx" in parts:
        g["q_idx"] = normal(s, TID_Q_IDX, (T, wl.H_I, D_I), 1 / math.sqrt(D_I), "f16")
    if "w" in parts:
        g["w"] = normal(s, TID_W, (T, wl.H_I), 1 / math.sqrt(wl.H_I), "f32")
    if "q_lat" in parts:
        g["q_lat"] = normal(s, TID_Q_LAT, (T, wl.H, D_L), 1 / math.sqrt(D_L), "bf16")
    if "q_rope" in parts:
        g["q_rope"] = normal(s, TID_Q_ROPE, (T, wl.H, D_R), 1 / math.sqrt(D_R), "bf16")
    if "kv_cache" in parts:
        g["kv_cache"] = normal(s, TID_KV_CACHE, (rows, D_ROW), 1 / math.sqrt(D_ROW), "bf16")
    return Inputs(**{k: g.get(k) for k in Inputs.__dataclass_fields__})


def batch_arrays(wl: Workload):
    """cu_q int32 [B+1], q_pos int32 [T], kv_off int64 [B] as numpy arrays."""
    return (np.asarray(wl.cu_q, dtype=np.int32),
            np.asarray(wl.q_pos, dtype=np.int32),
            np.asarray(wl.kv_off, dtype=np.int64))


# ---------------------------------------------------------------------------
# kpool indexer inputs (GLM-5.3-Flash DSA layers: MLA-NoPE latent rows of 512
# and packed indexer rows of 257 fp16 values, k | gate | valid)
# ---------------------------------------------------------------------------

KPOOL_ROW = 257


@dataclass
class KpoolInputs:
    """Host arrays of a kpool workload.

    rows      float16 [rows, 257]   packed indexer rows: k (N(0,1)/sqrt(128)) |
                                    gate (N(0,1)) | valid (1.0); the query
                                    tokens' own rows hold stale draws until
                                    the append writes them
    k_new     float16 [T, 128]      new indexer keys
    gate_new  float16 [T, 128]      new gate values
    ape       float32 [4, 128]      position-in-pool embedding, N(0,1)
    q_idx     float16 [T, H_I, 128] indexer queries
    w         float32 [T, H_I]      per-head indexer weights
    q_lat     uint16  [T, H, 512]   bf16 bits, latent queries
    kv_latent uint16  [rows, 512]   bf16 bits, latent rows (no rope tail)
    """
    rows: np.ndarray
    k_new: np.ndarray
    gate_new: np.ndarray
    ape: np.ndarray
    q_idx: np.ndarray
    w: np.ndarray
    q_lat: np.ndarray
    kv_latent: np.ndarray


def pack_kpool_rows(k: np.ndarray, gate: np.ndarray, valid=None) -> np.ndarray:
    """The packed row layout: k (128) | gate (128) | valid (1) as fp16."""
    n = k.shape[0]
    rows = np.empty((n, KPOOL_ROW), np.float16)
    rows[:, :D_I] = k
    rows[:, D_I:2 * D_I] = gate
    rows[:, 2 * D_I] = 1.0 if valid is None else valid
    return rows


def make_kpool_inputs(wl: Workload) -> KpoolInputs:
    s = wl.seed
    rows, T = wl.cache_rows, wl.T
    k = normal(s, TID_K_CACHE, (rows, D_I), 1 / math.sqrt(D_I), "f16")
    g = normal(s, TID_GATE_CACHE, (rows, D_I), 1.0, "f16")
    return KpoolInputs(
        rows=pack_kpool_rows(k, g),
        k_new=normal(s, TID_K_NEW, (T, D_I), 1 / math.sqrt(D_I), "f16"),
        gate_new=normal(s, TID_GATE_NEW, (T, D_I), 1.0, "f16"),
        ape=normal(s, TID_APE, (4, D_I), 1.0, "f32"),
        q_idx=normal(s, TID_Q_IDX, (T, wl.H_I, D_I), 1 / math.sqrt(D_I), "f16"),
        w=normal(s, TID_W, (T, wl.H_I), 1 / math.sqrt(wl.H_I), "f32"),
        q_lat=normal(s, TID_Q_LAT, (T, wl.H, D_L), 1 / math.sqrt(D_L), "bf16"),
        kv_latent=normal(s, TID_KV_CACHE, (rows, D_L), 1 / math.sqrt(D_L), "bf16"))
