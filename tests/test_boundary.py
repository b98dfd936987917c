"""The C-ABI library builds, loads and exports every symbol include/dsa.h
declares; host-side validation answers before anything touches a device."""
import ctypes as C
import os
import re

import pytest

import dsa_sparse_attention_score_gb300 as dsa
from dsa_sparse_attention_score_gb300 import build as dsa_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "dsa.h")


@pytest.fixture(scope="module")
def L():
    dsa_build.build()
    return dsa.lib()


def declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_path():
    names = declared()
    for n in ("dsa_indexer_k_append", "dsa_indexer_score", "dsa_topk", "dsa_sparse_mla_attn", "dsa_decode"):
        assert n in names


def test_exports_every_declared_symbol(L):
    for name in declared():
        assert hasattr(L, name), name
    assert set(declared()) == set(dsa.SIGNATURES), "binding and header disagree"


def test_binding_signatures_match_the_header_arity():
    """Every declaration's parameter count equals the binding's argtypes."""
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    decls = re.findall(r"\b(?:dsa_status_t|int|const char\s*\*)\s*(dsa_[a-z0-9_]+)\s*\(([^;]*?)\)\s*;", src,
                       flags=re.S)
    assert {n for n, _ in decls} == set(dsa.SIGNATURES)
    for name, params in decls:
        p = params.strip()
        n = 0 if p in ("", "void") else p.count(",") + 1
        assert n == len(dsa.SIGNATURES[name][1]), name


def test_device_status_bits_match_the_header():
    """The binding's DSA_DEV_* constants are the header's enum values."""
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    bits = {name: 1 << int(sh) for name, sh in re.findall(r"\b(DSA_DEV_[A-Z_]+)\s*=\s*1u\s*<<\s*(\d+)", src)}
    assert len(bits) >= 4
    for name, value in bits.items():
        assert getattr(dsa, name) == value, name
    assert len(set(bits.values())) == len(bits), "bits overlap"


def test_version_and_status_strings(L):
    assert dsa.dsa_version() == 10100
    for code in range(0, 7):
        assert dsa.dsa_status_string(code) not in ("", "unknown status")
    assert dsa.dsa_status_string(99) == "unknown status"


def _batch(**kw):
    d = dict(batch=2, total_q=2, max_q_per_seq=1, max_kv=100, cache_rows=200,
             cu_q=0x1000, q_pos=0x2000, kv_off=0x3000)
    d.update(kw)
    return dsa.dsa_batch_t(d["batch"], d["total_q"], d["max_q_per_seq"], d["max_kv"], d["cache_rows"],
                           d["cu_q"], d["q_pos"], d["kv_off"])


def test_workspace_sizes(L):
    n = C.c_size_t()
    b = _batch()
    for op in range(5):
        assert L.dsa_workspace_size(op, C.byref(b), 32, 64, 16, C.byref(n)) == dsa.DSA_OK
        assert n.value >= 256 and n.value % 256 == 0
    # decode: status + slab + idx + split partials
    assert L.dsa_workspace_size(dsa.DSA_OP_DECODE, C.byref(b), 32, 64, 2048, C.byref(n)) == 0
    assert n.value >= 256 + 2 * 100 * 4 + 2 * 2048 * 4
    assert L.dsa_workspace_size(7, C.byref(b), 32, 64, 16, C.byref(n)) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert L.dsa_workspace_size(dsa.DSA_OP_TOPK, C.byref(b), 32, 64, 0, C.byref(n)) == dsa.DSA_ERR_UNSUPPORTED
    assert L.dsa_workspace_size(0, None, 32, 64, 16, C.byref(n)) == dsa.DSA_ERR_INVALID_ARGUMENT


def test_split_partials_stay_within_what_the_combine_merges(L):
    """One token with k = 65536 (1024 row tiles) would ask for 147 splits;
    the layout caps them at the 128 the combine kernel merges, so the
    workspace holds exactly 128 bf16 partials of 64 heads (plus their (m, l)
    in float32)."""
    n = C.c_size_t()
    b = _batch(batch=1, total_q=1, max_kv=70000, cache_rows=70000)
    assert L.dsa_workspace_size(dsa.DSA_OP_SPARSE_ATTN, C.byref(b), 4, 8, 65536, C.byref(n)) == dsa.DSA_OK
    part_o, part_ml = 128 * 64 * 512 * 2, 128 * 64 * 2 * 4
    assert n.value == 256 + part_o + part_ml


def test_head_groups_size_the_partials(L):
    """More than 64 query heads run as two head groups of 64; the split
    partials hold both groups (8 tokens x 128 heads: 8 splits of 4 tiles)."""
    n = C.c_size_t()
    b = _batch(batch=8, total_q=8, max_kv=8192, cache_rows=8 * 8192)
    assert L.dsa_workspace_size(dsa.DSA_OP_SPARSE_ATTN, C.byref(b), 64, 128, 2048, C.byref(n)) == dsa.DSA_OK
    rows = 8 * 8 * 2 * 64
    assert n.value == 256 + rows * 512 * 2 + rows * 2 * 4
    assert L.dsa_workspace_size(dsa.DSA_OP_SPARSE_ATTN, C.byref(b), 64, 129, 2048, C.byref(n)) == \
        dsa.DSA_ERR_UNSUPPORTED


def test_test_fault_hook_is_a_host_setting(L):
    assert L.dsa_set_test_faults(2_000_000, 1) == dsa.DSA_OK
    assert L.dsa_set_test_faults(0, 0) == dsa.DSA_OK


def test_decode_launch_counts(L):
    """dsa_decode enqueues: an append unless every sequence has one token
    (then the score kernel appends), a score and a top-k per score window
    (1 GiB slab), the attention, and a combine when tokens are split."""
    n = C.c_int()
    cases = [
        (dict(batch=8, total_q=8, max_q_per_seq=1, max_kv=8192, cache_rows=8 * 8192), 2048, 4),
        (dict(batch=1, total_q=4096, max_q_per_seq=4096, max_kv=8192, cache_rows=8192), 2048, 4),
        (dict(batch=1, total_q=16384, max_q_per_seq=16384, max_kv=131072, cache_rows=131072), 2048, 18),
    ]
    for kw, k, want in cases:
        b = _batch(**kw)
        assert L.dsa_decode_launches(C.byref(b), 32, 64, k, C.byref(n)) == dsa.DSA_OK
        assert n.value == want, (kw, n.value)
    assert L.dsa_decode_launches(C.byref(_batch()), 32, 64, 0, C.byref(n)) == dsa.DSA_ERR_UNSUPPORTED
    assert L.dsa_decode_launches(None, 32, 64, 16, C.byref(n)) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert L.dsa_decode_launches(C.byref(_batch()), 32, 64, 16, None) == dsa.DSA_ERR_INVALID_ARGUMENT


def test_argument_validation_runs_before_any_launch(L):
    b = _batch()
    ws, nws = C.c_void_p(0x10000), 1 << 20
    fake = C.c_void_p(0x40000)          # never dereferenced: every call below fails validation
    # null pointers
    assert L.dsa_indexer_k_append(None, 0, C.byref(b), fake, 0, ws, nws, None) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert L.dsa_topk(fake, 100, None, 4, fake, ws, nws, None) == dsa.DSA_ERR_INVALID_ARGUMENT
    # bad dtype enum
    assert L.dsa_indexer_k_append(fake, 7, C.byref(b), fake, 0, ws, nws, None) == dsa.DSA_ERR_INVALID_ARGUMENT
    # unsupported dims
    assert L.dsa_indexer_score(fake, fake, fake, C.byref(b), 65, 0, fake, 100, ws, nws, None) == \
        dsa.DSA_ERR_UNSUPPORTED
    assert L.dsa_indexer_score(fake, fake, fake, C.byref(b), 0, 0, fake, 100, ws, nws, None) == \
        dsa.DSA_ERR_UNSUPPORTED
    assert L.dsa_topk(fake, 100, C.byref(b), 0, fake, ws, nws, None) == dsa.DSA_ERR_UNSUPPORTED
    assert L.dsa_topk(fake, 100, C.byref(b), 70000, fake, ws, nws, None) == dsa.DSA_ERR_UNSUPPORTED
    assert L.dsa_sparse_mla_attn(fake, fake, fake, C.byref(b), fake, 16, 129, 0.1, fake, None, ws, nws,
                                 None) == dsa.DSA_ERR_UNSUPPORTED
    assert L.dsa_sparse_mla_attn(fake, fake, fake, C.byref(b), fake, 16, 0, 0.1, fake, None, ws, nws,
                                 None) == dsa.DSA_ERR_UNSUPPORTED
    assert L.dsa_decode(fake, 0, fake, fake, fake, fake, fake, fake, C.byref(b), 32, 129, 16, 0.1, 0,
                        fake, None, None, ws, nws, None) == dsa.DSA_ERR_UNSUPPORTED
    # score row stride shorter than the visible span
    assert L.dsa_topk(fake, 99, C.byref(b), 4, fake, ws, nws, None) == dsa.DSA_ERR_INVALID_ARGUMENT
    # misaligned TMA operands
    odd = C.c_void_p(0x40008)
    assert L.dsa_sparse_mla_attn(odd, fake, fake, C.byref(b), fake, 16, 8, 0.1, fake, None, ws, nws,
                                 None) == dsa.DSA_ERR_MISALIGNED
    assert L.dsa_indexer_k_append(fake, 0, C.byref(b), odd, 0, ws, nws, None) == dsa.DSA_ERR_MISALIGNED
    # workspace
    assert L.dsa_topk(fake, 100, C.byref(b), 4, fake, ws, 16, None) == dsa.DSA_ERR_WORKSPACE_TOO_SMALL
    assert L.dsa_topk(fake, 100, C.byref(b), 4, fake, C.c_void_p(0x10010), nws, None) == dsa.DSA_ERR_MISALIGNED
    n = C.c_size_t()
    L.dsa_workspace_size(dsa.DSA_OP_DECODE, C.byref(b), 32, 64, 2048, C.byref(n))
    assert L.dsa_decode(fake, 0, fake, fake, fake, fake, fake, fake, C.byref(b), 32, 64, 2048, 0.1, 0,
                        fake, None, None, ws, n.value - 256, None) == dsa.DSA_ERR_WORKSPACE_TOO_SMALL
    # inconsistent batch bounds
    for kw in (dict(batch=0), dict(total_q=3, max_q_per_seq=1), dict(max_kv=0), dict(cache_rows=1 << 31),
               dict(q_pos=0)):
        bb = _batch(**kw)
        assert L.dsa_topk(fake, 100, C.byref(bb), 4, fake, ws, nws, None) == dsa.DSA_ERR_INVALID_ARGUMENT
    # attention sink: negative count, misaligned anchors
    assert L.dsa_topk_sink(fake, 100, C.byref(b), 4, -1, None, fake, ws, nws, None) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert L.dsa_topk_sink(fake, 100, C.byref(b), 4, 2, C.c_void_p(0x40002), fake, ws, nws, None) == \
        dsa.DSA_ERR_MISALIGNED
    assert L.dsa_decode_sink(fake, 0, fake, fake, fake, fake, fake, fake, C.byref(b), 32, 64, 2048, 0.1, 0, -1,
                             None, fake, None, None, ws, n.value, None) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert L.dsa_set_trace_events(None, -1) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert L.dsa_set_trace_events(None, 0) == dsa.DSA_OK
    assert L.dsa_workspace_init(None, 256, None) == dsa.DSA_ERR_INVALID_ARGUMENT
    assert L.dsa_workspace_init(ws, 100, None) == dsa.DSA_ERR_WORKSPACE_TOO_SMALL


def test_product_path_never_touches_the_oracle():
    """The library package imports nothing from oracle/ and ships no CPU path."""
    pkg = os.path.dirname(dsa.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(root, f)).read()
                assert "oracle" not in text.lower(), f


def test_binding_rejects_rows_of_the_wrong_width():
    """The binding checks each tensor's innermost extent before any call
    (a 576-wide cache passed where 512-wide latent rows are expected would
    otherwise be read with the wrong stride)."""
    import torch

    class Fake:                                # stands in for a CUDA tensor; no GPU needed
        is_cuda = True
        dtype = torch.bfloat16
        device = "cuda:0"

        def __init__(self, *shape):
            self.shape = shape

        def is_contiguous(self):
            return True

        def dim(self):
            return len(self.shape)

    dsa._req(Fake(100, 512), torch.bfloat16, "kv_latent")
    with pytest.raises(TypeError, match="rows of 512"):
        dsa._req(Fake(100, 576), torch.bfloat16, "kv_latent")
    with pytest.raises(TypeError, match="rows of 576"):
        dsa._req(Fake(100, 512), torch.bfloat16, "kv_cache")
    with pytest.raises(TypeError, match="rows of 64"):
        dsa._req(Fake(8, 64, 32), torch.bfloat16, "q_rope")
    dsa._req(Fake(8, 64), torch.bfloat16, "w")                  # no fixed width
