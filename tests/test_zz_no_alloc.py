"""dsa_decode_noalloc: the decode step for callers that cannot allocate device
memory (no workspace argument; the library's static scratch is used instead).

Checked against dsa_decode with a caller workspace on two calls in a row
(the first through the raw C ABI, the second through the Python binding),
within the tolerances of the other GPU tests (attention output 2e-3
max-abs, lse 1e-3; indices and appended keys exact).  This file is named so
that pytest collects it last.
"""
import ctypes as C

import numpy as np
import pytest

import dsa_synth as S
from _helpers import dev_batch, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    from dsa_sparse_attention_score_gb300 import build
    build.build()
    import dsa_sparse_attention_score_gb300 as m
    return m


def _p(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def test_noalloc_matches_workspace_decode_twice(dsa):
    import torch
    wl = S.config(2)                                   # batched decode, B=8, L=8192, top-2048
    inp = S.make_inputs(wl)
    b = dev_batch(wl)
    args = [to_dev(inp.k_new), to_dev(inp.q_idx), to_dev(inp.w), to_dev(inp.q_lat), to_dev(inp.q_rope)]
    kv = to_dev(inp.kv_cache)

    def outputs():
        return (torch.full((wl.T, wl.H, 512), float("nan"), device="cuda"),
                torch.full((wl.T, wl.H), float("nan"), device="cuda"),
                torch.full((wl.T, wl.top_k), -7, dtype=torch.int32, device="cuda"))

    # the existing entry point, with a workspace allocated by the caller
    kc_ref = to_dev(inp.k_cache)
    out_ref, lse_ref, idx_ref = outputs()
    ws = dsa.workspace(dsa.DSA_OP_DECODE, b, wl.H_I, wl.H, wl.top_k)
    dsa.dsa_decode(*args, kc_ref, kv, b, wl.top_k, wl.sm_scale, wl.hadamard, out_ref, lse_ref, idx_ref, ws)
    torch.cuda.synchronize()

    L = dsa.lib()
    desc = b.desc()
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        kc = to_dev(inp.k_cache)
        out, lse, idx = outputs()
        if call == 0:                                  # the raw C ABI
            rc = L.dsa_decode_noalloc(_p(args[0]), dsa.DSA_KEY_F32, _p(args[1]), _p(args[2]), _p(args[3]),
                                      _p(args[4]), _p(kc), _p(kv), C.byref(desc), wl.H_I, wl.H, wl.top_k,
                                      C.c_float(wl.sm_scale), int(wl.hadamard), _p(out), _p(lse), _p(idx), stream)
            assert rc == dsa.DSA_OK, dsa.dsa_status_string(rc)
        else:                                          # the Python binding of the same call
            dsa.dsa_decode_noalloc(*args, kc, kv, b, wl.top_k, wl.sm_scale, wl.hadamard, out, lse, idx)
        torch.cuda.synchronize()
        assert torch.equal(kc, kc_ref), f"call {call}: appended keys differ"
        assert torch.equal(idx, idx_ref), f"call {call}: selections differ"
        err_o = (out - out_ref).abs().max().item()
        err_l = (lse - lse_ref).abs().max().item()
        assert err_o <= 2e-3, f"call {call}: max |out diff| {err_o}"
        assert err_l <= 1e-3, f"call {call}: max |lse diff| {err_l}"


def test_noalloc_refuses_batches_beyond_its_scratch(dsa):
    """A prefill chunk of 4096 tokens needs more than the 64 MiB of static
    scratch: refused with DSA_ERR_WORKSPACE_TOO_SMALL before any launch."""
    wl = S.config(4)
    b = dev_batch(wl)
    assert dsa.dsa_workspace_size(dsa.DSA_OP_DECODE, b, wl.H_I, wl.H, wl.top_k) > 64 << 20
    desc = b.desc()
    fake = C.c_void_p(0x1000)        # never dereferenced: the size check answers first
    rc = dsa.lib().dsa_decode_noalloc(fake, 0, fake, fake, fake, fake, fake, fake, C.byref(desc), wl.H_I, wl.H,
                                      wl.top_k, C.c_float(wl.sm_scale), 0, fake, None, None, None)
    assert rc == dsa.DSA_ERR_WORKSPACE_TOO_SMALL
