"""A plain C program drives the library through the C ABI alone
(tests/c_caller/decode_from_files.c): it compiles and links against the
library with gcc (no GPU needed), and on a GPU its dsa_decode step matches
the oracle on the tiny and batched decode workloads."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import dsa_synth as S
from dsa_sparse_attention_score_gb300 import build as dsa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_caller", "decode_from_files.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _compile(tmp_path):
    if not shutil.which("gcc") or not os.path.exists(os.path.join(CUDA, "include", "cuda_runtime_api.h")):
        pytest.skip("gcc or the CUDA headers are missing")
    lib = dsa_build.build()
    exe = str(tmp_path / "decode_from_files")
    libdirs = [d for d in (os.path.join(CUDA, "lib64"), os.path.join(CUDA, "lib")) if os.path.isdir(d)]
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", SRC, "-I" + os.path.join(ROOT, "include"),
           "-I" + os.path.join(CUDA, "include"), "-L" + os.path.dirname(lib), "-ldsa_gb300",
           *["-L" + d for d in libdirs], "-lcudart", "-Wl,-rpath," + os.path.dirname(lib), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe, libdirs


def test_c_caller_compiles_and_links(tmp_path):
    _compile(tmp_path)


def _write_inputs(d, wl, inp):
    meta = np.array([wl.B, wl.T, wl.max_q_per_seq, wl.max_kv, wl.H_I, wl.H, wl.top_k, int(wl.hadamard)],
                    np.int32).tobytes() + np.array([wl.cache_rows], np.int64).tobytes() + \
        np.array([wl.sm_scale], np.float32).tobytes()
    (d / "meta.bin").write_bytes(meta)
    cu, qp, ko = S.batch_arrays(wl)
    for name, a in (("cu_q", cu), ("q_pos", qp), ("kv_off", ko), ("k_new", inp.k_new), ("q_idx", inp.q_idx),
                    ("w", inp.w), ("q_lat", inp.q_lat), ("q_rope", inp.q_rope), ("k_cache", inp.k_cache),
                    ("kv_cache", inp.kv_cache)):
        (d / f"{name}.bin").write_bytes(np.ascontiguousarray(a).tobytes())


@pytest.mark.gpu
@pytest.mark.parametrize("cfg", [1, 2])
def test_c_caller_decode_matches_oracle(tmp_path, cfg):
    import oracle
    from _helpers import check_attention, check_selection
    exe, libdirs = _compile(tmp_path)
    wl = S.config(cfg)
    inp = S.make_inputs(wl)
    d = tmp_path / "io"
    d.mkdir()
    _write_inputs(d, wl, inp)
    env = dict(os.environ)
    env["LD_LIBRARY_PATH"] = ":".join(libdirs + [env.get("LD_LIBRARY_PATH", "")])
    r = subprocess.run([exe, str(d)], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    out = np.fromfile(d / "out.bin", np.float32).reshape(wl.T, wl.H, 512)
    lse = np.fromfile(d / "lse.bin", np.float32).reshape(wl.T, wl.H)
    idx = np.fromfile(d / "idx.bin", np.int32).reshape(wl.T, wl.top_k)
    kc = np.fromfile(d / "k_cache_out.bin", np.float16).reshape(wl.cache_rows, 128)
    ref = oracle.decode(inp, wl)
    assert np.array_equal(kc.view(np.uint16), ref["k_cache"].view(np.uint16))
    for t in range(wl.T):
        n = wl.q_pos[t] + 1
        check_selection(idx[t], ref["idx"][t], ref["scores"][t, :n], wl.top_k)
    ref_o, ref_l = oracle.sparse_attn(inp.q_lat, inp.q_rope, inp.kv_cache, oracle.Batch.of(wl), idx, wl.sm_scale)
    check_attention(out, lse, ref_o, ref_l, name="C caller attention")
