#!/usr/bin/env python3
"""Throughput of the DSA hot path (indexer-key append, lightning-indexer
score, top-k, sparse MLA attention) on GB300.

One step = one fused dsa_decode call over one batch of synthetic inputs
already resident in HBM.  Headline workload: batched decode, 8 sequences of
8192 cached positions, 32 indexer heads x 128, 64 query heads, top-2048,
576-wide bf16 latent rows.  The same default run then measures the rest of
the metric the same way under "workloads": the ragged long-context decode
(32 sequences of 4k-64k positions, rotation on) and the two prefill
workloads (4096 tokens after 4096, 16384 after 114688).  Each step is the
library's own stream launches (--graph replays a CUDA graph of the step
instead); L2 is flushed (a 512 MB write, then a 512 MB read) before every
timed step and each step is timed with CUDA events on its stream.  Each
kernel's time inside the overlapped step comes from the library's device
timeline (globaltimer at the first CTA start and last CTA end of every
kernel), which gives the per-kernel rooflines.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--headline-only]
  python bench.py --impl reference ...    # the CPU oracle on the same workload

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(independent replicas, no data-path collective); the reported time is the
maximum over ranks and the value counts the tokens of all ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "DSA decode tok/s & prefill tok/s on 1 GB300; % of HBM / tensor roofline"
UNIT = "tok/s"
WORKLOADS = {"tiny_decode": 1, "batched_decode": 2, "ragged_decode": 3, "prefill_chunk": 4, "long_prefill": 5,
             "indexshare_decode": 2, "kpool_decode": 2}
STACK_LAYERS = 78
MAX_TRACE_WINDOWS = 32    # score windows whose top-k launch the trace events bracket


def index_share_full(il: int) -> bool:
    """ik_llama_opt commit log, "GLM-5.2 DSA: IndexShare (shared layers reuse
    full-layer top-k)": layer il computes its own top-k iff il <= 1 or
    il % 4 == 2 (21 of 78 layers); the others reuse the most recent full
    layer's selection."""
    return il <= 1 or il % 4 == 2
STAGES = ["k_append", "indexer_score", "topk", "sparse_attn", "attn_combine"]
KERNEL_OF_STAGE = {"k_append": "k_append_kernel", "indexer_score": "score_kernel", "topk": "topk_cluster_kernel",
                   "sparse_attn": "sparse_attn_kernel", "attn_combine": "attn_combine_kernel"}
SOURCE_OF_KERNEL = {"k_append_kernel": "k_append.cu", "score_kernel": "score.cu", "topk_cluster_kernel": "topk.cu",
                    "sparse_attn_kernel": "sparse_attn.cu", "attn_combine_kernel": "sparse_attn.cu"}


def parse():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["dsa", "reference"], default="dsa")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="batched_decode")
    ap.add_argument("--flush-mb", type=int, default=512)
    ap.add_argument("--e2e-steps", type=int, default=1000)
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="budget of the CPU-baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true",
                    help="measure only the chosen workload (by default the batched-decode run also measures the "
                         "ragged decode and the two prefill workloads)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="prefill workloads only: keep the last N query tokens of the chunk (same row lengths, "
                         "a smaller case of the same kernels, e.g. for an ncu capture)")
    ap.add_argument("--graph", action="store_true",
                    help="replay each step as a CUDA graph (default: the library's own stream launches, which "
                         "measured 2.8 us faster per batched-decode step on GB300: a graph replay adds "
                         "GPU-side launch latency, and the flush between steps keeps the host ahead)")
    return ap.parse_args()


# ---------------------------------------------------------------------------- helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def shrink(wl, tokens):
    """The last `tokens` query tokens of a one-sequence prefill workload,
    with the same cache and row lengths (0: the workload unchanged)."""
    if not tokens or tokens >= wl.T:
        return wl
    if wl.B != 1:
        raise SystemExit("--tokens applies to the prefill workloads only")
    import dsa_synth as S
    end = wl.q_pos[-1] + 1
    return S.prefill_workload(f"prefill_T{tokens}_after{end - tokens}", wl.seed, end - tokens, tokens,
                              H_I=wl.H_I, H=wl.H, top_k=wl.top_k, hadamard=wl.hadamard)


def algorithmic(wl):
    """Bytes each step must move and flops it must do (per kernel), from the
    workload shape: the indexer reads every visible key once per sequence
    (256 B a row) and does 2*128 flops per (visible key, query, head); the
    attention gathers the selected 1152-B latent rows once per query token
    and does 2*(576+512) flops per (selected row, head)."""
    key_rows = 0
    for b in range(wl.B):
        toks = range(wl.cu_q[b], wl.cu_q[b + 1])
        key_rows += max(wl.q_pos[t] for t in toks) + 1 if len(toks) else 0
    pairs = sum(p + 1 for p in wl.q_pos)
    sel = sum(min(wl.top_k, p + 1) for p in wl.q_pos)
    score_bytes = key_rows * 256
    attn_bytes = sel * 1152
    return dict(score_bytes=score_bytes, score_flops=pairs * wl.H_I * 256,
                attn_bytes=attn_bytes, attn_flops=sel * wl.H * 2 * (576 + 512),
                step_bytes=score_bytes + attn_bytes,
                topk_bytes=pairs * 4, append_bytes=wl.T * (512 + 256), out_bytes=wl.T * wl.H * 512 * 4)


def source_hash(kernel):
    path = os.path.join(ROOT, "dsa_sparse_attention_score_gb300", "csrc", SOURCE_OF_KERNEL[kernel])
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def ncu_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current source of that kernel and this workload; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path)).get(kernel, {}).get(workload)
    if not rec or rec.get("src_sha256_16") != source_hash(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.tmp = tempfile.NamedTemporaryFile(prefix="dsa_clocks_", suffix=".csv", delete=False)
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(gpu_index)], stdout=self.tmp, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.tmp.close()
        rows = []
        for line in open(self.tmp.name):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append(dict(sm=float(parts[2]), max=float(parts[3]), power=parts[4],
                                 hw=parts[6], hwt=parts[7], swt=parts[8], swp=parts[9]))
            except ValueError:
                continue
        os.unlink(self.tmp.name)
        return rows

    @staticmethod
    def summary(rows):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


def max_over_ranks(x: float) -> float:
    """The largest value of x over the ranks of the job (the job takes as
    long as its slowest replica); x itself outside a multi-rank job."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def stage_split(t, pairs):
    """Per-stage milliseconds of one traced step.

    t: elapsed ms from trace event 0 to events 1..5 (before the first score,
    before the first top-k, before the attention, before the combine, after
    the last launch).  pairs: elapsed ms to events (6 + 2j, 7 + 2j), which
    bracket the top-k of score window j; a pair outside [t[0], t[2]] is a
    slot this call did not record, and ends the windows.  With several
    windows the score stage is everything between the append and the
    attention that is not top-k.
    """
    win = []
    for a, b in pairs:
        if not (t[0] <= a <= b <= t[2]):
            break
        win.append((a, b))
    if not win:
        win = [(t[1], t[2])]
    topk = sum(b - a for a, b in win)
    return {"k_append": t[0], "indexer_score": t[2] - t[0] - topk, "topk": topk,
            "sparse_attn": t[3] - t[2], "attn_combine": t[4] - t[3]}


def job_throughput(world: int, tokens_per_step: int, steps: int, seconds: float) -> float:
    """Whole-job tokens per second: every rank runs its own replica of the
    workload (weak scaling), so the job processes world x tokens per step."""
    return world * tokens_per_step * steps / seconds


def gpu_index_for(device):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if device < len(ids) and ids[device].isdigit():
            return int(ids[device])
    return device


# ---------------------------------------------------------------------------- oracle (CPU) legs

def token_subs(wl, inp, tokens):
    """Single-token workloads: token t of wl decoded alone over its own
    sequence's keys 0..q_pos[t] (the same work it has in the full step)."""
    import numpy as np
    import dsa_synth as S
    subs = []
    for t in tokens:
        b = int(np.searchsorted(wl.cu_q, t, side="right") - 1)
        off, p = wl.kv_off[b], wl.q_pos[t]
        one = S.Workload(wl.name, wl.seed, [p + 1], [p], [0, 1], wl.H_I, wl.H, wl.top_k, wl.hadamard, wl.sm_scale)
        sl = slice(off, off + p + 1)
        subs.append((one, S.Inputs(k_cache=inp.k_cache[sl], k_new=inp.k_new[t:t + 1], q_idx=inp.q_idx[t:t + 1],
                                   w=inp.w[t:t + 1], q_lat=inp.q_lat[t:t + 1], q_rope=inp.q_rope[t:t + 1],
                                   kv_cache=inp.kv_cache[sl])))
    return subs


def run_oracle_sample(wl, inp, seconds):
    """Times the oracle on the host cores within a budget: whole steps of a
    decode batch, or, for a prefill chunk (whose full step would take
    minutes to hours), up to 64 of its tokens spread evenly over the chunk,
    each decoded alone over its full key range -- tokens per second
    extrapolate to the chunk by token count.  Also the middle token of the
    workload, decoded alone on a single thread."""
    import oracle
    cores = oracle.set_threads(0)
    if wl.T <= 64:
        def one(i):
            oracle.decode(inp, wl)
            return wl.T
        what = f"full steps of the {wl.name} workload ({wl.T} query tokens each)"
    else:
        subs = token_subs(wl, inp, range(0, wl.T, -(-wl.T // 64)))

        def one(i):
            o, si = subs[i % len(subs)]
            oracle.decode(si, o)
            return 1
        what = (f"tokens of {wl.name} ({len(subs)} spread evenly over the {wl.T}-token chunk, each decoded "
                f"alone over its full key range; extrapolated to the chunk by token count)")
    reps, toks, t0 = 0, 0, time.perf_counter()
    while True:
        toks += one(reps)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds or reps >= 50:
            break
    ((o1, s1),) = token_subs(wl, inp, [wl.T // 2])
    oracle.set_threads(1)
    t1 = time.perf_counter()
    oracle.decode(s1, o1)
    el1 = time.perf_counter() - t1
    oracle.set_threads(0)
    return dict(value=toks / el, unit=UNIT, cores=cores, kind="oracle",
                sample=f"{reps} {what}, {el:.1f} s of CPU time on {cores} OpenMP threads",
                single_thread={"value": 1.0 / el1, "unit": UNIT, "cores": 1,
                               "sample": f"token {wl.T // 2} of {wl.name} decoded alone over its full key "
                                         f"range on one thread, {el1:.2f} s"})


def reference_arm(args):
    """The CPU oracle as the reference implementation: each step decodes one
    query token of the workload (its own sequence, all its keys)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import dsa_synth as S
    import oracle
    wl = S.config(WORKLOADS[args.workload])
    inp = S.make_inputs(wl)
    cores = oracle.set_threads(0)
    subs = token_subs(wl, inp, range(min(wl.T, 64)))
    stack = args.workload == "indexshare_decode"

    def one_step(i):
        one, si = subs[i % len(subs)]
        if not stack:
            oracle.decode(si, one)
            return
        # one token through the layer stack: full layers decode, shared
        # layers attend over the last full layer's selection
        idx = None
        for il in range(STACK_LAYERS):
            if index_share_full(il):
                idx = oracle.decode(si, one)["idx"]
            else:
                oracle.sparse_attn(si.q_lat, si.q_rope, si.kv_cache, oracle.Batch.of(one), idx, one.sm_scale)

    for i in range(args.warmup):
        one_step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        one_step(i)
    el = time.perf_counter() - t0
    value = args.steps / el
    line = {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": (f"indexshare_decode_B8_L8192_{STACK_LAYERS}layers" if stack else wl.name),
                       "B": wl.B, "T": wl.T, "H_I": wl.H_I, "H": wl.H, "top_k": wl.top_k,
                       "step": "one query token of the workload (its sequence's full key range)"
                               + (f" through {STACK_LAYERS} layers" if stack else "")},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{args.steps} steps, one query token each, cycling over the "
                                       f"{len(subs)} first tokens of {wl.name}"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------- layer stack (IndexShare)

def layer_stack(args):
    """Decode through a stack of STACK_LAYERS layers of the batched-decode
    shapes.  Full layers run dsa_decode (append, score, top-k, attention) and
    keep their selection; shared layers run dsa_sparse_mla_attn on the most
    recent full layer's selection.  The same stack with every layer full is
    timed beside it.  Each layer has its own caches (about 92 MB), generated
    on the device from a seeded generator with the shapes and scales of the
    single-layer inputs, so no layer finds another's rows in L2."""
    import torch
    torch.cuda.set_device(0)
    dev = torch.cuda.current_device()
    from dsa_sparse_attention_score_gb300 import build as lib_build
    lib_build.build()
    import dsa_sparse_attention_score_gb300 as dsa
    import dsa_synth as S
    wl = S.config(2)
    g = torch.Generator(device="cuda")
    g.manual_seed(20260)

    def normal(shape, scale, dtype):
        return (torch.randn(shape, generator=g, device="cuda", dtype=torch.float32) * scale).to(dtype)

    rows, T = wl.cache_rows, wl.T
    # per-step inputs of every layer packed in one buffer (256-B aligned
    # slots), so the end-to-end loop moves them with one copy
    step_shapes = [("k_new", (T, 128), torch.float32, 128 ** -0.5), ("q_idx", (T, wl.H_I, 128), torch.float16, 128 ** -0.5),
                   ("w", (T, wl.H_I), torch.float32, wl.H_I ** -0.5), ("q_lat", (T, wl.H, 512), torch.bfloat16, 512 ** -0.5),
                   ("q_rope", (T, wl.H, 64), torch.bfloat16, 64 ** -0.5)]
    slot = []
    total = 0
    for name, shp, dt, _ in step_shapes:
        nb = math.prod(shp) * torch.empty((), dtype=dt).element_size()
        slot.append((total, nb))
        total += (nb + 255) // 256 * 256
    d_pack = torch.empty(STACK_LAYERS * total, dtype=torch.uint8, device="cuda")
    layers = []
    for il in range(STACK_LAYERS):
        L = dict(k_cache=normal((rows, 128), 128 ** -0.5, torch.float16),
                 kv_cache=normal((rows, 576), 576 ** -0.5, torch.bfloat16))
        for (name, shp, dt, sc), (off, nb) in zip(step_shapes, slot):
            v = d_pack[il * total + off: il * total + off + nb].view(dt).view(shp)
            v.copy_(normal(shp, sc, dt))
            L[name] = v
        layers.append(L)
    h_pack = d_pack.cpu().pin_memory()
    batch = dsa.Batch.from_host(wl.cu_q, wl.q_pos, wl.kv_off, wl.cache_rows, max_q_per_seq=1, max_kv=wl.max_kv)
    ws = dsa.workspace(dsa.DSA_OP_DECODE, batch, wl.H_I, wl.H, wl.top_k)
    out = torch.empty((T, wl.H, 512), device="cuda")
    lse = torch.empty((T, wl.H), device="cuda")
    idx = torch.empty((T, wl.top_k), dtype=torch.int32, device="cuda")
    flush = torch.empty(args.flush_mb << 20, dtype=torch.uint8, device="cuda")
    flush_r = torch.ones((args.flush_mb << 20) // 4, dtype=torch.float32, device="cuda")

    def step(share):
        for il, L in enumerate(layers):
            if not share or index_share_full(il):
                dsa.dsa_decode(L["k_new"], L["q_idx"], L["w"], L["q_lat"], L["q_rope"], L["k_cache"],
                               L["kv_cache"], batch, wl.top_k, wl.sm_scale, wl.hadamard, out, lse, idx, ws)
            else:
                dsa.dsa_sparse_mla_attn(L["q_lat"], L["q_rope"], L["kv_cache"], batch, idx, wl.sm_scale, out,
                                        lse, ws)

    res = {}
    for share in (True, False):
        step(share)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step(share)
        for i in range(args.warmup):
            flush.fill_(i & 0xFF)
            flush_r.amax()
            graph.replay()
        torch.cuda.synchronize()
        clocks = Clocks(gpu_index_for(dev))
        time.sleep(0.2)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            flush_r.amax()
            ev[i][0].record()
            graph.replay()
            ev[i][1].record()
        torch.cuda.synchronize()
        rows_c = clocks.stop()
        ms = statistics.fmean(a.elapsed_time(b) for a, b in ev)
        res[share] = (ms, Clocks.summary(rows_c))
        if dsa.dsa_read_device_status(ws) != 0:
            raise RuntimeError("device status flags set during the timed steps")
    # end to end through the public API: one pinned H2D copy of every layer's
    # step inputs, the IndexShare stack, a D2H read of the last layer's output
    graph = torch.cuda.CUDAGraph()
    step(True)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        step(True)
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_ms = []
    for i in range(min(args.steps, args.e2e_steps) + 3):
        flush.fill_(i & 0xFF)
        flush_r.amax()
        e0.record()
        d_pack.copy_(h_pack, non_blocking=True)
        step(True)
        h_out.copy_(out, non_blocking=True)
        e1.record()
        e1.synchronize()
        if i >= 3:
            e2e_ms.append(e0.elapsed_time(e1))
    e2e_step = statistics.fmean(e2e_ms)
    n_full = sum(index_share_full(il) for il in range(STACK_LAYERS))
    per_full = dsa.dsa_decode_launches(batch, wl.H_I, wl.H, wl.top_k)
    per_shared = per_full - 2                        # attention (+ combine) only
    alg = algorithmic(wl)
    step_bytes = n_full * alg["step_bytes"] + (STACK_LAYERS - n_full) * alg["attn_bytes"]
    ms, clk = res[True]
    pk = peaks()
    achieved = step_bytes / (ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": T / (ms * 1e-3), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp16+bf16 (f32 accumulate)",
        "data": "synthetic (device generator, seeded)",
        "config": {"workload": f"indexshare_decode_B8_L8192_{STACK_LAYERS}layers", "B": wl.B, "T": T,
                   "L": wl.max_kv, "H_I": wl.H_I, "H": wl.H, "top_k": wl.top_k, "layers": STACK_LAYERS,
                   "full_layers": n_full, "shared_layers": STACK_LAYERS - n_full,
                   "l2": f"flushed before every timed step ({args.flush_mb} MB write, then read)",
                   "launch": "CUDA graph replay of the whole stack", "parallelism": "replicas x1"},
        "clocks": clk,
        "gpu_launches": (n_full * per_full + (STACK_LAYERS - n_full) * per_shared) * args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / pk["hbm_gbs"], "algorithmic_bytes_per_step": step_bytes,
                     "kernel": "whole stack", "traffic": None},
        "all_full_layers": {"ms_per_step": res[False][0], "tok_s": T / (res[False][0] * 1e-3),
                            "clocks": res[False][1]},
        "index_share_speedup": res[False][0] / ms,
        "e2e": {"value": T / (e2e_step * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h_pack.numel(),
                "d2h_bytes_per_step": h_out.numel() * h_out.element_size(), "steps": len(e2e_ms),
                "path": "one pinned H2D copy of every layer's step inputs, the stack through the Python "
                        "binding (eager launches), D2H of the last layer's output"},
    }
    if not args.no_cpu_baseline:
        import oracle
        cores = oracle.set_threads(0)
        one = S.Workload(wl.name, wl.seed, [wl.q_pos[0] + 1], [wl.q_pos[0]], [0, 1], wl.H_I, wl.H, wl.top_k,
                         wl.hadamard, wl.sm_scale)
        si = S.make_inputs(one)
        t0 = time.perf_counter()
        idx1 = None
        for il in range(STACK_LAYERS):
            if index_share_full(il):
                idx1 = oracle.decode(si, one)["idx"]
            else:
                oracle.sparse_attn(si.q_lat, si.q_rope, si.kv_cache, oracle.Batch.of(one), idx1, one.sm_scale)
        el = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": 1.0 / el, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": f"one query token (L=8192) through the {STACK_LAYERS}-layer IndexShare "
                                          f"stack, {el:.1f} s on {cores} OpenMP threads"}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------- GPU arm

TIMELINE_ORDER = ["k_append", "indexer_score", "topk", "sparse_attn", "attn_combine"]
EXTRA_WORKLOADS = ["ragged_decode", "prefill_chunk", "long_prefill", "kpool_decode"]


def exclusive_spans(spans):
    """Per-kernel time inside one overlapped step, from the device timeline.

    spans: stage -> (first CTA start, last CTA end) in us.  A kernel launched
    with programmatic dependent launch starts its prologue while its
    predecessor still runs and then waits for it, so its own share of the
    step runs from the later of its first CTA start and the predecessor's last
    CTA end, to its own last CTA end.  The shares add up to the step's span.
    """
    out, prev_end = {}, None
    for st in TIMELINE_ORDER:
        if st not in spans:
            continue
        a, b = spans[st]
        lo = a if prev_end is None else max(a, prev_end)
        out[st] = max(0.0, b - lo)
        prev_end = b
    return out


def kernel_roofline(stage, ms, wl, alg, pk):
    """Roofline of one kernel over one step: decode contractions stream HBM
    (bytes they must read), prefill contractions run on the tensor cores
    (causal flops of the definition; fp16 and bf16 share one dense peak), the
    selection reads its score rows once, the combine writes the outputs."""
    decode = wl.max_q_per_seq == 1
    sec = ms * 1e-3
    if stage in ("indexer_score", "sparse_attn") and not decode:
        flops = alg["score_flops"] if stage == "indexer_score" else alg["attn_flops"]
        ach = flops / sec / 1e12
        return {"bound": "tensor", "achieved": ach, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": ach / pk["bf16_tflops"], "frac_of_sustained": ach / pk["bf16_tflops_sustained"],
                "dtype": "fp16" if stage == "indexer_score" else "bf16", "algorithmic_flops": flops}
    nbytes = {"indexer_score": alg["score_bytes"], "sparse_attn": alg["attn_bytes"], "topk": alg["topk_bytes"],
              "k_append": alg["append_bytes"], "attn_combine": alg["out_bytes"]}[stage]
    ach = nbytes / sec / 1e9
    return {"bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": ach / pk["hbm_gbs"],
            "algorithmic_bytes": nbytes}


def measure(dsa, torch, wl, steps, warmup, flush_mb, world=1, e2e_steps=0, graph=False):
    """Times one workload: `steps` steps (each on a cold L2, CUDA events on
    the launching stream), then per-kernel times from the device timeline of
    up to 200 more steps, and from the stage events.  Returns the measured
    numbers and, with e2e_steps, the end-to-end rate through the binding."""
    import numpy as np
    import dsa_synth as S
    inp = S.make_inputs(wl)

    def up(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).cuda()
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    # The per-step inputs live in one packed buffer (each tensor at a 256-B
    # aligned offset), so the end-to-end loop moves them with one copy.
    step_in = [(inp.k_new, torch.float32), (inp.q_idx, torch.float16), (inp.w, torch.float32),
               (inp.q_lat, torch.bfloat16), (inp.q_rope, torch.bfloat16)]
    offs, total = [], 0
    for a, _ in step_in:
        offs.append(total)
        total += (a.nbytes + 255) // 256 * 256
    h_pack = torch.zeros(total, dtype=torch.uint8).pin_memory()
    for (a, _), off in zip(step_in, offs):
        h_pack[off:off + a.nbytes] = torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).reshape(-1))
    d_pack = h_pack.cuda()
    k_new, q_idx, w, q_lat, q_rope = [d_pack[off:off + a.nbytes].view(dt).view(a.shape)
                                      for (a, dt), off in zip(step_in, offs)]
    k_cache, kv_cache = up(inp.k_cache), up(inp.kv_cache)
    del inp
    batch = dsa.Batch.from_host(wl.cu_q, wl.q_pos, wl.kv_off, wl.cache_rows, max_q_per_seq=wl.max_q_per_seq,
                                max_kv=wl.max_kv)
    ws = dsa.workspace(dsa.DSA_OP_DECODE, batch, wl.H_I, wl.H, wl.top_k)
    out = torch.empty((wl.T, wl.H, 512), device="cuda")
    lse = torch.empty((wl.T, wl.H), device="cuda")
    idx = torch.empty((wl.T, wl.top_k), dtype=torch.int32, device="cuda")
    flush = torch.empty(flush_mb << 20, dtype=torch.uint8, device="cuda")
    flush_r = torch.ones((flush_mb << 20) // 4, dtype=torch.float32, device="cuda")
    launches = dsa.dsa_decode_launches(batch, wl.H_I, wl.H, wl.top_k)
    trace = [torch.cuda.Event(enable_timing=True) for _ in range(6 + 2 * MAX_TRACE_WINDOWS)]
    tl_buf = torch.zeros(10, dtype=torch.int64, device="cuda")

    def flush_l2(i):
        # write a buffer larger than L2, then read another one, so the step
        # starts with a cold L2 that holds no dirty lines of the flush itself
        flush.fill_(i & 0xFF)
        flush_r.amax()

    def step():
        dsa.dsa_decode(k_new, q_idx, w, q_lat, q_rope, k_cache, kv_cache, batch, wl.top_k, wl.sm_scale,
                       wl.hadamard, out, lse, idx, ws)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    run = step
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        run = g.replay
    for i in range(warmup):
        flush_l2(i)
        run()
    torch.cuda.synchronize()
    if dsa.dsa_read_device_status(ws) != 0:
        raise RuntimeError(f"{wl.name}: device status flags set during warm-up")

    # ---- timed region: K steps, each on a cold L2, timed on the device
    clocks = Clocks(gpu_index_for(torch.cuda.current_device()))
    time.sleep(0.2)                                  # let the sampler start
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        flush_l2(i)
        ev[i][0].record()
        run()
        ev[i][1].record()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clock_rows = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]

    # ---- per-kernel times: the device timeline of the same step (earliest
    # CTA start / latest CTA end of each kernel), and stage events (which
    # serialise the kernels; used where score and top-k run in several windows)
    n_side = min(steps, 200)
    big = torch.iinfo(torch.int64).max
    excl = {st: [] for st in TIMELINE_ORDER}
    spans = {st: [] for st in TIMELINE_ORDER}
    for i in range(n_side):
        tl_buf[0::2] = big
        tl_buf[1::2] = 0
        flush_l2(i)
        dsa.dsa_set_timeline(tl_buf)
        step()
        dsa.dsa_set_timeline(None)
        torch.cuda.synchronize()
        v = tl_buf.tolist()
        t0 = min(x for x in v[0::2] if x != big)
        sp = {st: ((v[2 * j] - t0) / 1e3, (v[2 * j + 1] - t0) / 1e3)
              for j, st in enumerate(TIMELINE_ORDER) if v[2 * j] != big}
        for st, x in sp.items():
            spans[st].append(x)
        for st, x in exclusive_spans(sp).items():
            excl[st].append(x)
    stage_ms = {st: [] for st in STAGES}
    for i in range(n_side):
        flush_l2(i)
        dsa.dsa_set_trace_events(trace)
        step()
        dsa.dsa_set_trace_events(None)
        trace[5].synchronize()
        t = [trace[0].elapsed_time(trace[j]) for j in range(1, 6)]
        pairs = [(trace[0].elapsed_time(trace[6 + 2 * j]), trace[0].elapsed_time(trace[7 + 2 * j]))
                 for j in range(MAX_TRACE_WINDOWS)]
        for st, x in stage_split(t, pairs).items():
            stage_ms[st].append(x)
    torch.cuda.synchronize()
    windows = score_windows(dsa, batch)
    if windows == 1:
        kernel_ms = {st: statistics.median(v) / 1e3 for st, v in excl.items() if v}
        source = ("device timeline (globaltimer): each kernel's exclusive span in the overlapped step, from the "
                  "later of its first CTA start and its predecessor's last CTA end to its last CTA end; "
                  f"median of {n_side} steps")
    else:
        kernel_ms = {st: statistics.median(v) for st, v in stage_ms.items() if v and statistics.median(v) > 0}
        append = 0 if wl.max_q_per_seq == 1 else 1
        if launches - append - 2 * windows - 1 == 0:    # no split tokens: no combine kernel ran
            kernel_ms.pop("attn_combine", None)
        source = (f"stage events around each of the {windows} score windows' top-k launches (the score and "
                  f"top-k kernels alternate, so their timeline spans overlap); median of {n_side} steps")

    res = dict(step_ms=step_ms, kernel_ms=kernel_ms, kernel_source=source, launches=launches,
               clocks=Clocks.summary(clock_rows),
               timeline_us={st: [round(statistics.median(a for a, _ in v), 2),
                                 round(statistics.median(b for _, b in v), 2)] for st, v in spans.items() if v},
               stages_ms={st: round(statistics.median(v), 5) for st, v in stage_ms.items() if v})

    if e2e_steps:
        # ---- end to end through the public API with host buffers: one pinned
        # copy of every input of the step; the result lands in pinned host
        # memory, written there by the kernels themselves when the driver
        # maps that memory into the device's address space at the same
        # address (NVLink-C2C on Grace), else by copies after the step
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        m_out, m_lse = host_mapped_alias(torch, h_out), host_mapped_alias(torch, h_lse)
        zero_copy = m_out is not None and m_lse is not None
        # inputs: read from the mapped pinned buffer by the SMs (a copy kernel)
        # when it is mapped, else by the copy engine
        m_pack = host_mapped_alias(torch, h_pack.view(torch.int32)) if h_pack.numel() % 4 == 0 else None
        d_pack32 = d_pack.view(torch.int32)

        def copy_in():
            if m_pack is not None:
                torch.add(m_pack, 0, out=d_pack32)
            else:
                d_pack.copy_(h_pack, non_blocking=True)

        def step_e2e():
            if zero_copy:
                dsa.dsa_decode(k_new, q_idx, w, q_lat, q_rope, k_cache, kv_cache, batch, wl.top_k, wl.sm_scale,
                               wl.hadamard, m_out, m_lse, idx, ws)
            else:
                step()
                h_out.copy_(out, non_blocking=True)
                h_lse.copy_(lse, non_blocking=True)

        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2e_ms = []
        for i in range(e2e_steps + 3):
            flush_l2(i)
            e0.record()
            copy_in()                                 # every input of the step, one copy
            step_e2e()
            e1.record()
            e1.synchronize()
            if i >= 3:
                e2e_ms.append(e0.elapsed_time(e1))
        if not torch.equal(h_out, out.cpu()):
            raise RuntimeError(f"{wl.name}: end-to-end output differs from the device-resident run")
        res["e2e_ms"] = e2e_ms
        res["h2d"] = h_pack.numel()
        res["d2h"] = h_out.numel() * h_out.element_size() + h_lse.numel() * h_lse.element_size()
        res["e2e_path"] = ("one H2D copy of the step's packed inputs from pinned host memory ("
                           + ("read over the link by a copy kernel" if m_pack is not None else "copy engine")
                           + "), dsa_decode through the Python binding; "
                           + ("out and lse written by the kernels straight into pinned host memory (mapped at the "
                              "same address), no separate D2H copy" if zero_copy else "D2H copies of out and lse")
                           + "; caches stay resident")
    if dsa.dsa_read_device_status(ws) != 0:
        raise RuntimeError(f"{wl.name}: device status flags set during the timed steps")
    return res


def host_mapped_alias(torch, t):
    """A CUDA tensor over the pinned host tensor t's memory, if the driver
    maps that memory into the device's address space at the same address
    (asked with cuPointerGetAttribute); else None."""
    import ctypes
    try:
        cu = ctypes.CDLL("libcuda.so.1")
    except OSError:
        return None
    p = t.data_ptr()
    mtype, dptr = ctypes.c_uint32(0), ctypes.c_uint64(0)
    if cu.cuPointerGetAttribute(ctypes.byref(mtype), ctypes.c_int(2), ctypes.c_uint64(p)) != 0 or mtype.value != 1:
        return None                                  # not host memory the driver knows
    if cu.cuPointerGetAttribute(ctypes.byref(dptr), ctypes.c_int(3), ctypes.c_uint64(p)) != 0 or dptr.value != p:
        return None                                  # not mapped at the same address

    typestr = {torch.float32: "<f4", torch.int32: "<i4", torch.uint8: "|u1"}.get(t.dtype)
    if typestr is None:
        return None

    class _View:
        __cuda_array_interface__ = {"shape": tuple(t.shape), "typestr": typestr, "data": (p, False), "version": 2,
                                    "strides": None}
    a = torch.as_tensor(_View(), device="cuda")
    return a if a.data_ptr() == p and a.is_contiguous() else None


def score_windows(dsa, batch):
    """Score windows of one dsa_decode call (query tokens are scored in
    windows whose scores fit the workspace's 1 GiB slab).  The call launches
    an append (unless every sequence has one token), a score and a top-k per
    window, the attention, and a combine when tokens are split; with k = 1
    no token is split."""
    n = dsa.dsa_decode_launches(batch, 1, 64, 1)
    append = 0 if batch.max_q_per_seq == 1 else 1
    return (n - append - 1) // 2


def workload_line(wl, res, pk, steps, headline=False, alg=None):
    """The numbers of one workload: throughput, per-kernel rooflines, the
    dominant kernel (longest per-kernel time) and the whole step against the
    HBM roofline of the bytes it must move."""
    alg = alg or algorithmic(wl)
    ms = statistics.fmean(res["step_ms"])
    kernels = {st: dict(ms=round(m, 5), **kernel_roofline(st, m, wl, alg, pk)) for st, m in res["kernel_ms"].items()}
    if alg.get("kpool"):
        kernels.get("k_append", {})["kernel_name"] = "kpool_append_kernel"
    dom = max(res["kernel_ms"], key=res["kernel_ms"].get)
    roof = dict(kernels[dom])
    roof["kernel"] = KERNEL_OF_STAGE[dom]
    roof["ms_per_launch_note"] = res["kernel_source"]
    roof["peak_source"] = f"{pk['source']} (MEASURED_PEAKS.json)" if pk["source"] == "measured" else "fallback"
    roof["traffic"] = ncu_traffic(KERNEL_OF_STAGE[dom], wl.name)
    step_gbs = alg["step_bytes"] / (ms * 1e-3) / 1e9
    line = {"workload": wl.name, "kind": "decode" if wl.max_q_per_seq == 1 else "prefill", "B": wl.B, "T": wl.T,
            "L": wl.max_kv, "H_I": wl.H_I, "H": wl.H, "top_k": wl.top_k, "hadamard": wl.hadamard,
            "steps": steps, "ms_per_step": ms, "tok_s": wl.T / (ms * 1e-3),
            "roofline": roof, "kernels": kernels,
            "step_roofline": {"bound": "hbm", "algorithmic_bytes": alg["step_bytes"], "achieved": step_gbs,
                              "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": step_gbs / pk["hbm_gbs"]},
            "timeline_us": res["timeline_us"], "stages_ms": res["stages_ms"], "clocks": res["clocks"],
            "gpu_launches_per_step": res["launches"]}
    return line


def kpool_workload():
    """GLM-5.3-Flash DSA decode (vllm-rdna PR #2 "Glm5Next (GLM-5.3-Flash) on
    gfx1030": kpool indexer 32 heads x 128, top_k 2048 -> 2051 positions,
    MLA-NoPE attention on 512-d latents, 64 heads): 8 sequences of 8192
    positions, the batched-decode shapes without the rope tail."""
    import dsa_synth as S
    return S.Workload("kpool_decode_B8_L8192", 6, kv_len=[8192] * 8, q_pos=[8191] * 8, cu_q=list(range(9)),
                      H_I=32, H=64, top_k=2048)


def kpool_algorithmic(wl):
    """Bytes a kpool decode step must move: every visible pooled key of each
    sequence (256 B per pool) and each token's selected latent rows (1024 B
    each, at most 4 floor(top_k/4) + 3); flops of the pool scores and the
    attention."""
    pools = sum((p + 1) // 4 for p in wl.q_pos)
    width = (wl.top_k // 4) * 4 + 3
    sel = sum(min(width, p + 1) for p in wl.q_pos)
    return dict(score_bytes=pools * 256, attn_bytes=sel * 1024, step_bytes=pools * 256 + sel * 1024,
                score_flops=pools * wl.H_I * 256, attn_flops=sel * wl.H * 2 * (512 + 512),
                topk_bytes=pools * 4, append_bytes=wl.T * 2 * 514, out_bytes=wl.T * wl.H * 512 * 4)


def measure_kpool(dsa, torch, wl, steps, warmup, flush_mb, world=1):
    """dsa_decode_kpool steps, timed like measure(): the context's pooled keys
    are built first by appending every cached position."""
    import numpy as np
    import dsa_synth as S
    inp = S.make_kpool_inputs(wl)

    def up(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).cuda()
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    rows, kv_latent = up(inp.rows), up(inp.kv_latent)
    pool = torch.zeros(((wl.cache_rows + 3) // 4, 128), dtype=torch.float16, device="cuda")
    ape = up(inp.ape)
    # context: positions 0 .. p - 1 of every sequence, with the rows' own k and gate
    ctx_pos = [s for p in wl.q_pos for s in range(p)]
    ctx_cu = [0]
    for p in wl.q_pos:
        ctx_cu.append(ctx_cu[-1] + p)
    tok = [wl.kv_off[b] + s for b, p in enumerate(wl.q_pos) for s in range(p)]
    b_ctx = dsa.Batch.from_host(ctx_cu, ctx_pos, wl.kv_off, wl.cache_rows, max_q_per_seq=max(wl.q_pos),
                                max_kv=max(wl.q_pos))
    ws0 = dsa.workspace(dsa.DSA_OP_K_APPEND, b_ctx)
    dsa.dsa_kpool_append(up(np.ascontiguousarray(inp.rows[tok, :128])), up(np.ascontiguousarray(inp.rows[tok, 128:256])),
                         ape, b_ctx, rows, pool, ws0)
    torch.cuda.synchronize()
    batch = dsa.Batch.from_host(wl.cu_q, wl.q_pos, wl.kv_off, wl.cache_rows, max_q_per_seq=wl.max_q_per_seq,
                                max_kv=wl.max_kv)
    ws = dsa.workspace(dsa.DSA_OP_KPOOL, batch, wl.H_I, wl.H, wl.top_k)
    k_new, gate_new, q_idx, w, q_lat = (up(inp.k_new), up(inp.gate_new), up(inp.q_idx), up(inp.w), up(inp.q_lat))
    out = torch.empty((wl.T, wl.H, 512), device="cuda")
    lse = torch.empty((wl.T, wl.H), device="cuda")
    idx = torch.empty((wl.T, dsa.kpool_width(wl.top_k)), dtype=torch.int32, device="cuda")
    flush = torch.empty(flush_mb << 20, dtype=torch.uint8, device="cuda")
    flush_r = torch.ones((flush_mb << 20) // 4, dtype=torch.float32, device="cuda")
    tl_buf = torch.zeros(10, dtype=torch.int64, device="cuda")

    def flush_l2(i):
        flush.fill_(i & 0xFF)
        flush_r.amax()

    def step():
        dsa.dsa_decode_kpool(k_new, gate_new, ape, q_idx, w, q_lat, rows, pool, kv_latent, batch, wl.top_k,
                             wl.sm_scale, out, lse, idx, ws)

    for i in range(3 + warmup):
        flush_l2(i)
        step()
    torch.cuda.synchronize()
    if dsa.dsa_read_device_status(ws) != 0:
        raise RuntimeError(f"{wl.name}: device status flags set during warm-up")
    clocks = Clocks(gpu_index_for(torch.cuda.current_device()))
    time.sleep(0.2)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        flush_l2(i)
        ev[i][0].record()
        step()
        ev[i][1].record()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clock_rows = clocks.stop()
    big = torch.iinfo(torch.int64).max
    excl = {st: [] for st in TIMELINE_ORDER}
    spans = {st: [] for st in TIMELINE_ORDER}
    for i in range(min(steps, 200)):
        tl_buf[0::2] = big
        tl_buf[1::2] = 0
        flush_l2(i)
        dsa.dsa_set_timeline(tl_buf)
        step()
        dsa.dsa_set_timeline(None)
        torch.cuda.synchronize()
        v = tl_buf.tolist()
        t0 = min(x for x in v[0::2] if x != big)
        sp = {st: ((v[2 * j] - t0) / 1e3, (v[2 * j + 1] - t0) / 1e3)
              for j, st in enumerate(TIMELINE_ORDER) if v[2 * j] != big}
        for st, x in sp.items():
            spans[st].append(x)
        for st, x in exclusive_spans(sp).items():
            excl[st].append(x)
    if dsa.dsa_read_device_status(ws) != 0:
        raise RuntimeError(f"{wl.name}: device status flags set during the timed steps")
    # 2 appends? one (one token per sequence); then a score and top-k per
    # window, the expansion, the attention and (split tokens) the combine
    return dict(step_ms=[a.elapsed_time(b) for a, b in ev],
                kernel_ms={st: statistics.median(v) / 1e3 for st, v in excl.items() if v},
                kernel_source=("device timeline (globaltimer): exclusive spans in the overlapped step (the expansion "
                               "kernel between top-k and attention has no slot and falls in the attention's share)"),
                launches=6, clocks=Clocks.summary(clock_rows),
                timeline_us={st: [round(statistics.median(a for a, _ in v), 2),
                                  round(statistics.median(b for _, b in v), 2)] for st, v in spans.items() if v},
                stages_ms={})


def main():
    args = parse()
    if args.impl == "reference":
        return reference_arm(args)
    if args.workload == "indexshare_decode":
        return layer_stack(args)

    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)

    from dsa_sparse_attention_score_gb300 import build as lib_build
    if rank == 0 or world == 1:
        lib_build.build()
    if world > 1:
        torch.distributed.barrier()
    import dsa_sparse_attention_score_gb300 as dsa
    import dsa_synth as S

    pk = peaks()
    if args.workload == "kpool_decode":                  # the GLM-5.3-Flash step alone
        w2 = kpool_workload()
        r2 = measure_kpool(dsa, torch, w2, args.steps, args.warmup, args.flush_mb, world=world)
        line = workload_line(w2, r2, pk, args.steps, alg=dict(kpool_algorithmic(w2), kpool=True))
        line.update(metric=METRIC, unit=UNIT, value=job_throughput(world, w2.T, args.steps,
                                                                       max_over_ranks(sum(r2["step_ms"]) / 1e3)),
                    n_gpus=world, higher_is_better=True, scaling="weak", config={"workload": w2.name})
        if rank == 0:
            print(json.dumps(line), flush=True)
        return 0
    wl = shrink(S.config(WORKLOADS[args.workload]), args.tokens)
    n_e2e = max(1, min(args.e2e_steps, args.steps))
    res = measure(dsa, torch, wl, args.steps, args.warmup, args.flush_mb, world=world, e2e_steps=n_e2e,
                  graph=args.graph)
    total_s = max_over_ranks(sum(res["step_ms"]) / 1e3)
    ms_per_step = 1e3 * total_s / args.steps
    value = job_throughput(world, wl.T, args.steps, total_s)
    e2e_s = max_over_ranks(sum(res["e2e_ms"]) / 1e3)
    e2e_value = job_throughput(world, wl.T, n_e2e, e2e_s)
    head = workload_line(wl, res, pk, args.steps, headline=True)
    gpu_launches = res["launches"] * args.steps

    # ---- the rest of the metric: the ragged long-context decode and the two
    # prefill workloads, each on its own (fewer steps for the long ones)
    extra = {}
    if not args.headline_only and args.workload == "batched_decode":
        for name in EXTRA_WORKLOADS:
            torch.cuda.empty_cache()
            n2 = max(3, min(args.steps, 20 if name != "long_prefill" else 10))
            if name == "kpool_decode":
                w2 = kpool_workload()
                r2 = measure_kpool(dsa, torch, w2, n2, max(3, min(args.warmup, 5)), args.flush_mb, world=world)
                extra[name] = workload_line(w2, r2, pk, n2, alg=dict(kpool_algorithmic(w2), kpool=True))
                extra[name]["selection_width"] = dsa.kpool_width(w2.top_k)
            else:
                w2 = S.config(WORKLOADS[name])
                r2 = measure(dsa, torch, w2, n2, max(3, min(args.warmup, 5)), args.flush_mb, world=world)
                extra[name] = workload_line(w2, r2, pk, n2)
            extra[name]["ms_per_step"] = 1e3 * max_over_ranks(sum(r2["step_ms"]) / 1e3) / n2
            extra[name]["tok_s"] = job_throughput(world, w2.T, n2, 1e-3 * extra[name]["ms_per_step"] * n2)
            gpu_launches += r2["launches"] * n2
            del r2
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp16+bf16 (f32 accumulate)", "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "T": wl.T, "L": wl.max_kv, "H_I": wl.H_I, "H": wl.H,
                   "top_k": wl.top_k, "hadamard": wl.hadamard,
                   "l2": f"flushed before every timed step ({args.flush_mb} MB write, then {args.flush_mb} MB "
                         "read of another buffer)",
                   "launch": "CUDA graph replay" if args.graph else
                             "stream launches through the C ABI (programmatic dependent launch between kernels)",
                   "parallelism": f"replicas x{world}"},
        "clocks": res["clocks"],
        "gpu_launches": gpu_launches,
        "gpu_launches_note": "library kernels inside every timed step of the headline and of the workloads below",
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                "steps": n_e2e, "path": res.get("e2e_path") or "one pinned H2D copy of the step's packed inputs, dsa_decode through the Python "
                                        "binding, D2H of the output; caches stay resident"},
        "roofline": head["roofline"],
        "kernels": head["kernels"],
        "step_roofline": head["step_roofline"],
        "timeline_us": head["timeline_us"],
        "timeline_note": "median [first CTA start, last CTA end] of each kernel inside an overlapped step, from the "
                         "library's device timeline (globaltimer), relative to the first start",
        "stages_ms": head["stages_ms"],
        "stages_note": "per-stage times with events between the stages (they serialise the kernels and add launch "
                       "latency); the roofline uses the device timeline instead",
    }
    if extra:
        line["workloads"] = extra
        line["workloads_note"] = ("the other workloads of the metric, each measured like the headline (cold L2, "
                                  "CUDA events per step); prefill tok/s = query tokens of the chunk / step time")
    if world == 1 and not args.no_cpu_baseline:
        inp = S.make_inputs(wl)
        line["cpu_baseline"] = run_oracle_sample(wl, inp, args.cpu_seconds)
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
