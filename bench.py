#!/usr/bin/env python
"""Decode-step benchmark of the QSA sparse-attention path on GB300.

A step is one decode step of one QSA layer: pooled-key cache update, index score of every
pooled row, block-domain top-k, cell list, sparse attention over the selected cells.
Each step appends one token to its layer; steps rotate over ``--layers`` independent
layer sets (12 QSA layers per token in the pages' model), so successive steps never
re-read the same pooled cache from L2.

Prints one JSON line: decode steps/s at the primary context (255,181 tokens by default),
with the 61,789 / 126,253 / 255,181-token sweep, the HBM roofline of the score scan, an
end-to-end figure with host buffers, SM clocks sampled during the timed region and the
fp64 CPU oracle timed on a bounded sample as a baseline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun every rank runs an independent replica ("replicas only": the decode path
of one sequence does not shard); value = steps of all ranks / max time over ranks.
"""
from __future__ import annotations

import argparse
import functools
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "sparse-attn decode steps/s at 64k/128k/256k ctx; achieved HBM GB/s vs roofline"
CONTEXTS = {"64k": "decode_64k", "128k": "decode_128k", "256k": "decode_256k"}
SCORE_SRCS = [os.path.join(ROOT, "gather_qsa_pool_gb300", "csrc", f)
              for f in ("index_score.cu", "score_stream.cuh")]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "score_stream_256k_traffic.txt")
STEP_SCORE_SRCS = [os.path.join(ROOT, "gather_qsa_pool_gb300", "csrc", f)
                   for f in ("score_pool.cu", "score_stream.cuh", "qsa_internal.cuh")]
STEP_TRAFFIC_FILE = os.path.join(ROOT, "profiles", "score_pool_256k_traffic.txt")
# Kernels one qsa_decode_step launches when it appends a token: the fused pool-update +
# score scan, the top-k (whose last CTA also writes the cell list) and the attention
# kernel (split-K with the combine inside its cluster).
LAUNCHES_PER_DECODE_STEP = 3
SCORE_POOL_THREADS = 256  # block size of the step's score kernel (score_pool_kernel)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3072)
    ap.add_argument("--warmup", type=int, default=24)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--contexts", default="64k,128k,256k")
    ap.add_argument("--primary", default="256k")
    ap.add_argument("--layers", type=int, default=12)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-mask", action="store_true")
    ap.add_argument("--no-ablation", action="store_true",
                    help="skip the timing of the pages' earlier path, piece by piece")
    ap.add_argument("--prefill-reps", type=int, default=5)
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the bf16 pooled-cache and multi-query decode lines")
    ap.add_argument("--pooled", choices=["f32", "bf16"], default="f32",
                    help="pooled-key cache storage of the main sweep")
    ap.add_argument("--queries", type=int, default=1, choices=[1, 2, 3, 4],
                    help="query tokens per decode step of the main sweep")
    ap.add_argument("--union-only", action="store_true",
                    help="run only the grouped-union sweep (a profiling case; with "
                         "--union-queries / --union-depth / --union-shares)")
    ap.add_argument("--union-queries", type=int, default=1024)
    ap.add_argument("--union-depth", type=int, default=255181)
    ap.add_argument("--union-shares", default="0,0.5,0.75,0.85,0.9,0.95,1")
    return ap.parse_args()


# ----------------------------------------------------------------------------- plumbing

def dist_setup():
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi sampled every 20 ms while the timed region runs."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def mark(self):
        return time.time()

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self, t0: float, t1: float):
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts + frac, float(parts[2]), float(parts[3]), parts[6:10]))
            except Exception:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sel = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in sel for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[1] for r in sel),
                "sm_max_mhz": max(r[2] for r in sel), "reasons": reasons, "samples": len(sel)}


def traffic_per_launch(path, srcs, n_rows):
    """DRAM bytes per launch from a committed ncu summary (bytes per pooled row, scaled to
    n_rows), if it was taken on the current kernel sources ``srcs`` (else None)."""
    try:
        h = hashlib.sha256()
        for src in srcs:
            with open(src, "rb") as f:
                h.update(f.read())
        sha = h.hexdigest()[:16]
        kv = {}
        with open(path) as f:
            for ln in f:
                if "=" in ln and not ln.startswith("#"):
                    k, v = ln.split("=", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha256_16") != sha:
            return None
        return float(kv["dram_bytes_per_row"]) * n_rows
    except Exception:
        return None


# ----------------------------------------------------------------------------- GPU arm

def run_context(name, args, world, rank, local, want_clocks, pooled="f32", n_q=1, light=False,
                winners=False):
    """Decode steps at one context length over ``args.layers`` rotating layer sets.
    pooled: storage of the pooled-key cache ("f32" or "bf16"); n_q: query tokens per step
    (a token and its drafts, each step appending n_q tokens); light: skip the CUDA-graph
    replay and the end-to-end loop; winners: scores with clear winners (1% of the completed
    pooled rows leaning toward the queries' common direction, qsa_synth.clear_winners_torch)."""
    import torch

    import gather_qsa_pool_gb300 as qsa
    import qsa_synth

    shape = qsa_synth.CONFIGS[CONTEXTS[name]]
    L = args.layers
    K, W = args.steps, args.warmup
    k_kernel = max(L, min(K, 4 * L * 16))
    k_e2e = 0 if light else max(L, min(K, 1024))
    total_steps = W + K + k_e2e + 2
    extra = n_q * (total_steps // L + 2)
    dev = torch.device("cuda", local)
    n_q_pool = 32
    pdt = torch.bfloat16 if pooled == "bf16" else torch.float32

    layers, caches, win_rows = [], [], []
    for li in range(L):
        inp = qsa_synth.decode_inputs_torch(shape, seed=1000 * (rank + 1) + li, device=dev,
                                            extra_tokens=extra, n_steps=n_q_pool)
        lay = qsa.DecodeLayer(cap_tokens=shape.n_ctx + extra, H_idx=shape.H_idx,
                              d_idx=shape.d_idx, H_q=shape.H_q, H_kv=shape.H_kv, d=shape.d,
                              top_k_tokens=shape.top_k_tokens, eps=shape.eps,
                              rope_base=shape.rope_base, pooled_dtype=pdt, max_queries=n_q,
                              device=dev)
        lay.rebuild(inp["raw_k"], inp["norm_w"], shape.n_ctx - 1)
        if winners:
            cw = qsa_synth.clear_winners_torch((shape.n_ctx - 1) // 4, shape.H_idx * shape.d_idx,
                                               n_q_pool, seed=77 + 1000 * (rank + 1) + li,
                                               device=dev)
            lay.pooled[cw["rows"]] = (lay.pooled[cw["rows"]].float() + cw["add"]).to(pdt)
            inp["q_idx"] = cw["q_idx"]
            win_rows.append(cw["rows"])
        if not light:
            lay.enable_host_feed(inp["raw_k"].dtype, inp["K"].dtype)
        lay.bind(inp["raw_k"], inp["norm_w"], inp["K"], inp["V"])
        layers.append(lay)
        caches.append(inp)
        del inp
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    n_ctx = [shape.n_ctx] * L  # context length of each layer's next step
    q_ptrs = [([c["q_idx"][j].data_ptr() for j in range(n_q_pool)],
               [c["q"][j].data_ptr() for j in range(n_q_pool)]) for c in caches]

    def step(s):
        li = s % L
        j = (s // L) % (n_q_pool - n_q + 1)
        n_ctx[li] += n_q - 1
        layers[li].step_ptr(n_ctx[li], q_ptrs[li][0][j], q_ptrs[li][1][j], sp, n_q)
        n_ctx[li] += 1

    s = 0
    for _ in range(W):
        step(s)
        s += 1
    torch.cuda.synchronize()
    barrier(world)
    sampler = None
    if want_clocks:
        sampler = ClockSampler(local)
        sampler.start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(world)
    t_wall0 = time.time()
    ev0.record(stream)
    t_issue0 = time.perf_counter()
    for _ in range(K):
        step(s)
        s += 1
    t_issue = time.perf_counter() - t_issue0
    ev1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier(world)
    ms = ev0.elapsed_time(ev1)
    clocks = None
    if sampler is not None:
        sampler.stop()
        clocks = sampler.summary(t_wall0, t_wall1)
    ms_max = max_over_ranks(ms, world)

    # the same steps replayed from a CUDA graph (one captured step per layer set, context
    # lengths fixed at capture): launch issue leaves the host
    graph_us, graph_err = None, None
    if light:
        graph_err = "not run"
    try:
        if light:
            raise RuntimeError("not run")
        gs = torch.cuda.Stream(device=dev)
        gs.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(gs):
            with torch.cuda.graph(graph, stream=gs):
                for li in range(L):
                    layers[li].step_ptr(n_ctx[li] + n_q - 1, q_ptrs[li][0][0], q_ptrs[li][1][0],
                                        gs.cuda_stream, n_q)
            for li in range(L):
                layers[li].n_valid_full = (n_ctx[li] - 1) // 4
        torch.cuda.synchronize()
        reps = max(3, K // L)
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(torch.cuda.current_stream())
        for _ in range(reps):
            graph.replay()
        g1.record(torch.cuda.current_stream())
        torch.cuda.synchronize()
        graph_us = g0.elapsed_time(g1) * 1e3 / (reps * L)
        del graph
    except Exception as e:  # capture unsupported on this driver: report why
        if not light:
            graph_err = f"{type(e).__name__}: {e}"[:200]
        torch.cuda.synchronize()

    # the step's own score kernel (pool update of the new / open rows + scan of every row +
    # the top-k histogram), live: each layer set's step captured, all kernels but the score
    # kernel dropped from the graph, the rest replayed over the rotating layer sets
    step_score_us, step_score_err = None, None
    if not light:
        try:
            def cap_of(li):
                def cap(stream_ptr):
                    layers[li].step_ptr(n_ctx[li] + n_q - 1, q_ptrs[li][0][0], q_ptrs[li][1][0],
                                        stream_ptr, n_q)
                return cap

            step_score_us = step_kernel_us([cap_of(li) for li in range(L)], 0,
                                           SCORE_POOL_THREADS, max(3, K // L), dev)
        except Exception as e:
            step_score_err = f"{type(e).__name__}: {e}"[:200]
        finally:
            for li in range(L):
                layers[li].n_valid_full = (n_ctx[li] - 1) // 4
                # the replays added to the top-k histograms: start the next step from zero
                layers[li].workspace.zero_()
            torch.cuda.synchronize()

    # score kernel alone, back to back over the rotating layers (its average duration)
    n_rows = [(c + 3) // 4 for c in n_ctx]

    # the C call with its arguments marshalled once per layer set, so that issuing the
    # launches stays well ahead of the GPU even for the short scans
    lib = qsa.load()
    score_args = []
    for li in range(L):
        pdt_c = qsa.QSA_BF16 if pooled == "bf16" else qsa.QSA_F32
        score_args.append([(caches[li]["q_idx"][j].data_ptr(), n_q, shape.H_idx * shape.d_idx,
                            None, layers[li].pooled.data_ptr(), pdt_c, n_rows[li], shape.H_idx,
                            shape.d_idx, 1.0 / math.sqrt(shape.d_idx),
                            layers[li].scores.data_ptr(), n_rows[li], qsa.QSA_PREC_F32, None, 0,
                            sp) for j in range(n_q_pool - n_q + 1)])

    def score_only(i):
        a = score_args[i % L]
        st_ = lib.qsa_index_score(*a[i % len(a)])
        if st_ != 0:
            raise qsa.QSAError("qsa_index_score", st_)

    for i in range(L):
        score_only(i)
    torch.cuda.synchronize()
    ev2, ev3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev2.record(stream)
    for i in range(k_kernel):
        score_only(i)
    ev3.record(stream)
    torch.cuda.synchronize()
    score_us = ev2.elapsed_time(ev3) * 1e3 / k_kernel
    score_rows = sum(n_rows[i % L] for i in range(k_kernel)) / k_kernel

    # end to end through the C call with host buffers (qsa_decode_plan_step_host): per step
    # the new token's raw-key, K and V rows and both queries cross from page-locked host
    # memory (a copy kernel reads them in place), the step, the output crosses back (a copy
    # kernel writes it into page-locked host memory), and a wait for it
    h2d = d2h = 0
    if not light:
        g = torch.Generator()
        g.manual_seed(99)
        for lay in layers:
            hin = lay.host_inputs(1)
            for key in ("raw", "k", "v", "q_idx", "q"):
                hin[key].copy_(torch.randn(hin[key].shape, generator=g).to(hin[key].dtype))
        h2d = layers[0].host_inputs(1)["bytes"]
        d2h = shape.H_q * shape.d * 4
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(k_e2e):
        li = s % L
        layers[li].step_host(n_ctx[li], sp, 1)
        n_ctx[li] += 1
        s += 1
        stream.synchronize()
    t_e2e = time.perf_counter() - t0
    t_e2e = max_over_ranks(t_e2e, world)

    splits = qsa._binding.load()  # noqa: F841  (library already loaded)
    n_cells_last = int(layers[(s - 1) % L].n_cells[0].item())
    winner_share = None
    if winners:  # of the blocks the last step selected, the share that are leaning rows
        lw = layers[(s - 1) % L]
        sel = lw.blocks[0, :int(lw.counts[0].item())].long()
        winner_share = float(torch.isin(sel, win_rows[(s - 1) % L]).float().mean().item())
    res = {
        "ms": ms_max, "K": K, "W": W, "score_us": score_us, "score_rows": score_rows,
        "t_e2e": t_e2e, "k_e2e": k_e2e, "host_issue_us": t_issue * 1e6 / K, "h2d": h2d, "d2h": d2h, "clocks": clocks,
        "n_cells": n_cells_last, "shape": shape, "n_ctx_end": max(n_ctx),
        "graph_us": graph_us, "graph_err": graph_err, "pooled": pooled, "n_q": n_q,
        "step_score_us": step_score_us, "step_score_err": step_score_err,
        "step_score_rows": sum((c + n_q - 1 + 3) // 4 for c in n_ctx) / L,
        "winner_share": winner_share,
    }
    del layers, caches
    torch.cuda.empty_cache()
    return res


def graph_time_us(fns, reps, dev):
    """Device time per repetition of the calls fns (in order), captured reps times into one
    CUDA graph and replayed after a warm-up replay: the kernels' time, not the Python
    wrappers' issue time."""
    import torch

    gs = torch.cuda.Stream(device=dev)
    for fn in fns:
        fn()
    torch.cuda.synchronize()
    gs.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(gs):
        with torch.cuda.graph(graph, stream=gs):
            for _ in range(reps):
                for fn in fns:
                    fn()
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    graph.replay()
    b.record()
    torch.cuda.synchronize()
    del graph
    return a.elapsed_time(b) * 1e3 / reps


class _KernelNodeParams(__import__("ctypes").Structure):
    """CUDA_KERNEL_NODE_PARAMS_v2 of the driver API (the fields read here)."""
    import ctypes as _ct
    _fields_ = [("func", _ct.c_void_p), ("gridDimX", _ct.c_uint), ("gridDimY", _ct.c_uint),
                ("gridDimZ", _ct.c_uint), ("blockDimX", _ct.c_uint), ("blockDimY", _ct.c_uint),
                ("blockDimZ", _ct.c_uint), ("sharedMemBytes", _ct.c_uint),
                ("kernelParams", _ct.c_void_p), ("extra", _ct.c_void_p), ("kern", _ct.c_void_p),
                ("ctx", _ct.c_void_p)]


def step_kernel_us(captures, keep, block_x, reps, dev):
    """Live device time of one kernel of the decode step, as the step runs it: each function
    of ``captures`` issues one decode step (three kernels) on the stream it is given, which
    is captured into a CUDA graph through the driver API; a clone of each graph keeps only
    the kernel at position ``keep`` (checked by its block size, ``block_x``), and the
    one-kernel graphs are replayed round-robin between CUDA events on one stream (so they
    run one after another, as inside the steps).  Returns microseconds per kernel.  The kept
    kernels read and write exactly what they do inside the step."""
    import ctypes

    import torch

    cu = ctypes.CDLL("libcuda.so.1")
    V = ctypes.c_void_p

    def ck(r, what):
        if r != 0:
            raise RuntimeError(f"{what}: CUresult {r}")

    gs = torch.cuda.Stream(device=dev)
    gs.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    h = V(gs.cuda_stream)
    graphs, execs = [], []
    try:
        for capture in captures:
            graph = V()
            ck(cu.cuStreamBeginCapture_v2(h, ctypes.c_int(2)), "cuStreamBeginCapture")  # relaxed
            try:
                capture(gs.cuda_stream)
            finally:
                r_end = cu.cuStreamEndCapture(h, ctypes.byref(graph))
            ck(r_end, "cuStreamEndCapture")
            graphs.append(graph)
            n = ctypes.c_size_t(0)
            ck(cu.cuGraphGetNodes(graph, None, ctypes.byref(n)), "cuGraphGetNodes")
            nodes = (V * n.value)()
            ck(cu.cuGraphGetNodes(graph, nodes, ctypes.byref(n)), "cuGraphGetNodes")
            kern = []
            for i in range(n.value):
                t = ctypes.c_int(-1)
                ck(cu.cuGraphNodeGetType(V(nodes[i]), ctypes.byref(t)), "cuGraphNodeGetType")
                if t.value == 0:  # CU_GRAPH_NODE_TYPE_KERNEL
                    kern.append(nodes[i])
            if len(kern) != 3:
                raise RuntimeError(f"{len(kern)} kernel nodes in one step")
            kept = kern[keep]
            prm = _KernelNodeParams()
            ck(cu.cuGraphKernelNodeGetParams_v2(V(kept), ctypes.byref(prm)), "params")
            if prm.blockDimX != block_x:
                raise RuntimeError(f"kept kernel has {prm.blockDimX} threads, not {block_x}")
            clone = V()
            ck(cu.cuGraphClone(ctypes.byref(clone), graph), "cuGraphClone")
            graphs.append(clone)
            for i in range(n.value):
                if nodes[i] == kept:
                    continue
                cn = V()
                ck(cu.cuGraphNodeFindInClone(ctypes.byref(cn), V(nodes[i]), clone), "find")
                ck(cu.cuGraphDestroyNode(cn), "cuGraphDestroyNode")
            ex = V()
            ck(cu.cuGraphInstantiateWithFlags(ctypes.byref(ex), clone, ctypes.c_ulonglong(0)),
               "cuGraphInstantiate")
            execs.append(ex)
        for ex in execs:
            ck(cu.cuGraphLaunch(ex, h), "cuGraphLaunch")
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(gs)
        for _ in range(reps):
            for ex in execs:
                ck(cu.cuGraphLaunch(ex, h), "cuGraphLaunch")
        b.record(gs)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / (reps * len(execs))
    finally:
        torch.cuda.synchronize()
        for ex in execs:
            cu.cuGraphExecDestroy(ex)
        for g in graphs:
            cu.cuGraphDestroy(g)


def run_prefill(args, local, pooled_kind="f32"):
    """The prefill chunk: 1024 queries after 255,181 tokens.  Times (CUDA-graph replays after a
    warm-up) the tensor-core score contraction (which also writes each query's maxima of 32-row
    groups), the per-query top-k fed by those maxima, the cell lists and the gathered
    attention, one at a time and as one chained chunk; returns per-kernel microseconds, the
    chunk's and the score kernel's TFLOP/s, and (outside the chunk) the top-k that scans whole
    rows on the same scores.
    pooled_kind "bf16": the pooled cache is stored in bf16 and the contraction reads it in
    place (no conversion pass).  "f32_mirror": an fp32 cache kept together with a bf16 mirror
    (every pool update also writes the mirror's rows: bit for bit the cache's bf16 rounding),
    which the contraction reads in place; the chunk's own mirror update (its new rows) is
    timed as part of the chunk, in place of the rounding pass over the whole cache."""
    import torch

    import gather_qsa_pool_gb300 as qsa
    import qsa_synth

    shape = qsa_synth.CONFIGS["prefill_256k"]
    dev = torch.device("cuda", local)
    inp = qsa_synth.prefill_inputs_torch(shape, seed=4242, device=dev)
    H, d, n_q, n_rows = shape.H_idx, shape.d_idx, shape.n_q, shape.n_rows
    pdt = torch.bfloat16 if pooled_kind == "bf16" else torch.float32
    pooled = torch.zeros(n_rows, H * d, dtype=pdt, device=dev)
    qsa.pool_update(inp["raw_k"], shape.n_ctx, H, d, inp["norm_w"], shape.eps, shape.rope_base,
                    pooled, 0)
    score_src, score_dt = pooled, (qsa.QSA_BF16 if pooled_kind == "bf16" else qsa.QSA_F32)
    mirror = None
    if pooled_kind == "f32_mirror":
        # the mirror as it stood before the chunk; the chunk's rows go in inside the timing
        mirror = torch.zeros(n_rows, H * d, dtype=torch.bfloat16, device=dev)
        qsa.pool_update(inp["raw_k"], shape.depth, H, d, inp["norm_w"], shape.eps,
                        shape.rope_base, mirror, 0)
        score_src, score_dt = mirror, qsa.QSA_BF16
    scores = torch.empty(n_q, n_rows, device=dev)
    maxima = torch.empty(n_q, (n_rows + 31) // 32, device=dev)
    tws = torch.empty(qsa.topk_blocks_maxima_workspace_size(n_q), dtype=torch.uint8, device=dev)
    ws = torch.zeros(qsa.index_score_workspace_size(
        n_q, n_rows, H, d, qsa.QSA_PREC_BF16_TC, score_dt), dtype=torch.uint8, device=dev)
    blocks = torch.empty(n_q, shape.k_blk, dtype=torch.int32, device=dev)
    counts = torch.empty(n_q, dtype=torch.int32, device=dev)
    pos = torch.empty(n_q, shape.max_cells, dtype=torch.int32, device=dev)
    n_cells = torch.empty(n_q, dtype=torch.int32, device=dev)
    out = torch.empty(n_q, shape.H_q, shape.d, device=dev)
    aws = torch.empty(max(qsa.sparse_attn_workspace_size(n_q, shape.H_q, shape.H_kv, shape.d,
                                                          shape.max_cells) // 4, 1), device=dev)
    scale_idx, scale = 1.0 / math.sqrt(d), 1.0 / math.sqrt(shape.d)

    calls = []
    if mirror is not None:
        calls.append(("mirror_update",
                      lambda: qsa.pool_update(inp["raw_k"], shape.n_ctx, H, d, inp["norm_w"],
                                              shape.eps, shape.rope_base, mirror,
                                              shape.depth // 4)))
    calls += [
        ("score_tc", lambda: qsa.index_score_maxima(inp["q_idx"], score_src, n_rows, H, d,
                                                     scale_idx, scores, maxima,
                                                     q_pos=inp["q_pos"], workspace=ws)),
        ("topk", lambda: qsa.topk_blocks_maxima(scores, maxima, n_rows, shape.k_blk, blocks,
                                                counts, tws, q_pos=inp["q_pos"])),
        ("cells", lambda: qsa.gather_kv(blocks, counts, shape.k_blk, pos, n_cells, shape.max_cells,
                                        q_pos=inp["q_pos"], n_kv=shape.n_ctx)),
        ("attn", lambda: qsa.sparse_attn(inp["q"], inp["K"], inp["V"], n_cells, shape.max_cells,
                                         out, shape.H_kv, shape.d, shape.d, scale, pos=pos,
                                         workspace=aws)),
    ]
    w_blocks, w_counts = torch.empty_like(blocks), torch.empty_like(counts)
    whole_rows = ("topk_whole_rows", lambda: qsa.topk_blocks(scores, n_rows, shape.k_blk, w_blocks,
                                                             w_counts, q_pos=inp["q_pos"]))
    for _ in range(2):
        for _, fn in calls:
            fn()
    whole_rows[1]()
    torch.cuda.synchronize()
    same_selection = bool(torch.equal(blocks, w_blocks) and torch.equal(counts, w_counts))
    # each kernel's calls captured into a CUDA graph and replayed (device time), then the
    # whole chunk as one graph; plain CUDA events around direct calls if capture fails
    res, timing, chunk_graph = {}, "cuda graph replay", None
    try:
        for name, fn in calls:
            res[name] = graph_time_us([fn], args.prefill_reps, dev)
        chunk_graph = graph_time_us([fn for _, fn in calls], args.prefill_reps, dev)
        whole_us = graph_time_us([whole_rows[1]], args.prefill_reps, dev)
    except Exception as e:  # noqa: BLE001 -- reported in the JSON line
        timing = f"cuda events around direct calls (graph capture failed: {type(e).__name__})"
        torch.cuda.synchronize()
        for name, fn in calls:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(args.prefill_reps):
                fn()
            b.record()
            torch.cuda.synchronize()
            res[name] = a.elapsed_time(b) * 1e3 / args.prefill_reps
        whole_us = None
    flops = 2.0 * n_q * n_rows * H * d
    attn_flops = 2.0 * 2.0 * n_q * shape.H_q * shape.d * float(n_cells.float().mean().item())
    out_d = {
        "workload": (f"prefill chunk: {n_q} queries at positions {shape.depth:,}..{shape.n_ctx - 1:,}, "
                     f"indexer {H}x{d} ({pooled_kind.replace('_', ' with a bf16 ')} pooled cache), "
                     f"top-k {shape.top_k_tokens}, "
                     f"attention {shape.H_q}/{shape.H_kv}x{shape.d} bf16"),
        "us": {k: round(v, 1) for k, v in res.items()},
        "chunk_us": round(sum(res.values()), 1),
        "chunk_graph_us": None if chunk_graph is None else round(chunk_graph, 1),
        "topk_whole_rows_us": None if whole_us is None else round(whole_us, 1),
        "topk_same_selection": same_selection,
        "timing": timing,
        "score_tc_tflops": flops / (res["score_tc"] * 1e-6) / 1e12,
        "attn_tflops": attn_flops / (res["attn"] * 1e-6) / 1e12,
        "tokens_per_s": n_q / ((chunk_graph or sum(res.values())) * 1e-6),
    }
    del inp, pooled, mirror, score_src, scores, maxima, ws, pos, out, aws
    torch.cuda.empty_cache()
    return out_d


def run_grouped_union(args, local):
    """Grouped-union attention (qsa_sparse_attn_union) against the per-query kernel
    (qsa_sparse_attn) on the prefill chunk's shape -- 1024 queries after 255,181 tokens, 512
    selected blocks each plus the open tail -- over a sweep of how many of its blocks each
    query shares with the others of its group of 16 (qsa_synth.overlap_block_lists: the
    share of each query's blocks drawn from one common set per group, the rest drawn
    independently).  Each call captured in a CUDA graph and replayed; returns microseconds
    per call, the union's mean size per group and the share from which the union wins."""
    import torch

    import gather_qsa_pool_gb300 as qsa
    import qsa_synth

    shape = qsa_synth.shrink(qsa_synth.CONFIGS["prefill_256k"], n_q=args.union_queries,
                             depth=args.union_depth)
    dev = torch.device("cuda", local)
    n_q, n_ctx, d, H_kv, H_q = shape.n_q, shape.n_ctx, shape.d, shape.H_kv, shape.H_q
    g = torch.Generator(device=dev)
    g.manual_seed(5150)
    K = torch.randn(n_ctx, H_kv, d, generator=g, device=dev).to(torch.bfloat16)
    V = torch.randn(n_ctx, H_kv, d, generator=g, device=dev).to(torch.bfloat16)
    q = torch.randn(n_q, H_q, d, generator=g, device=dev)
    q_pos = shape.depth + np.arange(n_q)
    q_pos_d = torch.from_numpy(q_pos.astype(np.int32)).to(dev)
    scale = 1.0 / math.sqrt(d)
    ws = torch.empty(qsa.sparse_attn_union_workspace_size(n_q, shape.max_cells),
                     dtype=torch.uint8, device=dev)
    out_u = torch.empty(n_q, H_q, d, device=dev)
    out_r = torch.empty(n_q, H_q, d, device=dev)
    pos = torch.empty(n_q, shape.max_cells, dtype=torch.int32, device=dev)
    n_cells = torch.empty(n_q, dtype=torch.int32, device=dev)
    rows = []
    for share in (float(x) for x in args.union_shares.split(",")):
        blocks = qsa_synth.overlap_block_lists((q_pos + 1) // 4, shape.k_blk, 16, share,
                                               int(1000 * share) + 7)
        bl = np.zeros((n_q, shape.k_blk), np.int32)
        cnt = np.zeros(n_q, np.int32)
        for i, b in enumerate(blocks):
            bl[i, :b.shape[0]] = b
            cnt[i] = b.shape[0]
        qsa.gather_kv(torch.from_numpy(bl).to(dev), torch.from_numpy(cnt).to(dev), shape.k_blk,
                      pos, n_cells, shape.max_cells, q_pos=q_pos_d, n_kv=n_ctx)
        union = float(np.mean([np.unique(np.concatenate(blocks[i:i + 16])).shape[0]
                               for i in range(0, n_q, 16)]))
        u_us = graph_time_us([lambda: qsa.sparse_attn_union(q, K, V, n_cells, shape.max_cells,
                                                            out_u, H_kv, d, scale, pos,
                                                            workspace=ws)],
                             args.prefill_reps, dev)
        r_us = graph_time_us([lambda: qsa.sparse_attn(q, K, V, n_cells, shape.max_cells, out_r,
                                                      H_kv, d, d, scale, pos=pos)],
                             args.prefill_reps, dev)
        diff = float((out_u - out_r).abs().max().item())
        rows.append({"share": share, "union_blocks_per_group": round(union, 1),
                     "union_us": round(u_us, 1), "per_query_us": round(r_us, 1),
                     "max_abs_diff": diff})
    wins = [r["share"] for r in rows if r["union_us"] < r["per_query_us"]]
    del K, V, q, ws, out_u, out_r, pos, n_cells
    torch.cuda.empty_cache()
    return {"workload": (f"{n_q} queries at positions {shape.depth:,}..{n_ctx - 1:,}, "
                         f"{shape.k_blk} blocks + tail each, groups of 16, attention "
                         f"{H_q}/{H_kv}x{d} bf16"),
            "timing": "cuda graph replay", "sweep": rows,
            "union_wins_from_share": min(wins) if wins else None}


def run_ablation(args, local):
    """The pages' A/B on this GPU at 255,181 tokens: each piece of the QSA decode step next
    to the piece it replaced -- the full pooled-cache rebuild (before the incremental cache),
    the block score expanded to cells and a cell-level top-k (before the block-domain
    top-k), attention over every cell of the context (before the selected-K/V gather) -- and
    the gather itself as the pages run it (the listed K/V rows copied into a compact buffer,
    then attention over that buffer), which the decode step replaces by reading the rows in
    place.  CUDA events over a few repetitions after a warm-up call; returns microseconds."""
    import torch

    import gather_qsa_pool_gb300 as qsa
    import qsa_synth

    shape = qsa_synth.CONFIGS["decode_256k"]
    dev = torch.device("cuda", local)
    inp = qsa_synth.decode_inputs_torch(shape, seed=777, device=dev)
    H, d, n_ctx = shape.H_idx, shape.d_idx, shape.n_ctx
    n_rows, n_full, k_blk = shape.n_rows, shape.n_full, shape.k_blk
    lay = qsa.DecodeLayer(cap_tokens=n_ctx, H_idx=H, d_idx=d, H_q=shape.H_q, H_kv=shape.H_kv,
                          d=shape.d, top_k_tokens=shape.top_k_tokens, eps=shape.eps,
                          rope_base=shape.rope_base, device=dev)
    raw, w, K, V = inp["raw_k"], inp["norm_w"], inp["K"], inp["V"]
    lay.rebuild(raw, w, n_ctx - 1)
    lay.step(raw, w, K, V, n_ctx, inp["q_idx"][0], inp["q"][0])
    q = inp["q"][:1]
    scores = lay.scores_of(1, n_ctx)
    blocks = torch.empty(1, k_blk, dtype=torch.int32, device=dev)
    counts = torch.empty(1, dtype=torch.int32, device=dev)
    cells = torch.empty(1, 4 * n_full, device=dev)
    cell_sel = torch.empty(1, 4 * k_blk, dtype=torch.int32, device=dev)
    out = torch.empty(1, shape.H_q, shape.d, device=dev)
    all_pos = torch.arange(n_ctx, dtype=torch.int32, device=dev).view(1, n_ctx)
    all_n = torch.tensor([n_ctx], dtype=torch.int32, device=dev)
    ws = torch.zeros(max(qsa.sparse_attn_workspace_size(1, shape.H_q, shape.H_kv, shape.d, n_ctx)
                         // 4, 1), device=dev)
    scale_idx, scale = 1.0 / math.sqrt(d), 1.0 / math.sqrt(shape.d)
    mc = lay.max_cells
    Kc = torch.empty(mc, shape.H_kv, shape.d, dtype=K.dtype, device=dev)
    Vc = torch.empty(mc, shape.H_kv, shape.d, dtype=V.dtype, device=dev)
    g_pos = torch.empty(1, mc, dtype=torch.int32, device=dev)
    g_n = torch.empty(1, dtype=torch.int32, device=dev)
    pieces = [
        ("pool_full_rebuild", lambda: qsa.pool_update(raw, n_ctx, H, d, w, shape.eps,
                                                      shape.rope_base, lay.pooled, 0)),
        ("pool_incremental", lambda: qsa.pool_update(raw, n_ctx, H, d, w, shape.eps,
                                                     shape.rope_base, lay.pooled, n_full - 1)),
        ("score_scan", lambda: qsa.index_score(inp["q_idx"][:1], lay.pooled, n_rows, H, d,
                                               scale_idx, scores)),
        ("block_topk", lambda: qsa.topk_blocks(scores, n_full, k_blk, blocks, counts)),
        ("expand_to_cells", lambda: qsa.expand_block_scores(scores, n_full, cells)),
        ("cell_topk", lambda: qsa.topk_blocks(cells, 4 * n_full, 4 * k_blk, cell_sel, counts)),
        ("attn_listed_cells", lambda: qsa.sparse_attn(q, K, V, lay.n_cells[:1], lay.max_cells,
                                                      out, shape.H_kv, shape.d, shape.d, scale,
                                                      pos=lay.pos[:1], workspace=lay.workspace)),
        ("attn_full_kv", lambda: qsa.sparse_attn(q, K, V, all_n, n_ctx, out, shape.H_kv, shape.d,
                                                 shape.d, scale, pos=all_pos, workspace=ws)),
        ("gather_rows", lambda: qsa.gather_kv(blocks, counts, k_blk, g_pos, g_n, mc, n_ctx=n_ctx,
                                              K=K, V=V, K_out=Kc, V_out=Vc, H_kv=shape.H_kv,
                                              d_k=shape.d, d_v=shape.d)),
        ("attn_gathered_rows", lambda: qsa.sparse_attn(q, Kc, Vc, g_n, mc, out, shape.H_kv,
                                                       shape.d, shape.d, scale,
                                                       workspace=lay.workspace)),
    ]
    # each piece captured (reps calls) into a CUDA graph and replayed, so the device time is
    # measured rather than the Python wrapper's issue time
    res = {name: round(graph_time_us([fn], 5, dev), 1) for name, fn in pieces}
    n_listed = int(lay.n_cells[0].item())
    n_gathered = int(g_n[0].item())
    gather_bytes = 2 * n_gathered * shape.H_kv * shape.d * K.element_size() * 2  # read + write
    out_d = {
        "workload": (f"one layer at {n_ctx:,} tokens: {n_rows:,} pooled rows, {n_listed} listed "
                     f"cells of {n_ctx:,}"),
        "us": res,
        "old_path_us": round(res["pool_full_rebuild"] + res["score_scan"] + res["expand_to_cells"]
                             + res["cell_topk"] + res["attn_full_kv"], 1),
        "qsa_pieces_us": round(res["pool_incremental"] + res["score_scan"] + res["block_topk"]
                               + res["attn_listed_cells"], 1),
        "gather_rows_GBps": round(gather_bytes / res["gather_rows"] / 1e3, 1),
        "gather_then_attend_us": round(res["gather_rows"] + res["attn_gathered_rows"], 1),
        "note": ("pieces timed one at a time from CUDA-graph replays (the fused decode step "
                 "overlaps them and uses the histogram-fed top-k); the old path is the sum of "
                 "the pieces it ran; gather_rows copies the selected blocks' K and V rows (and "
                 "the open tail) into a compact buffer, gather_then_attend_us adds the "
                 "attention over that buffer, against attn_listed_cells reading the rows in "
                 "place"),
    }
    del lay, inp, cells, ws, Kc, Vc
    torch.cuda.empty_cache()
    return out_d


def run_mask(args, local):
    """The mask-driven variant at 32,768 keys: mask -> position list (qsa_mask_to_list) and
    attention of 16 query heads over the listed keys (DKQ 576, d_v 512, bf16), separately,
    back to back, and as the one call qsa_mask_sparse_attn.  Eight rotating input sets
    (about 300 MB of K/V) keep consecutive calls out of L2.  Returns microseconds per call
    and GB/s of the bytes each call must read."""
    import torch

    import gather_qsa_pool_gb300 as qsa
    import qsa_synth

    shape = qsa_synth.CONFIGS["mask_32k"]
    dev = torch.device("cuda", local)
    n_sets = 8
    g = torch.Generator(device=dev)
    g.manual_seed(32768)
    sets = []
    for i in range(n_sets):
        m = torch.from_numpy(qsa_synth.mask_rows(shape.n_q, shape.n_kv, seed=100 + i)).to(dev)
        KV = torch.randn(shape.n_kv, shape.d_k, device=dev, generator=g).to(torch.bfloat16)
        q = torch.randn(shape.n_q, shape.H_q, shape.d_k, device=dev, generator=g)
        sets.append((m, KV, q))
    pos = torch.empty(shape.n_q, shape.max_list, dtype=torch.int32, device=dev)
    counts = torch.empty(shape.n_q, dtype=torch.int32, device=dev)
    out = torch.empty(shape.n_q, shape.H_q, shape.d_v, device=dev)
    ws_n = qsa.sparse_attn_workspace_size(shape.n_q, shape.H_q, 1, shape.d_v, shape.max_list)
    ws = torch.empty(max(ws_n // 4, 1), device=dev)
    scale = 1.0 / math.sqrt(shape.d_k)

    def to_list(i):
        qsa.mask_to_list(sets[i % n_sets][0], shape.max_list, pos, counts)

    def attend(i):
        _, KV, q = sets[i % n_sets]
        qsa.sparse_attn(q, KV, KV, counts, shape.max_list, out, 1, shape.d_k, shape.d_v, scale,
                        pos=pos, workspace=ws, ld_k=shape.d_k, ld_v=shape.d_k)

    def fused(i):
        m, KV, q = sets[i % n_sets]
        qsa.mask_sparse_attn(q, KV, m, shape.max_list, out, scale, counts_out=counts)

    # reps calls (rotating sets) captured into one CUDA graph and replayed: device time per
    # call; plain CUDA events around direct calls if capture fails
    reps = 8 * n_sets
    res, timing = {}, "cuda graph replay"
    for name, fns in (("mask_to_list", (to_list,)), ("attn", (attend,)),
                      ("both", (to_list, attend)), ("one_call", (fused,))):
        calls = [functools.partial(fn, i) for i in range(reps) for fn in fns]
        try:
            res[name] = graph_time_us(calls, 1, dev) / reps
        except Exception as e:  # noqa: BLE001 -- reported in the JSON line
            timing = f"cuda events around direct calls (graph capture failed: {type(e).__name__})"
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for c in calls:
                c()
            b.record()
            torch.cuda.synchronize()
            res[name] = a.elapsed_time(b) * 1e3 / reps
    n_listed = float(counts.float().mean().item())
    mask_bytes = shape.n_q * shape.n_kv
    kv_bytes = shape.n_q * n_listed * (shape.d_k + shape.d_v) * 2
    out_d = {
        "workload": (f"mask mode: {shape.n_q} query tokens x {shape.H_q} heads, {shape.n_kv:,} "
                     f"keys, DKQ {shape.d_k} / d_v {shape.d_v} bf16, list of {shape.max_list}, "
                     f"{n_sets} rotating input sets"),
        "mean_listed": n_listed,
        "us": {k: round(v, 2) for k, v in res.items()},
        "timing": timing,
        "mask_to_list_GBps": mask_bytes / (res["mask_to_list"] * 1e-6) / 1e9,
        "attn_GBps": kv_bytes / (res["attn"] * 1e-6) / 1e9,
        "algorithmic_bytes": {"mask": mask_bytes, "kv": kv_bytes},
    }
    del sets, pos, out, ws
    torch.cuda.empty_cache()
    return out_d


def algorithmic_bytes(shape, n_rows, n_cells, pooled_esize=4, n_q=1):
    """Pooled-cache scan (read once for all queries) + each query's selected K/V rows, per
    decode step."""
    esize = 2 if shape.dtype == "bf16" else 4
    return (n_rows * shape.H_idx * shape.d_idx * pooled_esize
            + n_q * n_cells * shape.H_kv * 2 * shape.d * esize)


def summarize(r, world, layers, peak):
    """Per-context figures of one run_context result."""
    sh = r["shape"]
    n_q = r["n_q"]
    pes = 2 if r["pooled"] == "bf16" else 4
    n_rows_avg = (sh.n_ctx + sh.n_ctx + n_q * r["K"] // layers) // 2 // 4
    steps_s = world * r["K"] / (r["ms"] / 1e3)
    bytes_step = algorithmic_bytes(sh, n_rows_avg, r["n_cells"], pes, n_q)
    out = {
        "n_ctx": sh.n_ctx, "steps_per_s": steps_s, "us_per_step": r["ms"] * 1e3 / r["K"],
        "algorithmic_MB_per_step": bytes_step / 1e6,
        "achieved_GBps_step": bytes_step * steps_s / world / 1e9,
        "frac_of_hbm_peak_step": bytes_step * steps_s / world / 1e9 / peak,
        "score_kernel_us": r["score_us"],
        "score_kernel_GBps": r["score_rows"] * sh.H_idx * sh.d_idx * pes / r["score_us"] / 1e3,
        "host_issue_us_per_step": r["host_issue_us"],
    }
    if n_q == 1:
        out["tokens_per_s_12_layers"] = steps_s / 12.0
    else:
        out["query_tokens_per_step"] = n_q
        out["query_tokens_per_s"] = n_q * steps_s
    if r["k_e2e"]:
        out["e2e_steps_per_s"] = world * r["k_e2e"] / r["t_e2e"]
    if r.get("winner_share") is not None:
        out["selected_winner_share"] = r["winner_share"]
    if r["graph_us"] is not None:
        out["graph_us_per_step"] = r["graph_us"]
    elif r["graph_err"] and r["graph_err"] != "not run":
        out["graph_err"] = r["graph_err"]
    return out


# ----------------------------------------------------------------------------- CPU oracle

def oracle_prepare(shape, n_steps: int, seed: int = 7):
    """The oracle's decode inputs and its pooled cache built up to the first step (untimed)."""
    from oracle import oracle
    import qsa_synth

    inp = qsa_synth.decode_inputs(shape, seed=seed, extra_tokens=n_steps + 1, n_steps=4)
    n0 = shape.n_ctx - 1
    cap = (shape.n_ctx + n_steps + 4) // 4
    pooled = np.zeros((cap, shape.H_idx * shape.d_idx), np.float32)
    oracle.pool_rows(inp["raw_k"], n0, shape.H_idx, shape.d_idx, inp["norm_w"], shape.eps,
                     shape.rope_base, 0, (n0 + 3) // 4, pooled)
    return inp, pooled


def oracle_steps(shape, inp, pooled, n_steps: int, budget_s: float, first_q: int = 0,
                 start: int = 0):
    """Consecutive oracle decode steps (incremental pool update of the new rows, score of
    every row, full sort, attention) on ``pooled`` for up to n_steps steps or budget_s
    seconds, continuing after ``start`` steps already taken on it.  Returns (steps,
    seconds)."""
    from oracle import oracle

    valid = (shape.n_ctx - 1 + start) // 4
    done, t = 0, 0.0
    while done < n_steps and t < budget_s:
        n_ctx = shape.n_ctx + start + done
        j = (first_q + done) % 4
        t0 = time.perf_counter()
        oracle.decode_step(inp["raw_k"], n_ctx, shape.H_idx, shape.d_idx, inp["norm_w"], shape.eps,
                           shape.rope_base, pooled, valid, inp["q_idx"][j], shape.top_k_tokens,
                           inp["q"][j], inp["K"], inp["V"], shape.H_q, shape.H_kv, shape.d)
        t += time.perf_counter() - t0
        valid = n_ctx // 4
        done += 1
    return done, t


def oracle_decode_sample(shape, n_steps: int, budget_s: float, seed: int = 7):
    """Single-threaded oracle decode steps after an untimed build of its pooled cache."""
    inp, pooled = oracle_prepare(shape, n_steps, seed)
    return oracle_steps(shape, inp, pooled, n_steps, budget_s)


def _oracle_worker(shape_name, folder, rank, n_steps, budget_s, start, results):
    """One process of the all-cores oracle timing: its own copy of the pooled cache, the
    shared inputs read from files."""
    sys.path.insert(0, ROOT)
    import qsa_synth

    shape = qsa_synth.CONFIGS[shape_name]
    inp = {k: np.load(os.path.join(folder, k + ".npy"), mmap_mode="r")
           for k in ("raw_k", "norm_w", "K", "V", "q_idx", "q")}
    inp = {k: np.ascontiguousarray(v) if k in ("norm_w", "q_idx", "q") else v
           for k, v in inp.items()}
    pooled = np.array(np.load(os.path.join(folder, "pooled.npy"), mmap_mode="r"))
    start.wait(timeout=600)
    done, _ = oracle_steps(shape, inp, pooled, n_steps, budget_s, first_q=rank)
    results.put(done)


def oracle_all_cores_sample(shape_name, n_proc: int, n_steps: int, budget_s: float):
    """The oracle as it stands (single-threaded C) run as n_proc independent processes, one
    per host core, each stepping its own copy of the same layer: aggregate steps/s over the
    wall time from a common start.  Inputs are built once and shared through files."""
    import multiprocessing as mp
    import shutil
    import tempfile

    import qsa_synth

    shape = qsa_synth.CONFIGS[shape_name]
    inp, pooled = oracle_prepare(shape, n_steps)
    base = "/dev/shm" if os.path.isdir("/dev/shm") else None
    folder = tempfile.mkdtemp(prefix="qsa_oracle_", dir=base)
    try:
        for k in ("raw_k", "norm_w", "K", "V", "q_idx", "q"):
            np.save(os.path.join(folder, k + ".npy"), inp[k])
        np.save(os.path.join(folder, "pooled.npy"), pooled)
        del inp, pooled
        ctx = mp.get_context("spawn")
        start = ctx.Barrier(n_proc + 1)
        results = ctx.Queue()
        procs = [ctx.Process(target=_oracle_worker,
                             args=(shape_name, folder, r, n_steps, budget_s, start, results))
                 for r in range(n_proc)]
        for p in procs:
            p.start()
        try:
            start.wait(timeout=600)
            t0 = time.perf_counter()
            total = sum(results.get(timeout=600) for _ in range(n_proc))
            wall = time.perf_counter() - t0
        except Exception:  # a worker that died or stalled: no all-cores figure
            total, wall = None, None
        for p in procs:
            p.join(60)
            if p.is_alive():
                p.kill()
        return total, wall
    finally:
        shutil.rmtree(folder, ignore_errors=True)


def host_description() -> str:
    """Core count and CPU model of this host (the CPU baseline's machine)."""
    model = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.split(":")[0].strip() in ("Model name", "Model"):
                model = ln.split(":", 1)[1].strip()
                if ln.startswith("Model name"):
                    break
    except Exception:
        pass
    import platform

    return f"host {os.cpu_count()} cores, {model or platform.processor() or platform.machine()}"


def config_for(shape, layers, pooled="f32", n_q=1):
    pes = 2 if pooled == "bf16" else 4
    step = "+1 token per step" if n_q == 1 else f"{n_q} query tokens (+{n_q} tokens) per step"
    return {
        "workload": (f"bf16 decode, one QSA layer per step at {shape.n_ctx:,}-token context, "
                     f"{step}, {layers} rotating layer sets"),
        "n_ctx": shape.n_ctx, "indexer": f"{shape.H_idx} heads x {shape.d_idx}",
        "attention": f"{shape.H_q} q heads / {shape.H_kv} kv heads x {shape.d}",
        "top_k_tokens": shape.top_k_tokens, "layers": layers, "queries_per_step": n_q,
        "storage": f"bf16 K/V and raw indexer keys, {pooled} pooled-key cache",
        "l2": (f"inputs larger than L2: {layers} rotating layer sets of "
               f"{shape.n_rows * shape.H_idx * shape.d_idx * pes / 1e6:.0f} MB pooled cache each"),
    }


def main():
    args = parse_args()
    import qsa_synth

    primary = qsa_synth.CONFIGS[CONTEXTS[args.primary]]

    if args.union_only:
        import torch

        torch.cuda.set_device(0)
        import gather_qsa_pool_gb300 as qsa

        qsa.load()
        print(json.dumps({"grouped_union": run_grouped_union(args, 0)}))
        return

    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        if rank != 0:
            return
        # W untimed warm-up steps (at least three; bounded to ~30 s), then up to K timed
        # ones on the same appending context, bounded to ~90 s
        W = max(args.warmup, 3)
        K = max(1, args.steps)
        inp, pooled = oracle_prepare(primary, W + K)
        W, _ = oracle_steps(primary, inp, pooled, W, budget_s=30.0)
        n_done, t = oracle_steps(primary, inp, pooled, K, budget_s=90.0, first_q=W, start=W)
        steps = n_done
        value = n_done / t
        line = {
            "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world,
            "steps": steps, "warmup": W, "ms_per_step": 1e3 * t / n_done,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_for(primary, args.layers), "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "steps/s", "cores": 1, "kind": "oracle",
                             "sample": f"{n_done} consecutive oracle decode steps of one layer "
                                       f"at {primary.n_ctx:,} tokens (bounded to ~90 s), after "
                                       f"an untimed build of its pooled cache and {W} untimed "
                                       f"warm-up steps; single-threaded C; "
                                       f"{host_description()}"},
            "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line))
        return

    world, rank, local = dist_setup()
    import torch

    import gather_qsa_pool_gb300 as qsa

    qsa.load()
    names = [c for c in args.contexts.split(",") if c]
    if args.primary not in names:
        names.append(args.primary)
    results = {}
    for name in names:
        results[name] = run_context(name, args, world, rank, local,
                                    want_clocks=(name == args.primary and rank == 0),
                                    pooled=args.pooled, n_q=args.queries,
                                    light=args.queries > 1)
    peak, peak_kind = load_peaks()

    sweep = {name: summarize(r, world, args.layers, peak) for name, r in results.items()}
    # Next to the headline: the pooled-key cache stored in bf16 (half the scan's bytes),
    # and steps carrying a token with two drafts (three queries, one scan).
    variants = {}
    if not args.no_variants:
        for label, ctx, pooled, n_q, win in (("bf16_pooled_64k", "64k", "bf16", 1, False),
                                             ("bf16_pooled_128k", "128k", "bf16", 1, False),
                                             ("bf16_pooled_256k", "256k", "bf16", 1, False),
                                             ("three_queries_256k", "256k", "f32", 3, False),
                                             ("three_queries_bf16_pooled_256k", "256k", "bf16", 3,
                                              False),
                                             ("clear_winners_256k", "256k", "f32", 1, True)):
            rv = run_context(ctx, args, world, rank, local, want_clocks=False, pooled=pooled,
                             n_q=n_q, light=True, winners=win)
            variants[label] = dict(summarize(rv, world, args.layers, peak),
                                   pooled_cache=pooled, queries_per_step=n_q)
            if win:
                variants[label]["scores"] = ("1% of the completed pooled rows lean toward the "
                                             "queries' common direction (+3 sd)")
        if not args.no_prefill:
            variants["prefill_bf16_pooled"] = run_prefill(args, local, "bf16")
            variants["prefill_f32_pooled_bf16_mirror"] = run_prefill(args, local, "f32_mirror")
    r = results[args.primary]
    sh = r["shape"]
    value = sweep[args.primary]["steps_per_s"]
    pes = 2 if args.pooled == "bf16" else 4
    default_form = args.pooled == "f32" and args.queries == 1

    def row_bytes(rows):
        # per pooled row: the row read once, one fp32 score written per query
        return rows * (sh.H_idx * sh.d_idx * pes + args.queries * 4)

    # the standalone scan (qsa_index_score) and, when it could be timed, the step's own
    # fused score kernel (the step's dominant kernel)
    scan_GBps = row_bytes(r["score_rows"]) / (r["score_us"] * 1e-6) / 1e9
    scan = {"kernel": "score_stream_kernel (qsa_index_score alone)", "us": r["score_us"],
            "rows": r["score_rows"], "achieved": scan_GBps, "frac": scan_GBps / peak,
            "traffic": traffic_per_launch(TRAFFIC_FILE, SCORE_SRCS, r["score_rows"])
            if default_form else None}
    in_step = None
    if r.get("step_score_us"):
        st_GBps = row_bytes(r["step_score_rows"]) / (r["step_score_us"] * 1e-6) / 1e9
        in_step = {"kernel": "score_pool_kernel (inside qsa_decode_step: open-row update, "
                             "scan, top-k histogram)",
                   "us": r["step_score_us"], "rows": r["step_score_rows"], "achieved": st_GBps,
                   "frac": st_GBps / peak,
                   "traffic": traffic_per_launch(STEP_TRAFFIC_FILE, STEP_SCORE_SRCS,
                                                 r["step_score_rows"]) if default_form else None}
    main_k = in_step or scan
    peak_src = (f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                if peak_kind == "measured" else "fallback 6.8 TB/s")
    roofline = {"bound": "hbm", "achieved": main_k["achieved"], "peak": peak, "unit": "GB/s",
                "frac": main_k["frac"], "traffic": main_k["traffic"],
                "kernel": f"{main_k['kernel']}; {args.pooled} cache, {args.queries} "
                          f"quer{'y' if args.queries == 1 else 'ies'}",
                "us_per_launch": main_k["us"], "peak_source": peak_src,
                "scan_alone": scan, "in_step": in_step,
                "in_step_err": r.get("step_score_err")}

    prefill = None if args.no_prefill else run_prefill(args, local)
    mask = None if args.no_mask else run_mask(args, local)
    ablation = None if args.no_ablation else run_ablation(args, local)
    grouped_union = None if args.no_prefill else run_grouped_union(args, local)

    cpu_baseline = None
    cpu_all_cores = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n_done, t = oracle_decode_sample(sh, n_steps=40, budget_s=20.0)
        cpu_baseline = {"value": n_done / t, "unit": "steps/s", "cores": 1, "kind": "oracle",
                        "sample": f"{n_done} consecutive fp64 oracle decode steps of one layer at "
                                  f"{sh.n_ctx:,} tokens (pool update, score of all "
                                  f"{sh.n_rows:,} rows, full sort, attention), after an untimed "
                                  f"build of its pooled cache; single-threaded C; "
                                  f"{host_description()}"}
        n_proc = os.cpu_count() or 1
        total = wall = None
        if n_proc > 1:
            total, wall = oracle_all_cores_sample(CONTEXTS[args.primary], n_proc, 40, 12.0)
        if n_proc > 1 and total:
            cpu_all_cores = {"value": total / wall, "unit": "steps/s", "cores": n_proc,
                             "kind": "oracle",
                             "sample": f"{n_proc} processes (one per host core), each running "
                                       f"up to 40 of the same single-threaded oracle steps "
                                       f"(or 12 s) on its own copy of the layer; {total} steps "
                                       f"in {wall:.1f} s of wall time; {host_description()}"}

    line = {
        "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world,
        "steps": r["K"], "warmup": r["W"], "ms_per_step": r["ms"] / r["K"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded N(0,1) keys/values/queries, 1% of blocks +3 on raw indexer keys)",
        "config": config_for(sh, args.layers, args.pooled, args.queries),
        "roofline": roofline,
        "e2e": ({"value": sweep[args.primary]["e2e_steps_per_s"], "unit": "steps/s",
                 "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]}
                if "e2e_steps_per_s" in sweep[args.primary] else None),
        "gpu_launches": r["K"] * LAUNCHES_PER_DECODE_STEP,
        "clocks": r["clocks"],
        "sweep": sweep,
        "variants": variants or None,
        "prefill": prefill,
        "mask": mask,
        "ablation": ablation,
        "grouped_union": grouped_union,
        "cpu_baseline": cpu_baseline,
        "cpu_baseline_all_cores": cpu_all_cores,
    }
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
