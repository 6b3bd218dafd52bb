#!/usr/bin/env python
"""Benchmark of the block-sparse decode step on GB300.

One step = kt_sparse_decode_step on one layer: score every Context block
against its representatives, select the top-k, and attend over Initial +
selected + Local blocks.  For the benchmarked shapes this is one cooperative
launch of the attention kernel with the selection inside it
(kt_sparse_decode_step_kernels reports the launches per step); the two-kernel
path (selection, then attention) is timed beside it.

Default workload: the InternLM2.5-7B-1M-shaped 128K layer (32 query heads, 8 KV
heads, head_dim 128, 131072 fp16 tokens in 128-token blocks, Initial 128,
Local 4096, Quest reps, SHARED top-32), seeded synthetic data, eight distinct
layers rotated so that the touched working set (8 x 38 MB) is larger than twice
the L2 cache.  Further legs: the Quest rep build and the dense decode over the
same layers; decoding over the eight layers under selection-reuse policies
(kt_decode_layer: dense layers, layer_step, token_step); the 1M-token, 4-layer
workload (SEPARATE top-32 per KV head, Quest and Max reps); the batched paged
workload (16 sequences, every rep method and head mode); the 128K layers with
K/V stored as Q8_0 and with K/V in host memory read over NVLink-C2C; the
Dynamic rep build and step at 128K (with its gap to dense attention); the
preselection and the step restricted to it.  --phase-stamps adds per-phase
timings of single step launches (kt_set_phase_stamps).

value = algorithmic bytes per step (reps of every Context block + K/V of the
attended tokens) / device time per step, in GB/s; us_per_step and
ms_per_step give the time.  Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "sparse decode attention µs/step and achieved HBM GB/s at 128K and 1M context"
BLOCK = 128
D = 128


# ----------------------------------------------------------------------------- sizes

def step_bytes(w: synth.Workload) -> dict:
    """Algorithmic bytes of one decode step: representative rows of every Context
    block (each read once) + K and V of every attended valid token per KV head."""
    p = w.params
    R = p.reps_per_block()
    rep_elem = 4 if p.rep == synth.REP_MEAN else 2
    H_kv = w.num_kv_heads
    reps = kv = 0
    for n in w.seq_lens:
        n = int(n)
        nb = (n + BLOCK - 1) // BLOCK
        c0 = min(p.initial_blocks, nb)
        c1 = max(c0, nb - p.local_blocks)
        C = c1 - c0
        k = min(p.top_k, C)
        reps += C * H_kv * R * D * rep_elem
        tokens = c0 * BLOCK + k * BLOCK + (n - c1 * BLOCK)
        kv += tokens * H_kv * D * 2 * 2
    return {"reps": reps, "kv": kv, "total": reps + kv}


# ----------------------------------------------------------------------------- device side

class Layer:
    """One layer's KV cache, reps and step buffers on the GPU."""

    def __init__(self, w: synth.Workload, extra_reps=(), keep_host=False):
        import torch

        import block_sparse_long_quest_gb300 as kt
        self.w = w

        def dev(a):
            if a.dtype == np.uint16:
                return torch.from_numpy(a.view(np.int16)).view(torch.float16).cuda()
            return torch.from_numpy(a).cuda()

        self.k, self.v = dev(w.k_pool), dev(w.v_pool)
        if not keep_host:  # free the host copy, keep the (heads, block, dim) shape
            w.k_pool = w.v_pool = np.empty((0,) + w.k_pool.shape[1:], dtype=np.uint16)
        self.table, self.lens, self.q = dev(w.block_table), dev(w.seq_lens), dev(w.q)
        self.kv = kt.paged_kv(self.k, self.v, self.table, self.lens)
        self.variants = {}
        for rep in (w.params.rep, *extra_reps):
            p = w.params
            params = kt.sparse_params(p.num_q_heads, p.initial_blocks, p.local_blocks, p.top_k,
                                      rep, p.head_mode, num_reps=p.num_reps,
                                      fix_stride=p.fix_stride, softmax_scale=p.softmax_scale)
            reps = torch.zeros(kt.kt_reps_pool_bytes(self.kv, params), dtype=torch.uint8,
                               device="cuda")
            if rep != synth.REP_DYNAMIC:  # Dynamic reps need the local queries
                kt.kt_build_block_reps(self.kv, params, 0, w.max_blocks, reps)
            SEL = 1 if p.head_mode == synth.HEAD_SHARED else w.num_kv_heads
            self.variants[rep] = dict(
                params=params, reps=reps,
                sel=torch.zeros((w.batch, SEL, p.top_k), dtype=torch.int32, device="cuda"),
                cnt=torch.zeros((w.batch, SEL), dtype=torch.int32, device="cuda"),
                out=torch.zeros((w.batch, p.num_q_heads, D), dtype=torch.float32, device="cuda"),
                ws=kt.workspace(kt.KT_OP_SPARSE_STEP, self.kv, params))

    def step(self, rep):
        import block_sparse_long_quest_gb300 as kt
        v = self.variants[rep]
        kt.kt_sparse_decode_step(self.q, self.kv, v["reps"], v["params"], v["sel"], v["cnt"],
                                 v["out"], v["ws"])

    def select(self, rep):
        import block_sparse_long_quest_gb300 as kt
        v = self.variants[rep]
        kt.kt_score_select_blocks(self.q, self.kv, v["reps"], v["params"], v["sel"], v["cnt"],
                                  None, v["ws"])

    def attend(self, rep):
        import block_sparse_long_quest_gb300 as kt
        v = self.variants[rep]
        kt.kt_sparse_decode_attn(self.q, self.kv, v["params"], v["sel"], v["cnt"], v["out"],
                                 v["ws"])


def graph_time(fn_list, count, warmup, stream, chunk=1000, sampler=None, replays=None):
    """Device seconds for `count` calls cycling through fn_list, captured in CUDA
    graphs (chunks of `chunk` calls + a remainder graph), timed with events.
    With `replays` (a list), the device seconds of each full-chunk replay are
    appended to it as well (events between replays; no work is added)."""
    import torch
    with torch.cuda.stream(stream):
        for i in range(warmup):
            fn_list[i % len(fn_list)]()
    stream.synchronize()
    graphs = []
    c = min(chunk, count)
    reps, rem = divmod(count, c)
    for n in ([c] if reps else []) + ([rem] if rem else []):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                fn_list[i % len(fn_list)]()
        graphs.append((g, n))
    plan = [graphs[0][0]] * reps + ([graphs[-1][0]] if rem else [])
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(len(plan) + 1)] \
        if replays is not None else []
    with torch.cuda.stream(stream):  # replay() launches on the current stream
        for g, _ in graphs:  # one untimed replay of each graph
            g.replay()
        stream.synchronize()
        if sampler:
            sampler.mark_start()
        start.record(stream)
        for i, g in enumerate(plan):
            if marks:
                marks[i].record(stream)
            g.replay()
        if marks:
            marks[-1].record(stream)
        end.record(stream)
    end.synchronize()
    if sampler:
        sampler.mark_end()
    if marks:
        for i in range(reps):  # the full chunks (the remainder graph is shorter)
            replays.append(marks[i].elapsed_time(marks[i + 1]) / 1e3)
    return start.elapsed_time(end) / 1e3


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 20):
        self.index, self.period_ms = index, period_ms
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def mark_start(self):
        self.t_start = time.perf_counter()

    def mark_end(self):
        self.t_end = time.perf_counter()

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        t0 = getattr(self, "t_start", 0.0)
        t1 = getattr(self, "t_end", float("inf"))
        rows = []
        for ts, l in self.lines:
            parts = [x.strip() for x in l.split(",")]
            if len(parts) == 7 and t0 <= ts <= t1 + 0.05:
                rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[3 + i] == "Active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from
# one ncu capture of the 128K workload, per kernel, valid only for the kernel
# code it was taken from (sha256 over KERNEL_SOURCES without comments); null
# otherwise.
KERNEL_SOURCES = ("attn.cu", "select_common.cuh", "kt_internal.cuh")
KERNEL_TRAFFIC = {
    "attn_kernel<fused step>": {
        "bytes": 38268416 + 202496,
        "sources_sha256": "9e5f3fe5ea560d61adca72955d9f4a08518731b640cfdb388d3c981fb46db3dc"},
}


def _code_only(text: str) -> str:
    """The source without comments and blank lines: the record follows the code."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_sources_sha():
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        path = os.path.join(ROOT, "block_sparse_long_quest_gb300", "csrc", name)
        try:
            h.update(_code_only(open(path, encoding="utf-8").read()).encode())
        except OSError:
            return None
    return h.hexdigest()


def kernel_traffic(kernel):
    rec = KERNEL_TRAFFIC.get(kernel)
    if rec is None:
        return None
    return rec["bytes"] if kernel_sources_sha() == rec["sources_sha256"] else None


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def workload_config(w, seq_len: int) -> dict:
    """The `config` both arms print for the 128K workload (identical dicts)."""
    return {"workload": w.name, "batch": w.batch, "seq_len": seq_len, "q_heads": 32,
            "kv_heads": 8, "head_dim": 128, "block_size": 128, "initial_tokens": 128,
            "local_tokens": 4096, "top_k": 32, "rep": "quest", "head_mode": "shared",
            "bytes_per_step": step_bytes(w)}


# ----------------------------------------------------------------------------- CPU baseline

def cpu_baseline(w: synth.Workload, budget_s: float = 12.0) -> dict:
    """The oracle (single-threaded C) on the same work as one GPU step: score,
    select and attend for one 128K layer, reps built beforehand (untimed)."""
    import oracle
    kv = oracle.KV.of(w)
    st = oracle.StepTimer(kv, w.params, w.q_local)
    st.step(w.q)  # warm
    n, t0 = 0, time.perf_counter()
    while True:
        st.step(w.q)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or n >= 200:
            break
    per = el / n
    return {"value": step_bytes(w)["total"] / per / 1e9, "unit": "GB/s", "cores": 1,
            "kind": "oracle", "us_per_step": per * 1e6,
            "sample": f"oracle score+select+attend, {w.name}, 1 layer, reps prebuilt "
                      f"(untimed), {n} steps in {el:.1f} s"}


def host_info():
    try:
        model = [l.split(":", 1)[1].strip() for l in open("/proc/cpuinfo")
                 if l.lower().startswith(("model name", "cpu part"))][:1]
    except OSError:
        model = []
    return {"nproc": os.cpu_count(), "cpu": model[0] if model else None}


# ----------------------------------------------------------------------------- main

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    """Max of a float over all ranks (identity for one rank)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def run_reference(args, world, rank):
    """The oracle on the host cores, same workload/metric; rank 0 only."""
    if rank != 0:
        return
    import oracle
    w = synth.long128k(seq_len=args.seq_len)
    kv = oracle.KV.of(w)
    st = oracle.StepTimer(kv, w.params)
    for _ in range(max(0, args.warmup)):
        st.step(w.q)
        break  # one warm step: each step takes a fraction of a second
    t_one = time.perf_counter()
    st.step(w.q)
    t_one = time.perf_counter() - t_one
    cap = max(1, int(90.0 / max(t_one, 1e-6)))
    steps = min(args.steps, cap)
    t0 = time.perf_counter()
    for _ in range(steps):
        st.step(w.q)
    el = time.perf_counter() - t0
    per = el / steps
    value = step_bytes(w)["total"] / per / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": world, "steps": steps, "steps_requested": args.steps, "warmup": args.warmup,
        "ms_per_step": per * 1e3, "us_per_step": per * 1e6, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, args.seq_len),
        "parallelism": "single-thread CPU",
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"oracle score+select+attend on one {w.name} layer, reps "
                                   f"prebuilt, {steps} steps (capped to ~90 s)"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "host": host_info(),
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=8, help="rotated 128K layers")
    ap.add_argument("--seq-len", type=int, default=131072)
    ap.add_argument("--no-1m", action="store_true")
    ap.add_argument("--seq-len-1m", type=int, default=1048576,
                    help="tokens per layer of the SEPARATE leg (smaller for profiling)")
    ap.add_argument("--layers-1m", type=int, default=4)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-dynamic", action="store_true")
    ap.add_argument("--no-kv-sources", action="store_true",
                    help="skip the Q8_0 and host-memory KV legs")
    ap.add_argument("--no-batched", action="store_true", help="skip the batched paged leg")
    ap.add_argument("--phase-stamps", action="store_true",
                    help="add per-phase timings of single step launches (phase_us)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    import torch

    import block_sparse_long_quest_gb300 as kt  # fails loudly without libkt.so
    torch.cuda.set_device(local)
    stream = torch.cuda.Stream()

    # ---- 128K workload: `layers` independent layers, rotated every step
    layers = []
    for l in range(args.layers):
        w = synth.long128k(layer=l, seq_len=args.seq_len)
        layers.append(Layer(w, keep_host=(l == 0)))
    w0 = layers[0].w
    rep = w0.params.rep
    l2_bytes = torch.cuda.get_device_properties(local).L2_cache_size
    bytes_step = step_bytes(w0)
    torch.cuda.synchronize()

    # correctness guard: every layer's device status word is clean after a step
    for L in layers:
        L.step(rep)
    for L in layers:
        st = kt.kt_read_device_status(L.variants[rep]["ws"])
        if st != kt.KT_OK:
            raise RuntimeError(f"device status {kt.status_string(st)}")

    # ---- timed region: exactly `steps` decode steps
    steps_fns = [lambda L=L: L.step(rep) for L in layers]
    n_layers = len(layers)
    barrier(world)
    torch.cuda.synchronize()
    replay_s, replay_steps = [], min(args.steps, 1000)
    with ClockSampler(local) as clocks:
        t_step = graph_time(steps_fns, args.steps, args.warmup, stream, sampler=clocks,
                            replays=replay_s)
    torch.cuda.synchronize()
    barrier(world)
    t_step = max_over_ranks(t_step, world)
    per_step = t_step / args.steps
    if per_step < 5e-7:
        raise RuntimeError("timed region recorded no work")
    value = world * bytes_step["total"] * args.steps / t_step / 1e9

    # ---- per-kernel device time.  With one launch per step the step kernel is
    # the dominant (only) kernel: its algorithmic bytes are the reps it scores
    # plus the KV it attends, its duration the event-timed step above.  The
    # two-kernel path (selection, then attention) is timed beside it.
    v0 = layers[0].variants[rep]
    launches = kt.kt_sparse_decode_step_kernels(layers[0].kv, v0["params"])
    n_k = min(args.steps, 20000)
    t_attn = graph_time([lambda L=L: L.attend(rep) for L in layers], n_k, args.warmup, stream)
    t_sel = graph_time([lambda L=L: L.select(rep) for L in layers], n_k, args.warmup, stream)
    attn_us, sel_us = t_attn / n_k * 1e6, t_sel / n_k * 1e6
    peak, peak_kind = measured_peak()
    if launches == 1:
        roof_kernel, roof_bytes, roof_us = "attn_kernel<fused step>", bytes_step["total"], per_step * 1e6
    else:
        roof_kernel, roof_bytes, roof_us = "attn_kernel", bytes_step["kv"], attn_us
    roof_gbs = roof_bytes / (roof_us * 1e-6) / 1e9

    # ---- end to end through the host-buffer entry point, query and output in
    # page-locked host memory that the step kernel reads and writes over the
    # link (every step moves the query in and the output out)
    q_host = torch.empty_like(layers[0].q, device="cpu").pin_memory()
    out_host = torch.empty_like(v0["out"], device="cpu").pin_memory()
    q_host.copy_(layers[0].q.cpu())
    q_dev = [torch.empty_like(L.q) for L in layers]
    n_e2e = min(args.steps, 3000)
    for i in range(args.warmup):
        L = layers[i % len(layers)]
        v = L.variants[rep]
        kt.kt_sparse_decode_step_host(q_host, None, L.kv, v["reps"], v["params"], v["sel"],
                                      v["cnt"], None, out_host, v["ws"], stream)
    barrier(world)
    t0 = time.perf_counter()
    for i in range(n_e2e):
        L = layers[i % len(layers)]
        v = L.variants[rep]
        kt.kt_sparse_decode_step_host(q_host, None, L.kv, v["reps"], v["params"], v["sel"],
                                      v["cnt"], None, out_host, v["ws"], stream)
    t_e2e = max_over_ranks(time.perf_counter() - t0, world)
    e2e_value = world * bytes_step["total"] * n_e2e / t_e2e / 1e9
    e2e_parts = e2e_breakdown(layers, rep, q_host, out_host, q_dev, stream, per_step)

    extra = {}
    if args.phase_stamps:
        extra["phase_us"] = {"128k": phase_stamps_leg(steps_fns)}

    # ---- representative build (amortised, outside the step): Quest reps of one
    # 128K layer; algorithmic bytes = K read once + reps written
    L0 = layers[0]
    v0q = L0.variants[rep]
    n_rb = 20
    t_rb = graph_time([lambda: kt.kt_build_block_reps(L0.kv, v0q["params"], 0, w0.max_blocks,
                                                      v0q["reps"])], n_rb, args.warmup, stream)
    rb_bytes = int(L0.k.numel() * 2 + v0q["reps"].numel())
    extra["rep_build_128k_quest"] = {"us": t_rb / n_rb * 1e6,
                                     "gbs": rb_bytes / (t_rb / n_rb) / 1e9,
                                     "bytes": rb_bytes}
    # ---- dense decode over all 131072 tokens (the full scan the method avoids):
    # the attention kernel alone on K/V of every token, layers rotated
    n_d = 200
    dense_fns = []
    for L in layers:
        vL = L.variants[rep]
        ws_d = kt.workspace(kt.KT_OP_DENSE_ATTN, L.kv, vL["params"])
        dense_fns.append(lambda L=L, vL=vL, ws_d=ws_d: kt.kt_dense_decode_attn(
            L.q, L.kv, w0.params.num_q_heads, w0.params.softmax_scale, vL["out"], ws_d))
    torch.cuda.nvtx.range_push("dense_128k")  # lets a profiler select this leg's launches
    t_d = graph_time(dense_fns, n_d, args.warmup, stream)
    torch.cuda.nvtx.range_pop()
    d_bytes = int(w0.seq_lens.sum()) * w0.num_kv_heads * D * 2 * 2
    extra["dense_128k"] = {"us": t_d / n_d * 1e6, "gbs": d_bytes / (t_d / n_d) / 1e9,
                           "frac_of_hbm_peak": d_bytes / (t_d / n_d) / 1e9 / peak,
                           "bytes": d_bytes, "l2_note": f"{n_layers} layers rotated"}

    # ---- decoding over the rotated layers with selection reuse
    extra["decode_reuse_128k"] = decode_reuse_leg(stream, layers, rep)
    # ---- the other KV sources over the same rotated layers: Q8_0 pools in HBM,
    # and fp16 pools in host memory read over NVLink-C2C
    if not args.no_kv_sources:
        extra["q8_0_128k"] = q8_leg(args, stream, layers, rep)
        extra["host_kv_128k"] = hostkv_leg(args, stream, layers, rep)

    # ---- 1M-token leg: 4 layers back to back, Quest and Max reps
    if world == 1 and not args.no_1m:
        del layers, steps_fns, q_dev
        torch.cuda.empty_cache()
        big = []
        for l in range(args.layers_1m):
            wb = synth.long1m(layer=l, rep=synth.REP_QUEST, seq_len=args.seq_len_1m)
            big.append(Layer(wb, extra_reps=(synth.REP_MAX,)))
        res = {}
        for r, name in ((synth.REP_QUEST, "quest"), (synth.REP_MAX, "max")):
            for L in big:
                L.step(r)
            for L in big:
                if kt.kt_read_device_status(L.variants[r]["ws"]) != kt.KT_OK:
                    raise RuntimeError("device status after 1M step")
            n1 = 2000
            t1 = graph_time([lambda L=L, r=r: L.step(r) for L in big], n1, args.warmup, stream)
            wq = big[0].w
            wq.params.rep = r
            b1 = step_bytes(wq)
            per_layer = t1 / n1
            res[name] = {"us_per_layer_step": per_layer * 1e6,
                         f"us_per_{args.layers_1m}layer_step": args.layers_1m * per_layer * 1e6,
                         "gbs": b1["total"] / per_layer / 1e9,
                         "bytes_per_layer_step": b1["total"]}
            wq.params.rep = synth.REP_QUEST
            if args.phase_stamps:
                extra.setdefault("phase_us", {})[f"1m_{name}"] = phase_stamps_leg(
                    [lambda L=L, r=r: L.step(r) for L in big])
        extra["at_1m"] = {"workload": f"1m-gqa4-separate-k32 ({args.layers_1m} layers, "
                                      f"{args.seq_len_1m} tokens each)",
                          **res}
        del big
        torch.cuda.empty_cache()
    if world == 1 and not args.no_batched:
        extra["batched_paged"] = batched_leg(args, stream)
    if world == 1 and not args.no_dynamic:
        extra["at_dynamic_128k"] = dynamic_leg(args, stream)
        extra["preselect_128k"] = preselect_leg(args, stream)

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3,
        "us_per_step": per_step * 1e6, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": workload_config(w0, args.seq_len),
        "l2": f"{n_layers} layers rotated, touched set {n_layers * bytes_step['total'] / 1e6:.0f} MB "
              f"vs L2 {l2_bytes / 1e6:.0f} MB (inputs larger than L2 between steps)",
        "parallelism": f"replicas x{world}",
        "replays": {"steps_per_replay": replay_steps, "count": len(replay_s),
                    "median_us_per_step": float(np.median(replay_s)) / replay_steps * 1e6
                    if replay_s else None,
                    "min_us_per_step": float(np.min(replay_s)) / replay_steps * 1e6
                    if replay_s else None},
        "roofline": {"bound": "hbm", "kernel": roof_kernel, "achieved": roof_gbs,
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": roof_gbs / peak, "traffic": kernel_traffic(roof_kernel),
                     "algorithmic_bytes_per_launch": roof_bytes,
                     "us_per_launch": roof_us},
        "kernels_us": {roof_kernel: roof_us,
                       "two_kernel_path": {"select_kernel": sel_us, "attn_kernel": attn_us}},
        "launches_per_step": launches,
        "e2e": {"value": e2e_value, "unit": "GB/s", "us_per_step": t_e2e / n_e2e * 1e6,
                "steps": n_e2e, "h2d_bytes_per_step": int(layers_q_bytes(w0)),
                "d2h_bytes_per_step": int(w0.batch * w0.params.num_q_heads * D * 4),
                "transfer": "kt_sparse_decode_step_host with q and out in page-locked host "
                            "memory, read and written by the step kernel over NVLink-C2C; "
                            "the call returns after a stream sync",
                "breakdown": e2e_parts},
        "gpu_launches": launches * args.steps,
        "clocks": clocks.summary(),
        **extra,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w0)
        line["host"] = host_info()
    if rank == 0:
        print(json.dumps(line), flush=True)
    barrier(world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def dynamic_leg(args, stream, nl=8):
    """Dynamic reps at 128K: the rep build (two passes over K, tensor-core
    contraction of the 64 local queries x 4 heads against every key, timed on
    one layer) and the decode step that scores blocks by max q.rep over 4 reps,
    over `nl` rotated layers.  The gap to dense attention over the same KV is
    reported (max and median row relative error, and the share of each query
    head's dense attention mass that the attended blocks hold)."""
    import torch

    import block_sparse_long_quest_gb300 as kt
    layers = []
    for l in range(nl):
        w = synth.dynamic128k(layer=l)
        L = Layer(w, keep_host=(l == 0))  # no reps yet: Dynamic reps need the local queries
        v = L.variants[synth.REP_DYNAMIC]
        L.q_local = torch.from_numpy(w.q_local.view(np.int16)).view(torch.float16).cuda()
        L.ws_dyn = kt.workspace(kt.KT_OP_DYNAMIC_REPS, L.kv, v["params"], w.q_local.shape[1])
        kt.kt_build_dynamic_reps(L.kv, v["params"], L.q_local, w.q_local.shape[1], 0,
                                 w.max_blocks, v["reps"], None, L.ws_dyn)
        layers.append(L)
    L0 = layers[0]
    w0 = L0.w
    v0 = L0.variants[synth.REP_DYNAMIC]
    T = w0.q_local.shape[1]
    build = lambda: kt.kt_build_dynamic_reps(L0.kv, v0["params"], L0.q_local, T, 0, w0.max_blocks,
                                             v0["reps"], None, L0.ws_dyn)
    n_b = 10
    t_b = graph_time([build], n_b, 3, stream)
    rows = T * w0.params.num_q_heads
    flops = 2 * 2 * rows * int(w0.seq_lens[0]) * D  # two passes of Q K^T
    n_s = 2000
    t_s = graph_time([lambda L=L: L.step(synth.REP_DYNAMIC) for L in layers], n_s, args.warmup,
                     stream)
    b = step_bytes(w0)
    # sparse vs dense on layer 0
    L0.step(synth.REP_DYNAMIC)
    sparse = v0["out"].cpu().numpy().astype(np.float64)
    sel, cnt = v0["sel"].cpu().numpy(), v0["cnt"].cpu().numpy()
    ws_d = kt.workspace(kt.KT_OP_DENSE_ATTN, L0.kv, v0["params"])
    dense_t = torch.zeros_like(v0["out"])
    kt.kt_dense_decode_attn(L0.q, L0.kv, 32, w0.params.softmax_scale, dense_t, ws_d)
    dense = dense_t.cpu().numpy().astype(np.float64)
    gap = np.abs(sparse - dense).max(-1) / np.abs(dense).max(-1)
    mass = attention_mass(w0, sel, cnt)
    return {"workload": f"{w0.name}, {nl} layers rotated for the step",
            "rep_build_us": t_b / n_b * 1e6, "rep_build_tflops": flops / (t_b / n_b) / 1e12,
            "rep_build_k_bytes_read": 2 * int(L0.k.numel()) * 2,
            "step_us": t_s / n_s * 1e6, "step_gbs": b["total"] / (t_s / n_s) / 1e9,
            "step_bytes": b["total"],
            "l2_note": f"{nl} layers rotated, touched set {nl * b['total'] / 1e6:.0f} MB",
            "dynamic_vs_dense": {
                "max_row_rel_err": float(gap.max()), "median_row_rel_err": float(np.median(gap)),
                "attention_mass_of_attended_tokens": {"min": float(mass.min()),
                                                      "median": float(np.median(mass))},
                "note": "synthetic N(0,1) keys and queries: dense attention is spread over "
                        "all 131072 tokens, so the 8320 attended tokens (Initial 128 + 32 "
                        "blocks + Local 4096) hold about their share of it, 1/16"}}


def attention_mass(w, sel, cnt):
    """Per query head, the share of dense softmax(q K^T / sqrt(d)) mass on the
    tokens a step attends (Initial + selected + Local), from the host K."""
    n = int(w.seq_lens[0])
    p = w.params
    nb = (n + 127) // 128
    c0 = min(p.initial_blocks, nb)
    c1 = max(c0, nb - p.local_blocks)
    G = p.num_q_heads // w.num_kv_heads
    out = np.zeros(p.num_q_heads)
    for h in range(w.num_kv_heads):
        K = w.k_pool[w.block_table[0, :nb], h].reshape(-1, D)[:n].view(np.float16)
        K = K.astype(np.float32)
        keep = np.zeros(nb, dtype=bool)
        keep[:c0] = True
        keep[c1:] = True
        for g in range(G):
            hq = h * G + g
            u = 0 if p.head_mode == synth.HEAD_SHARED else h
            kk = keep.copy()
            kk[sel[0, u, :int(cnt[0, u])]] = True
            q = w.q[0, hq].view(np.float16).astype(np.float32)
            lg = (K @ q).astype(np.float64) * p.softmax_scale
            pr = np.exp(lg - lg.max())
            pr /= pr.sum()
            out[hq] = pr[np.repeat(kk, 128)[:n]].sum()
    return out


def decode_reuse_leg(stream, layers, rep):
    """Decoding over the rotated 128K layers under selection-reuse policies
    (dense layers, layer_step, token_step of the pages' parameter list): one
    kt_decode_layer call per (token, layer) over one token_step window,
    captured in graphs; the KV cache is not appended to, so every window
    repeats the same work."""
    import torch

    import block_sparse_long_quest_gb300 as kt
    nl = len(layers)
    p = layers[0].w.params
    res = {}
    for name, (dense, lstep, tstep) in (("select_every_layer_and_token", (0, 1, 1)),
                                        ("layer_step2_token_step4", (0, 2, 4)),
                                        ("dense2_layer_step1_token_step100", (2, 1, 100))):
        if dense >= nl:  # needs more layers than are rotated
            continue
        pol = kt.reuse_policy(nl, dense, lstep, tstep)
        slots = max(1, kt.kt_decode_history_slots(pol))
        SEL = layers[0].variants[rep]["sel"].shape[1]
        hs = torch.zeros((slots, 1, SEL, p.top_k), dtype=torch.int32, device="cuda")
        hc = torch.zeros((slots, 1, SEL), dtype=torch.int32, device="cuda")
        fns, actions = [], []
        for t in range(tstep):
            for l, Ly in enumerate(layers):
                v = Ly.variants[rep]
                actions.append(kt.kt_decode_layer_action(pol, t, l)[0])
                fns.append(lambda t=t, l=l, Ly=Ly, v=v, pol=pol, hs=hs, hc=hc: kt.kt_decode_layer(
                    pol, t, l, Ly.q, Ly.kv, v["reps"], v["params"], hs, hc, v["out"], v["ws"]))
        per = len(fns)
        count = per * max(1, 800 // per)
        sec = graph_time(fns, count, per, stream, chunk=per * max(1, 1000 // per))
        tokens = count // nl
        res[name] = {"dense_layer_num": dense, "layer_step": lstep, "token_step": tstep,
                     "us_per_token_all_layers": sec / tokens * 1e6,
                     "selections_per_token": actions.count(kt.KT_LAYER_SELECT) / tstep,
                     "dense_layers_per_token": actions.count(kt.KT_LAYER_DENSE) / tstep}
    return {"workload": f"128k-gqa4-quest-shared-k32, {nl} layers", **res}


def preselect_leg(args, stream, nl=8):
    """Preselection at 128K (the 96 blocks of the pages' YAML, pool window 5,
    64 local queries): its one-off cost (it reads K twice: 2 x 268 MB, past
    the L2), and the Quest SHARED top-32 step restricted to it over `nl`
    rotated layers.  The restricted step scores every Context block (only the
    preselected ones compete), so its bytes count every Context block's reps."""
    import torch

    import block_sparse_long_quest_gb300 as kt
    layers = []
    for l in range(nl):
        w = synth.dynamic128k(layer=l)
        w.params.rep = synth.REP_QUEST
        L = Layer(w)
        v = L.variants[synth.REP_QUEST]
        q_local = torch.from_numpy(w.q_local.view(np.int16)).view(torch.float16).cuda()
        T = w.q_local.shape[1]
        SEL = 1 if w.params.head_mode == synth.HEAD_SHARED else w.num_kv_heads
        mw = kt.kt_preselect_mask_words(L.kv)
        L.mask = torch.zeros((w.batch, SEL, mw), dtype=torch.int32, device="cuda")
        L.pcnt = torch.zeros((w.batch, SEL), dtype=torch.int32, device="cuda")
        L.ws_p = kt.workspace(kt.KT_OP_PRESELECT, L.kv, v["params"], T)
        L.run_p = lambda L=L, v=v, q_local=q_local, T=T: kt.kt_preselect_blocks(
            L.kv, v["params"], q_local, T, 5, 96, L.mask, L.pcnt, L.ws_p)
        L.run_p()
        if kt.kt_read_device_status(L.ws_p) != kt.KT_OK:
            raise RuntimeError("device status after preselection")
        layers.append(L)
    n_p = 10
    t_p = graph_time([layers[0].run_p], n_p, 3, stream)

    def step(L):
        v = L.variants[synth.REP_QUEST]
        kt.kt_sparse_decode_step_presel(L.q, L.kv, v["reps"], v["params"], L.mask, L.pcnt,
                                        v["sel"], v["cnt"], v["out"], v["ws"])

    n_s = 2000
    t_s = graph_time([lambda L=L: step(L) for L in layers], n_s, args.warmup, stream)
    b = step_bytes(layers[0].w)
    return {"workload": "128k-gqa4-quest-shared-k32, preselect 96 blocks (pool 5, 64 local "
                        f"queries), {nl} layers rotated",
            "preselect_us": t_p / n_p * 1e6, "step_us": t_s / n_s * 1e6,
            "step_gbs": b["total"] / (t_s / n_s) / 1e9, "step_bytes": b["total"],
            "note": "the restricted step reads the reps of every Context block and attends "
                    "the top-32 of the 96 preselected"}


def e2e_breakdown(layers, rep, q_host, out_host, q_dev, stream, device_s, n=500):
    """Host wall time per step of the parts around the host-buffer call, each
    timed alone: the same call with device staging buffers (query upload,
    step, output download, sync; the layers rotated as in the timed loop), the
    query upload alone (pinned -> device, then a stream sync), the output
    download alone, one step on device buffers launched and synchronised, and
    the host time to launch a step (enqueue only); device_us is the
    event-timed step."""
    import torch

    import block_sparse_long_quest_gb300 as kt
    L = layers[0]
    v = L.variants[rep]

    def per_call(fn):
        fn()
        stream.synchronize()
        t0 = time.perf_counter()
        for _ in range(n):
            fn()
        return (time.perf_counter() - t0) / n * 1e6

    ring = {"i": 0}

    def staged_call():
        # the host-buffer call with device staging buffers, rotating the
        # layers like the timed e2e loop
        Li = layers[ring["i"] % len(layers)]
        vi = Li.variants[rep]
        kt.kt_sparse_decode_step_host(q_host, q_dev[ring["i"] % len(layers)], Li.kv, vi["reps"],
                                      vi["params"], vi["sel"], vi["cnt"], vi["out"], out_host,
                                      vi["ws"], stream)
        ring["i"] += 1

    with torch.cuda.stream(stream):
        staged = per_call(staged_call)
        h2d = per_call(lambda: (q_dev[0].copy_(q_host, non_blocking=True), stream.synchronize()))
        d2h = per_call(lambda: (out_host.copy_(v["out"], non_blocking=True), stream.synchronize()))
        step = per_call(lambda: (kt.kt_sparse_decode_step(L.q, L.kv, v["reps"], v["params"],
                                                          v["sel"], v["cnt"], v["out"], v["ws"],
                                                          stream), stream.synchronize()))
        stream.synchronize()
        t0 = time.perf_counter()
        for _ in range(200):
            kt.kt_sparse_decode_step(L.q, L.kv, v["reps"], v["params"], v["sel"], v["cnt"],
                                     v["out"], v["ws"], stream)
        launch = (time.perf_counter() - t0) / 200 * 1e6
        stream.synchronize()
    return {"staged_call_us": staged, "h2d_and_sync_us": h2d, "d2h_and_sync_us": d2h,
            "step_and_sync_us": step, "launch_host_us": launch, "device_us": device_s * 1e6}


def batched_leg(args, stream):
    """The batched paged workload: 16 sequences of 8K-64K tokens whose pages are
    permuted in one pool, GQA 32/8, Local 2048, top-16; one step per rep method
    (Max, Mean, Quest, Fix stride 32) and head mode (SHARED, SEPARATE) on the
    same KV.  The touched set of one step (~300 MB) exceeds twice the L2."""
    import torch

    import block_sparse_long_quest_gb300 as kt
    w = synth.batched(rep=synth.REP_QUEST, head_mode=synth.HEAD_SHARED)
    L = Layer(w, extra_reps=(synth.REP_MAX, synth.REP_MEAN, synth.REP_FIX))
    p = w.params
    res = {}
    for mode, mname in ((synth.HEAD_SHARED, "shared"), (synth.HEAD_SEPARATE, "separate")):
        SEL = 1 if mode == synth.HEAD_SHARED else w.num_kv_heads
        for r, rname in ((synth.REP_MAX, "max"), (synth.REP_MEAN, "mean"),
                         (synth.REP_QUEST, "quest"), (synth.REP_FIX, "fix32")):
            params = kt.sparse_params(p.num_q_heads, p.initial_blocks, p.local_blocks, p.top_k, r,
                                      mode, num_reps=p.num_reps, fix_stride=p.fix_stride,
                                      softmax_scale=p.softmax_scale)
            reps = L.variants[r]["reps"]
            sel = torch.zeros((w.batch, SEL, p.top_k), dtype=torch.int32, device="cuda")
            cnt = torch.zeros((w.batch, SEL), dtype=torch.int32, device="cuda")
            out = torch.zeros((w.batch, p.num_q_heads, D), dtype=torch.float32, device="cuda")
            ws = kt.workspace(kt.KT_OP_SPARSE_STEP, L.kv, params)
            fn = lambda params=params, reps=reps, sel=sel, cnt=cnt, out=out, ws=ws: \
                kt.kt_sparse_decode_step(L.q, L.kv, reps, params, sel, cnt, out, ws)
            fn()
            if kt.kt_read_device_status(ws) != kt.KT_OK:
                raise RuntimeError("device status after a batched step")
            n = 1000
            t = graph_time([fn], n, args.warmup, stream) / n
            w.params.rep, w.params.head_mode = r, mode
            b = step_bytes(w)
            res[f"{rname}_{mname}"] = {"us_per_step": t * 1e6, "gbs": b["total"] / t / 1e9,
                                       "bytes_per_step": b["total"],
                                       "launches": kt.kt_sparse_decode_step_kernels(L.kv, params)}
    w.params.rep, w.params.head_mode = synth.REP_QUEST, synth.HEAD_SHARED
    peak, _ = measured_peak()
    best = max(v["gbs"] for v in res.values())
    return {"workload": "batched16-paged-k16 (16 sequences, 8K-64K tokens, pages permuted)",
            "sequence_lengths": [int(x) for x in w.seq_lens], **res,
            "best_frac_of_hbm_peak": best / peak,
            "l2_note": "one step touches ~300 MB, more than twice the L2"}


def q8_leg(args, stream, layers, rep):
    """Q8_0 K/V for the rotated 128K layers: each layer's fp16 pools quantised
    once (timed on one layer), then per step the one-launch step over the
    codes (selection from the fp16 reps), beside the attention alone and the
    two-kernel path; bytes per attended (block, KV head) are 2 x (16 KiB codes
    + 1 KiB scales) instead of 64 KiB."""
    import torch

    import block_sparse_long_quest_gb300 as kt
    pools = []
    for L in layers:
        P, H, bs, d = L.k.shape
        kc = torch.empty((P, H, bs, d), dtype=torch.int8, device="cuda")
        vc = torch.empty_like(kc)
        ks = torch.empty((P, H, bs, d // 32), dtype=torch.float16, device="cuda")
        vs = torch.empty_like(ks)
        kt.kt_quantize_kv_q8_0(L.kv, kc, ks, vc, vs)
        pools.append(dict(kc=kc, vc=vc, ks=ks, vs=vs,
                          kvq=kt.paged_kv_q8(kc, ks, vc, vs, L.table, L.lens)))
    L0, p0 = layers[0], pools[0]
    n_q = 10
    t_q = graph_time([lambda: kt.kt_quantize_kv_q8_0(L0.kv, p0["kc"], p0["ks"], p0["vc"],
                                                     p0["vs"])], n_q, 3, stream) / n_q
    q_bytes = 2 * L0.k.numel() * 2 + 2 * (p0["kc"].numel() + p0["ks"].numel() * 2)

    def attend(L, pq):
        v = L.variants[rep]
        kt.kt_sparse_decode_attn_q8_0(L.q, pq["kvq"], v["params"], v["sel"], v["cnt"], v["out"],
                                      v["ws"])

    for L in layers:  # a selection for every layer first
        L.select(rep)
    n = 2000
    t_att = graph_time([lambda L=L, pq=pq: attend(L, pq) for L, pq in zip(layers, pools)], n,
                       args.warmup, stream) / n
    t_step = graph_time([lambda L=L, pq=pq: (L.select(rep), attend(L, pq))
                         for L, pq in zip(layers, pools)], n, args.warmup, stream) / n

    def step(L, pq):
        v = L.variants[rep]
        kt.kt_sparse_decode_step_q8_0(L.q, pq["kvq"], v["reps"], v["params"], v["sel"],
                                      v["cnt"], v["out"], v["ws"])

    t_one = graph_time([lambda L=L, pq=pq: step(L, pq) for L, pq in zip(layers, pools)], n,
                       args.warmup, stream) / n
    w = layers[0].w
    b = step_bytes(w)
    kv_q8 = b["kv"] * (2 * (16384 + 1024)) // (2 * 32768)
    peak, _ = measured_peak()
    return {"workload": f"{w.name}, {len(layers)} layers rotated, K/V stored as Q8_0",
            "quantise_us_per_layer": t_q * 1e6, "quantise_gbs": q_bytes / t_q / 1e9,
            "attention_us": t_att * 1e6, "attention_kv_bytes": int(kv_q8),
            "attention_gbs": kv_q8 / t_att / 1e9,
            "attention_frac_of_hbm_peak": kv_q8 / t_att / 1e9 / peak,
            "fp16_attention_kv_bytes": int(b["kv"]),
            "step_us (one launch)": t_one * 1e6,
            "step_us (select + attention)": t_step * 1e6,
            "step_bytes": int(b["reps"] + kv_q8),
            "step_gbs": (b["reps"] + kv_q8) / t_one / 1e9,
            "step_frac_of_hbm_peak": (b["reps"] + kv_q8) / t_one / 1e9 / peak}


def hostkv_leg(args, stream, layers, rep):
    """The rotated 128K layers with their K/V pools copied into page-locked host
    memory: per step the selection (reps stay on the GPU) and the attention,
    which reads the attended (block, KV head) pairs over NVLink-C2C."""
    import torch

    import block_sparse_long_quest_gb300 as kt
    host = []
    for L in layers:
        hk = torch.empty(L.k.shape, dtype=L.k.dtype, device="cpu", pin_memory=True)
        hv = torch.empty(L.v.shape, dtype=L.v.dtype, device="cpu", pin_memory=True)
        hk.copy_(L.k)
        hv.copy_(L.v)
        host.append((hk, hv, kt.paged_kv(hk, hv, L.table, L.lens)))

    def attend(L, kvh):
        v = L.variants[rep]
        kt.kt_sparse_decode_attn_hostkv(L.q, kvh, v["params"], v["sel"], v["cnt"], v["out"],
                                        v["ws"])

    for L in layers:
        L.select(rep)
    n = 400
    t_att = graph_time([lambda L=L, h=h: attend(L, h[2]) for L, h in zip(layers, host)], n,
                       args.warmup, stream) / n
    t_step = graph_time([lambda L=L, h=h: (L.select(rep), attend(L, h[2]))
                         for L, h in zip(layers, host)], n, args.warmup, stream) / n
    b = step_bytes(layers[0].w)
    del host
    return {"workload": f"{layers[0].w.name}, {len(layers)} layers rotated, K/V in host memory",
            "attention_us": t_att * 1e6, "attended_kv_bytes_over_c2c": int(b["kv"]),
            "c2c_gbs": b["kv"] / t_att / 1e9,
            "step_us (select + attention)": t_step * 1e6,
            "note": "reps and the selection stay in HBM; only attended K/V cross NVLink-C2C"}


PHASES = ("entry", "slice_pages", "slice_reps_landed", "slice_scored", "slice_published",
          "unit_slices_seen", "selection_picked", "first_kv_load", "first_selected_load",
          "last_block_attended", "partial_published", "partials_seen", "output_written")


def phase_stamps_leg(step_fns, launches=40):
    """Per-CTA phase stamps (kt_set_phase_stamps) of single step launches, in
    us after the launch's first CTA entry: for each phase the median over CTAs
    (and the latest CTA), each the median over `launches` launches."""
    import torch

    import block_sparse_long_quest_gb300 as kt
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    buf = torch.zeros(sms * 16, dtype=torch.int64, device="cuda")
    med = {ph: [] for ph in PHASES}
    last = {ph: [] for ph in PHASES}
    kt.kt_set_phase_stamps(buf, sms)
    try:
        for i in range(launches + 5):
            buf.zero_()
            step_fns[i % len(step_fns)]()
            torch.cuda.synchronize()
            if i < 5:
                continue
            st = buf.view(sms, 16).cpu().numpy().astype(np.float64)
            t0 = st[:, 0][st[:, 0] > 0].min()
            for k, ph in enumerate(PHASES):
                col = st[:, k]
                col = col[col > 0]
                if col.size:
                    med[ph].append(float(np.median(col - t0)) / 1e3)
                    last[ph].append(float((col - t0).max()) / 1e3)
    finally:
        kt.kt_set_phase_stamps(None)
    return {ph: {"median_cta_us": round(float(np.median(med[ph])), 3),
                 "last_cta_us": round(float(np.median(last[ph])), 3)}
            for ph in PHASES if med[ph]}


def layers_q_bytes(w):
    return w.batch * w.params.num_q_heads * D * 2


if __name__ == "__main__":
    main()
