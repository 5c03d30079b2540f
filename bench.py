#!/usr/bin/env python
"""Benchmark: one decode step (append + paged decode attention, every layer) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload gqa8b] [--block-size 16]
    python bench.py --impl reference ...      # the float64 CPU oracle on the host cores

A step is the whole hot path over one batch: for each of the 32 layers, the new token's K/V is
written into its slot and decode attention runs over every cached token (split into 1024-token
partitions, 512 for the long-context workload, + log-sum-exp merge where a context needs it).
The default workload is the largest single-GPU configuration, the 8B-shaped GQA decode: batch
64, 32 layers, 32 q / 8 kv heads, head_dim 128, block_size 16, 2048 prefilled tokens per
request and 128 consecutive decode steps (step t appends position 2047 + t; timed steps cycle
through them), fp16 K/V ~ N(0, 1), physical blocks a seeded permutation of the pool.  Each
layer has its own ~570 MB cache, so every step streams ~17 GB: far larger than L2, no flush
needed.  --workload mha7b | shared_prefix | long_context | tiny select the other shapes.

Printed (rank 0, one JSON line): decode-attention HBM GB/s over the whole step (value), the
step time, tokens/s, the dominant kernel's roofline (algorithmic bytes / its CUDA-event time,
against the measured HBM copy bandwidth), the end-to-end rate through the C ABI with host
buffers (inputs copied host->device and outputs device->host inside the timed region), SM
clocks sampled during the timed region, and the CPU oracle's rate on a bounded sample.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attention HBM GB/s & % of GB300 roofline; tokens/s per step at 1 GPU"
LAYERS = 32
FALLBACK_HBM_GBS = 6800.0

WORKLOAD_TEXT = {
    "mha7b": "7B-shaped MHA decode: batch 16, 32 layers, 32 q / 32 kv heads, head_dim 128, block_size {bs}, "
             "context U[200,4000] per request (seeded), fp16 K/V ~N(0,1), one append+decode per layer",
    "gqa8b": "8B-shaped GQA decode: batch 64, 32 layers, 32 q / 8 kv heads, head_dim 128, block_size {bs}, "
             "2048 prefilled tokens, decode step t appends position 2047+t (steps cycle 1..128)",
    "shared_prefix": "shared-prefix batch: batch 32, 32 layers, 32 q / 8 kv heads, head_dim 128, block_size 16, "
                     "1024-token common prefix (64 shared blocks) + private suffix U[128,1024]",
    "long_context": "long context: batch 4, 32 layers, 32 q / 8 kv heads, head_dim 128, context 32768, "
                    "block_size {bs}, 1% of K rows x8 (peaky softmax), 512-token split partitions",
    "tiny": "tiny: batch 1, 1 layer, 32 q = 32 kv heads, head_dim 128, context 512, block_size 16",
}


# ----------------------------------------------------------------------------- helpers

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_over_ranks(ms_per_step: float, units: float, world: int):
    """Whole-job timing: the slowest rank's time, the sum of every rank's units."""
    if world <= 1:
        return ms_per_step, units
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([ms_per_step], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            peaks = json.load(f)
        return float(peaks["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, STREAM-style copy)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, one earlier GB300 copy measurement)"


def _code_only(text: str) -> str:
    """C++ source without comments and with whitespace collapsed (string literals of the kernel
    sources hold no comment markers)."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(workload: str = "") -> str:
    """Hash of the code (comments and layout ignored) of the kernel sources a workload's timed
    launches come from (the shared-prefix step also runs the prefix kernel)."""
    h = hashlib.sha256()
    names = ["pkv_decode.cu", "pkv_engine.cuh", "pkv_device.cuh"] + \
        (["pkv_prefix.cu"] if workload.startswith("shared_prefix") else [])
    for name in names:
        with open(os.path.join(ROOT, "paged_kv_cache_278_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def read_traffic(workload: str, bs: int):
    """DRAM bytes per launch of the partition kernel from a committed ncu summary, valid only
    while the kernel source is unchanged since the capture (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    want = kernel_source_hash(workload)
    with open(path, encoding="utf-8") as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            fields = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
            if fields.get("workload") == workload and int(fields.get("block_size", "0")) == bs \
                    and fields.get("kernel_sha") == want:
                return float(fields["dram_bytes_per_launch"])
    return None


class ClockSampler:
    """nvidia-smi samples (every 100 ms) of SM clock and throttle reasons, with host timestamps."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self, windows):
        inside = [s for t, s in self.samples if any(a <= t <= b for a, b in windows)]
        used = inside if inside else [s for _, s in self.samples]
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(s[0]) for s in used if num(s[0]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in used:
            for name, val in zip(names, s[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(used[0][1]),
                "power_w_max": max((num(s[2]) or 0.0) for s in used),
                "reasons": sorted(reasons),
                "samples": len(used), "samples_in_timed_region": len(inside)}


def gpu_uuid(dev_index: int) -> str:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev_index).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[dev_index] if vis else str(dev_index)


# ----------------------------------------------------------------------------- workload set-up

def make_layer(workload: str, layer: int, bs: int, device, step: int = 1):
    import workloads
    if workload == "mha7b":
        return workloads.mha7b(layer, device=device)
    if workload == "gqa8b":
        return workloads.gqa8b(layer, step, bs, device=device)
    if workload == "shared_prefix":
        return workloads.shared_prefix(layer, device=device)
    if workload == "long_context":
        return workloads.long_context(layer, bs, device=device)
    if workload == "tiny":
        return workloads.tiny(device=device)
    raise ValueError(workload)


def decode_bytes(ctx, num_kv_heads, num_q_heads, head_dim, bs, unique_prefix_tokens=0, num_seqs=None,
                 kv="fp16", q_len=1):
    """Algorithmic bytes of one decode-attention call: K and V of every cached token read once
    (a shared prefix once), q read, out written, block-table entries and context lengths read.
    kv="int8k": a key row is head_dim int8 codes plus one float32 scale; kv="int8kv": value rows too;
    kv="fp8kv": as int8kv with 8-bit floating-point (E4M3) codes."""
    b = len(ctx) if num_seqs is None else num_seqs
    tokens = sum(ctx) - unique_prefix_tokens * (b - 1) if unique_prefix_tokens else sum(ctx)
    k_row = head_dim + 4 if kv in ("int8k", "int8kv", "fp8kv") else head_dim * 2
    v_row = head_dim + 4 if kv in ("int8kv", "fp8kv") else head_dim * 2
    kv = tokens * num_kv_heads * (k_row + v_row)
    qo = 2 * b * q_len * num_q_heads * head_dim * 2
    tables = sum(-(-c // bs) for c in ctx) * 4 + 4 * b
    return kv + qo + tables


# ----------------------------------------------------------------------------- our arm

def run_ours(args):
    import numpy as np
    import torch

    import paged_kv_cache_278_gb300 as pkv
    from paged_kv_cache_278_gb300.build import build

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    build()
    dev = torch.device("cuda", local)

    bs = args.block_size
    n_layers = 1 if args.workload == "tiny" else (args.layers or LAYERS)
    steps_cycle = 128 if args.workload == "gqa8b" else 1

    # per-layer caches (distinct, like a real model) and per-layer new-token inputs in one block
    cases = [make_layer(args.workload, l, bs, dev) for l in range(n_layers)]
    c0 = cases[0]
    cpu_sample = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.query_len == 1:
        # host copies taken before any of our kernels run (the oracle baseline times single-token steps)
        cpu_sample = {k: getattr(c0, k).cpu().numpy() for k in
                      ("q", "k_cache", "v_cache", "k_new", "v_new", "block_tables", "context_lens", "positions")}
    int8k = args.kv == "int8k"
    int8kv = args.kv == "int8kv"
    fp8kv = args.kv == "fp8kv"
    if int8kv or fp8kv:
        # 8-bit K + V cache per layer (int8 or E4M3 codes): every pool row of the generated fp16 keys and values
        # quantised by the library's own append kernel (set-up, outside the timed regions)
        empty = pkv.empty_fp8kv_cache if fp8kv else pkv.empty_int8kv_cache
        append_q = pkv.append_fp8kv if fp8kv else pkv.append_int8kv
        for c in cases:
            nb_, hkv_, bs_, d_ = c.k_cache.shape
            c.k_codes, c.k_scale, c.v_codes, c.v_scale = empty(nb_, hkv_, bs_, dev)
            rows_k = c.k_cache.permute(0, 2, 1, 3).reshape(nb_ * bs_, hkv_, d_).contiguous()
            rows_v = c.v_cache.permute(0, 2, 1, 3).reshape(nb_ * bs_, hkv_, d_).contiguous()
            append_q(c.k_codes, c.k_scale, c.v_codes, c.v_scale, torch.arange(nb_ * bs_, device=dev), rows_k, rows_v)
            del rows_k, rows_v
            c.k_cache = c.v_cache = None
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
    if int8k:
        # int8-key cache per layer: every pool row of the generated fp16 keys quantised by the library's own
        # append kernel (set-up, outside the timed regions); V stays as generated
        for c in cases:
            nb_, hkv_, bs_, d_ = c.k_cache.shape
            c.k_codes, c.k_scale, _ = pkv.empty_int8k_cache(nb_, hkv_, bs_, dev)
            rows_k = c.k_cache.permute(0, 2, 1, 3).reshape(nb_ * bs_, hkv_, d_).contiguous()
            rows_v = c.v_cache.permute(0, 2, 1, 3).reshape(nb_ * bs_, hkv_, d_).contiguous()
            pkv.append_int8k(c.k_codes, c.k_scale, c.v_cache, torch.arange(nb_ * bs_, device=dev), rows_k, rows_v)
            del rows_k, rows_v
            c.k_cache = None
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
    B, Hq, Hkv, D = c0.num_seqs, c0.num_q_heads, c0.num_kv_heads, c0.head_dim
    bs = c0.block_size
    nq = args.query_len
    if nq > 1:
        # several new tokens per request (a draft being verified): seeded q / K / V for all of them
        g = torch.Generator(device=dev)
        g.manual_seed(7000 + nq)
        for c in cases:
            c.q = torch.randn((B * nq, Hq, D), generator=g, device=dev).half()
            c.k_new = torch.randn((B * nq, Hkv, D), generator=g, device=dev).half()
            c.v_new = torch.randn((B * nq, Hkv, D), generator=g, device=dev).half()
    q_all = torch.stack([c.q for c in cases])
    kn_all = torch.stack([c.k_new for c in cases])
    vn_all = torch.stack([c.v_new for c in cases])
    for l, c in enumerate(cases):
        c.q, c.k_new, c.v_new = q_all[l], kn_all[l], vn_all[l]
    out_all = torch.empty_like(q_all)
    block_tables = c0.block_tables.clone()
    max_ctx_cap = c0.max_blocks_per_seq * bs

    # context lengths / slots of each step of the cycle (host pool logic -> device, once)
    if args.workload == "gqa8b":
        import workloads
        ctx_steps = [[workloads.GQA_PREFILL + t] * B for t in range(1, steps_cycle + 1)]
    else:
        ctx_steps = [c0.context_lens.cpu().tolist()]
    ctx_dev = torch.tensor(ctx_steps, dtype=torch.int32, device=dev)
    # slots of the step's new tokens: positions ctx - nq .. ctx - 1 of every request (request-major)
    slot_dev = torch.stack([
        torch.stack([pkv.slot_mapping(block_tables.cpu(), torch.tensor(c, dtype=torch.int32) - nq + i, bs)
                     for i in range(nq)], 1).reshape(-1) for c in ctx_steps]).to(dev)
    query_start = torch.arange(0, (B + 1) * nq, nq, dtype=torch.int32, device=dev)
    ctx_cur = ctx_dev[0].clone()
    slot_cur = slot_dev[0].clone()
    cascade = args.workload == "shared_prefix" and not args.no_cascade
    prefix_len = 1024 if cascade else 0
    # the long-context workload is defined with 512-token split partitions; the others take the library's
    # default (PKV_DEFAULT_PARTITION)
    part = 512 if (args.workload == "long_context" and nq == 1 and args.kv == "fp16"
                   and not args.separate_append) else 0
    if args.partition:
        part = args.partition
    ws = pkv.make_step_workspace(B, Hq, max_ctx_cap, prefix_len, dev, partition_size=part) if nq == 1 else \
        pkv.make_multi_workspace(B, B * nq, nq, Hq, Hkv, max_ctx_cap, dev)

    # Each layer's step reads its own caches, which the kernel before it (the previous layer's step)
    # never writes, so every step call may stream its cache history while that kernel drains.
    overlap = not args.no_overlap

    def decode(l, c, attention_only=False):
        """One layer of the step: the append is fused into the decode kernel (pkv_decode_step) unless
        --separate-append asks for the two-call path (pkv_append + attention).  attention_only skips a
        separate append launch (the kernel-only timing region)."""
        if nq > 1:
            if args.separate_append:
                if not attention_only:
                    pkv.append(c.k_cache, c.v_cache, slot_cur, c.k_new, c.v_new)
                pkv.decode_attention_multi(out_all[l], c.q, c.k_cache, c.v_cache, block_tables, ctx_cur, query_start,
                                           nq, c.scale, workspace=ws)
            else:
                pkv.decode_step_multi(out_all[l], c.q, c.k_new, c.v_new, c.k_cache, c.v_cache, block_tables, ctx_cur,
                                      query_start, nq, c.scale, workspace=ws, overlap=overlap)
        elif int8kv:
            if args.separate_append:
                if not attention_only:
                    pkv.append_int8kv(c.k_codes, c.k_scale, c.v_codes, c.v_scale, slot_cur, c.k_new, c.v_new)
                pkv.decode_attention_int8kv(out_all[l], c.q, c.k_codes, c.k_scale, c.v_codes, c.v_scale, block_tables,
                                            ctx_cur, c.scale, workspace=ws)
            else:
                pkv.decode_step_int8kv(out_all[l], c.q, c.k_new, c.v_new, c.k_codes, c.k_scale, c.v_codes, c.v_scale,
                                       block_tables, ctx_cur, c.scale, workspace=ws, overlap=overlap)
        elif fp8kv:
            if args.separate_append:
                if not attention_only:
                    pkv.append_fp8kv(c.k_codes, c.k_scale, c.v_codes, c.v_scale, slot_cur, c.k_new, c.v_new)
                pkv.decode_attention_fp8kv(out_all[l], c.q, c.k_codes, c.k_scale, c.v_codes, c.v_scale, block_tables,
                                           ctx_cur, c.scale, workspace=ws)
            else:
                pkv.decode_step_fp8kv(out_all[l], c.q, c.k_new, c.v_new, c.k_codes, c.k_scale, c.v_codes, c.v_scale,
                                      block_tables, ctx_cur, c.scale, workspace=ws, overlap=overlap)
        elif int8k:
            if args.separate_append:
                if not attention_only:
                    pkv.append_int8k(c.k_codes, c.k_scale, c.v_cache, slot_cur, c.k_new, c.v_new)
                pkv.decode_attention_int8k(out_all[l], c.q, c.k_codes, c.k_scale, c.v_cache, block_tables, ctx_cur,
                                           c.scale, workspace=ws)
            else:
                pkv.decode_step_int8k(out_all[l], c.q, c.k_new, c.v_new, c.k_codes, c.k_scale, c.v_cache,
                                      block_tables, ctx_cur, c.scale, workspace=ws, overlap=overlap)
        elif args.separate_append:
            if not attention_only:
                pkv.append(c.k_cache, c.v_cache, slot_cur, c.k_new, c.v_new)
            if cascade:
                pkv.decode_attention_shared_prefix(out_all[l], c.q, c.k_cache, c.v_cache, block_tables, ctx_cur,
                                                   c.scale, prefix_len, ws)
            else:
                pkv.decode_attention(out_all[l], c.q, c.k_cache, c.v_cache, block_tables, ctx_cur, c.scale,
                                     workspace=ws)
        else:
            pkv.decode_step(out_all[l], c.q, c.k_new, c.v_new, c.k_cache, c.v_cache, block_tables, ctx_cur, c.scale,
                            prefix_len, ws, partition_size=part, overlap=overlap)

    prefix_tokens = 1024 if args.workload == "shared_prefix" else 0
    bytes_per_step = [n_layers * decode_bytes(c, Hkv, Hq, D, bs, prefix_tokens, kv=args.kv, q_len=nq)
                      for c in ctx_steps]
    logical_bytes_per_step = [n_layers * decode_bytes(c, Hkv, Hq, D, bs, kv=args.kv, q_len=nq) for c in ctx_steps]

    # per layer: the decode kernel (append and the split's merge fused in), plus the prefix kernel and the
    # merge kernel with the cascade, plus the append kernel on the two-call path
    launches_per_step = n_layers * (1 + (2 if cascade else 0) + (1 if args.separate_append else 0))

    def step():
        for l, c in enumerate(cases):
            decode(l, c)

    def attention_only():
        for l, c in enumerate(cases):
            decode(l, c, attention_only=True)

    def set_step(i):
        j = i % steps_cycle
        if steps_cycle > 1:
            ctx_cur.copy_(ctx_dev[j], non_blocking=True)
            slot_cur.copy_(slot_dev[j], non_blocking=True)
        return j

    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 1)):
            set_step(i)
            step()
    torch.cuda.synchronize(dev)
    graph = kernel_graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
        kernel_graph = torch.cuda.CUDAGraph()  # the attention launches alone (no separate append)
        with torch.cuda.graph(kernel_graph, stream=stream):
            attention_only()
        with torch.cuda.stream(stream):
            for i in range(args.warmup):
                set_step(i)
                graph.replay()
        torch.cuda.synchronize(dev)
    assert pkv.device_error() == pkv.PKV_DEV_OK
    assert torch.isfinite(out_all.float()).all()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    clocks = ClockSampler(gpu_uuid(local))
    clocks.start()
    time.sleep(0.3)
    windows = []

    # ---- timed region 1: K whole steps (CUDA-graph replay of all layers)
    barrier()
    t0 = time.time()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    step_bytes = 0
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(args.steps):
            j = set_step(i)
            step_bytes += bytes_per_step[j % len(bytes_per_step)]
            if graph is not None:
                graph.replay()
            else:
                step()
        e1.record(stream)
    barrier()
    windows.append((t0, time.time()))
    ms_total = e0.elapsed_time(e1)
    ms_per_step = ms_total / args.steps

    # ---- timed region 2: the dominant kernel alone.  A pkv_decode_step call is exactly one launch of
    # the decode kernel (the append and the split's log-sum-exp merge run inside it; the cascade adds
    # its prefix kernel and its merge kernel); a separate append launch is left out here.  Per step the layers'
    # launches are replayed back to back from a CUDA graph (no host launch gaps) between one pair of
    # CUDA events on the launching stream: average launch duration = event interval / launches.
    kt_steps = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(kt_steps)]
    kernel_bytes = 0
    barrier()
    t0 = time.time()
    with torch.cuda.stream(stream):
        for i in range(kt_steps):
            j = set_step(i)
            a, b = ev[i]
            a.record(stream)
            if kernel_graph is not None:
                kernel_graph.replay()
            else:
                attention_only()
            b.record(stream)
            kernel_bytes += bytes_per_step[j % len(bytes_per_step)]
    barrier()
    windows.append((t0, time.time()))
    kernel_ms = sum(a.elapsed_time(b) for a, b in ev)
    kernel_launches = kt_steps * n_layers

    # ---- timed region 3: end to end through the public API with host buffers.  Run like a serving
    # loop (with graphs): two sets of per-step device inputs and outputs, each with its own graph of
    # the step; a copy stream uploads step i + 1's inputs while step i runs and reads step i's
    # outputs back while step i + 1 runs, events ordering every reuse of a set.  Every copy of
    # every step is inside the timed region.
    q_h = q_all.cpu().pin_memory()
    kn_h = kn_all.cpu().pin_memory()
    vn_h = vn_all.cpu().pin_memory()
    bt_h = block_tables.cpu().pin_memory()
    ctx_h = ctx_dev.cpu().pin_memory()
    slot_h = slot_dev.cpu().pin_memory()
    out_h = torch.empty(out_all.shape, dtype=out_all.dtype).pin_memory()
    h2d = (q_h.numel() + kn_h.numel() + vn_h.numel()) * 2 + bt_h.numel() * 4 + ctx_h[0].numel() * 4 + \
        slot_h[0].numel() * 8
    d2h = out_h.numel() * 2
    e2e_bytes = 0
    x0 = torch.cuda.Event(enable_timing=True)
    x1 = torch.cuda.Event(enable_timing=True)
    if graph is not None:
        set0 = (q_all, kn_all, vn_all, block_tables, ctx_cur, slot_cur, out_all)
        set1 = tuple(t.clone() for t in set0)
        # capture the step once more on the second set (decode() reads these names at call time)
        out_all, block_tables, ctx_cur, slot_cur = set1[6], set1[3], set1[4], set1[5]
        for l, c in enumerate(cases):
            c.q, c.k_new, c.v_new = set1[0][l], set1[1][l], set1[2][l]
        graph1 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph1, stream=stream):
            step()
        out_all, block_tables, ctx_cur, slot_cur = set0[6], set0[3], set0[4], set0[5]
        for l, c in enumerate(cases):
            c.q, c.k_new, c.v_new = q_all[l], kn_all[l], vn_all[l]
        sets, graphs = (set0, set1), (graph, graph1)
        copy_stream = torch.cuda.Stream(device=dev)
        ev_in = (torch.cuda.Event(), torch.cuda.Event())
        ev_done = (torch.cuda.Event(), torch.cuda.Event())

        def upload(i, st):
            j = i % steps_cycle
            st[0].copy_(q_h, non_blocking=True)
            st[1].copy_(kn_h, non_blocking=True)
            st[2].copy_(vn_h, non_blocking=True)
            st[3].copy_(bt_h, non_blocking=True)
            st[4].copy_(ctx_h[j], non_blocking=True)
            st[5].copy_(slot_h[j], non_blocking=True)

        torch.cuda.synchronize(dev)
        barrier()
        t0 = time.time()
        with torch.cuda.stream(copy_stream):
            x0.record(copy_stream)
            upload(0, sets[0])
            ev_in[0].record(copy_stream)
        for i in range(args.steps):
            s, ns = i % 2, (i + 1) % 2
            with torch.cuda.stream(stream):
                stream.wait_event(ev_in[s])
                graphs[s].replay()
                ev_done[s].record(stream)
            with torch.cuda.stream(copy_stream):
                if i + 1 < args.steps:
                    if i >= 1:
                        copy_stream.wait_event(ev_done[ns])  # step i - 1 is done with set ns
                    upload(i + 1, sets[ns])
                    ev_in[ns].record(copy_stream)
                copy_stream.wait_event(ev_done[s])
                out_h.copy_(sets[s][6], non_blocking=True)
            e2e_bytes += bytes_per_step[(i % steps_cycle) % len(bytes_per_step)]
        stream.wait_stream(copy_stream)
        x1.record(stream)
        x1.synchronize()
    else:
        barrier()
        t0 = time.time()
        with torch.cuda.stream(stream):
            x0.record(stream)
            for i in range(args.steps):
                j = i % steps_cycle
                q_all.copy_(q_h, non_blocking=True)
                kn_all.copy_(kn_h, non_blocking=True)
                vn_all.copy_(vn_h, non_blocking=True)
                block_tables.copy_(bt_h, non_blocking=True)
                ctx_cur.copy_(ctx_h[j], non_blocking=True)
                slot_cur.copy_(slot_h[j], non_blocking=True)
                step()
                out_h.copy_(out_all, non_blocking=True)
                e2e_bytes += bytes_per_step[j % len(bytes_per_step)]
            x1.record(stream)
        x1.synchronize()
    barrier()
    windows.append((t0, time.time()))
    e2e_ms = x0.elapsed_time(x1)
    clocks.stop()
    assert pkv.device_error() == pkv.PKV_DEV_OK
    assert torch.isfinite(out_h.float()).all()

    # ---- whole-job numbers
    ms_job, bytes_job = reduce_over_ranks(ms_per_step, step_bytes / args.steps, world)
    e2e_ms_job, e2e_bytes_job = reduce_over_ranks(e2e_ms / args.steps, e2e_bytes / args.steps, world)
    kernel_avg_ms = kernel_ms / kernel_launches
    kernel_bytes_avg = kernel_bytes / kernel_launches
    if rank != 0:
        return

    peak, peak_src = read_peaks()
    gbs = bytes_job / (ms_job * 1e-3) / 1e9
    achieved = kernel_bytes_avg / (kernel_avg_ms * 1e-3) / 1e9
    traffic = read_traffic(args.workload + ("" if args.kv == "fp16" else "/" + args.kv) + (f"/q{nq}" if nq > 1 else ""),
                           bs)
    both8 = int8kv or fp8kv
    layer_cache_bytes = (cases[0].k_codes.numel() * (2 if both8 else 1) + cases[0].k_scale.numel() * 4
                         * (2 if both8 else 1) + (0 if both8 else cases[0].v_cache.numel() * 2)
                         if args.kv != "fp16" else cases[0].v_cache.numel() * 4)
    line = {
        "metric": METRIC,
        "value": round(gbs, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_job, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": KV_DTYPE[args.kv],
        "accumulate": "f32",
        "data": "synthetic (seeded N(0,1) fp16 K/V/q, seeded block permutation)",
        "config": {
            "workload": WORKLOAD_TEXT[args.workload].format(bs=bs),
            "layers": n_layers,
            "batch": B,
            "num_q_heads": Hq,
            "num_kv_heads": Hkv,
            "head_dim": D,
            "block_size": bs,
            "partition_size": ("prefix: 128-token chunks; suffix: picked per call (64-512 tokens)" if cascade
                               else part or pkv.PKV_DEFAULT_PARTITION),
            "kv_cache": KV_TEXT[args.kv],
            "l2": "inputs larger than L2: every layer has its own cache (%.0f MB), %.1f GB streamed per step"
                  % (layer_cache_bytes / 1e6, bytes_job / 1e9),
            "timing": "CUDA-graph replay of the whole step" if graph is not None else "eager launches",
            "decode_call": ((f"pkv_append + pkv_decode_attention_multi ({nq} new tokens per request, causal)"
                             if args.separate_append else
                             f"pkv_decode_step_multi ({nq} new tokens per request appended and attended causally"
                             f" in one launch)") if nq > 1 else
                            ("pkv_append" + KV_SUFFIX[args.kv] + " + " if args.separate_append
                             else "pkv_decode_step" + KV_SUFFIX[args.kv] + " ")
                            + ("shared prefix 1024 tokens" if cascade else "")
                            + (" with PKV_STEP_OVERLAP (each layer streams its cache history while the previous "
                               "layer's kernel drains)" if overlap and not args.separate_append else "")),
        },
        "tokens_per_s": round(B * nq * world / (ms_job * 1e-3), 1),
        "pct_of_hbm_peak": round(100 * gbs / peak, 1),
        "decode_bytes_per_step": int(bytes_job),
        "logical_bytes_per_step": int(sum(logical_bytes_per_step) / len(logical_bytes_per_step)),
        "roofline": {
            "kernel": f"decode_partition_kernel (packed-GQA paged decode, {part or pkv.PKV_DEFAULT_PARTITION}-token "
                      "partitions, fused LSE merge)"
                      + (" + prefix_kernel + merge_groups_kernel (timed together)" if cascade else ""),
            "timing": "CUDA events around graph replays of the layers' attention launches"
                      if kernel_graph is not None else "CUDA events around eager attention launches",
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_source": peak_src,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "algorithmic_bytes_per_launch": int(kernel_bytes_avg),
            "avg_launch_us": round(kernel_avg_ms * 1e3, 2),
            "launches_timed": kernel_launches,
        },
        "e2e": {
            "value": round(e2e_bytes_job / (e2e_ms_job * 1e-3) / 1e9, 1),
            "unit": "GB/s",
            "ms_per_step": round(e2e_ms_job, 4),
            "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h),
            "note": "KV cache is device-resident state; each step copies the new tokens' q/k/v for all layers, "
                    "block tables, context lengths and slots from pinned host memory and reads every layer's "
                    "output back" + (", double-buffered on a copy stream (step i + 1's upload and step i's "
                                     "readback overlap the neighbouring steps)" if graph is not None else ""),
        },
        "gpu_launches": launches_per_step * args.steps + (2 * args.steps if steps_cycle > 1 else 0),
        "clocks": clocks.summary(windows),
        "kernel_source": kernel_source_hash(args.workload if cascade else ""),
        "gpu": torch.cuda.get_device_name(dev),
    }
    if cpu_sample is not None:
        line["cpu_baseline"] = cpu_baseline(cpu_sample, c0, bs, Hkv, Hq, D, budget_s=args.cpu_budget, kv=args.kv)
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- CPU oracle

KV_DTYPE = {"fp16": "f16", "int8k": "i8 keys (f32 row scales), f16 values",
            "int8kv": "i8 keys and values (f32 row scales)", "fp8kv": "e4m3 keys and values (f32 row scales)"}
KV_TEXT = {"fp16": "fp16 K and V", "int8k": "int8 keys + float32 scale per (token, kv head), fp16 values",
           "int8kv": "int8 keys and values, each + float32 scale per (token, kv head)",
           "fp8kv": "fp8 (E4M3) keys and values, each + float32 scale per (token, kv head)"}
KV_SUFFIX = {"fp16": "", "int8k": "_int8k", "int8kv": "_int8kv", "fp8kv": "_fp8kv"}


def oracle_int8kv_pool(h):
    """Host int8 K + V pool (k_codes, k_scale, v_codes, v_scale) of the sample's fp16 rows, quantised
    by the oracle."""
    import numpy as np

    import oracle
    nb, hkv, bs, d = h["k_cache"].shape
    pool = (np.zeros((nb, hkv, bs, d), np.int8), np.zeros((nb, hkv, bs), np.float32),
            np.zeros((nb, hkv, bs, d), np.int8), np.zeros((nb, hkv, bs), np.float32))
    rows = lambda a: np.ascontiguousarray(a.transpose(0, 2, 1, 3).reshape(nb * bs, hkv, d))
    oracle.append_quant_kv(*pool, np.arange(nb * bs, dtype=np.int64), rows(h["k_cache"]), rows(h["v_cache"]))
    return pool


def oracle_fp8kv_pool(h):
    """Host fp8 K + V pool (k_codes, k_scale, v_codes, v_scale) of the sample's fp16 rows, quantised
    by the oracle."""
    import numpy as np

    import oracle
    nb, hkv, bs, d = h["k_cache"].shape
    pool = (np.zeros((nb, hkv, bs, d), np.uint8), np.zeros((nb, hkv, bs), np.float32),
            np.zeros((nb, hkv, bs, d), np.uint8), np.zeros((nb, hkv, bs), np.float32))
    rows = lambda a: np.ascontiguousarray(a.transpose(0, 2, 1, 3).reshape(nb * bs, hkv, d))
    oracle.append_fp8_kv(*pool, np.arange(nb * bs, dtype=np.int64), rows(h["k_cache"]), rows(h["v_cache"]))
    return pool


def oracle_int8k_pool(h):
    """Host int8-key pool (codes, scales) of the sample's fp16 keys, quantised by the oracle."""
    import numpy as np

    import oracle
    nb, hkv, bs, d = h["k_cache"].shape
    codes = np.zeros((nb, hkv, bs, d), np.int8)
    scales = np.zeros((nb, hkv, bs), np.float32)
    v = h["v_cache"].copy()
    rows = lambda a: np.ascontiguousarray(a.transpose(0, 2, 1, 3).reshape(nb * bs, hkv, d))
    oracle.append_quant_k(codes, scales, v, np.arange(nb * bs, dtype=np.int64), rows(h["k_cache"]),
                          rows(h["v_cache"]))
    return codes, scales


def cpu_baseline(h, case, bs, hkv, hq, d, budget_s=15.0, max_requests=None, kv="fp16"):
    """The oracle (single-threaded C, float64) on a bounded sample of the workload: one layer's
    append + decode for as many requests (in order) as fit the time budget."""
    import numpy as np

    import oracle
    ctx = h["context_lens"].tolist()
    b = len(ctx)
    slots = oracle.slot_mapping(h["block_tables"], h["positions"], bs)
    if kv == "int8kv":
        pool = oracle_int8kv_pool(h)
        t0 = time.perf_counter()
        oracle.append_quant_kv(*pool, slots, h["k_new"], h["v_new"])
        decode_one = lambda sl: oracle.decode_quant_kv(h["q"][sl], *pool, h["block_tables"][sl],
                                                       h["context_lens"][sl], case.scale)
    elif kv == "fp8kv":
        pool = oracle_fp8kv_pool(h)
        t0 = time.perf_counter()
        oracle.append_fp8_kv(*pool, slots, h["k_new"], h["v_new"])
        decode_one = lambda sl: oracle.decode_fp8_kv(h["q"][sl], *pool, h["block_tables"][sl],
                                                     h["context_lens"][sl], case.scale)
    elif kv == "int8k":
        codes, scales = oracle_int8k_pool(h)
        t0 = time.perf_counter()
        oracle.append_quant_k(codes, scales, h["v_cache"], slots, h["k_new"], h["v_new"])
        decode_one = lambda sl: oracle.decode_quant_k(h["q"][sl], codes, scales, h["v_cache"], h["block_tables"][sl],
                                                      h["context_lens"][sl], case.scale)
    else:
        t0 = time.perf_counter()
        oracle.append(h["k_cache"], h["v_cache"], slots, h["k_new"], h["v_new"])
        decode_one = lambda sl: oracle.decode(h["q"][sl], h["k_cache"], h["v_cache"], h["block_tables"][sl],
                                              h["context_lens"][sl], case.scale)
    done, nbytes, tokens = 0, 0, 0
    limit = b if max_requests is None else min(b, max_requests)
    # requests of layer 0 in order, cycling, until the time budget is spent (at least one pass)
    while done < limit or time.perf_counter() - t0 < budget_s:
        i = done % b
        decode_one(slice(i, i + 1))
        nbytes += decode_bytes(ctx[i:i + 1], hkv, hq, d, bs, kv=kv)
        tokens += ctx[i]
        done += 1
        if max_requests is not None and done >= limit:
            break
    dt = time.perf_counter() - t0
    return {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"layer 0: append of all {b} requests, then {done} single-request decodes cycling over "
                      f"the {b} requests ({tokens} cached tokens attended), single-threaded C float64, {dt:.1f} s",
            "cpu": cpu_model()}


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part", "hardware")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


# ----------------------------------------------------------------------------- reference arm

def run_reference(args):
    """The oracle as it stands on the host cores: each step = append + decode of a bounded set of
    requests of one layer of the same workload; steps sized so the run ends within minutes."""
    rank, world, local = dist_env()
    if rank != 0:
        return
    import numpy as np
    import oracle

    bs = args.block_size
    case = make_layer(args.workload, 0, bs, "cpu")
    bs = case.block_size
    h = {k: getattr(case, k).numpy() for k in
         ("q", "k_cache", "v_cache", "k_new", "v_new", "block_tables", "context_lens", "positions")}
    ctx = h["context_lens"].tolist()
    b = len(ctx)
    # calibrate: one request
    t0 = time.perf_counter()
    oracle.decode(h["q"][:1], h["k_cache"], h["v_cache"], h["block_tables"][:1], h["context_lens"][:1], case.scale)
    per_token = (time.perf_counter() - t0) / max(ctx[0], 1)
    per_step_budget = args.cpu_budget * 8 / max(args.steps + args.warmup, 1)
    n_req, tok = 0, 0
    while n_req < b and (tok + ctx[n_req]) * per_token <= per_step_budget:
        tok += ctx[n_req]
        n_req += 1
    n_req = max(n_req, 1)
    sl = slice(0, n_req)
    slots = oracle.slot_mapping(h["block_tables"][sl], h["positions"][sl], bs)

    if args.kv == "int8kv":
        pool = oracle_int8kv_pool(h)

        def one():
            oracle.append_quant_kv(*pool, slots, h["k_new"][sl], h["v_new"][sl])
            oracle.decode_quant_kv(h["q"][sl], *pool, h["block_tables"][sl], h["context_lens"][sl], case.scale)
    elif args.kv == "fp8kv":
        pool = oracle_fp8kv_pool(h)

        def one():
            oracle.append_fp8_kv(*pool, slots, h["k_new"][sl], h["v_new"][sl])
            oracle.decode_fp8_kv(h["q"][sl], *pool, h["block_tables"][sl], h["context_lens"][sl], case.scale)
    elif args.kv == "int8k":
        codes, scales = oracle_int8k_pool(h)

        def one():
            oracle.append_quant_k(codes, scales, h["v_cache"], slots, h["k_new"][sl], h["v_new"][sl])
            oracle.decode_quant_k(h["q"][sl], codes, scales, h["v_cache"], h["block_tables"][sl],
                                  h["context_lens"][sl], case.scale)
    else:
        def one():
            oracle.append(h["k_cache"], h["v_cache"], slots, h["k_new"][sl], h["v_new"][sl])
            oracle.decode(h["q"][sl], h["k_cache"], h["v_cache"], h["block_tables"][sl], h["context_lens"][sl],
                          case.scale)

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    dt = time.perf_counter() - t0
    nbytes = decode_bytes(ctx[:n_req], case.num_kv_heads, case.num_q_heads, case.head_dim, bs, kv=args.kv)
    value = nbytes * args.steps / dt / 1e9
    sample = (f"per step: layer 0, append + decode of {n_req} of {b} requests ({sum(ctx[:n_req])} cached tokens), "
              f"single-threaded C float64")
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1) fp16 K/V/q, seeded block permutation)",
        "config": {"workload": WORKLOAD_TEXT[args.workload].format(bs=bs), "block_size": bs,
                   "kv_cache": KV_TEXT[args.kv]},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample, "cpu": cpu_model()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOAD_TEXT), default="gqa8b")
    ap.add_argument("--block-size", type=int, default=16)
    ap.add_argument("--layers", type=int, default=0, help="layers per step (default 32; fewer only for profiling)")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-cascade", action="store_true", help="shared_prefix: plain decode instead of the cascade")
    ap.add_argument("--separate-append", action="store_true",
                    help="two calls per layer (pkv_append, then attention) instead of pkv_decode_step")
    ap.add_argument("--kv", choices=["fp16", "int8k", "int8kv", "fp8kv"], default="fp16",
                    help="cache format: fp16 K/V; int8 keys with float32 row scales and fp16 values; "
                         "int8 keys and values, each with float32 row scales; or the same with fp8 (E4M3) codes")
    ap.add_argument("--query-len", type=int, default=1,
                    help="new tokens per request per step (>1: append them, then causal multi-token attention)")
    ap.add_argument("--partition", type=int, default=0,
                    help="split-context partition in tokens for the fused fp16 step (0: the workload's default)")
    ap.add_argument("--no-overlap", action="store_true",
                    help="step calls without PKV_STEP_OVERLAP (no layer streams its cache before the previous drains)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.query_len > 1 and (args.kv != "fp16" or args.workload == "shared_prefix"):
        ap.error("--query-len > 1 runs the fp16 multi-token path on mha7b, gqa8b, long_context or tiny")
    if args.query_len > 16 and not args.separate_append:
        ap.error("the one-launch several-token step takes up to 16 new tokens; use --separate-append beyond")
    if args.partition and (args.partition % 16 or not 16 <= args.partition <= 4096 or args.kv != "fp16"
                           or args.query_len > 1 or args.separate_append
                           or (args.workload == "shared_prefix" and not args.no_cascade)):
        ap.error("--partition (a multiple of 16 in [16, 4096]) applies to the fused fp16 single-token step")
    if args.query_len > 1 and args.impl == "reference":
        ap.error("the reference arm times single-token steps")
    if args.kv != "fp16" and args.workload == "shared_prefix" and not args.no_cascade:
        ap.error("the shared-prefix cascade reads fp16 K/V; use --no-cascade with an int8 cache")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)
    rank, world, _ = dist_env()
    if world > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.barrier()
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
