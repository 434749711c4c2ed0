#!/usr/bin/env python
"""Benchmark of the Llama-3-style decoder block on GB300.

Default workload: one Llama-3 8B-shaped decode block step at batch 32 with 1000
cached positions (pos = 1000, keys 0..1000 read), bf16, seeded synthetic
weights N(0, 0.02), x and cache N(0, 1).  A "step" is one full pass of the
block (RMSNorm, QKV + RoPE + KV append, attention, O + residual, RMSNorm,
gate/up + SwiGLU, down + residual) for every sequence of the batch; it rewrites
cache row 1000, so steps are idempotent.  The weights (436 MB) are larger than
L2 (126 MB), so every step streams them from HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--batch B] [--impl ours|reference]

Prints one JSON line.  `--impl reference` times the CPU oracle (the plain
NumPy definition of the block) on a bounded sample of the same workload on the
host cores.  Under torchrun each rank runs an independent replica (the path
needs no exchange between GPUs): value = tokens of all ranks / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "decode block tok/s & HBM-roofline frac; prefill block TFLOP/s vs bf16 peak"
POS = 1000
MAX_SEQ = 1024
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0)), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


# ----------------------------------------------------------------------------- algorithmic work

def decode_step_bytes(dims, B, pos):
    from_bytes = 2
    d, f = dims.d_model, dims.d_ff
    q, kv = dims.n_heads * dims.head_dim, dims.n_kv_heads * dims.head_dim
    weights = d * (q + 2 * kv) + q * d + 3 * d * f + 2 * d
    kv_read = 2 * B * dims.n_kv_heads * (pos + 1) * dims.head_dim
    kv_write = 2 * B * kv
    act = 2 * B * d
    return from_bytes * (weights + kv_read + kv_write + act)


def decode_seqpos_bytes(dims, positions):
    """decode_step_bytes with a position per sequence: each sequence reads its own
    pos + 1 cache rows."""
    d, f = dims.d_model, dims.d_ff
    q, kv = dims.n_heads * dims.head_dim, dims.n_kv_heads * dims.head_dim
    B = len(positions)
    weights = d * (q + 2 * kv) + q * d + 3 * d * f + 2 * d
    kv_read = sum(2 * dims.n_kv_heads * (p + 1) * dims.head_dim for p in positions)
    return 2 * (weights + kv_read + 2 * B * kv + 2 * B * d)


def gateup_launch_bytes(dims, B):
    """Algorithmic bytes of one gate/up projection launch: both weight matrices once,
    the normalised input read, the SwiGLU output written."""
    return 2 * (2 * dims.d_ff * dims.d_model + B * dims.d_model + B * dims.d_ff)


def prefill_stage_flops(dims, B, T):
    """Algorithmic FLOPs of each tensor-core stage of a causal prefill step."""
    d, f = dims.d_model, dims.d_ff
    q, kv = dims.n_heads * dims.head_dim, dims.n_kv_heads * dims.head_dim
    n = B * T
    return {"qkv": 2 * n * d * (q + 2 * kv), "attention": B * 4 * dims.n_heads * dims.head_dim * (T * (T + 1) // 2),
            "o_proj": 2 * n * q * d, "gate_up": 2 * n * d * 2 * f, "down": 2 * n * f * d}


def prefill_flops(dims, B, T):
    d, f = dims.d_model, dims.d_ff
    q, kv = dims.n_heads * dims.head_dim, dims.n_kv_heads * dims.head_dim
    macs = d * (q + 2 * kv) + q * d + 3 * d * f
    pairs = T * (T + 1) // 2
    return B * (2 * macs * T + 4 * dims.n_heads * dims.head_dim * pairs)


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, flags in rows for i, fl in enumerate(flags) if fl == "Active"})
        top = max(r[0] for r in rows)
        loaded = [r[0] for r in rows if r[0] >= 0.5 * top] or [r[0] for r in rows]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows)}


# ----------------------------------------------------------------------------- traffic from the committed ncu summary

def kernel_source_digest():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_decoder_block_gb300", "csrc")
    # the kernel and the host code that fixes its schedule (the K-segment choice)
    for f in ("gemm_tc.cuh", "gemm_ws.cuh", "gemm_weight_stream.cu", "gemm_host.cu", "ptx.cuh", "common.cuh"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel_key: str):
    """dram read+write bytes per launch recorded in profiles/ for this kernel, or None
    when there is none or the kernel source changed since it was captured."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    digest = kernel_source_digest()
    for f in sorted(os.listdir(pdir)):
        if not f.endswith((".md", ".txt")):
            continue
        text = open(os.path.join(pdir, f)).read()
        m = re.search(rf"traffic\[{re.escape(kernel_key)}\]\s*=\s*([0-9.eE+]+)\s+bytes per launch,\s*source\s+([0-9a-f]+)",
                      text)
        if m and m.group(2) == digest:
            return float(m.group(1))
    return None


# ----------------------------------------------------------------------------- ranks

def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of every rank's x (each rank's timed region: the job takes as long
    as its slowest replica); x itself on a single rank."""
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- our arm

def run_ours(args, rank, world, device):
    import dense_decoder_block_gb300 as ddb
    ddb.lib()
    dims = workloads.LLAMA3_8B
    B = args.batch
    wts = workloads.make_weights(dims, weight_std=0.02)
    inp = workloads.make_block_inputs(dims, B, 1, cache_len=POS, max_seq=MAX_SEQ, weights=wts)
    w = {k: v.to(device) for k, v in inp.weights.items()}
    g = {k: v.to(device) for k, v in inp.gains.items()}
    blk = ddb.LlamaBlock(dims, w, g, MAX_SEQ)
    kc, vc = inp.k_cache.to(device), inp.v_cache.to(device)
    kv = ddb.KVCache(kc, vc)
    x = inp.x.to(device)
    y = torch.empty_like(x)
    ws = blk.workspace(B, 1)
    stream = torch.cuda.current_stream(device)

    pos_dev = torch.tensor([POS], dtype=torch.int32, device=device)

    def eager_step():
        blk.decode(x, kv, POS, y, ws)

    # One decode step captured once as a CUDA graph (position read on the device),
    # replayed per step: no host work between the block's kernels.
    for _ in range(args.warmup):
        eager_step()
    torch.cuda.synchronize(device)
    assert blk.poll_error() == 0
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(device)
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        blk.decode_devpos(x, kv, pos_dev, y, ws, cap)
        with torch.cuda.graph(graph, stream=cap):
            blk.decode_devpos(x, kv, pos_dev, y, ws, cap)
    stream.wait_stream(cap)
    torch.cuda.synchronize(device)

    def step():
        graph.replay()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)
    assert blk.poll_error() == 0

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(device)

    # --- timed region: K steps, device-side events on the launching stream
    gpu_index = device.index if device.index is not None else 0
    visible = os.environ.get("CUDA_VISIBLE_DEVICES")
    if visible:
        try:
            gpu_index = int(visible.split(",")[gpu_index])
        except (ValueError, IndexError):
            pass
    with ClockSampler(gpu_index) as clk:
        time.sleep(0.3)
        barrier()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(args.steps):
            step()
        t1.record(stream)
        barrier()
        ms = t0.elapsed_time(t1)
    clocks = clk.summary()
    ms_step = ms / args.steps
    if world > 1:
        ms = max_over_ranks(ms, world, device)
        ms_step = ms / args.steps
    tokens = B * world * args.steps
    value = tokens / (ms / 1e3)

    # --- per-stage durations (second pass, events between the block's kernels)
    stage_ms = stage_profile(blk, lambda st: blk.decode_devpos(x, kv, pos_dev, y, ws, st), device, args.steps)

    # --- end to end through the public API with host buffers.  The input of every step is
    # in pinned host memory and its result must land there.  Main figure: the block's
    # kernels read x from and write y to that host memory themselves (device addresses
    # from llama_device_ptr_of_host; NVLink-C2C on a Grace host), one graph replay per
    # step.  Also reported: the same step between a host-to-device and a
    # device-to-host copy call.
    xh = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    xh.copy_(inp.x)
    yh = torch.empty(y.shape, dtype=y.dtype, pin_memory=True)
    xm, ym = ddb.HostMapped(xh), ddb.HostMapped(yh)
    graph_h = torch.cuda.CUDAGraph()
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        blk.decode_devpos(xm, kv, pos_dev, ym, ws, cap)
        with torch.cuda.graph(graph_h, stream=cap):
            blk.decode_devpos(xm, kv, pos_dev, ym, ws, cap)
    stream.wait_stream(cap)
    torch.cuda.synchronize(device)
    for _ in range(args.warmup):
        graph_h.replay()
    barrier()
    assert torch.equal(yh, y.cpu()), "host-memory decode differs from the device-memory decode"

    def timed(fn):
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        barrier()
        return max_over_ranks(e0.elapsed_time(e1), world, device)

    e2e_ms = timed(graph_h.replay)

    def copy_step():
        x.copy_(xh, non_blocking=True)
        step()
        yh.copy_(y, non_blocking=True)

    for _ in range(args.warmup):
        copy_step()
    e2e_copy_ms = timed(copy_step)
    e2e_value = tokens / (e2e_ms / 1e3)
    assert blk.poll_error() == 0

    n_launch = blk_launches(blk)
    hbm, bf16_peak, _, peak_kind = peaks()
    step_bytes = decode_step_bytes(dims, B, POS)
    gu_bytes = gateup_launch_bytes(dims, B)
    gu_ms = stage_ms.get("gate_up")
    roof = None
    if gu_ms:
        ach = gu_bytes / (gu_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": "gate/up projection + SwiGLU (weight-streaming tcgen05)",
                "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s", "frac": round(ach / hbm, 4),
                "peak_kind": f"{peak_kind} HBM copy bandwidth",
                "traffic": committed_traffic("gate_up_decode_b%d" % B),
                "algorithmic_bytes_per_launch": gu_bytes, "avg_launch_us": round(gu_ms * 1e3, 2)}
    step_ach = step_bytes / (ms_step / 1e3) / 1e9
    out = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "tok/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,0.02) weights, N(0,1) x and KV cache)",
        "config": {"workload": f"Llama-3 8B-shaped decode block, batch {B}, 1000 cached positions (pos 1000)",
                   "batch": B, "pos": POS, "keys_read": POS + 1, "d_model": dims.d_model,
                   "heads": f"{dims.n_heads}q/{dims.n_kv_heads}kv", "head_dim": dims.head_dim, "d_ff": dims.d_ff,
                   "l2": "inputs larger than L2: 436 MB of weights streamed per step (L2 126 MB)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "step_hbm": {"algorithmic_bytes": step_bytes, "achieved_gbs": round(step_ach, 1),
                     "frac": round(step_ach / hbm, 4), "peak_gbs": hbm, "peak_kind": peak_kind},
        "roofline": roof,
        "stages_us": {k: round(v * 1e3, 2) for k, v in stage_ms.items()},
        "clocks": clocks,
        "e2e": {"value": round(e2e_value, 1), "unit": "tok/s", "h2d_bytes_per_step": x.numel() * x.element_size(),
                "d2h_bytes_per_step": y.numel() * y.element_size(),
                "mode": "x and y in pinned host memory, read and written by the kernels (llama_device_ptr_of_host)",
                "with_copy_calls": {"value": round(tokens / (e2e_copy_ms / 1e3), 1), "unit": "tok/s"}},
        "gpu_launches": args.steps * n_launch,
        "launch": "one CUDA graph per step (llama_block_decode_devpos captured once)",
    }
    if args.extra and rank == 0:
        out["extra"] = extra_measurements(ddb, dims, wts, device, hbm, bf16_peak, peak_kind)
        del wts
        out["extra"]["llama31_70b"] = extra_70b(ddb, device, hbm, bf16_peak, peak_kind)
        st = stack_measurements(device)
        out["extra"]["stack_8b_32_layers"] = {k: st[k] for k in ("workload", "decode", "prefill", "clocks")}
    return out


def run_prefill(args, rank, world, device):
    """The 8B-shaped causal prefill block (batch 1, T = --tokens): TFLOP/s against the
    measured bf16 peak.  One step = one prefill of the whole block."""
    import dense_decoder_block_gb300 as ddb
    ddb.lib()
    dims = workloads.LLAMA3_8B
    T = args.tokens
    wts = workloads.make_weights(dims, weight_std=0.02)
    inp = workloads.make_block_inputs(dims, 1, T, max_seq=T, weights=wts, poison_tail=False)
    w = {k: v.to(device) for k, v in inp.weights.items()}
    g = {k: v.to(device) for k, v in inp.gains.items()}
    blk = ddb.LlamaBlock(dims, w, g, T)
    kv = ddb.KVCache(inp.k_cache.to(device), inp.v_cache.to(device))
    x = inp.x.to(device)
    y = torch.empty_like(x)
    ws = blk.workspace(1, T)
    stream = torch.cuda.current_stream(device)
    ms = time_region(lambda: blk.prefill(x, kv, y, ws), args.steps, args.warmup, stream)
    assert blk.poll_error() == 0
    n_launch = blk_launches(blk)
    stage_ms = stage_profile(blk, lambda st: blk.prefill(x, kv, y, ws, st), device, max(3, args.steps))
    _, bf16_peak, _, peak_kind = peaks()
    fl = prefill_flops(dims, 1, T)
    tf = fl / (ms / 1e3) / 1e12
    return {"metric": METRIC, "value": round(T * world / (ms / 1e3), 1), "unit": "tok/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,0.02) weights, N(0,1) x)",
            "config": {"workload": f"Llama-3 8B-shaped causal prefill block, batch 1, T={T}", "tokens": T},
            "tflops": round(tf, 1), "frac_of_bf16_peak": round(tf / bf16_peak, 4), "peak_kind": peak_kind,
            "stages_us": {k: round(v * 1e3, 2) for k, v in stage_ms.items()},
            "stage_tflops": {k: round(v / (stage_ms[k] / 1e3) / 1e12, 1)
                             for k, v in prefill_stage_flops(dims, 1, T).items()},
            "gpu_launches": args.steps * n_launch}


def run_stack(args, rank, world, device):
    """The 8B-shaped decoder stack: 32 blocks, token embedding, final RMSNorm + LM head
    + greedy choice; batch 32, a 1024-token prefill, then 256 decode steps that feed
    each chosen id back (one step = one captured graph replay).  `value` is the
    decode throughput; the prefill is reported beside it."""
    r = stack_measurements(device)
    steps, B = r["decode_steps"], r["batch"]
    return {"metric": METRIC, "value": round(r["decode"]["tok_s"] * world, 1), "unit": "tok/s", "n_gpus": world,
            "steps": steps, "warmup": 3, "ms_per_step": round(r["decode"]["us_per_step"] / 1e3, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,0.02) weights drawn on the device, uniform token ids)",
            "config": {"workload": r["workload"], "layers": r["layers"], "batch": B,
                       "prefill_tokens": r["prefill_tokens"], "decode_steps": steps,
                       "l2": "inputs larger than L2: 15.9 GB of weights per decode step"},
            "decode": r["decode"], "prefill": r["prefill"], "clocks": r["clocks"],
            "gpu_launches": r["gpu_launches"],
            "launch": "one CUDA graph per decode step (embedding, 32 blocks, head, position update)"}


def stack_measurements(device):
    """Config 5 measured: build the stack, time its prefill and its greedy decode steps."""
    import dense_decoder_block_gb300 as ddb
    from dense_decoder_block_gb300.stack import LlamaStack
    ddb.lib()
    cfg = workloads.STACK_8B
    dims, L, B, T, steps, V = cfg["dims"], cfg["n_layers"], cfg["batch"], cfg["prefill_tokens"], \
        cfg["decode_steps"], cfg["vocab"]
    std = cfg["weight_std"]
    max_seq = T + steps

    def draw(shape, seed):
        gen = torch.Generator(device=device)
        gen.manual_seed(seed)
        return torch.randn(shape, generator=gen, device=device).mul_(std).to(torch.bfloat16)

    shapes = dims.weight_shapes()
    layers = []
    for l in range(L):
        w = {name: draw(shapes[name], 1000 + 16 * l + i) for i, name in enumerate(workloads.WEIGHT_NAMES)}
        g = {name: torch.ones(dims.d_model, dtype=torch.bfloat16, device=device) for name in workloads.GAIN_NAMES}
        layers.append((w, g))
    w_embed = draw((V, dims.d_model), 7)
    w_out = draw((V, dims.d_model), 8)
    g_final = torch.ones(dims.d_model, dtype=torch.bfloat16, device=device)
    st = LlamaStack(dims, layers, w_embed, g_final, w_out, batch=B, max_seq=max_seq, prefill_tokens=T)
    ids = workloads.make_token_ids(B, T, V, seed=9).to(device)
    stream = torch.cuda.current_stream(device)

    # prefill: warm-up once, then time a few
    n_pre = 3
    pre_ms = time_region(lambda: st.prefill(ids), n_pre, 1, stream)
    n_pre_launch = blk_launches(st.blocks[0])
    assert st.poll_error() == 0 and int(st.err.item()) == 0
    pre_flops = L * prefill_flops(dims, B, T) + 2 * B * dims.d_model * V

    # decode: capture one step, replay `steps` times after a fresh prefill
    side = torch.cuda.Stream(device)
    side.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        st.decode_step(side)                   # warm-up outside the capture
        torch.cuda.synchronize(device)
        with torch.cuda.graph(graph, stream=side):
            st.decode_step(side)
    torch.cuda.synchronize(device)
    n_dec = blk_launches(st.blocks[0])
    st.prefill(ids)
    torch.cuda.synchronize(device)
    for _ in range(3):                         # warm-up replays, then restart from the prefill
        graph.replay()
    st.prefill(ids)
    torch.cuda.synchronize(device)
    sampler = ClockSampler(device.index or 0)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with sampler:
        a.record(stream)
        for _ in range(steps):
            graph.replay()
        b.record(stream)
        torch.cuda.synchronize(device)
    dec_ms = a.elapsed_time(b)
    assert st.poll_error() == 0 and int(st.err.item()) == 0
    assert int(st.pos.item()) == T + steps
    ids_last = st.ids.cpu()
    assert int(ids_last.min()) >= 0 and int(ids_last.max()) < V
    # the prefill is a long step (about half a second of tensor-core work): sustained bf16 peak
    hbm, _, bf16_sustained, peak_kind = peaks()
    bf16_peak = bf16_sustained if bf16_sustained > 0 else peaks()[1]
    step_bytes = [L * decode_step_bytes(dims, B, T + k) + 2 * V * dims.d_model + 2 * B * dims.d_model
                  for k in range(steps)]
    dec_bytes = sum(step_bytes)
    tok_s = B * steps / (dec_ms / 1e3)
    res = {"workload": f"Llama-3 8B-shaped stack: {L} blocks + embedding + LM head (V={V}), batch {B}, "
                       f"{T}-token prefill then {steps} greedy decode steps",
           "layers": L, "batch": B, "prefill_tokens": T, "decode_steps": steps,
           "decode": {"tok_s": round(tok_s, 1), "us_per_step": round(dec_ms / steps * 1e3, 1),
                      "hbm_frac": round(dec_bytes / (dec_ms / 1e3) / 1e9 / hbm, 4),
                      "algorithmic_bytes_per_step": round(dec_bytes / steps), "peak_gbs": hbm},
           "prefill": {"ms": round(pre_ms, 2), "tok_s": round(B * T / (pre_ms / 1e3), 1),
                       "tflops": round(pre_flops / (pre_ms / 1e3) / 1e12, 1),
                       "frac_of_bf16_peak": round(pre_flops / (pre_ms / 1e3) / 1e12 / bf16_peak, 4),
                       "peak_tflops": bf16_peak, "peak_kind": peak_kind + " (sustained)"},
           "clocks": sampler.summary(),
           "gpu_launches": steps * (2 + L * n_dec + 3) + (n_pre + 1) * (1 + L * n_pre_launch + 3)}
    del graph, st, layers, w_embed, w_out
    torch.cuda.empty_cache()
    return res


def blk_launches(blk):
    """Kernels the block's last prefill or decode call enqueued, as the library counted
    them (8B shapes: prefill 8 -- rmsnorm_1, QKV, RoPE, attention, O, rmsnorm_2,
    gate/up, down; decode 10 -- rmsnorm_1, QKV + reduction, attention + combine,
    O + reduction with rmsnorm_2, gate/up in one K-segment, down + reduction)."""
    n = blk.launch_count()
    assert n > 0
    return n


STAGES = ("rmsnorm_1", "qkv", "attention", "o_proj", "rmsnorm_2", "gate_up", "down")


def stage_profile(blk, launch, device, steps):
    """Average device time of each stage of one block step (`launch(stream)` runs
    it).  The library records CUDA events between its kernels on the launching
    stream; the step (with those event records) is captured as a graph and
    replayed, so the stages run back to back as in the timed region."""
    import dense_decoder_block_gb300 as ddb
    n = len(STAGES) + 1
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    cap = torch.cuda.Stream(device)
    for ev in evs:           # torch creates the CUDA event on first record
        ev.record(cap)
    torch.cuda.synchronize(device)
    g = torch.cuda.CUDAGraph()
    ddb.llama_block_set_stage_events(blk.h, evs)
    try:
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                launch(cap)
    finally:
        ddb.llama_block_set_stage_events(blk.h, None)
    sums = [0.0] * len(STAGES)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize(device)
    for _ in range(steps):
        g.replay()
        torch.cuda.synchronize(device)
        for i in range(len(STAGES)):
            sums[i] += evs[i].elapsed_time(evs[i + 1])
    return {name: sums[i] / steps for i, name in enumerate(STAGES)}


def time_region(fn, steps, warmup, stream):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def extra_measurements(ddb, dims, wts, device, hbm, bf16_peak, peak_kind):
    """Other batch sizes of the decode workload and the prefill workload (T = 512,
    2048, 8192), each timed on its own."""
    res = {}
    w = {k: v.to(device) for k, v in wts[0].items()}
    g = {k: v.to(device) for k, v in wts[1].items()}
    stream = torch.cuda.current_stream(device)
    for B in (1, 8):
        inp = workloads.make_block_inputs(dims, B, 1, cache_len=POS, max_seq=MAX_SEQ, weights=wts)
        blk = ddb.LlamaBlock(dims, w, g, MAX_SEQ)
        kv = ddb.KVCache(inp.k_cache.to(device), inp.v_cache.to(device))
        x = inp.x.to(device)
        y = torch.empty_like(x)
        ws = blk.workspace(B, 1)
        ms = time_region(lambda: blk.decode(x, kv, POS, y, ws), 50, 5, stream)
        by = decode_step_bytes(dims, B, POS)
        res[f"decode_b{B}"] = {"tok_s": round(B / (ms / 1e3), 1), "us_per_step": round(ms * 1e3, 2),
                               "hbm_frac": round(by / (ms / 1e3) / 1e9 / hbm, 4)}
    res["decode_b32_seqpos"] = extra_seqpos(ddb, dims, wts, device, hbm)
    for T in (512, 2048, 8192):
        inp = workloads.make_block_inputs(dims, 1, T, max_seq=T, weights=wts, poison_tail=False)
        blk = ddb.LlamaBlock(dims, w, g, T)
        kv = ddb.KVCache(inp.k_cache.to(device), inp.v_cache.to(device))
        x = inp.x.to(device)
        y = torch.empty_like(x)
        ws = blk.workspace(1, T)
        steps = 10 if T < 8192 else 3
        ms = time_region(lambda: blk.prefill(x, kv, y, ws), steps, 2, stream)
        fl = prefill_flops(dims, 1, T)
        tf = fl / (ms / 1e3) / 1e12
        # per stage, events between the kernels (a second pass; the step's own time is above)
        stage_ms = stage_profile(blk, lambda st: blk.prefill(x, kv, y, ws, st), device, steps)
        st_tf = {k: v / (stage_ms[k] / 1e3) / 1e12 for k, v in prefill_stage_flops(dims, 1, T).items()}
        res[f"prefill_t{T}"] = {"tok_s": round(T / (ms / 1e3), 1), "ms": round(ms, 3), "tflops": round(tf, 1),
                                "frac_of_bf16_peak": round(tf / bf16_peak, 4), "peak_kind": peak_kind,
                                "stages_us": {k: round(v * 1e3, 2) for k, v in stage_ms.items()},
                                "stage_tflops": {k: round(v, 1) for k, v in st_tf.items()},
                                "stage_frac_of_bf16_peak": {k: round(v / bf16_peak, 4) for k, v in st_tf.items()}}
    res["sample_b32"] = extra_sample(ddb, device, stream)
    return res


def extra_sample(ddb, device, stream):
    """The sampling head (llama_sample) on batch-32 rows of 128,256 fp32 logits:
    temperature 1 then top-p 0.9 (Meta's 8B reference setting), and top-k 50 with it."""
    gen = torch.Generator(device=device)
    gen.manual_seed(3)
    z = torch.randn(32, workloads.VOCAB, generator=gen, device=device) * 3
    u = torch.rand(32, generator=gen, device=device)
    ids = torch.empty(32, dtype=torch.int32, device=device)
    out = {}
    calls = 20
    for name, k, p in (("top_p_0.9", 0, 0.9), ("top_k_50_top_p_0.9", 50, 0.9)):
        # device time: the calls captured once in a CUDA graph and replayed (the
        # Python marshalling of an eager call takes about as long as the kernel)
        cap = torch.cuda.Stream(device)
        for _ in range(3):
            ddb.llama_sample(z, 32, workloads.VOCAB, 1.0, k, p, u, ids, stream=cap)
        torch.cuda.synchronize(device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                for _ in range(calls):
                    ddb.llama_sample(z, 32, workloads.VOCAB, 1.0, k, p, u, ids, stream=cap)
        ms = time_region(g.replay, 5, 2, stream) / calls
        eager = time_region(lambda: ddb.llama_sample(z, 32, workloads.VOCAB, 1.0, k, p, u, ids), calls, 3, stream)
        out[name] = {"us_per_call": round(ms * 1e3, 2), "us_per_eager_call": round(eager * 1e3, 2),
                     "logits_mb": round(32 * workloads.VOCAB * 4 / 1e6, 2),
                     "hbm_frac": round(32 * workloads.VOCAB * 4 / (ms / 1e3) / 1e9 / 6760.6, 4)}
    return out


def extra_seqpos(ddb, dims, wts, device, hbm):
    """Batch 32 with a position per sequence (llama_block_decode_seqpos): positions
    spread evenly over 500..1500 (mean 1000, the main line's), timed on its own."""
    B = 32
    positions = [500 + (b * 1000) // (B - 1) for b in range(B)]
    w = {k: v.to(device) for k, v in wts[0].items()}
    g = {k: v.to(device) for k, v in wts[1].items()}
    stream = torch.cuda.current_stream(device)
    max_seq = 2048
    inp = workloads.make_block_inputs(dims, B, 1, cache_len=max(positions), max_seq=max_seq, weights=wts)
    blk = ddb.LlamaBlock(dims, w, g, max_seq)
    kv = ddb.KVCache(inp.k_cache.to(device), inp.v_cache.to(device))
    x = inp.x.to(device)
    y = torch.empty_like(x)
    ws = blk.workspace(B, 1)
    pos_seq = torch.tensor(positions, dtype=torch.int32, device=device)
    ms = time_region(lambda: blk.decode_seqpos(x, kv, pos_seq, y, ws), 50, 5, stream)
    assert blk.poll_error() == 0
    by = decode_seqpos_bytes(dims, positions)
    return {"tok_s": round(B / (ms / 1e3), 1), "us_per_step": round(ms * 1e3, 2),
            "hbm_frac": round(by / (ms / 1e3) / 1e9 / hbm, 4), "algorithmic_bytes": by,
            "positions": f"{positions[0]}..{positions[-1]} (one per sequence, mean {sum(positions) / B:.0f})"}


def extra_70b(ddb, device, hbm, bf16_peak, peak_kind):
    """The 70B-shaped block: decode at batch 16 with 8192 cached positions and a
    4096-token prefill, each timed on its own (fresh seeded weights, N(0, 0.01))."""
    cfg = workloads.BLOCK_70B
    dims = cfg["dims"]
    wts = workloads.make_weights(dims, weight_std=cfg["weight_std"])
    w = {k: v.to(device) for k, v in wts[0].items()}
    g = {k: v.to(device) for k, v in wts[1].items()}
    stream = torch.cuda.current_stream(device)
    res = {}
    B, P = cfg["decode_batch"], cfg["cache_len"]
    inp = workloads.make_block_inputs(dims, B, 1, cache_len=P, max_seq=P + 8, weights=wts)
    blk = ddb.LlamaBlock(dims, w, g, P + 8)
    kv = ddb.KVCache(inp.k_cache.to(device), inp.v_cache.to(device))
    x = inp.x.to(device)
    y = torch.empty_like(x)
    ws = blk.workspace(B, 1)
    ms = time_region(lambda: blk.decode(x, kv, P, y, ws), 20, 3, stream)
    assert blk.poll_error() == 0
    by = decode_step_bytes(dims, B, P)
    res["decode_b16_pos8192"] = {"tok_s": round(B / (ms / 1e3), 1), "us_per_step": round(ms * 1e3, 2),
                                 "algorithmic_bytes": by, "hbm_frac": round(by / (ms / 1e3) / 1e9 / hbm, 4)}
    del inp, kv, x, y, ws, blk
    T = cfg["prefill_tokens"]
    inp = workloads.make_block_inputs(dims, 1, T, max_seq=T, weights=wts, poison_tail=False)
    blk = ddb.LlamaBlock(dims, w, g, T)
    kv = ddb.KVCache(inp.k_cache.to(device), inp.v_cache.to(device))
    x = inp.x.to(device)
    y = torch.empty_like(x)
    ws = blk.workspace(1, T)
    ms = time_region(lambda: blk.prefill(x, kv, y, ws), 5, 2, stream)
    assert blk.poll_error() == 0
    fl = prefill_flops(dims, 1, T)
    tf = fl / (ms / 1e3) / 1e12
    res[f"prefill_t{T}"] = {"tok_s": round(T / (ms / 1e3), 1), "ms": round(ms, 3), "tflops": round(tf, 1),
                            "frac_of_bf16_peak": round(tf / bf16_peak, 4), "peak_kind": peak_kind}
    return res


TRACE_NAMES = {1: "rmsnorm", 2: "gemm_ws", 3: "gemm_tt", 4: "reduce_qkv", 5: "reduce_resid", 6: "reduce_swiglu",
               7: "reduce_resid_norm", 8: "attn_decode", 9: "attn_combine", 10: "attn_prefill", 11: "rope",
               12: "attn_wide"}


def timeline_stages(rec, order):
    """Per-launch figures from a per-CTA trace of one step.  `order` lists the
    step's launches as (stage name, kernel id) in launch order; launches sharing an
    id are told apart by CTA index: a launch's CTA i starts before CTA i of the
    next launch of that kernel, which is several launches later."""
    rows = sorted(zip(rec["kernel"], rec["t_start"], rec["t_release"], rec["t_end"], rec["cta"]), key=lambda r: r[1])
    t0 = min(r[1] for r in rows)
    uses = {}
    for name, kid in order:
        uses.setdefault(kid, []).append(name)
    groups = {name: [] for name, _ in order}
    seen = {}
    for r in rows:   # the j-th record of a (kernel, CTA index) in time belongs to the j-th launch of that kernel
        names = uses.get(r[0])
        if not names:
            continue
        j = seen.get((r[0], r[4]), 0)
        seen[(r[0], r[4])] = j + 1
        if j < len(names):
            groups[names[j]].append(r)
    out = {}
    prev_end = None
    for name, _ in order:
        rs = groups[name]
        if not rs:
            out[name] = {"ctas": 0}
            continue
        first = min(r[1] for r in rs) - t0
        last = max(r[3] for r in rs) - t0
        rel = [r[2] - t0 for r in rs if r[2]]
        durs = sorted(r[3] - r[1] for r in rs)
        out[name] = {"ctas": len(rs), "first_start_us": round(first / 1e3, 2), "last_end_us": round(last / 1e3, 2),
                     "span_us": round((last - first) / 1e3, 2),
                     "last_release_us": round(max(rel) / 1e3, 2) if rel else None,
                     "cta_us_median": round(durs[len(durs) // 2] / 1e3, 2),
                     "start_after_previous_end_us": None if prev_end is None else round((first - prev_end) / 1e3, 2)}
        prev_end = last
    out["step_us"] = round((max(r[3] for r in rows) - t0) / 1e3, 2)
    return out


def run_timeline(args, rank, world, device):
    """One replayed decode step (the default workload: 8B block, batch 32, pos 1000)
    and one prefill of --tokens tokens (2048 by default), each traced CTA by CTA (llama_trace_begin, in the
    library's trace build): when each launch's first CTA starts, its last ends and
    its CTAs' durations -- from kernel start, not from the dependency release.  A
    traced step runs a few microseconds longer than the product build's."""
    from dense_decoder_block_gb300 import _native
    from dense_decoder_block_gb300 import build as _build
    _native.load(_build.build(trace=True))   # the trace build of the same sources
    import dense_decoder_block_gb300 as ddb
    dims = workloads.LLAMA3_8B
    B = args.batch
    wts = workloads.make_weights(dims, weight_std=0.02)
    inp = workloads.make_block_inputs(dims, B, 1, cache_len=POS, max_seq=MAX_SEQ, weights=wts)
    w = {k: v.to(device) for k, v in inp.weights.items()}
    g = {k: v.to(device) for k, v in inp.gains.items()}
    blk = ddb.LlamaBlock(dims, w, g, MAX_SEQ)
    kv = ddb.KVCache(inp.k_cache.to(device), inp.v_cache.to(device))
    x = inp.x.to(device)
    y = torch.empty_like(x)
    ws = blk.workspace(B, 1)
    pos_dev = torch.tensor([POS], dtype=torch.int32, device=device)
    cap = torch.cuda.Stream(device)
    for _ in range(args.warmup):
        blk.decode(x, kv, POS, y, ws)
    torch.cuda.synchronize(device)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            blk.decode_devpos(x, kv, pos_dev, y, ws, cap)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize(device)
    decode_order = [("rmsnorm_1", 1), ("qkv", 2), ("qkv_reduce", 4), ("attention", 8), ("attention_combine", 9),
                    ("o_proj", 2 | 1 << 8), ("o_reduce_rmsnorm_2", 7), ("gate_up", 2 | 2 << 8),
                    ("down", 2 | 1 << 8), ("down_reduce", 5)]
    steps = []
    for _ in range(max(1, min(args.steps, 5))):
        with ddb.Trace(1 << 14, device) as tr:
            graph.replay()
            torch.cuda.synchronize(device)
        steps.append(timeline_stages(tr.records(), decode_order))
    assert blk.poll_error() == 0
    best = min(steps, key=lambda st: st["step_us"])
    by = decode_step_bytes(dims, B, POS)
    hbm = peaks()[0]
    res = {"metric": "per-CTA timeline of one replayed decode step and one prefill", "workload": "timeline",
           "decode_8b_b32_pos1000": best, "decode_steps_traced": [st["step_us"] for st in steps],
           "decode_step_hbm_frac": round(by / (best["step_us"] / 1e6) / 1e9 / hbm, 4)}
    del graph, blk, kv, w
    torch.cuda.empty_cache()

    T = args.tokens
    pinp = workloads.make_block_inputs(dims, 1, T, max_seq=T, weights=wts)
    w = {k: v.to(device) for k, v in pinp.weights.items()}
    g = {k: v.to(device) for k, v in pinp.gains.items()}
    pblk = ddb.LlamaBlock(dims, w, g, T)
    pkv = ddb.KVCache(pinp.k_cache.to(device), pinp.v_cache.to(device))
    px = pinp.x.to(device)
    py = torch.empty_like(px)
    pws = pblk.workspace(1, T)
    for _ in range(args.warmup):
        pblk.prefill(px, pkv, py, pws)
    torch.cuda.synchronize(device)
    prefill_order = [("rmsnorm_1", 1), ("qkv", 3), ("rope", 11), ("attention", 10), ("o_proj", 3 | 1 << 8),
                     ("rmsnorm_2", 1), ("gate_up", 3 | 2 << 8), ("down", 3 | 1 << 8)]
    if pblk.launch_count() > len(prefill_order):   # few tokens: the down projection split, then its reduction
        prefill_order[-1] = ("down", 3 | 1 << 8 | 1 << 12)
        prefill_order.append(("down_reduce", 5))
    with ddb.Trace(1 << 16, device) as tr:
        pblk.prefill(px, pkv, py, pws)
        torch.cuda.synchronize(device)
    assert pblk.poll_error() == 0
    res[f"prefill_8b_t{T}"] = timeline_stages(tr.records(), prefill_order)
    return res


def run_survey(args, rank, world, device):
    """One call of each kernel family the default line does not time on its own, each
    after a warm-up call, for a per-kernel launch list under a profiler (every input
    is a few GB at most): the 70B-shaped decode block (batch 16, 8192 cached
    positions: two-segment gate/up, its reduction, 8 query heads per KV head), the
    LM head with the greedy choice and the sampling head (batch 32, 128,256
    logits), the embedding gather, decode with 16 query heads per KV head (the
    wide-group attention), the fp32 tiny block (CUDA-core kernels) and the 8B
    prefill at 512 tokens (split down projection and its reduction)."""
    import dense_decoder_block_gb300 as ddb
    ddb.lib()
    stream = torch.cuda.current_stream(device)
    calls = {}

    def timed(name, fn, launches=None):
        fn()
        torch.cuda.synchronize(device)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize(device)
        calls[name] = {"us": round(a.elapsed_time(b) * 1e3, 2)}
        if launches is not None:
            calls[name]["kernels"] = launches()

    def block_case(name, dims, B, T, P, dtype=torch.bfloat16, std=0.02):
        wts = workloads.make_weights(dims, dtype=dtype, weight_std=std)
        inp = workloads.make_block_inputs(dims, B, T, dtype=dtype, cache_len=P, max_seq=P + T + 8, weights=wts)
        blk = ddb.LlamaBlock(dims, {k: v.to(device) for k, v in wts[0].items()},
                             {k: v.to(device) for k, v in wts[1].items()}, P + T + 8)
        kv = ddb.KVCache(inp.k_cache.to(device), inp.v_cache.to(device))
        x = inp.x.to(device)
        y = torch.empty_like(x)
        ws = blk.workspace(B, T)
        if T == 1:
            timed(name, lambda: blk.decode(x, kv, P, y, ws), blk.launch_count)
        else:
            timed(name, lambda: blk.prefill_at(x, kv, P, y, ws), blk.launch_count)
        assert blk.poll_error() == 0

    cfg70 = workloads.BLOCK_70B
    block_case("decode_70b_b16_pos8192", cfg70["dims"], cfg70["decode_batch"], 1, cfg70["cache_len"],
               std=cfg70["weight_std"])
    block_case("decode_wide_group_16q_per_kv_b4_pos1000",
               workloads.BlockDims(d_model=2048, n_heads=16, n_kv_heads=1, head_dim=128, d_ff=4096), 4, 1, 1000)
    block_case("decode_tiny_fp32_pos16", workloads.TINY, 1, 1, 16, dtype=torch.float32)
    block_case("prefill_8b_t512", workloads.LLAMA3_8B, 1, 512, 0)

    d, V, B = 4096, workloads.VOCAB, 32
    gen = torch.Generator(device=device)
    gen.manual_seed(5)
    h = torch.randn(B, d, generator=gen, device=device).to(torch.bfloat16)
    g_f = torch.ones(d, dtype=torch.bfloat16, device=device)
    w_out = torch.randn(V, d, generator=gen, device=device).mul_(0.02).to(torch.bfloat16)
    ids = torch.empty(B, dtype=torch.int32, device=device)
    logits = torch.empty(B, V, dtype=torch.float32, device=device)
    hws = torch.empty(ddb.llama_lmhead_workspace_bytes(B, d, V), dtype=torch.uint8, device=device)
    timed("lmhead_argmax_b32", lambda: ddb.llama_lmhead_argmax(h, B, d, g_f, w_out, V, d, 1e-5, ids, logits, hws,
                                                               hws.numel()))
    u = torch.rand(B, generator=gen, device=device)
    timed("sample_b32_top_p_0.9", lambda: ddb.llama_sample(logits, B, V, 1.0, 0, 0.9, u, ids))
    tok = workloads.make_token_ids(B, 1, V, seed=3).to(device).view(-1)
    x = torch.empty(B, d, dtype=torch.bfloat16, device=device)
    timed("embed_b32", lambda: ddb.llama_embed(tok, B, w_out, V, d, x))
    return {"metric": METRIC, "workload": "kernel survey (one call of each kernel family, after a warm-up call)",
            "unit": "us per call", "calls": calls}


# ----------------------------------------------------------------------------- oracle timing

def oracle_decode_sample(dims, wts32, seqs: int):
    """Time the oracle (fp32 arrays, bf16 rounding points emulated) on `seqs`
    sequences of the decode workload; returns (seconds, tokens)."""
    from oracle import block as ob
    from oracle.bf16 import round_bf16
    inp = workloads.make_block_inputs(dims, seqs, 1, cache_len=POS, max_seq=MAX_SEQ,
                                      weights=wts32["torch"], poison_tail=False)
    x = inp.x.float().numpy()
    kc = inp.k_cache.float().numpy()
    vc = inp.v_cache.float().numpy()
    t0 = time.perf_counter()
    ob.block_forward(x, wts32["w"], wts32["g"], dims, kc, vc, POS, round_bf16)
    return time.perf_counter() - t0, seqs


def oracle_weights32(dims):
    wts = workloads.make_weights(dims, weight_std=0.02)
    return {"torch": wts, "w": {k: v.float().numpy() for k, v in wts[0].items()},
            "g": {k: v.float().numpy() for k, v in wts[1].items()}}


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count()


def cpu_baseline_line(dims, seqs=4, min_seconds=10.0, max_reps=400):
    w32 = oracle_weights32(dims)
    oracle_decode_sample(dims, w32, 1)   # warm caches / BLAS threads
    tot_s, tot_tok, reps = 0.0, 0, 0
    while reps < max_reps and (reps == 0 or tot_s < min_seconds):
        s, t = oracle_decode_sample(dims, w32, seqs)
        tot_s += s
        tot_tok += t
        reps += 1
    return {"value": round(tot_tok / tot_s, 3), "unit": "tok/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{reps} x {seqs} sequences of the batch-32 decode step at pos 1000 (fp32 NumPy oracle, "
                      f"bf16 rounding emulated), {tot_s:.1f} s of CPU time"}


def run_reference(args):
    dims = workloads.LLAMA3_8B
    w32 = oracle_weights32(dims)
    for _ in range(args.warmup):
        oracle_decode_sample(dims, w32, 1)
    t_total, tok = 0.0, 0
    for _ in range(args.steps):
        s, t = oracle_decode_sample(dims, w32, 1)
        t_total += s
        tok += t
    value = tok / t_total
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tok/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * t_total / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded N(0,0.02) weights, N(0,1) x and KV cache)",
        "config": {"workload": f"Llama-3 8B-shaped decode block, batch {args.batch}, 1000 cached positions "
                               f"(pos 1000); each reference step is one sequence of that batch",
                   "batch": args.batch, "pos": POS},
        "cpu_baseline": {"value": round(value, 3), "unit": "tok/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"{args.steps} steps x 1 sequence of the decode step, fp32 NumPy oracle"},
        "e2e": {"value": round(value, 3), "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--batch", type=int, default=32)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=("decode", "prefill", "stack", "survey", "timeline"), default="decode",
                    help="decode: the 8B decode block (default); prefill: the 8B causal prefill block at --tokens; "
                         "stack: 32 blocks + embedding + LM head, prefill then greedy decode; survey: one call of "
                         "each other kernel family, for a per-kernel profile; timeline: one decode step and one "
                         "prefill traced CTA by CTA")
    ap.add_argument("--tokens", type=int, default=2048, help="prefill tokens (with --workload prefill or timeline)")
    ap.add_argument("--no-extra", dest="extra", action="store_false")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    run = {"decode": run_ours, "prefill": run_prefill, "stack": run_stack, "survey": run_survey,
           "timeline": run_timeline}[args.workload]
    out = run(args, rank, world, device)
    if rank == 0 and args.cpu_baseline and world == 1 and args.workload not in ("survey", "timeline"):
        out["cpu_baseline"] = cpu_baseline_line(workloads.LLAMA3_8B)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
