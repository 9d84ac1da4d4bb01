#!/usr/bin/env python
"""Benchmark of one paged-KV engine step on GB300.

A step is one pass of the whole hot path over one batch: pa_plan (host),
pa_slot_mapping, pa_write_kv and pa_attention (split-KV decode, tensor-core
extend / shared-prefix tiles, partial merge).  The default workload is the
decode-only Llama-3-8B-shaped layer (64 requests, seq_len U[512, 4096],
Hq=32, Hkv=8, D=128); ``--workload`` selects another of the five.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the fp64 CPU
oracle on the host cores instead (bounded samples of the same workload).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
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

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_16_gb300 import binding, build, workloads  # noqa: E402
from paged_kv_cache_16_gb300.step import DeviceStep, GraphStep, NativeGraphStep  # noqa: E402
from paged_kv_cache_16_gb300.workloads import bf16_bits  # noqa: E402

METRIC = "paged-attn step tokens/s; decode KV GB/s & prefill TFLOPS as % GB300 roofline"
L2_FLUSH_BYTES = 256 << 20

WORKLOADS = {
    "decode": ("decode-only Llama-3-8B-shaped layer: 64 requests x 1 token, seq_len U[512,4096], "
               "Hq=32 Hkv=8 D=128 bf16, block_size 16, 20000-block permuted pool",
               lambda seed, dev, kv: workloads.decode(seed=seed, device=dev, pool_device=dev, kv_cache_dtype=kv)),
    "tiny": ("tiny mixed step (reading 1B): Hq=4 Hkv=2 D=64, 2 decodes + 8-token chunk over 9 cached + "
             "33-token prefill, 64-block pool",
             lambda seed, dev, kv: workloads.tiny("1B", seed=seed, device=dev)),
    "mixed": ("mixed continuous-batching step: 256 decodes seq_len U[1024,8192] (32 share a 1024-token "
              "prefix) + 2048-token chunk from 0 + 2048-token chunk over 4096 cached; Hq=32 Hkv=8 D=128",
              lambda seed, dev, kv: workloads.mixed(seed=seed, device=dev, pool_device=dev, kv_cache_dtype=kv)),
    "prefill": ("the two chunked-prefill requests of the mixed step alone: a 2048-token chunk from 0 and a "
                "2048-token chunk over 4096 cached tokens; Hq=32 Hkv=8 D=128",
                lambda seed, dev, kv: workloads.mixed(seed=seed, n_decode=0, n_shared=0, device=dev, pool_device=dev,
                                                        kv_cache_dtype=kv)),
    "long": ("long-context decode, 70B-shaped layer: 8 requests x 131072 tokens, Hq=64 Hkv=8 D=128",
             lambda seed, dev, kv: workloads.long_context(seed=seed, device=dev, pool_device=dev, kv_cache_dtype=kv)),
    "cascade": ("cascade shared-prefix decode: 128 decodes over a 4096-token common prefix "
                "(num_common_prefix_blocks=256) + private suffixes U[64,1024]; Hq=32 Hkv=8 D=128",
                lambda seed, dev, kv: workloads.cascade(seed=seed, device=dev, pool_device=dev, kv_cache_dtype=kv)),
    "verify": ("speculative-decoding verify step: 64 requests x 4 query tokens (1 + 3 drafts), seq_len "
               "U[512,4096], Hq=32 Hkv=8 D=128 (rows of 2..8 tokens run on the split-KV decode kernel)",
               lambda seed, dev, kv: workloads.verify(seed=seed, device=dev, pool_device=dev, kv_cache_dtype=kv)),
    "cascade-off": ("the cascade workload on the plain route (num_common_prefix_blocks=0)",
                    lambda seed, dev, kv: workloads.cascade(seed=seed, device=dev, pool_device=dev,
                                                            use_cascade=False, kv_cache_dtype=kv)),
}

# Per-launch DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of the
# dominant kernel from one ncu capture, valid only while the kernel source is
# unchanged (sha256 of the file).  Filled in from profiles/.
TRAFFIC = {
    # (kernel, workload, kv dtype, source sha) -> bytes per launch (fused-write variant, the one the
    # default step runs); profiles/decode_kernel_decode-workload.md, profiles/extend_kernel_prefill-workload.md,
    # profiles/decode_kernel_e4m3_decode-workload.md
    ("decode", "decode", "bf16", "92b11a045f4b2f7c"): 645_422_592,
    ("decode", "decode", "fp8", "92b11a045f4b2f7c"): 325_470_720,
    ("extend", "prefill", "bf16", "e6cbabdc09e6bede"): 74_034_176,
}
KERNEL_SOURCES = {"decode": "paged_kv_cache_16_gb300/csrc/k_decode.cu",
                  "extend": "paged_kv_cache_16_gb300/csrc/k_extend.cu"}


def source_sha(kind: str) -> str:
    with open(os.path.join(ROOT, KERNEL_SOURCES[kind]), "rb") as fh:
        return hashlib.sha256(fh.read()).hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        rows = []
        with open(self.file.name) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value: float, device) -> float:
    if world == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(world, value: float, device) -> float:
    if world == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ oracle --

def oracle_sample(batch, host, budget_s: float, seed: int = 0):
    """Time the oracle (write + attention) on a bounded sample of the workload.

    Returns (tokens, seconds, description, threads).  Requests are taken in a
    seeded random order, pass after pass over the whole batch, until the
    measured time reaches the budget (rewriting a slot is idempotent)."""
    from oracle.oracle import default as default_oracle
    orc = default_oracle()
    rng = np.random.default_rng(seed)
    order = [int(r) for r in rng.permutation(batch.num_reqs) if batch.q_lens[r] > 0]
    kc, vc = host["kc"], host["vc"]
    slots = orc.slot_mapping(batch.query_start_loc, batch.num_computed, batch.block_table, batch.block_size)
    tokens, seconds, taken = 0, 0.0, 0
    while order and seconds < budget_s:
        for r in order:
            a, b = int(batch.query_start_loc[r]), int(batch.query_start_loc[r + 1])
            rows = np.arange(a, b, dtype=np.int32)
            t0 = time.perf_counter()
            common = dict(query_start_loc=batch.query_start_loc, seq_lens=batch.seq_lens,
                          num_computed=batch.num_computed, block_table=batch.block_table, q=host["q"],
                          key_cache=kc, value_cache=vc, softmax_scale=batch.softmax_scale, rows=rows)
            if batch.kv_cache_dtype == "fp8":
                orc.write_kv_fp8(host["key"][a:b], host["value"][a:b], slots[a:b], kc, vc, batch.k_scale,
                                 batch.v_scale)
                orc.attention_fp8(k_scale=batch.k_scale, v_scale=batch.v_scale, **common)
            else:
                orc.write_kv(host["key"][a:b], host["value"][a:b], slots[a:b], kc, vc)
                orc.attention(**common)
            seconds += time.perf_counter() - t0
            tokens += b - a
            taken += 1
            if seconds >= budget_s:
                break
    full = taken // max(1, len(order))
    desc = (f"{full} full pass(es) over the {len(order)} requests + {taken - full * len(order)} more requests "
            f"({tokens} query tokens in {seconds:.1f} s), write + attention, fp64")
    return tokens, seconds, desc, orc.num_threads()


def host_copies(batch):
    def cache(t):
        return t.detach().cpu().numpy().copy() if t.dtype == torch.uint8 else np.array(bf16_bits(t))
    return {"q": bf16_bits(batch.q), "key": bf16_bits(batch.key), "value": bf16_bits(batch.value),
            "kc": cache(batch.key_cache), "vc": cache(batch.value_cache)}


# ---------------------------------------------------------------- reference --

def run_reference(args, world, rank):
    if rank != 0:
        return 0
    desc, maker = WORKLOADS[args.workload]
    batch = maker(args.seed, "cpu", args.kv_dtype)
    host = host_copies(batch)
    per_step = max(0.02, min(2.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(batch, host, per_step, seed=args.seed + 1)
    toks, secs = 0, 0.0
    sample_desc, cores = "", 1
    t_wall = time.perf_counter()
    for k in range(args.steps):
        t, s, sample_desc, cores = oracle_sample(batch, host, per_step, seed=args.seed + 2 + k)
        toks += t
        secs += s
    wall = time.perf_counter() - t_wall
    value = toks / secs if secs > 0 else 0.0
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * wall / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16 inputs, no dataset)",
        "config": {"workload": desc, "seed": args.seed},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"per step: {sample_desc}"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# --------------------------------------------------------------------- ours --

def step_desc(graph_mode: bool, fused: bool) -> str:
    body = "pa_attention_with_kv_update" if fused else "pa_slot_mapping + pa_write_kv + pa_attention"
    if graph_mode:
        body = ("pa_attention_with_kv_update_launch" if fused else
                "pa_slot_mapping + pa_write_kv + pa_attention_launch")
        return (f"pa_plan_fixed + pa_plan_copy_metadata (host) + CUDA-graph replay of pa_upload_metadata_from "
                f"+ {body}")
    return f"pa_plan (host) + {body}"


def run_ours(args, world, rank, local):
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the CUDA library has no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    build.build()
    binding.load()
    desc, maker = WORKLOADS[args.workload]
    batch = maker(args.seed + rank, dev, args.kv_dtype)
    T = batch.num_tokens
    st = DeviceStep(batch, dev)
    q, key, value = batch.q.to(dev), batch.key.to(dev), batch.value.to(dev)
    kc, vc = batch.key_cache.to(dev), batch.value_cache.to(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def flush_l2():
        # write a buffer larger than L2, then read it back: L2 ends up full of
        # clean lines of the flush buffer, so the step neither hits in L2 nor
        # pays for writing back the flush's dirty lines
        flush.fill_(1)
        flush.view(torch.int32).max()
    stream = torch.cuda.current_stream(dev)
    info = st.plan.info()

    fused = args.write == "fused"

    def one_step(plans, timing, plan=None):
        plan = plan or st.make_plan()
        if timing:
            plan.enable_timing(True)
        plans.append(plan)
        if fused:
            st.run_fused(q, key, value, kc, vc, stream, plan=plan)
        else:
            st.slot_mapping(stream)
            st.write(key, value, kc, vc, stream)
            st.attend(q, kc, vc, stream, plan=plan)

    keep = []
    for _ in range(args.warmup):
        flush_l2()
        one_step(keep, False)
    torch.cuda.synchronize(dev)
    if st.check_errors():
        raise SystemExit("device error during warm-up")
    keep.clear()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    stops = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    plans = []
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clocks:
        t_wall = time.perf_counter()
        for i in range(args.steps):
            plan = st.make_plan()              # host planning overlaps the previous GPU work
            flush_l2()                         # L2 flush between timed steps (not timed)
            starts[i].record(stream)
            one_step(plans, True, plan)
            stops[i].record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t_wall
    barrier(world)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, stops)]
    ms = sum(step_ms) / len(step_ms)
    ms_all = max_over_ranks(world, ms, dev)
    tokens_all = sum_over_ranks(world, float(T), dev)
    bits = st.check_errors()

    # per-kernel device times from the plans' events
    k_ms = [0.0] * 4
    k_n = [0] * 4
    for p in plans:
        t, n = p.kernel_times()
        for k in range(4):
            k_ms[k] += t[k]
            k_n[k] += n[k]
    # our kernels per step: the attention call's, the upload kernel, and the
    # separate slot-mapping + write launches (fused: one extend write kernel
    # when the step has extend rows)
    per_step = info["kernels_per_call"] + 1 + ((1 if info["num_extend_rows"] else 0) if fused else 2)
    launches = args.steps * per_step
    plans.clear()

    hbm, bf16, bf16_sus, peak_src = measured_peaks()
    if info["decode_kv_bytes"] and k_n[0]:
        kind = "decode"
        t_launch = k_ms[0] / k_n[0] / 1000.0
        q_out_bytes = 2 * info["num_decode_rows"] * batch.num_heads_q * batch.head_dim * 2
        algo = info["decode_kv_bytes"] + q_out_bytes
        achieved = algo / t_launch / 1e9
        sha = source_sha("decode")
        traffic = TRAFFIC.get(("decode", args.workload, args.kv_dtype, sha))
        roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                    "traffic": traffic, "kernel": "decode_kernel", "peak_source": f"{peak_src} hbm_gbs",
                    "algorithmic_bytes_per_launch": algo, "launch_ms": t_launch * 1e3}
    elif k_n[1]:
        kind = "extend"
        t_launch = k_ms[1] / k_n[1] / 1000.0
        flops = info["extend_flops"] + info["prefix_flops"]
        achieved = flops / t_launch / 1e12
        sha = source_sha("extend")
        traffic = TRAFFIC.get(("extend", args.workload, args.kv_dtype, sha))
        roofline = {"bound": "tensor", "achieved": achieved, "peak": bf16, "unit": "TFLOP/s",
                    "frac": achieved / bf16, "traffic": traffic, "kernel": "extend_kernel",
                    "peak_source": f"{peak_src} bf16_tflops (burst)", "algorithmic_flops_per_launch": flops,
                    "launch_ms": t_launch * 1e3}
    else:
        kind, roofline = "none", None
    kernels = {"decode": {"ms_per_launch": k_ms[0] / k_n[0] if k_n[0] else None, "launches": k_n[0]},
               "extend": {"ms_per_launch": k_ms[1] / k_n[1] if k_n[1] else None, "launches": k_n[1]},
               "merge": {"ms_per_launch": k_ms[2] / k_n[2] if k_n[2] else None, "launches": k_n[2]},
               "metadata_copy": {"ms_per_launch": k_ms[3] / k_n[3] if k_n[3] else None, "launches": k_n[3]}}
    if info["extend_flops"] + info["prefix_flops"] and k_n[1]:
        tf = (info["extend_flops"] + info["prefix_flops"]) / (k_ms[1] / k_n[1] / 1e3) / 1e12
        kernels["extend"]["tflops"] = tf
        kernels["extend"]["frac_of_bf16_peak"] = tf / bf16
    if info["decode_kv_bytes"] and k_n[0]:
        kernels["decode"]["gbs"] = info["decode_kv_bytes"] / (k_ms[0] / k_n[0] / 1e3) / 1e9

    # ---- the same step replayed from one CUDA graph (fixed-shape plan) ----
    # Capacities are this workload's own sizes; the eager plan and the
    # fixed-shape plan cut the work identically, so the kernels (timed per
    # launch above) are the same ones the graph replays.
    gs_args = dict(num_heads_q=batch.num_heads_q, num_heads_kv=batch.num_heads_kv, head_dim=batch.head_dim,
                   num_blocks=batch.num_blocks, max_blocks_per_req=batch.block_table.shape[1],
                   softmax_scale=batch.softmax_scale, max_tokens=max(T, 1), max_reqs=max(batch.num_reqs, 1),
                   max_extend_tiles=info["num_extend_tiles"], max_dequant_blocks=info["num_dequant_blocks"],
                   max_partial_slots=max(info["num_partial_slots"], 1), kv_cache_dtype=batch.kv_cache_dtype,
                   k_scale=batch.k_scale, v_scale=batch.v_scale, device=dev, fused=fused)
    gs = GraphStep(**gs_args)
    first = gs.make_plan(batch)
    gs.load(batch, first, q, key, value)
    gs.capture(first, kc, vc)

    def graph_step(keep_plans):
        plan = gs.make_plan(batch)
        gs.replay(plan)

    for _ in range(args.warmup):
        flush_l2()
        graph_step(keep)
    torch.cuda.synchronize(dev)
    if gs.check_errors():
        raise SystemExit("device error during graph warm-up")
    keep.clear()
    g_starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    g_stops = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as g_clocks:
        for i in range(args.steps):
            # host planning and the metadata image overlap the previous GPU
            # work (as in an engine, where the next step is planned while the
            # current one runs); the events time the replay
            gs.prepare_replay(gs.make_plan(batch))
            flush_l2()
            g_starts[i].record(stream)
            gs.launch_replay()
            g_stops[i].record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    keep.clear()
    g_ms_all = max_over_ranks(world, statistics.mean(s.elapsed_time(e) for s, e in zip(g_starts, g_stops)), dev)
    bits |= gs.check_errors()
    graph_mode = args.launch == "graph"
    modes = {"eager": {"ms_per_step": ms_all, "value": tokens_all / (ms_all / 1e3)},
             "graph": {"ms_per_step": g_ms_all, "value": tokens_all / (g_ms_all / 1e3)}}
    if graph_mode:
        ms_all, clocks = g_ms_all, g_clocks

    # ---- end to end through the C ABI with host buffers ----
    e2e_steps = max(3, min(args.steps, 200))
    e2e_times = []
    if graph_mode:
        # the step's inputs sit in a page-locked image (q, key, value and the
        # request metadata in one layout); each replay copies it in, runs the
        # step and copies the output back to page-locked memory
        gh = NativeGraphStep(**gs_args, key_cache=kc, value_cache=vc, host_io=True)
        for i in (0, 1):
            gh.fill_host_image(i, batch, batch.q, batch.key, batch.value)
        h2d = gh.host_in[0].numel()
        d2h = gh.host_out[0].numel() * 2
        R = batch.num_reqs
        for i in range(e2e_steps + 2):
            flush_l2()
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            gh.launch(R, batch.num_common_prefix_blocks)
            out_host = gh.output(T)
            if i >= 2:
                e2e_times.append(time.perf_counter() - t0)
        if not torch.equal(out_host, gs.out[:T].cpu()):
            raise SystemExit("host-to-host step differs from the device-resident replay")
        bits |= gh.check_errors()
        gh.destroy()
    else:
        pin = lambda t: t.cpu().pin_memory()  # noqa: E731
        q_h, key_h, val_h = pin(batch.q), pin(batch.key), pin(batch.value)
        meta_h = [pin(torch.as_tensor(a)) for a in (batch.query_start_loc, batch.num_computed, batch.block_table)]
        meta_d = [st.qsl, st.num_computed, st.block_table]
        out_h = torch.empty((max(T, 1), batch.num_heads_q, batch.head_dim), dtype=torch.bfloat16).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in (q_h, key_h, val_h, *meta_h))
        d2h = T * batch.num_heads_q * batch.head_dim * 2
        for i in range(e2e_steps + 2):
            flush_l2()
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            q.copy_(q_h, non_blocking=True)
            key.copy_(key_h, non_blocking=True)
            value.copy_(val_h, non_blocking=True)
            for d_, h_ in zip(meta_d, meta_h):
                d_.copy_(h_, non_blocking=True)
            plan = st.make_plan()
            if fused:
                st.run_fused(q, key, value, kc, vc, stream, plan=plan)
            else:
                st.slot_mapping(stream)
                st.write(key, value, kc, vc, stream)
                st.attend(q, kc, vc, stream, plan=plan)
            out_h[:T].copy_(st.out[:T], non_blocking=True)
            torch.cuda.synchronize(dev)
            if i >= 2:
                e2e_times.append(time.perf_counter() - t0)
            plan.destroy()
    e2e_s = max_over_ranks(world, statistics.mean(e2e_times), dev)
    e2e = {"value": tokens_all / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "ms_per_step": e2e_s * 1e3,
           "path": ("pa_graph_step (the library's graph executor, one C call: fixed plan from the host metadata, "
                    "metadata image, graph launch); the graph copies the page-locked input image to the device, "
                    "uploads the metadata, runs the step kernels and copies the output to page-locked memory; "
                    "wall clock to the output's arrival" if graph_mode else
                    "per-tensor copies from page-locked memory, host plan, eager launches, output copy back; "
                    "wall clock to the output's arrival")}

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N=1) ----
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host = host_copies(batch)
        toks, secs, sdesc, cores = oracle_sample(batch, host, args.cpu_budget, seed=args.seed)
        cpu = {"value": toks / secs, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sdesc,
               "seconds": secs}

    if rank == 0:
        line = {
            "metric": METRIC, "value": tokens_all / (ms_all / 1e3), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_all, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if args.kv_dtype == "bf16" else "bf16 q/out, e4m3 kv",
            "data": "synthetic (seeded N(0,1) bf16 q/k/v and cache pool, seeded lengths and block permutation)",
            "config": {"workload": desc, "name": args.workload, "tokens_per_step": T, "seed": args.seed,
                       "kv_cache_dtype": args.kv_dtype,
                       "l2": "flushed between timed steps (256 MiB write + read-back, outside the step events)",
                       "step": step_desc(graph_mode, fused), "write": args.write,
                       "host_plan": "made before the step's events (overlapping the previous GPU work, as an engine "
                                    "plans the next step); e2e includes it",
                       "launch": args.launch, "modes": modes,
                       "kernel_times": "eager pass, CUDA events around each launch (same kernels and work cut)",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
            "clocks": clocks.summary(), "kernels": kernels, "device_error_bits": bits,
            "wall_s_timed_loop": wall, "plan": {k: info[k] for k in ("num_decode_ctas", "num_decode_items",
                                                                     "num_extend_tiles", "num_prefix_tiles",
                                                                     "num_merge_rows", "kernels_per_call")},
        }
        print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="decode")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--kv-dtype", choices=["bf16", "fp8"], default="bf16",
                    help="KV cache element type (fp8 = E4M3 codes with per-tensor scales)")
    ap.add_argument("--launch", choices=["graph", "eager"], default="graph",
                    help="time the step as a CUDA-graph replay (fixed-shape plan) or as eager launches")
    ap.add_argument("--write", choices=["fused", "separate"], default="fused",
                    help="cache write inside the attention call (pa_attention_with_kv_update) or as its own launches")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            return run_reference(args, world, rank)
        return run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
