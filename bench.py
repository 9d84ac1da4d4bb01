#!/usr/bin/env python
"""Benchmark of one paged-KV engine step on GB300.

A step is one pass of the whole hot path over one batch: the host plan, the
cache write of the step's new K/V and attention (split-KV decode, tensor-core
extend / shared-prefix tiles, partial merge).  The default workload is the
mixed continuous-batching step (256 decode rows + two 2048-token
chunked-prefill rows, Hq=32, Hkv=8, D=128); ``--workload`` selects another.
Beside the main workload the run also measures the other configurations
(``per_config``): the tiny mixed step (both readings), the decode-only layer
(bf16 and E4M3 caches), long-context decode, the shared-prefix step on the
cascade route and on the plain route (their time ratio), the prefill half of
the mixed step alone and the mixed step over E4M3 caches.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the fp64 CPU
oracle on the host cores instead (bounded samples of the same workload).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
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
    "mixed": ("mixed continuous-batching step (token budget 8192): 256 decodes seq_len U[1024,8192] (32 share a "
              "1024-token prefix) + 2048-token chunk from 0 + 2048-token chunk over 4096 cached; Hq=32 Hkv=8 D=128 "
              "bf16, block_size 16",
              lambda seed, dev, kv: workloads.mixed(seed=seed, device=dev, pool_device=dev, kv_cache_dtype=kv)),
    "decode": ("decode-only Llama-3-8B-shaped layer: 64 requests x 1 token, seq_len U[512,4096], "
               "Hq=32 Hkv=8 D=128 bf16, block_size 16, 20000-block permuted pool",
               lambda seed, dev, kv: workloads.decode(seed=seed, device=dev, pool_device=dev, kv_cache_dtype=kv)),
    "tiny": ("tiny mixed step (reading 1B): Hq=4 Hkv=2 D=64, 2 decodes + 8-token chunk over 9 cached + "
             "33-token prefill, 64-block pool",
             lambda seed, dev, kv: workloads.tiny("1B", seed=seed, device=dev)),
    "tiny-1A": ("tiny mixed step (reading 1A): Hq=4 Hkv=2 D=64, decodes of 5 and 17 + prefills of 8 and 33 "
                "from 0, 64-block pool",
                lambda seed, dev, kv: workloads.tiny("1A", seed=seed, device=dev)),
    "prefill": ("the two chunked-prefill requests of the mixed step alone: a 2048-token chunk from 0 and a "
                "2048-token chunk over 4096 cached tokens; Hq=32 Hkv=8 D=128",
                lambda seed, dev, kv: workloads.mixed(seed=seed, n_decode=0, n_shared=0, device=dev, pool_device=dev,
                                                        kv_cache_dtype=kv)),
    "long": ("long-context decode, 70B-shaped layer: 8 requests x 131072 tokens, Hq=64 Hkv=8 D=128",
             lambda seed, dev, kv: workloads.long_context(seed=seed, device=dev, pool_device=dev, kv_cache_dtype=kv)),
    "cascade": ("cascade shared-prefix decode: 128 decodes over a 4096-token common prefix "
                "(num_common_prefix_blocks=256) + private suffixes U[64,1024]; Hq=32 Hkv=8 D=128",
                lambda seed, dev, kv: workloads.cascade(seed=seed, device=dev, pool_device=dev, kv_cache_dtype=kv)),
    "cascade-off": ("the cascade workload on the plain route (num_common_prefix_blocks=0)",
                    lambda seed, dev, kv: workloads.cascade(seed=seed, device=dev, pool_device=dev,
                                                            use_cascade=False, kv_cache_dtype=kv)),
    "verify": ("speculative-decoding verify step: 64 requests x 4 query tokens (1 + 3 drafts), seq_len "
               "U[512,4096], Hq=32 Hkv=8 D=128 (rows of 2..8 tokens run on the split-KV decode kernel)",
               lambda seed, dev, kv: workloads.verify(seed=seed, device=dev, pool_device=dev, kv_cache_dtype=kv)),
}

# The configurations measured beside the main workload: (entry, workload, kv dtype).
PER_CONFIG = [("tiny-1A", "tiny-1A", "bf16"), ("tiny-1B", "tiny", "bf16"), ("decode", "decode", "bf16"),
              ("decode-e4m3", "decode", "fp8"), ("long", "long", "bf16"), ("cascade", "cascade", "bf16"),
              ("cascade-off", "cascade-off", "bf16"), ("prefill", "prefill", "bf16"), ("mixed-e4m3", "mixed", "fp8"),
              ("long-e4m3", "long", "fp8"), ("verify", "verify", "bf16"), ("verify-e4m3", "verify", "fp8")]

# Per-launch DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of a
# kernel from one ncu capture, valid only while the kernel source is
# unchanged (sha256 prefix of the file); the summaries are under profiles/.
TRAFFIC = {
    # profiles/decode_kernel_decode-workload.md, profiles/decode_kernel_e4m3_decode-workload.md,
    # profiles/step_launches_mixed-workload.md, profiles/extend_kernel_prefill-workload.md
    ("decode", "decode", "bf16", "d98510bbbb11bb79"): 643_372_032,
    ("decode", "decode", "fp8", "d98510bbbb11bb79"): 323_800_832,
    ("decode", "mixed", "bf16", "d98510bbbb11bb79"): 4_686_585_600,
    ("extend", "prefill", "bf16", "8be8aea7e2cb901b"): 76_740_864,
    # profiles/dram_traffic_decode-and-extend_per-workload.md
    ("decode", "long", "bf16", "d98510bbbb11bb79"): 4_299_878_400,
    ("decode", "long", "fp8", "d98510bbbb11bb79"): 2_150_972_416,
    ("decode", "cascade", "bf16", "d98510bbbb11bb79"): 316_145_408,
    ("extend", "cascade", "bf16", "8be8aea7e2cb901b"): 17_895_424,
    ("decode", "cascade-off", "bf16", "d98510bbbb11bb79"): 334_178_560,
    ("decode", "verify", "bf16", "d98510bbbb11bb79"): 674_436_608,
    ("decode", "verify", "fp8", "d98510bbbb11bb79"): 341_064_704,
    ("decode", "mixed", "fp8", "d98510bbbb11bb79"): 2_336_910_080,
    ("extend", "mixed", "bf16", "8be8aea7e2cb901b"): 78_454_272,
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


# ------------------------------------------------------------------ clocks --

class NvmlClocks:
    """SM clock and throttle reasons read through NVML (read-only queries)
    every ~2 ms from a thread while the timed region runs; None if NVML
    cannot be loaded (then nvidia-smi sampling is used)."""
    REASONS = {"hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40,
               "sw_power_cap": 0x4}

    def __init__(self, gpu_index: int):
        self.lib = None
        for name in ("libnvidia-ml.so.1", "libnvidia-ml.so"):
            try:
                self.lib = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if self.lib is None or self.lib.nvmlInit_v2() != 0:
            raise OSError("NVML unavailable")
        self.handle = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(gpu_index), ctypes.byref(self.handle)) != 0:
            raise OSError("NVML device handle")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(self.lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        self.samples = []
        self.max_mhz = None
        mx = ctypes.c_uint()
        if self.lib.nvmlDeviceGetMaxClockInfo(self.handle, ctypes.c_int(1), ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        self._stop = threading.Event()
        self._thread = None

    def _read(self):
        clk = ctypes.c_uint()
        reasons = ctypes.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.handle, ctypes.c_int(1), ctypes.byref(clk)) != 0:
            return None
        if self.reasons_fn(self.handle, ctypes.byref(reasons)) != 0:
            reasons.value = 0
        return float(clk.value), int(reasons.value)

    def _run(self):
        while not self._stop.is_set():
            r = self._read()
            if r is not None:
                self.samples.append(r)
            time.sleep(0.002)

    def __enter__(self):
        self._thread = threading.Thread(target=self._run, daemon=True)
        self._thread.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        self._thread.join(timeout=5)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no samples"], "samples": 0,
                    "source": "nvml"}
        sm = [s[0] for s in self.samples]
        reasons = sorted({k for _, bits in self.samples for k, v in self.REASONS.items() if bits & v})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(self.samples), "source": "nvml, every ~2 ms during the timed steps"}


class SmiClocks:
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
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "source": "nvidia-smi -lms 50"}


def clock_sampler(gpu_index: int):
    try:
        return NvmlClocks(gpu_index)
    except (OSError, AttributeError):
        return SmiClocks(gpu_index)


# ------------------------------------------------------------ distributed --

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

def oracle_sample(batch, host, budget_s: float, seed: int = 0, threads: int | None = None):
    """Time the oracle (write + attention) on a bounded sample of the workload.

    Returns (tokens, seconds, description, threads).  Requests are taken in a
    seeded random order, pass after pass over the whole batch, until the
    measured time reaches the budget (rewriting a slot is idempotent).
    ``threads`` limits the oracle's OpenMP threads for this sample."""
    from oracle.oracle import default as default_oracle
    orc = default_oracle()
    all_threads = orc.num_threads()
    if threads is not None:
        orc.set_num_threads(threads)
    try:
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
        used = orc.num_threads()
    finally:
        orc.set_num_threads(all_threads)
    full = taken // max(1, len(order))
    desc = (f"{full} full pass(es) over the {len(order)} requests + {taken - full * len(order)} more requests "
            f"({tokens} query tokens in {seconds:.1f} s), write + attention, fp64")
    return tokens, seconds, desc, used


def host_copies(batch):
    def cache(t):
        return t.detach().cpu().numpy().copy() if t.dtype == torch.uint8 else np.array(bf16_bits(t))
    return {"q": bf16_bits(batch.q), "key": bf16_bits(batch.key), "value": bf16_bits(batch.value),
            "kc": cache(batch.key_cache), "vc": cache(batch.value_cache)}


def cpu_baseline(batch, budget_s: float, seed: int, one_core: bool = False):
    host = host_copies(batch)
    toks, secs, sdesc, cores = oracle_sample(batch, host, budget_s, seed=seed)
    out = {"value": toks / secs if secs > 0 else 0.0, "unit": "tokens/s", "cores": cores, "kind": "oracle",
           "sample": sdesc, "seconds": secs}
    if one_core:
        # the first sample rewrote the step's slots with the same values
        t1, s1, d1, c1 = oracle_sample(batch, host, budget_s, seed=seed, threads=1)
        out["one_core"] = {"value": t1 / s1 if s1 > 0 else 0.0, "unit": "tokens/s", "cores": c1, "sample": d1}
    return out


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
        "config": {"workload": desc, "name": args.workload, "seed": args.seed},
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


def unique_decode_bytes(batch, info) -> int:
    """K+V bytes of the decode rows' keys with every physical block counted
    once: per physical block, the most tokens any decode row reads from it
    (a prefix shared by several rows is one set of blocks in HBM).  On the
    cascade route the decode rows read only the keys past the prefix."""
    el = 1 if batch.kv_cache_dtype == "fp8" else 2
    row = batch.num_heads_kv * batch.head_dim * el * 2
    kb = batch.num_common_prefix_blocks * batch.block_size
    used = {}
    q = batch.q_lens
    per_unit = max(1, 16 // (batch.num_heads_q // batch.num_heads_kv))   # tokens of one decode-kernel unit
    for r in range(batch.num_reqs):
        if not 1 <= q[r] <= per_unit:
            continue   # rows of the tensor-core tiles
        L = int(batch.seq_lens[r])
        for lb in range(kb // batch.block_size, (L + batch.block_size - 1) // batch.block_size):
            n = min(batch.block_size, L - lb * batch.block_size)
            b = int(batch.block_table[r, lb])
            used[b] = max(used.get(b, 0), n)
    return sum(used.values()) * row


def flush_l2_fn(dev):
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def flush_l2():
        # write a buffer larger than L2, then read it back: L2 ends up full of
        # clean lines of the flush buffer, so the step neither hits in L2 nor
        # pays for writing back the flush's dirty lines
        flush.fill_(1)
        flush.view(torch.int32).max()
    return flush_l2


def measure(name, batch, dev, steps, warmup, fused, world=1, clocks=None, e2e_steps=0, peaks=None):
    """Graph-replayed step time (the headline), per-kernel times from an eager
    pass, rooflines, host planning time and optionally the end-to-end step
    from host memory to host memory."""
    T = batch.num_tokens
    flush_l2 = flush_l2_fn(dev)
    stream = torch.cuda.current_stream(dev)
    st = DeviceStep(batch, dev)
    q, key, value = batch.q.to(dev), batch.key.to(dev), batch.value.to(dev)
    kc, vc = batch.key_cache.to(dev), batch.value_cache.to(dev)
    info = st.plan.info()

    # ---- eager pass: per-kernel CUDA-event times (same kernels and cut) ----
    def eager_step(plan):
        if fused:
            st.run_fused(q, key, value, kc, vc, stream, plan=plan)
        else:
            st.slot_mapping(stream)
            st.write(key, value, kc, vc, stream)
            st.attend(q, kc, vc, stream, plan=plan)
    for _ in range(warmup):
        flush_l2()
        eager_step(st.make_plan())
    torch.cuda.synchronize(dev)
    if st.check_errors():
        raise SystemExit(f"{name}: device error during warm-up")
    e_starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    e_stops = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    plans = []
    for i in range(steps):
        plan = st.make_plan()
        plan.enable_timing(True)
        plans.append(plan)
        flush_l2()
        e_starts[i].record(stream)
        eager_step(plan)
        e_stops[i].record(stream)
    torch.cuda.synchronize(dev)
    eager_ms = statistics.mean(s.elapsed_time(e) for s, e in zip(e_starts, e_stops))
    k_ms, k_n = [0.0] * 4, [0] * 4
    for p in plans:
        t, n = p.kernel_times()
        for k in range(4):
            k_ms[k] += t[k]
            k_n[k] += n[k]
    plans.clear()
    bits = st.check_errors()
    kern = [k_ms[k] / k_n[k] if k_n[k] else None for k in range(4)]

    # ---- the same step replayed from one CUDA graph (fixed-shape plan) ----
    gs_args = dict(num_heads_q=batch.num_heads_q, num_heads_kv=batch.num_heads_kv, head_dim=batch.head_dim,
                   num_blocks=batch.num_blocks, max_blocks_per_req=batch.block_table.shape[1],
                   softmax_scale=batch.softmax_scale, max_tokens=max(T, 1), max_reqs=max(batch.num_reqs, 1),
                   max_extend_tiles=info["num_extend_tiles"], max_dequant_blocks=info["num_dequant_blocks"],
                   max_partial_slots=max(info["num_partial_slots"], 1), kv_cache_dtype=batch.kv_cache_dtype,
                   k_scale=batch.k_scale, v_scale=batch.v_scale, device=dev, fused=fused)
    gs = GraphStep(**gs_args)
    first = gs.make_plan(batch)
    fixed_info = first.info()
    gs.load(batch, first, q, key, value)
    gs.capture(first, kc, vc)
    for _ in range(warmup):
        flush_l2()
        gs.replay(gs.make_plan(batch))
    torch.cuda.synchronize(dev)
    if gs.check_errors():
        raise SystemExit(f"{name}: device error during graph warm-up")
    g_starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    g_stops = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    host_plan_s = []
    barrier(world)
    torch.cuda.synchronize(dev)
    ctx = clocks if clocks is not None else _NoClocks()
    with ctx:
        for i in range(steps):
            # host planning and the metadata image overlap the previous GPU
            # work (as in an engine, where the next step is planned while the
            # current one runs); the events time the replay
            t0 = time.perf_counter()
            gs.prepare_replay(gs.make_plan(batch))
            host_plan_s.append(time.perf_counter() - t0)
            flush_l2()
            g_starts[i].record(stream)
            gs.launch_replay()
            g_stops[i].record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    graph_ms = statistics.mean(s.elapsed_time(e) for s, e in zip(g_starts, g_stops))
    bits |= gs.check_errors()
    if not torch.equal(gs.out[:T], st.out[:T]):
        raise SystemExit(f"{name}: graph replay output differs from the eager step")

    # ---- rooflines of the two bounds of the step ----
    hbm, bf16, _, peak_src = peaks or measured_peaks()
    roof = {}
    if info["decode_kv_bytes"] and kern[0]:
        t_launch = kern[0] / 1e3
        q_out = 2 * info["num_decode_rows"] * batch.num_heads_q * batch.head_dim * 2
        algo = info["decode_kv_bytes"] + q_out
        uniq = unique_decode_bytes(batch, info) + q_out
        achieved = uniq / t_launch / 1e9
        roof["decode"] = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                          "traffic": TRAFFIC.get(("decode", name, batch.kv_cache_dtype, source_sha("decode"))),
                          "kernel": "decode_kernel", "peak_source": f"{peak_src} hbm_gbs (of measured)",
                          "bytes_used_for_frac": "unique: each physical block once (+ q/out)",
                          "unique_bytes_per_launch": uniq, "algorithmic_bytes_per_launch": algo,
                          "algorithmic_gbs": algo / t_launch / 1e9, "launch_ms": kern[0],
                          "sms": info["num_decode_ctas"] if info["side_by_side"] else None}
    flops = info["extend_flops"] + info["prefix_flops"]
    if flops and kern[1]:
        t_launch = kern[1] / 1e3
        achieved = flops / t_launch / 1e12
        sms = info["num_extend_ctas"]
        roof["extend"] = {"bound": "tensor", "achieved": achieved, "peak": bf16, "unit": "TFLOP/s",
                          "frac": achieved / bf16,
                          "traffic": TRAFFIC.get(("extend", name, batch.kv_cache_dtype, source_sha("extend"))),
                          "kernel": "extend_kernel", "peak_source": f"{peak_src} bf16_tflops (burst, of measured)",
                          "algorithmic_flops_per_launch": flops, "launch_ms": kern[1], "sms": sms,
                          "frac_of_its_sms": achieved / (bf16 * sms / 152.0) if sms else None}
    kernels = {"decode": kern[0], "extend": kern[1], "merge": kern[2], "metadata_upload": kern[3]}

    out = {"T": T, "graph_ms": graph_ms, "eager_ms": eager_ms, "kernels_ms": kernels, "roofline": roof,
           "bits": bits, "info": info, "fixed_info": fixed_info,
           "host_plan_ms": 1e3 * statistics.median(host_plan_s), "c_planner_ms": c_planner_ms(gs, batch),
           "launches_per_step": fixed_info["kernels_per_call"] + 1 + (1 if fused and fixed_info["num_extend_rows"]
                                                                      else 0 if fused else 2)}

    # ---- end to end through the C ABI with host buffers ----
    if e2e_steps:
        # the leading one-token and short rows (the decode stream's) come in
        # first; the chunks' rows after them, while the decode stream runs
        q_lens = np.diff(batch.query_start_loc)
        lead = int(np.argmax(q_lens > 8)) if (q_lens > 8).any() else len(q_lens)
        prefix = int(batch.query_start_loc[lead])
        staged = prefix if 0 < prefix < T and not (q_lens[lead:] <= 8).any() else 0
        gh = NativeGraphStep(**gs_args, key_cache=kc, value_cache=vc, host_io=True, decode_prefix_tokens=staged)
        for i in (0, 1):
            gh.fill_host_image(i, batch, batch.q, batch.key, batch.value)
        h2d = gh.host_in[0].numel()
        d2h = gh.host_out[0].numel() * 2
        R = batch.num_reqs
        times = []
        for i in range(e2e_steps + 2):
            flush_l2()
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            gh.launch(R, batch.num_common_prefix_blocks)
            out_host = gh.output(T)
            if i >= 2:
                times.append(time.perf_counter() - t0)
        # a staged plan's SM split (and so its decode cut and merge rounding)
        # may differ from the device-resident plan's; otherwise bit for bit
        diff = float((out_host.float() - gs.out[:T].cpu().float()).abs().max()) if T else 0.0
        if (diff > 0.05) if staged else not torch.equal(out_host, gs.out[:T].cpu()):
            raise SystemExit(f"{name}: host-to-host step differs from the device-resident replay ({diff})")
        out["bits"] |= gh.check_errors()
        gh.destroy()
        out["e2e"] = {"s": statistics.mean(times), "h2d": h2d, "d2h": d2h, "decode_prefix_tokens": staged}
    del gs, st
    return out


def c_planner_ms(gs, batch, reps=50) -> float:
    """Median time of the C planner alone (pa_plan_fixed + pa_plan_destroy)
    for this step on this host's core: the descriptor and its arrays are
    made once, outside the timing."""
    bt = batch.block_table
    mb = gs.model["max_blocks_per_req"]
    if bt.shape[1] != mb:
        padded = np.zeros((bt.shape[0], mb), dtype=np.int32)
        padded[:, :bt.shape[1]] = bt
        bt = padded
    d, keep = binding.make_desc(query_start_loc=batch.query_start_loc, seq_lens=batch.seq_lens,
                                num_computed_tokens=batch.num_computed, block_table_host=bt,
                                num_common_prefix_blocks=batch.num_common_prefix_blocks, **gs.model)
    fs = binding._fixed_shape(**gs.shape)
    lib = binding.load()
    times = []
    for _ in range(reps):
        h = ctypes.c_void_p()
        ws = ctypes.c_size_t()
        t0 = time.perf_counter()
        st = lib.pa_plan_fixed(ctypes.byref(d), ctypes.byref(fs), ctypes.byref(h), ctypes.byref(ws))
        lib.pa_plan_destroy(h.value)
        times.append(time.perf_counter() - t0)
        if st != binding.PA_OK:
            raise SystemExit(f"pa_plan_fixed failed: {st}")
    del keep
    return 1e3 * statistics.median(times)


class _NoClocks:
    def __enter__(self):
        return self

    def __exit__(self, *exc):
        return False


def per_config_entry(name, wl, kv, args, dev, peaks):
    desc, maker = WORKLOADS[wl]
    batch = maker(args.seed, dev, kv)
    steps = max(3, min(args.steps, 200))
    m = measure(wl, batch, dev, steps, args.warmup, args.write == "fused", peaks=peaks)
    dom = m["roofline"].get("decode") or m["roofline"].get("extend")
    entry = {"workload": desc, "kv_cache_dtype": kv, "tokens_per_step": m["T"],
             "value": m["T"] / (m["graph_ms"] / 1e3), "unit": "tokens/s", "ms_per_step": m["graph_ms"],
             "eager_ms_per_step": m["eager_ms"], "steps": steps, "roofline": dom, "rooflines": m["roofline"],
             "kernels_ms": m["kernels_ms"], "host_plan_ms": {"c_planner": m["c_planner_ms"],
                                                              "python_step_prep": m["host_plan_ms"]},
             "side_by_side": bool(m["fixed_info"]["side_by_side"]), "device_error_bits": m["bits"]}
    if not args.no_cpu_baseline:
        entry["cpu_baseline"] = cpu_baseline(batch, args.cpu_budget_config, args.seed,
                                             one_core=name in ("tiny-1A", "tiny-1B", "decode"))
    del batch
    torch.cuda.empty_cache()
    return entry


def run_ours(args, world, rank, local):
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the CUDA library has no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    build.build()
    binding.load()
    peaks = measured_peaks()
    fused = args.write == "fused"
    desc, maker = WORKLOADS[args.workload]
    batch = maker(args.seed + rank, dev, args.kv_dtype)
    T = batch.num_tokens
    clocks = clock_sampler(local)
    t_wall = time.perf_counter()
    m = measure(args.workload, batch, dev, args.steps, args.warmup, fused, world=world, clocks=clocks,
                e2e_steps=max(3, min(args.steps, 200)), peaks=peaks)
    wall = time.perf_counter() - t_wall
    ms_all = max_over_ranks(world, m["graph_ms"] if args.launch == "graph" else m["eager_ms"], dev)
    eager_all = max_over_ranks(world, m["eager_ms"], dev)
    graph_all = max_over_ranks(world, m["graph_ms"], dev)
    tokens_all = sum_over_ranks(world, float(T), dev)
    e2e_s = max_over_ranks(world, m["e2e"]["s"], dev)
    e2e = {"value": tokens_all / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": m["e2e"]["h2d"],
           "d2h_bytes_per_step": m["e2e"]["d2h"], "ms_per_step": e2e_s * 1e3,
           "host_plan_ms_per_step": {"c_planner": m["c_planner_ms"], "python_step_prep": m["host_plan_ms"],
                                     "what": "c_planner: pa_plan_fixed alone on one host core; python_step_prep: "
                                             "the bench's per-step plan through the Python binding plus the "
                                             "metadata image copy (not on the e2e path, which plans in C)"},
           "decode_prefix_tokens": m["e2e"]["decode_prefix_tokens"],
           "path": "pa_graph_step (the library's graph executor, one C call: fixed plan from the host metadata, "
                   "metadata image, graph launch); the graph copies the page-locked input image to the device "
                   "(with decode_prefix_tokens > 0: the decode rows and metadata first, the chunk rows after "
                   "them on a second stream, the decode stream starting in between), uploads the metadata and "
                   "runs the step kernels, which store the output rows straight into page-locked host memory "
                   "through its device mapping (d2h bytes: the output); wall clock to the output's arrival"}
    roof = m["roofline"]
    dominant = roof.get("decode") or roof.get("extend")

    cpu = None
    per_config = {}
    if rank == 0 and world == 1:
        if not args.no_cpu_baseline:
            cpu = cpu_baseline(batch, args.cpu_budget, args.seed)
        del batch
        torch.cuda.empty_cache()
        if not args.no_per_config:
            for name, wl, kv in PER_CONFIG:
                if wl == args.workload and kv == args.kv_dtype:
                    continue
                per_config[name] = per_config_entry(name, wl, kv, args, dev, peaks)
            if "cascade" in per_config and "cascade-off" in per_config:
                per_config["cascade"]["plain_over_cascade_time"] = (per_config["cascade-off"]["ms_per_step"] /
                                                                    per_config["cascade"]["ms_per_step"])

    if rank == 0:
        info = m["info"]
        line = {
            "metric": METRIC, "value": tokens_all / (ms_all / 1e3), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_all, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if args.kv_dtype == "bf16" else "bf16 q/out, e4m3 kv",
            "data": "synthetic (seeded N(0,1) bf16 q/k/v and cache pool, seeded lengths and block permutation)",
            "config": {"workload": desc, "name": args.workload, "tokens_per_step": T, "seed": args.seed,
                       "kv_cache_dtype": args.kv_dtype,
                       "l2": "flushed between timed steps (256 MiB write + read-back, outside the step events)",
                       "step": step_desc(args.launch == "graph", fused), "write": args.write,
                       "host_plan": "made before the step's events (overlapping the previous GPU work, as an engine "
                                    "plans the next step); e2e includes it",
                       "launch": args.launch,
                       "modes": {"eager": {"ms_per_step": eager_all, "value": tokens_all / (eager_all / 1e3)},
                                 "graph": {"ms_per_step": graph_all, "value": tokens_all / (graph_all / 1e3)}},
                       "kernel_times": "eager pass, CUDA events around each launch (same kernels and work cut)",
                       "side_by_side": bool(m["fixed_info"]["side_by_side"]),
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": dominant, "roofline_extend": roof.get("extend"), "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": args.steps * m["launches_per_step"], "clocks": clocks.summary(),
            "kernels_ms": m["kernels_ms"], "device_error_bits": m["bits"], "wall_s_main_workload": wall,
            "plan": {k: info[k] for k in ("num_decode_ctas", "num_extend_ctas", "num_decode_items", "num_extend_tiles",
                                          "num_prefix_tiles", "num_merge_rows", "kernels_per_call", "side_by_side")},
            "per_config": per_config or None,
        }
        print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="mixed")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--kv-dtype", choices=["bf16", "fp8"], default="bf16",
                    help="KV cache element type (fp8 = E4M3 codes with per-tensor scales)")
    ap.add_argument("--launch", choices=["graph", "eager"], default="graph",
                    help="report the step as a CUDA-graph replay (fixed-shape plan) or as eager launches")
    ap.add_argument("--write", choices=["fused", "separate"], default="fused",
                    help="cache write inside the attention call (pa_attention_with_kv_update) or as its own launches")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--cpu-budget-config", type=float, default=2.0,
                    help="seconds of oracle time for each per_config entry's cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="measure the main workload only")
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
