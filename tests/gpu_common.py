"""Shared helpers of the GPU parity tests: run a batch through the C ABI and
through the oracle, and compare."""
from __future__ import annotations

import numpy as np
import torch

from oracle.oracle import default as default_oracle
from paged_kv_cache_16_gb300 import binding, build
from paged_kv_cache_16_gb300.step import DeviceStep
from paged_kv_cache_16_gb300.workloads import Batch, bf16_bits

# attention output tolerance against the fp64 oracle (bf16 inputs)
MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def ensure_library():
    build.build()
    return binding.load()


class GpuRun:
    def __init__(self, out, key_cache, value_cache, slots, bits, step):
        self.out = out
        self.key_cache = key_cache
        self.value_cache = value_cache
        self.slots = slots
        self.bits = bits
        self.step = step


def run_gpu(batch: Batch, num_sms: int = 0, block_table=None) -> GpuRun:
    """Whole step through the C ABI on cuda:0 (caches copied, inputs untouched)."""
    dev = torch.device("cuda")
    st = DeviceStep(batch, dev, num_sms=num_sms)
    if block_table is not None:
        st.block_table = torch.as_tensor(block_table, device=dev)
    q = batch.q.to(dev)
    key = batch.key.to(dev)
    value = batch.value.to(dev)
    kc = batch.key_cache.to(dev, copy=True)
    vc = batch.value_cache.to(dev, copy=True)
    out = st.run(q, key, value, kc, vc)
    torch.cuda.synchronize()
    bits = st.check_errors()
    return GpuRun(out.clone(), kc, vc, st.slot_mapping().clone() if batch.num_tokens else None, bits, st)


def cache_bits(t: torch.Tensor) -> np.ndarray:
    """Host copy of a cache as its raw element patterns (uint16 bf16 / uint8 E4M3)."""
    return t.detach().cpu().numpy() if t.dtype == torch.uint8 else bf16_bits(t)


def run_oracle(batch: Batch, rows=None):
    """(key_cache, value_cache, slot_mapping, out) from the fp64 oracle."""
    orc = default_oracle()
    common = dict(query_start_loc=batch.query_start_loc, seq_lens=batch.seq_lens,
                  num_computed=batch.num_computed, block_table=batch.block_table, q=bf16_bits(batch.q),
                  key=bf16_bits(batch.key), value=bf16_bits(batch.value),
                  key_cache=cache_bits(batch.key_cache), value_cache=cache_bits(batch.value_cache),
                  softmax_scale=batch.softmax_scale, rows=rows)
    if batch.kv_cache_dtype == "fp8":
        return orc.step_fp8(k_scale=batch.k_scale, v_scale=batch.v_scale, **common)
    return orc.step(**common)


def attention_error(gpu_out: torch.Tensor, oracle_out: np.ndarray, rows=None):
    g = gpu_out.float().cpu().numpy().astype(np.float64)
    o = oracle_out
    if rows is not None:
        g = g[rows]
        o = o[rows]
    assert np.all(np.isfinite(g)), "non-finite attention output"
    err = np.abs(g - o)
    return float(err.max(initial=0.0)), float(err.mean()) if err.size else 0.0


def assert_close(gpu_out, oracle_out, rows=None, what=""):
    mx, mean = attention_error(gpu_out, oracle_out, rows)
    assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{what}: max-abs {mx:.3e}, mean-abs {mean:.3e}"
    return mx, mean
