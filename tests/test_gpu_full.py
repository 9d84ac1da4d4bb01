"""The five workloads at full size, in the launch configuration the
benchmark times (needs a GB300).

The cache write is compared with the oracle over the whole cache and the
slot mapping over every token.  Attention is compared element by element
with the oracle on every query row of every workload (tiny, decode, mixed,
long-context, shared prefix on both routes; bf16 and E4M3 caches).
"""
import numpy as np
import pytest
import torch

from gpu_common import assert_close, cache_bits, ensure_library, run_gpu, run_oracle
from paged_kv_cache_16_gb300 import workloads

pytestmark = pytest.mark.gpu

# oracle outputs computed once per (workload, kv dtype) in this module
_ORACLE_OUT = {}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_library()


def oracle_output(key, batch):
    if key not in _ORACLE_OUT:
        _ORACLE_OUT[key] = run_oracle(batch)[3]
    return _ORACLE_OUT[key]


def check_full(key, batch):
    g = run_gpu(batch)
    assert g.bits == 0, f"device error bits {g.bits:#x}"
    kc, vc, slots, out = run_oracle(batch)     # every token
    _ORACLE_OUT[key] = out
    assert batch.num_tokens > 0
    assert np.array_equal(g.slots.cpu().numpy(), slots)
    assert np.array_equal(cache_bits(g.key_cache), kc)
    assert np.array_equal(cache_bits(g.value_cache), vc)
    return assert_close(g.out, out, None, batch.name)


MAKERS = {
    "decode": lambda kv: workloads.decode(device="cuda", pool_device="cuda", kv_cache_dtype=kv),
    "mixed": lambda kv: workloads.mixed(device="cuda", pool_device="cuda", kv_cache_dtype=kv),
    "long": lambda kv: workloads.long_context(device="cuda", pool_device="cuda", kv_cache_dtype=kv),
    "cascade": lambda kv: workloads.cascade(device="cuda", pool_device="cuda", kv_cache_dtype=kv),
    "cascade-off": lambda kv: workloads.cascade(device="cuda", pool_device="cuda", use_cascade=False,
                                                kv_cache_dtype=kv),
}


@pytest.mark.parametrize("reading", ["1A", "1B"])
def test_full_tiny(reading):
    check_full(("tiny", reading), workloads.tiny(reading))


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_full_decode(kv):
    check_full(("decode", kv), MAKERS["decode"](kv))


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_full_mixed(kv):
    check_full(("mixed", kv), MAKERS["mixed"](kv))


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_full_long(kv):
    check_full(("long", kv), MAKERS["long"](kv))


@pytest.mark.parametrize("name", ["cascade", "cascade-off"])
def test_full_cascade(name):
    check_full((name, "bf16"), MAKERS[name]("bf16"))


@pytest.mark.parametrize("maker,kv", [("decode", "bf16"), ("decode", "fp8"), ("mixed", "bf16"), ("mixed", "fp8"),
                                      ("cascade", "bf16")])
def test_full_bench_path(maker, kv):
    """The benchmark's own path at full size: fused write + attention in the
    library's graph executor, host memory to host memory (page-locked input
    image in, output back).  Output and caches equal the eager separate path
    bit for bit, and every row is within tolerance of the oracle."""
    from paged_kv_cache_16_gb300.step import NativeGraphStep
    batch = MAKERS[maker](kv)
    ref = run_gpu(batch)
    assert ref.bits == 0
    info = ref.step.plan.info()
    dev = torch.device("cuda")
    kc = batch.key_cache.to(dev, copy=True)
    vc = batch.value_cache.to(dev, copy=True)
    ns = NativeGraphStep(num_heads_q=batch.num_heads_q, num_heads_kv=batch.num_heads_kv, head_dim=batch.head_dim,
                         num_blocks=batch.num_blocks, max_blocks_per_req=batch.block_table.shape[1],
                         softmax_scale=batch.softmax_scale, max_tokens=batch.num_tokens, max_reqs=batch.num_reqs,
                         max_extend_tiles=info["num_extend_tiles"], max_dequant_blocks=info["num_dequant_blocks"],
                         max_partial_slots=max(info["num_partial_slots"], 1), kv_cache_dtype=batch.kv_cache_dtype,
                         k_scale=batch.k_scale, v_scale=batch.v_scale, key_cache=kc, value_cache=vc, device=dev,
                         fused=True, host_io=True)
    out = ns.run(batch, batch.q, batch.key, batch.value).clone()
    torch.cuda.synchronize()
    assert ns.check_errors() == 0
    assert torch.equal(out, ref.out.cpu()), "graph executor output differs from the eager path"
    assert torch.equal(kc, ref.key_cache) and torch.equal(vc, ref.value_cache)
    assert torch.equal(ns.slot_mapping[:batch.num_tokens], ref.slots)
    assert_close(out, oracle_output((maker, kv), batch), None, batch.name)
    ns.destroy()
