"""The five workloads at full size, in the launch configuration the
benchmark times (needs a GB300).

Attention is compared with the oracle on sampled query rows (all heads),
the cache write over the whole cache, the slot mapping over every token.
"""
import numpy as np
import pytest
import torch

from gpu_common import assert_close, cache_bits, ensure_library, run_gpu, run_oracle
from oracle.oracle import default as default_oracle
from paged_kv_cache_16_gb300 import workloads
from paged_kv_cache_16_gb300.workloads import bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_library()


def sample_rows(batch, n_decode=8, n_per_chunk=16, seed=0):
    rng = np.random.default_rng(seed)
    q = batch.q_lens
    rows = []
    dec = [int(batch.query_start_loc[r]) for r in range(batch.num_reqs) if q[r] == 1]
    if dec:
        lens = [int(batch.seq_lens[r]) for r in range(batch.num_reqs) if q[r] == 1]
        rows += [dec[int(np.argmax(lens))], dec[int(np.argmin(lens))]]
        rows += list(rng.choice(dec, size=min(n_decode, len(dec)), replace=False))
    for r in range(batch.num_reqs):
        if q[r] > 1:
            a, b = int(batch.query_start_loc[r]), int(batch.query_start_loc[r + 1])
            rows += [a, b - 1] + list(rng.integers(a, b, size=n_per_chunk))
    return np.array(sorted(set(int(x) for x in rows)), dtype=np.int32)


def check_full(batch, n_decode=8):
    g = run_gpu(batch)
    assert g.bits == 0, f"device error bits {g.bits:#x}"
    rows = sample_rows(batch, n_decode=n_decode)
    kc, vc, slots, out = run_oracle(batch, rows=rows)
    assert np.array_equal(g.slots.cpu().numpy(), slots)
    assert np.array_equal(cache_bits(g.key_cache), kc)
    assert np.array_equal(cache_bits(g.value_cache), vc)
    return assert_close(g.out, out, rows, batch.name)


def test_full_tiny():
    for reading in ("1A", "1B"):
        check_full(workloads.tiny(reading))


def test_full_decode():
    check_full(workloads.decode(device="cuda", pool_device="cuda"))


def test_full_mixed():
    check_full(workloads.mixed(device="cuda", pool_device="cuda"))


def test_full_long():
    check_full(workloads.long_context(device="cuda", pool_device="cuda"), n_decode=2)


@pytest.mark.parametrize("use_cascade", [True, False])
def test_full_cascade(use_cascade):
    check_full(workloads.cascade(device="cuda", pool_device="cuda", use_cascade=use_cascade))


@pytest.mark.parametrize("maker", ["decode", "long", "mixed"])
def test_full_fp8(maker):
    """The decode, long-context and mixed workloads over E4M3 caches."""
    fn = {"decode": workloads.decode, "long": workloads.long_context, "mixed": workloads.mixed}[maker]
    check_full(fn(device="cuda", pool_device="cuda", kv_cache_dtype="fp8"), n_decode=2 if maker == "long" else 8)


@pytest.mark.parametrize("maker,kv", [("decode", "bf16"), ("decode", "fp8"), ("mixed", "bf16"), ("cascade", "bf16")])
def test_full_bench_path(maker, kv):
    """The benchmark's own path at full size: fused write + attention in the
    library's graph executor, host memory to host memory (page-locked input
    image in, output back).  Output and caches equal the eager separate path
    bit for bit; sampled rows are within tolerance of the oracle."""
    from paged_kv_cache_16_gb300.step import NativeGraphStep
    fn = {"decode": workloads.decode, "mixed": workloads.mixed, "cascade": workloads.cascade}[maker]
    batch = fn(device="cuda", pool_device="cuda", kv_cache_dtype=kv) if maker != "cascade" else \
        fn(device="cuda", pool_device="cuda")
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
    rows = sample_rows(batch, n_decode=4)
    _, _, _, oout = run_oracle(batch, rows=rows)
    assert_close(out, oout, rows, batch.name)
    ns.destroy()
