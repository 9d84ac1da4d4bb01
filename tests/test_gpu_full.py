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
