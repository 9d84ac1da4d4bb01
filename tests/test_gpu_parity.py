"""CUDA path against the fp64 oracle, element by element (needs a GB300).

Covers: slot mapping (bit-exact), the cache write (whole cache bit-exact),
attention on the tiny mixed step (both readings, finite and NaN poison),
shrunken versions of the decode / mixed / long / cascade workloads, the
supported head shapes, and ragged and degenerate batches.
"""
import numpy as np
import pytest
import torch

from gpu_common import assert_close, cache_bits, ensure_library, run_gpu, run_oracle
from oracle.oracle import default as default_oracle
from paged_kv_cache_16_gb300 import binding, workloads
from paged_kv_cache_16_gb300.workloads import bf16_bits, make_batch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_library()


def check_batch(batch, rows=None, num_sms=0, what=""):
    g = run_gpu(batch, num_sms=num_sms)
    kc, vc, slots, out = run_oracle(batch, rows=rows)
    assert g.bits == 0, f"device error bits {g.bits:#x}"
    if batch.num_tokens:
        assert np.array_equal(g.slots.cpu().numpy(), slots), "slot mapping differs"
    assert np.array_equal(cache_bits(g.key_cache), kc), "key cache differs after the write"
    assert np.array_equal(cache_bits(g.value_cache), vc), "value cache differs after the write"
    if batch.num_tokens:
        assert_close(g.out, out, rows, what or batch.name)
    return g


@pytest.mark.parametrize("reading", ["1A", "1B"])
@pytest.mark.parametrize("poison", ["finite", "nan"])
def test_tiny_mixed_step(reading, poison):
    check_batch(workloads.tiny(reading, poison=poison))


@pytest.mark.parametrize("seed", [1, 2])
def test_tiny_more_seeds(seed):
    check_batch(workloads.tiny("1B", seed=seed))


def test_decode_small():
    check_batch(workloads.decode(batch=16, lo=20, hi=700, num_blocks=1200, seed=3))


def test_decode_small_nan_poison():
    check_batch(workloads.decode(batch=12, lo=1, hi=300, num_blocks=400, seed=4, poison="nan"))


def test_mixed_small():
    check_batch(workloads.mixed(n_decode=24, n_shared=4, shared_tokens=64, lo=65, hi=900, chunk=300,
                                chunk_b_cached=500, seed=5))


def test_long_small():
    check_batch(workloads.long_context(batch=2, context=20000, num_blocks=2600, seed=6))


@pytest.mark.parametrize("use_cascade", [True, False])
def test_cascade_small(use_cascade):
    check_batch(workloads.cascade(batch=24, prefix_tokens=1024, lo=1, hi=300, num_blocks=900, seed=7,
                                  use_cascade=use_cascade))


def test_cascade_with_extend_rows():
    """Cascade route with chunked-prefill rows as well as decodes."""
    n = 8
    q_lens = [1] * 6 + [40, 150]
    seq = [300, 129, 513, 800, 200, 640, 300, 700]
    b = make_batch(name="cascade-mixed", num_heads_q=32, num_heads_kv=8, head_dim=128, q_lens=q_lens,
                   seq_lens=seq, num_blocks=400, seed=8, shared_prefix=[(list(range(8)), n)],
                   num_common_prefix_blocks=n)
    check_batch(b)


@pytest.mark.parametrize("hq,hkv,d", [(8, 8, 128), (16, 8, 64), (16, 4, 128), (32, 4, 64), (64, 4, 128),
                                      (4, 1, 128), (16, 1, 64), (32, 16, 128), (48, 3, 64), (6, 6, 64),
                                      (28, 4, 128), (24, 8, 64), (12, 2, 128), (40, 8, 128), (80, 8, 64),
                                      (32, 1, 128), (64, 1, 64), (128, 1, 128)])
def test_head_shapes(hq, hkv, d):
    """Group sizes 1..16 (powers of two and 3, 5, 6, 7, 10: 128 not a multiple
    of G leaves padding rows in the tiles), 32..128 (every row on the tiles),
    head dims 64/128, kv-head counts that are not a power of two and more
    than 8 kv heads (several decode head groups)."""
    q_lens = [1, 1, 37, 1, 129, 3, 1]
    seq = [1, 77, 37, 300, 400, 19, 64]
    b = make_batch(name=f"heads-{hq}-{hkv}-{d}", num_heads_q=hq, num_heads_kv=hkv, head_dim=d, q_lens=q_lens,
                   seq_lens=seq, num_blocks=120, seed=hq * 7 + hkv + d)
    check_batch(b)


@pytest.mark.parametrize("q_len,cached", [(2, 0), (31, 0), (32, 0), (33, 5), (127, 1), (128, 128), (129, 15),
                                          (200, 1000), (513, 0)])
def test_extend_ragged(q_len, cached):
    """Chunks that fill, miss or straddle 128-row and 128-key tiles."""
    b = make_batch(name="ragged", num_heads_q=32, num_heads_kv=8, head_dim=128, q_lens=[q_len, 1],
                   seq_lens=[cached + q_len, 50], num_blocks=200, seed=q_len + cached)
    check_batch(b)


def test_empty_and_idle_rows():
    """q_len = 0 requests between active ones; a batch with no tokens."""
    b = make_batch(name="idle", num_heads_q=8, num_heads_kv=2, head_dim=64, q_lens=[0, 1, 0, 20, 0],
                   seq_lens=[10, 33, 0, 40, 5], num_blocks=40, seed=9)
    check_batch(b)
    empty = make_batch(name="empty", num_heads_q=8, num_heads_kv=2, head_dim=64, q_lens=[0],
                       seq_lens=[7], num_blocks=4, seed=10)
    check_batch(empty)


def test_write_kv_slots_direct():
    """The scatter on its own: a random slot permutation with skipped (-1)
    tokens, compared with the oracle's write over the whole cache."""
    rng = np.random.default_rng(11)
    nb, hkv, d, T = 50, 8, 128, 300
    kc = torch.randn(nb, 16, hkv, d).to(torch.bfloat16)
    vc = torch.randn(nb, 16, hkv, d).to(torch.bfloat16)
    key = torch.randn(T, hkv, d).to(torch.bfloat16)
    val = torch.randn(T, hkv, d).to(torch.bfloat16)
    slots = rng.permutation(nb * 16)[:T].astype(np.int64)
    slots[rng.choice(T, 17, replace=False)] = -1
    okc, ovc = bf16_bits(kc).copy(), bf16_bits(vc).copy()
    assert default_oracle().write_kv(bf16_bits(key), bf16_bits(val), slots, okc, ovc) == 0
    dev = torch.device("cuda")
    gkc, gvc = kc.to(dev), vc.to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    binding.pa_write_kv(key.to(dev), val.to(dev), torch.as_tensor(slots, device=dev), gkc, gvc, err)
    torch.cuda.synchronize()
    assert binding.pa_check_device_errors(err) == 0
    assert np.array_equal(bf16_bits(gkc), okc) and np.array_equal(bf16_bits(gvc), ovc)


def test_write_kv_out_of_range_slot_reported():
    """A slot past the cache is skipped by the kernel's bounds check and
    reported in the error word; every other row is still written."""
    dev = torch.device("cuda")
    nb, hkv, d, T = 4, 2, 64, 5
    kc = torch.zeros(nb, 16, hkv, d, dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    key = torch.randn(T, hkv, d, device=dev).to(torch.bfloat16)
    val = torch.randn(T, hkv, d, device=dev).to(torch.bfloat16)
    slots = torch.tensor([0, 5, nb * 16, 7, 63], dtype=torch.int64, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    binding.pa_write_kv(key, val, slots, kc, vc, err)
    bits = binding.pa_check_device_errors(err)
    assert bits & binding.PA_DEVERR_SLOT_RANGE
    flat = kc.view(-1, hkv, d)
    for t, s in enumerate([0, 5, None, 7, 63]):
        if s is not None:
            assert torch.equal(flat[s], key[t])
    assert binding.pa_check_device_errors(err) == 0  # cleared by the read


@pytest.mark.parametrize("q_gain", [8.0, 40.0])
def test_extend_wide_score_range(q_gain):
    """Queries scaled up so that a row's scores span hundreds of powers of
    two: most weights underflow to zero and the running max moves many
    times along a row."""
    b = make_batch(name="wide", num_heads_q=32, num_heads_kv=8, head_dim=128, q_lens=[300, 1, 77, 2],
                   seq_lens=[700, 900, 77, 260], num_blocks=200, seed=11)
    b.q = (b.q.float() * q_gain).to(torch.bfloat16)
    check_batch(b, what=f"wide x{q_gain}")
