"""FP8 (E4M3) KV caches: the CUDA path against the oracle (needs a GB300).

The quantising write must match the oracle's codes bit for bit over the
whole cache; attention over E4M3 caches (native E4M3 decode, bf16 copies
for the tensor-core tiles) must match the oracle's attention over the
dequantised values within the same tolerance as bf16 caches.
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


def check(batch, rows=None, what="", num_sms=0):
    g = run_gpu(batch, num_sms=num_sms)
    kc, vc, slots, out = run_oracle(batch, rows=rows)
    assert g.bits == 0, f"device error bits {g.bits:#x}"
    assert np.array_equal(g.slots.cpu().numpy(), slots)
    assert np.array_equal(cache_bits(g.key_cache), kc), "key codes differ"
    assert np.array_equal(cache_bits(g.value_cache), vc), "value codes differ"
    assert_close(g.out, out, rows, what or batch.name)
    return g


def test_fp8_write_codes_bitexact():
    """Quantising write of ordinary, tiny, huge and NaN inputs, K and V with
    different scales, a random slot permutation with skipped tokens."""
    rng = np.random.default_rng(40)
    nb, hkv, d, T = 40, 8, 128, 200
    key = torch.randn(T, hkv, d) * 3
    val = torch.randn(T, hkv, d)
    key[0, 0, :8] = torch.tensor([1e6, -1e6, 1e-7, -3e-5, 0.0, -0.0, float("nan"), 448.5])
    key = key.to(torch.bfloat16)
    val = val.to(torch.bfloat16)
    kc = torch.zeros(nb, 16, hkv, d, dtype=torch.uint8)
    vc = torch.zeros_like(kc)
    slots = rng.permutation(nb * 16)[:T].astype(np.int64)
    slots[rng.choice(T, 11, replace=False)] = -1
    slots[0] = 3
    okc, ovc = kc.numpy().copy(), vc.numpy().copy()
    assert default_oracle().write_kv_fp8(bf16_bits(key), bf16_bits(val), slots, okc, ovc, 0.0173, 0.0021) == 0
    dev = torch.device("cuda")
    gkc, gvc = kc.to(dev), vc.to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    binding.pa_write_kv_fp8(key.to(dev), val.to(dev), torch.as_tensor(slots, device=dev), gkc, gvc, 0.0173,
                            0.0021, err)
    torch.cuda.synchronize()
    assert binding.pa_check_device_errors(err) == 0
    assert np.array_equal(gkc.cpu().numpy(), okc) and np.array_equal(gvc.cpu().numpy(), ovc)


def test_fp8_decode_small():
    check(workloads.decode(batch=16, lo=1, hi=700, num_blocks=1200, seed=41, kv_cache_dtype="fp8"))


def test_fp8_decode_nan_poison():
    check(workloads.decode(batch=12, lo=1, hi=300, num_blocks=400, seed=42, poison="nan", kv_cache_dtype="fp8"))


@pytest.mark.parametrize("num_sms", [1, 7, 40, 152, 400])
def test_fp8_partition_count(num_sms):
    """Split-KV cuts at every granularity: page runs of odd and even length
    that end inside a request, lone last blocks, single-block runs."""
    check(workloads.decode(batch=12, lo=1, hi=300, num_blocks=400, seed=46, kv_cache_dtype="fp8"),
          what=f"num_sms={num_sms}", num_sms=num_sms)


def test_fp8_mixed_small():
    check(workloads.mixed(n_decode=24, n_shared=4, shared_tokens=64, lo=65, hi=900, chunk=300,
                          chunk_b_cached=500, seed=43, kv_cache_dtype="fp8"))


@pytest.mark.parametrize("use_cascade", [True, False])
def test_fp8_cascade_small(use_cascade):
    check(workloads.cascade(batch=24, prefix_tokens=1024, lo=1, hi=300, num_blocks=900, seed=44,
                            use_cascade=use_cascade, kv_cache_dtype="fp8"))


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (16, 4), (64, 4), (4, 1), (32, 16), (48, 3), (28, 4), (40, 8),
                                     (32, 1)])
def test_fp8_head_shapes(hq, hkv):
    q_lens = [1, 1, 37, 1, 129, 3, 1]
    seq = [1, 77, 37, 300, 400, 19, 64]
    check(make_batch(name=f"fp8-{hq}-{hkv}", num_heads_q=hq, num_heads_kv=hkv, head_dim=128, q_lens=q_lens,
                     seq_lens=seq, num_blocks=120, seed=hq + hkv, kv_cache_dtype="fp8", k_scale=0.03,
                     v_scale=0.007))


def test_fp8_block_permutation_bitwise():
    from test_gpu_invariants import replace_blocks
    b = workloads.mixed(n_decode=20, n_shared=4, shared_tokens=64, lo=65, hi=700, chunk=200, chunk_b_cached=300,
                        seed=45, kv_cache_dtype="fp8")
    a = run_gpu(b)
    c = run_gpu(replace_blocks(b, 7))
    assert a.bits == 0 and c.bits == 0
    assert torch.equal(a.out, c.out)


def test_fp8_head_dim_64_unsupported():
    b = workloads.tiny("1A")
    st = binding.pa_plan_status(num_heads_q=4, num_heads_kv=2, head_dim=64, num_blocks=b.num_blocks,
                                query_start_loc=b.query_start_loc, seq_lens=b.seq_lens,
                                num_computed_tokens=b.num_computed, block_table_host=b.block_table,
                                softmax_scale=0.125, num_sms=152, kv_cache_dtype=binding.PA_KV_FP8_E4M3,
                                k_scale=0.1, v_scale=0.1)
    assert st == binding.PA_ERR_UNSUPPORTED
