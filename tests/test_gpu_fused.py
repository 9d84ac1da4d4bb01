"""pa_attention_with_kv_update (cache write fused into attention) against the
oracle and against the separate write + attention path (needs a GB300).

The fused call must leave the caches bit for bit as the oracle's write does
(decode rows are stored by the decode kernel, extend rows by one write kernel
before the tiles), report every token's slot, and give the output of the
separate path bit for bit (the decode kernel computes on the same values, only
taken from on-chip memory for the new row).
"""
import numpy as np
import pytest
import torch

from gpu_common import assert_close, cache_bits, ensure_library, run_gpu, run_oracle
from paged_kv_cache_16_gb300 import workloads
from paged_kv_cache_16_gb300.step import DeviceStep
from paged_kv_cache_16_gb300.workloads import make_batch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_library()


def run_fused(batch, num_sms=0):
    dev = torch.device("cuda")
    st = DeviceStep(batch, dev, num_sms=num_sms)
    kc = batch.key_cache.to(dev, copy=True)
    vc = batch.value_cache.to(dev, copy=True)
    out = st.run_fused(batch.q.to(dev), batch.key.to(dev), batch.value.to(dev), kc, vc).clone()
    torch.cuda.synchronize()
    return out, kc, vc, st.slots[:batch.num_tokens].clone(), st.check_errors()


def check(batch, num_sms=0):
    out, kc, vc, slots, bits = run_fused(batch, num_sms)
    assert bits == 0, f"device error bits {bits:#x}"
    okc, ovc, oslots, oout = run_oracle(batch)
    assert np.array_equal(cache_bits(kc), okc), "key cache differs from the oracle's write"
    assert np.array_equal(cache_bits(vc), ovc), "value cache differs from the oracle's write"
    if batch.num_tokens:
        assert np.array_equal(slots.cpu().numpy(), oslots), "slot mapping differs"
        assert_close(out, oout, what=batch.name)
        sep = run_gpu(batch, num_sms=num_sms)
        assert torch.equal(sep.out, out), "fused and separate paths differ"


@pytest.mark.parametrize("reading", ["1A", "1B"])
@pytest.mark.parametrize("poison", ["finite", "nan"])
def test_fused_tiny(reading, poison):
    check(workloads.tiny(reading, poison=poison))


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("num_sms", [0, 7, 400])
def test_fused_decode(kv, num_sms):
    """Decode rows split at several CTA counts: the new row's page is held by
    exactly one CTA per head group, whatever the cut."""
    check(workloads.decode(batch=16, lo=1, hi=700, num_blocks=1200, seed=21, poison="nan", kv_cache_dtype=kv),
          num_sms)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_fused_mixed(kv):
    check(workloads.mixed(n_decode=24, n_shared=4, shared_tokens=64, lo=65, hi=900, chunk=300, chunk_b_cached=500,
                          seed=22, kv_cache_dtype=kv))


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_fused_cascade(kv):
    check(workloads.cascade(batch=24, prefix_tokens=1024, lo=1, hi=300, num_blocks=900, seed=23, kv_cache_dtype=kv))


@pytest.mark.parametrize("hq,hkv,d", [(8, 8, 128), (16, 8, 64), (64, 4, 128), (32, 16, 128), (48, 3, 64)])
def test_fused_head_shapes(hq, hkv, d):
    """More than 8 kv heads (several head groups write one row each), D=64."""
    q_lens = [1, 1, 37, 1, 129, 3, 1]
    seq = [1, 77, 37, 300, 400, 19, 64]
    check(make_batch(name=f"fused-{hq}-{hkv}-{d}", num_heads_q=hq, num_heads_kv=hkv, head_dim=d, q_lens=q_lens,
                     seq_lens=seq, num_blocks=120, seed=hq + hkv + d))


@pytest.mark.parametrize("seq", [1, 15, 16, 17, 32, 33])
def test_fused_block_boundaries(seq):
    """The new token at the first, last and next slot of a block."""
    check(make_batch(name=f"edge-{seq}", num_heads_q=32, num_heads_kv=8, head_dim=128, q_lens=[1, 1],
                     seq_lens=[seq, seq + 16], num_blocks=20, seed=seq, poison="nan"))
