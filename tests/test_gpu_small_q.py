"""Rows of 2..8 query tokens (speculative verify, "vLLM 源码完全拆解（十六）"
second walk-through: c_i > 1 draft tokens after prefill) on the split-KV
decode kernel, against the oracle (needs a GB300).

Each row is cut into units of 16 / G tokens whose (token, head) pairs fill one
MMA tile; token i of a row sees keys up to its own position.  Covered: every
group size, both head dims, ragged last units, NaN in unwritten slots,
several CTA counts (units split into partials), E4M3 caches, the cascade
route and the fused write.
"""
import numpy as np
import pytest
import torch

from gpu_common import assert_close, cache_bits, ensure_library, run_gpu, run_oracle
from paged_kv_cache_16_gb300 import binding, workloads
from paged_kv_cache_16_gb300.step import DeviceStep
from paged_kv_cache_16_gb300.workloads import make_batch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_library()


def check(batch, num_sms=0, fused=False):
    if fused:
        dev = torch.device("cuda")
        st = DeviceStep(batch, dev, num_sms=num_sms)
        kc, vc = batch.key_cache.to(dev, copy=True), batch.value_cache.to(dev, copy=True)
        out = st.run_fused(batch.q.to(dev), batch.key.to(dev), batch.value.to(dev), kc, vc).clone()
        torch.cuda.synchronize()
        bits = st.check_errors()
    else:
        g = run_gpu(batch, num_sms=num_sms)
        out, kc, vc, bits = g.out, g.key_cache, g.value_cache, g.bits
    assert bits == 0, f"device error bits {bits:#x}"
    okc, ovc, _, oout = run_oracle(batch)
    assert np.array_equal(cache_bits(kc), okc) and np.array_equal(cache_bits(vc), ovc)
    assert_close(out, oout, what=batch.name)
    return out


def verify_batch(hq, hkv, d, q_lens, seq, seed, **kw):
    return make_batch(name=f"verify-{hq}-{hkv}-{d}", num_heads_q=hq, num_heads_kv=hkv, head_dim=d, q_lens=q_lens,
                      seq_lens=seq, num_blocks=kw.pop("num_blocks", 300), seed=seed, **kw)


@pytest.mark.parametrize("hq,hkv,d", [(8, 8, 128), (16, 8, 128), (32, 8, 128), (64, 8, 128), (16, 1, 64),
                                      (32, 2, 64), (48, 3, 128)])
def test_verify_rows_all_group_sizes(hq, hkv, d):
    """q_len 2..8 next to decode rows and a 40-token chunk; G = 1..16."""
    q_lens = [2, 1, 3, 4, 5, 8, 1, 6, 7, 40]
    seq = [17, 300, 16, 33, 700, 1000, 5, 130, 64, 200]
    b = verify_batch(hq, hkv, d, q_lens, seq, seed=hq + hkv + d, poison="nan")
    info = binding.pa_plan(num_heads_q=hq, num_heads_kv=hkv, head_dim=d, num_blocks=b.num_blocks,
                           query_start_loc=b.query_start_loc, seq_lens=b.seq_lens,
                           num_computed_tokens=b.num_computed, block_table_host=b.block_table,
                           softmax_scale=b.softmax_scale, num_sms=152).info()
    assert info["num_small_q_rows"] == 7 and info["num_extend_rows"] == 1
    check(b)


@pytest.mark.parametrize("num_sms", [1, 5, 152, 600])
def test_verify_rows_split(num_sms):
    """Units cut into partials at several CTA counts (per-token merge rows)."""
    b = verify_batch(32, 8, 128, [4, 8, 3, 1], [2000, 1500, 900, 1200], seed=11, num_blocks=400)
    check(b, num_sms=num_sms)


@pytest.mark.parametrize("q_len", [2, 3, 4, 5, 8])
def test_verify_row_alone_long_context(q_len):
    """One verify row over 20k keys: the decode path spreads it over every SM."""
    b = verify_batch(32, 8, 128, [q_len], [20000], seed=q_len, num_blocks=1300)
    check(b)


def test_verify_rows_fp8():
    b = verify_batch(32, 8, 128, [2, 1, 3, 4, 5, 8, 1, 40], [17, 300, 16, 33, 700, 1000, 5, 200], seed=12,
                     poison="nan", kv_cache_dtype="fp8")
    check(b)
    check(b, num_sms=7)


def test_verify_rows_cascade():
    """Verify rows behind a shared prefix: prefix tiles + suffix units + merge."""
    n = 8
    q_lens = [1, 3, 4, 1, 2, 1]
    seq = [300, 200, 513, 140, 131, 640]
    b = make_batch(name="verify-cascade", num_heads_q=32, num_heads_kv=8, head_dim=128, q_lens=q_lens,
                   seq_lens=seq, num_blocks=300, seed=13, shared_prefix=[(list(range(6)), n)],
                   num_common_prefix_blocks=n)
    check(b)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_verify_rows_fused(kv):
    """The fused call stores the verify rows' new tokens before the decode
    kernel reads them (units of one row read each other's new keys)."""
    b = verify_batch(32, 8, 128, [2, 1, 3, 8, 5, 1], [17, 300, 16, 1000, 70, 1], seed=14, poison="nan",
                     kv_cache_dtype=kv)
    out = check(b, fused=True)
    sep = run_gpu(b)
    assert torch.equal(sep.out, out)


def test_verify_rows_deterministic_and_placement_free():
    from test_gpu_invariants import replace_blocks
    b = verify_batch(32, 8, 128, [3, 1, 8, 2], [400, 77, 900, 18], seed=15)
    a1, a2 = run_gpu(b), run_gpu(b)
    c = run_gpu(replace_blocks(b, 3))
    assert torch.equal(a1.out, a2.out) and torch.equal(a1.out, c.out)
