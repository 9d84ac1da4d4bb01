"""Properties of the CUDA path that the pages fix (needs a GB300).

* physical block placement changes addressing only: bitwise-equal output;
* repeated runs are bitwise identical (no floating-point atomics);
* the split-KV partition count does not change the result beyond rounding;
* the cascade route equals the plain route on identical inputs;
* a decode step equals the last row of a prefill over the same context;
* a prefix-hit chunk equals recomputing the whole prompt;
* device-side bounds checks report a bad block id instead of faulting.
"""
import numpy as np
import pytest
import torch

from gpu_common import MAX_ABS, assert_close, attention_error, ensure_library, run_gpu, run_oracle
from paged_kv_cache_16_gb300 import binding, workloads
from paged_kv_cache_16_gb300.step import DeviceStep
from paged_kv_cache_16_gb300.workloads import make_batch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_library()


def replace_blocks(batch, seed):
    """The same logical batch with every physical block moved to a new id."""
    perm = np.random.default_rng(seed).permutation(batch.num_blocks)
    kc = torch.empty_like(batch.key_cache)
    vc = torch.empty_like(batch.value_cache)
    kc[torch.as_tensor(perm)] = batch.key_cache
    vc[torch.as_tensor(perm)] = batch.value_cache
    bt = perm[batch.block_table].astype(np.int32)
    import copy
    b2 = copy.copy(batch)
    b2.key_cache, b2.value_cache, b2.block_table = kc, vc, bt
    return b2


@pytest.mark.parametrize("maker", ["tiny", "mixed", "cascade"])
def test_block_permutation_bitwise(maker):
    if maker == "tiny":
        b = workloads.tiny("1B")
    elif maker == "mixed":
        b = workloads.mixed(n_decode=20, n_shared=4, shared_tokens=64, lo=65, hi=700, chunk=200,
                            chunk_b_cached=300, seed=12)
    else:
        b = workloads.cascade(batch=16, prefix_tokens=512, lo=1, hi=200, num_blocks=400, seed=13)
    a = run_gpu(b)
    c = run_gpu(replace_blocks(b, 99))
    assert a.bits == 0 and c.bits == 0
    assert torch.equal(a.out, c.out)


def test_repeat_bitwise():
    b = workloads.mixed(n_decode=20, n_shared=4, shared_tokens=64, lo=65, hi=700, chunk=200,
                        chunk_b_cached=300, seed=14)
    a = run_gpu(b)
    c = run_gpu(b)
    assert torch.equal(a.out, c.out)


@pytest.mark.parametrize("num_sms", [1, 7, 152, 400])
def test_partition_count_invariance(num_sms):
    """Different persistent-grid sizes cut the keys into different
    partitions; every result stays within tolerance of the oracle."""
    b = workloads.decode(batch=10, lo=1, hi=2000, num_blocks=1400, seed=15)
    g = run_gpu(b, num_sms=num_sms)
    assert g.bits == 0
    _, _, _, out = run_oracle(b)
    assert_close(g.out, out, what=f"num_sms={num_sms}")


def test_cascade_equals_plain():
    on = workloads.cascade(batch=32, prefix_tokens=1024, lo=1, hi=400, num_blocks=1000, seed=16)
    off = workloads.cascade(batch=32, prefix_tokens=1024, lo=1, hi=400, num_blocks=1000, seed=16,
                            use_cascade=False)
    a, c = run_gpu(on), run_gpu(off)
    assert a.bits == 0 and c.bits == 0
    _, _, _, out = run_oracle(on)
    assert_close(a.out, out, what="cascade")
    assert_close(c.out, out, what="plain")
    assert float((a.out.float() - c.out.float()).abs().max()) <= 2 * MAX_ABS


def test_decode_equals_last_prefill_row():
    """Request A prefills L tokens; request B decodes token L-1 over the same
    L-1 cached tokens (same blocks, same q row): outputs agree."""
    L = 300
    b = make_batch(name="dec-vs-pre", num_heads_q=32, num_heads_kv=8, head_dim=128, q_lens=[L, 1],
                   seq_lens=[L, L], num_blocks=60, seed=17, shared_prefix=[([0, 1], (L - 1) // 16)])
    # B shares A's first blocks (A's write fills them this step); B's own last
    # block already holds A's new rows for positions 288..298, and B's new
    # token and query row are A's last ones
    shared = (L - 1) // 16 * 16
    own = int(b.block_table[1, shared // 16])
    b.key_cache[own, :L - 1 - shared] = b.key[shared:L - 1]
    b.value_cache[own, :L - 1 - shared] = b.value[shared:L - 1]
    b.key[L] = b.key[L - 1]
    b.value[L] = b.value[L - 1]
    b.q[L] = b.q[L - 1]
    g = run_gpu(b)
    assert g.bits == 0
    mx, _ = attention_error(g.out[L:L + 1], g.out[L - 1:L].float().cpu().numpy().astype(np.float64))
    assert mx <= MAX_ABS


def test_prefix_hit_equals_recompute():
    """A chunk over a 128-token prefix hit equals the tail of a full prefill."""
    L, hit = 400, 128
    full = make_batch(name="full", num_heads_q=32, num_heads_kv=8, head_dim=128, q_lens=[L], seq_lens=[L],
                      num_blocks=40, seed=18)
    g_full = run_gpu(full)
    hitb = make_batch(name="hit", num_heads_q=32, num_heads_kv=8, head_dim=128, q_lens=[L - hit],
                      seq_lens=[L], num_blocks=40, seed=18)
    # same physical blocks and data: the first 128 tokens come from the cache,
    # which full's run wrote
    hitb.block_table = full.block_table.copy()
    hitb.key_cache = g_full.key_cache.cpu()
    hitb.value_cache = g_full.value_cache.cpu()
    hitb.q, hitb.key, hitb.value = full.q[hit:].clone(), full.key[hit:].clone(), full.value[hit:].clone()
    g_hit = run_gpu(hitb)
    assert g_hit.bits == 0
    mx, _ = attention_error(g_hit.out, g_full.out[hit:].float().cpu().numpy().astype(np.float64))
    assert mx <= MAX_ABS


@pytest.mark.parametrize("where", ["decode", "extend"])
def test_bad_block_id_reported(where):
    """An out-of-range id in the device block table (host copy not given to
    pa_plan) is caught by the kernel's own check: no load is issued for it and
    PA_DEVERR_BLOCK_RANGE is raised."""
    q_lens, seq = ([1], [100]) if where == "decode" else ([50], [100])
    b = make_batch(name="bad", num_heads_q=8, num_heads_kv=2, head_dim=64, q_lens=q_lens, seq_lens=seq,
                   num_blocks=20, seed=19)
    dev = torch.device("cuda")
    st = DeviceStep(b, dev, plan=False)
    st.plan = binding.pa_plan(num_heads_q=8, num_heads_kv=2, head_dim=64, num_blocks=20,
                              query_start_loc=b.query_start_loc, seq_lens=b.seq_lens,
                              num_computed_tokens=b.num_computed, max_blocks_per_req=b.max_blocks_per_req,
                              softmax_scale=b.softmax_scale)
    st.workspace = torch.zeros(st.plan.workspace_bytes, dtype=torch.uint8, device=dev)
    bt = b.block_table.copy()
    bt[0, 1] = 20 + 5                       # a cached block (tokens 16..31), not written this step
    st.block_table = torch.as_tensor(bt, device=dev)
    kc, vc = b.key_cache.to(dev), b.value_cache.to(dev)
    st.run(b.q.to(dev), b.key.to(dev), b.value.to(dev), kc, vc)
    bits = st.check_errors()
    assert bits & binding.PA_DEVERR_BLOCK_RANGE
    assert not bits & binding.PA_DEVERR_TIMEOUT
