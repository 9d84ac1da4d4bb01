"""pa_attention_no_alloc against pa_attention (needs a GB300).

The no-allocation entry point serves callers that cannot allocate device
memory (an engine whose KV pool already holds nearly all free memory, or a
hot path that must not call cudaMalloc/cudaFree because they can
synchronise the device).  It runs the same kernels with a library-owned
scratch array instead of a caller workspace.  This file is collected last
so that a failure here never hides the other tests; it also passes when run
alone in a fresh process.
"""
import numpy as np
import pytest
import torch

from gpu_common import MAX_ABS, MEAN_ABS, ensure_library
from paged_kv_cache_16_gb300 import binding, workloads
from paged_kv_cache_16_gb300.step import DeviceStep

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_library()


def _prepared(batch):
    """A step whose caches already hold the new rows (write done)."""
    dev = torch.device("cuda")
    st = DeviceStep(batch, dev)
    q = batch.q.to(dev)
    kc = batch.key_cache.to(dev, copy=True)
    vc = batch.value_cache.to(dev, copy=True)
    st.slot_mapping()
    st.write(batch.key.to(dev), batch.value.to(dev), kc, vc)
    return st, q, kc, vc


def _close(a: torch.Tensor, b: torch.Tensor):
    """Within the attention tolerance of the other tests, and in fact equal:
    both entry points run the same kernels on the same work cut, so stale
    partials left in the shared array by an earlier call would show here."""
    d = (a.float() - b.float()).abs()
    assert torch.isfinite(a.float()).all()
    assert float(d.max()) <= MAX_ABS and float(d.mean()) <= MEAN_ABS
    assert torch.equal(a, b)


def _batches():
    return [workloads.mixed(n_decode=24, n_shared=4, shared_tokens=64, lo=65, hi=900, chunk=300,
                            chunk_b_cached=500, seed=21),
            workloads.cascade(batch=16, prefix_tokens=512, lo=1, hi=300, num_blocks=400, seed=22),
            # E4M3 caches: the tiles' bf16 block copies live in the shared array too
            workloads.mixed(n_decode=24, n_shared=4, shared_tokens=64, lo=65, hi=900, chunk=300,
                            chunk_b_cached=500, seed=23, kv_cache_dtype="fp8")]


def test_no_alloc_matches_workspace_entry_point_twice():
    """Calls in a row (different batches, so each runs over the previous
    one's leftovers in the shared array) match pa_attention."""
    dev = torch.device("cuda")
    for batch in _batches():
        st, q, kc, vc = _prepared(batch)
        assert st.plan.workspace_bytes <= binding.NO_ALLOC_SCRATCH_BYTES
        T = batch.num_tokens
        ref = st.attend(q, kc, vc).clone()
        out = torch.full_like(st.out, float("nan"))
        err = torch.full((1,), -1, dtype=torch.int32, device=dev)
        binding.pa_attention_no_alloc(st.plan, q, kc, vc, st.block_table, out, err)
        torch.cuda.synchronize()
        assert binding.pa_check_device_errors(err) == 0
        _close(out[:T], ref)


FIRST_CALL = r"""
import sys, torch
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
from paged_kv_cache_16_gb300 import binding, workloads
from test_zz_no_alloc import _prepared
binding.load()
batch = workloads.mixed(n_decode=24, n_shared=4, shared_tokens=64, lo=65, hi=900, chunk=300,
                        chunk_b_cached=500, seed=31)
st, q, kc, vc = _prepared(batch)
T = batch.num_tokens
out = torch.full_like(st.out, float("nan"))
err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
binding.pa_attention_no_alloc(st.plan, q, kc, vc, st.block_table, out, err)   # first attention call
torch.cuda.synchronize()
assert binding.pa_check_device_errors(err) == 0
ref = st.attend(q, kc, vc).clone()
torch.cuda.synchronize()
assert torch.equal(out[:T], ref), "no-alloc output differs"
print("ok")
"""


def test_no_alloc_first_call_in_fresh_process():
    """In a new process, pa_attention_no_alloc is the first attention call
    (its one-time look-up of the array's address and the kernels' first
    attribute set-up happen there); pa_attention afterwards gives the same
    output."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    proc = subprocess.run([sys.executable, "-c", FIRST_CALL, root], capture_output=True, text=True, timeout=600)
    assert proc.returncode == 0, proc.stderr[-3000:]
    assert proc.stdout.strip().endswith("ok")


def test_no_alloc_rejects_plans_beyond_the_array():
    """A plan whose workspace exceeds the array is refused before anything is
    enqueued, with PA_ERR_WORKSPACE_TOO_SMALL."""
    T = 4096
    n = 64
    seq = np.full(T, n * 16 + 1, dtype=np.int32)
    plan = binding.pa_plan(num_heads_q=64, num_heads_kv=8, head_dim=128, num_blocks=n + T,
                           query_start_loc=np.arange(T + 1, dtype=np.int32), seq_lens=seq,
                           num_computed_tokens=seq - 1, max_blocks_per_req=n + 1, num_common_prefix_blocks=n,
                           softmax_scale=0.088, num_sms=152)
    assert plan.workspace_bytes > binding.NO_ALLOC_SCRATCH_BYTES
    dev = torch.device("cuda")
    dummy = torch.zeros(64, dtype=torch.bfloat16, device=dev)
    bt = torch.zeros(1, dtype=torch.int32, device=dev)
    with pytest.raises(binding.PaError) as exc:
        binding.pa_attention_no_alloc(plan, dummy, dummy, dummy, bt, dummy)
    assert exc.value.status == binding.PA_ERR_WORKSPACE_TOO_SMALL
