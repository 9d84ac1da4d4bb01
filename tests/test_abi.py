"""The C ABI on the CPU: the library loads, exports what pa.h declares, and
pa_plan validates metadata and decomposes work (no kernel is launched)."""
import math
import os
import re

import numpy as np
import pytest

from paged_kv_cache_16_gb300 import binding, build, workloads
from paged_kv_cache_16_gb300.workloads import make_batch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_header_symbols_exported(lib):
    names = declared_functions()
    assert "pa_attention" in names and "pa_plan" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in pa.h but not exported"
    assert sorted(binding.EXPORTED) == names


def test_status_strings(lib):
    for s in range(7):
        assert binding.status_string(s) != "unknown status"
    assert binding.status_string(99) == "unknown status"


def desc(batch, **over):
    kw = dict(num_heads_q=batch.num_heads_q, num_heads_kv=batch.num_heads_kv, head_dim=batch.head_dim,
              num_blocks=batch.num_blocks, query_start_loc=batch.query_start_loc, seq_lens=batch.seq_lens,
              num_computed_tokens=batch.num_computed, block_table_host=batch.block_table,
              num_common_prefix_blocks=batch.num_common_prefix_blocks, softmax_scale=batch.softmax_scale,
              num_sms=152)
    kw.update(over)
    return kw


@pytest.fixture(scope="module")
def tiny():
    return workloads.tiny("1B")


def test_valid_plan(lib, tiny):
    assert binding.pa_plan_status(**desc(tiny)) == binding.PA_OK


@pytest.mark.parametrize("case", [
    "qsl_start", "qsl_decreasing", "length_identity", "too_many_blocks", "block_id_range",
    "block_id_negative", "heads_indivisible", "scale_zero", "scale_nan", "negative_prefix",
    "prefix_not_computed", "prefix_not_shared", "zero_heads", "negative_sms"])
def test_invalid_metadata(lib, tiny, case):
    b = tiny
    kw = desc(b)
    qsl = b.query_start_loc.copy()
    nc = b.num_computed.copy()
    bt = b.block_table.copy()
    if case == "qsl_start":
        kw["query_start_loc"] = qsl + 1
    elif case == "qsl_decreasing":
        qsl[2] = qsl[3] + 1
        kw["query_start_loc"] = qsl
    elif case == "length_identity":
        nc[1] += 1
        kw["num_computed_tokens"] = nc
    elif case == "too_many_blocks":
        kw["block_table_host"] = bt[:, :1]
    elif case == "block_id_range":
        bt[0, 0] = b.num_blocks
        kw["block_table_host"] = bt
    elif case == "block_id_negative":
        bt[3, 1] = -1
        kw["block_table_host"] = bt
    elif case == "heads_indivisible":
        kw["num_heads_q"] = 5
    elif case == "scale_zero":
        kw["softmax_scale"] = 0.0
    elif case == "scale_nan":
        kw["softmax_scale"] = float("nan")
    elif case == "negative_prefix":
        kw["num_common_prefix_blocks"] = -1
    elif case == "prefix_not_computed":
        kw["num_common_prefix_blocks"] = 1     # requests with num_computed 0
    elif case == "prefix_not_shared":
        c = workloads.cascade(batch=4, lo=64, hi=80, num_blocks=400)
        bt2 = c.block_table.copy()
        bt2[2, [0, 1]] = bt2[2, [1, 0]]        # same ids, different order in one row
        kw = desc(c, block_table_host=bt2)
    elif case == "zero_heads":
        kw["num_heads_kv"] = 0
    elif case == "negative_sms":
        kw["num_sms"] = -1
    assert binding.pa_plan_status(**kw) == binding.PA_ERR_INVALID_ARGUMENT


@pytest.mark.parametrize("over", [dict(head_dim=96), dict(block_size=32), dict(num_heads_q=256, num_heads_kv=1)])
def test_unsupported_shapes(lib, tiny, over):
    kw = desc(tiny, **over)
    if "block_size" in over:
        # keep the metadata consistent with 32-token blocks
        kw["block_table_host"] = tiny.block_table[:, :2]
    assert binding.pa_plan_status(**kw) == binding.PA_ERR_UNSUPPORTED


@pytest.mark.parametrize("hq,hkv", [(6, 2), (28, 4), (64, 2), (32, 1), (128, 1)])
def test_any_group_size_plans(lib, hq, hkv):
    """Any Hq % Hkv == 0 up to 128 query heads per kv head: groups of at most
    16 keep decode rows on the split-KV kernel, larger ones run every row on
    the tensor-core tiles (a sub-tile holds 128 // G tokens)."""
    G = hq // hkv
    b = workloads.make_batch(name="g", num_heads_q=hq, num_heads_kv=hkv, head_dim=64, q_lens=[1, 5, 1, 40],
                             seq_lens=[30, 70, 200, 90], num_blocks=80, seed=G)
    info = binding.pa_plan(**desc(b)).info()
    if G <= 16:
        assert info["num_decode_rows"] == 2 and info["num_extend_rows"] + info["num_small_q_rows"] == 2
    else:
        assert info["num_decode_rows"] == 0 and info["num_small_q_rows"] == 0 and info["num_extend_rows"] == 4
        tpt = 2 * (128 // G)
        assert info["num_extend_tiles"] == hkv * sum(-(-q // tpt) for q in (1, 5, 1, 40))


def test_mixed_batch_example_metadata(lib):
    """The R0/R1/R2 worked example (decode, prefix-hit chunk, spec verify)."""
    qsl = np.array([0, 1, 257, 260], np.int32)
    seq = np.array([1025, 768, 603], np.int32)
    nc = np.array([1024, 512, 600], np.int32)
    kw = dict(num_heads_q=8, num_heads_kv=2, head_dim=128, num_blocks=200, query_start_loc=qsl, seq_lens=seq,
              num_computed_tokens=nc, max_blocks_per_req=65, softmax_scale=0.1, num_sms=152)
    plan = binding.pa_plan(**kw)
    info = plan.info()
    # R0 decode; R1's 256-token chunk on the tiles; R2's 3-token verify row on
    # the decode kernel (3 tokens x G = 4 heads fill one 16-row MMA tile)
    assert info["num_decode_rows"] == 1 and info["num_extend_rows"] == 1 and info["num_small_q_rows"] == 1
    # 256 query tokens, G = 4 -> 64 tokens per CTA tile: 4 tiles per kv head
    assert info["num_extend_tiles"] == 2 * 4
    row_bytes = 2 * 128 * 4
    assert info["decode_kv_bytes"] == (1025 + 603) * row_bytes
    bad = nc.copy()
    bad[1] = 511
    assert binding.pa_plan_status(**{**kw, "num_computed_tokens": bad}) == binding.PA_ERR_INVALID_ARGUMENT


@pytest.mark.parametrize("maker", ["decode", "long", "mixed", "cascade", "cascade_off"])
def test_plan_decomposition(lib, maker):
    """Row classification, tile counts, byte and FLOP counts, cascade slots
    and launch counts of the plan agree with the batch (host-side view)."""
    if maker == "decode":
        b = workloads.decode(batch=16, num_blocks=5000)
    elif maker == "long":
        b = workloads.long_context(batch=2, context=16384, num_blocks=2100)
    elif maker == "mixed":
        b = workloads.mixed(n_decode=24, n_shared=4, chunk=300, chunk_b_cached=500, lo=100, hi=900)
    elif maker == "cascade":
        b = workloads.cascade(batch=8, num_blocks=1000)
    else:
        b = workloads.cascade(batch=8, num_blocks=1000, use_cascade=False)
    plan = binding.pa_plan(**desc(b))
    info = plan.info()
    q_lens = b.q_lens
    n_prefix = b.num_common_prefix_blocks
    kb = n_prefix * 16
    dec = [r for r in range(b.num_reqs) if q_lens[r] == 1]
    ext = [r for r in range(b.num_reqs) if q_lens[r] > 1]
    assert info["num_decode_rows"] == len(dec) and info["num_extend_rows"] == len(ext)
    row_bytes = b.num_heads_kv * b.head_dim * 4
    assert info["decode_kv_bytes"] == sum((int(b.seq_lens[r]) - kb) * row_bytes for r in dec)
    G = b.num_heads_q // b.num_heads_kv
    tpt = 2 * (128 // G)        # tokens per CTA tile (two 128-row sub-tiles)
    n_ext_tiles = sum(math.ceil(q_lens[r] / tpt) for r in ext) * b.num_heads_kv
    assert info["num_extend_tiles"] == n_ext_tiles + info["num_prefix_tiles"]
    if n_prefix:
        assert info["num_prefix_tiles"] > 0
        assert info["prefix_kv_bytes"] == kb * row_bytes
        assert info["num_merge_rows"] == b.num_tokens
    else:
        assert info["num_prefix_tiles"] == 0
    assert plan.workspace_bytes % 256 == 0
    assert info["kernels_per_call"] == (info["num_decode_items"] > 0) + (info["num_extend_tiles"] > 0) + \
        (info["num_merge_rows"] > 0)
    assert info["num_decode_ctas"] <= 152


def test_plan_is_deterministic_and_placement_free(lib):
    """The plan depends on lengths only: a different physical placement of
    the same batch gives the same decomposition and workspace size."""
    a = workloads.decode(batch=16, num_blocks=5000, seed=0)
    b = workloads.decode(batch=16, num_blocks=5000, seed=0)
    b_bt = np.random.default_rng(9).permutation(5000)[: a.block_table.size].reshape(a.block_table.shape)
    pa = binding.pa_plan(**desc(a))
    pb = binding.pa_plan(**desc(b, block_table_host=b_bt.astype(np.int32)))
    assert pa.info() == pb.info() and pa.workspace_bytes == pb.workspace_bytes


def test_empty_batch(lib):
    kw = dict(num_heads_q=4, num_heads_kv=2, head_dim=64, num_blocks=4,
              query_start_loc=np.zeros(1, np.int32), seq_lens=np.zeros(0, np.int32),
              num_computed_tokens=np.zeros(0, np.int32), max_blocks_per_req=1, softmax_scale=0.125,
              num_sms=152)
    plan = binding.pa_plan(**kw)
    assert plan.info()["num_tokens"] == 0 and plan.info()["kernels_per_call"] == 0


def test_idle_requests_and_zero_lengths(lib):
    """q_len = 0 rows (and a zero-length request) plan to no work."""
    kw = dict(num_heads_q=4, num_heads_kv=2, head_dim=64, num_blocks=8,
              query_start_loc=np.array([0, 0, 1, 1], np.int32), seq_lens=np.array([5, 3, 0], np.int32),
              num_computed_tokens=np.array([5, 2, 0], np.int32), max_blocks_per_req=1,
              softmax_scale=0.125, num_sms=152)
    info = binding.pa_plan(**kw).info()
    assert info["num_decode_rows"] == 1 and info["num_extend_rows"] == 0 and info["num_tokens"] == 1


# ------------------------------------------------------ fixed-shape plans --
def fixed(batch, **shape):
    return binding.pa_plan_fixed(**shape, **desc(batch))


def test_fixed_plan_layout_depends_on_shape_only(lib):
    """Plans of one fixed shape have the same workspace size and launches
    whatever the step's lengths and request count; the decode cut itself is
    the eager plan's."""
    shape = dict(max_tokens=96, max_reqs=96)
    plans = [fixed(workloads.decode(batch=n, lo=lo, hi=hi, num_blocks=4000, seed=n), **shape)
             for n, lo, hi in ((8, 20, 300), (64, 100, 700), (96, 1, 100), (1, 1, 1))]
    sizes = {p.workspace_bytes for p in plans}
    assert len(sizes) == 1
    for p in plans:
        i = p.info()
        assert i["num_decode_ctas"] == 152 and i["kernels_per_call"] == 2
    b = workloads.decode(batch=64, lo=100, hi=700, num_blocks=4000, seed=64)
    e, f = binding.pa_plan(**desc(b)).info(), fixed(b, **shape).info()
    for k in ("num_decode_items", "num_partial_slots", "num_merge_rows", "decode_kv_bytes"):
        assert e[k] == f[k], k


def test_fixed_plan_mixed_shape(lib):
    """With tile room, extend rows and cascade prefixes fit; the tile and
    merge launches are always made."""
    b = workloads.mixed(n_decode=24, n_shared=4, chunk=300, chunk_b_cached=500, lo=100, hi=900)
    eager = binding.pa_plan(**desc(b)).info()
    p = fixed(b, max_tokens=1024, max_reqs=64, max_extend_tiles=128)
    i = p.info()
    assert i["num_extend_tiles"] == eager["num_extend_tiles"] and i["kernels_per_call"] == 3
    d = workloads.decode(batch=8, lo=100, hi=700, num_blocks=4000)
    j = fixed(d, max_tokens=1024, max_reqs=64, max_extend_tiles=128)
    assert j.info()["kernels_per_call"] == 3 and j.workspace_bytes == p.workspace_bytes


def test_metadata_image_for_captured_uploads(lib):
    """pa_plan_metadata_bytes / pa_plan_copy_metadata: one image size per
    fixed shape, an image per step, too small a buffer refused;
    pa_upload_metadata_from checks its arguments before any CUDA call."""
    import torch
    shape = dict(max_tokens=96, max_reqs=96)
    a = fixed(workloads.decode(batch=8, lo=20, hi=300, num_blocks=4000, seed=1), **shape)
    b = fixed(workloads.decode(batch=64, lo=100, hi=700, num_blocks=4000, seed=2), **shape)
    n = binding.pa_plan_metadata_bytes(a)
    assert n > 0 and n % 16 == 0 and n == binding.pa_plan_metadata_bytes(b)
    ia, ib = torch.zeros(n, dtype=torch.uint8), torch.zeros(n, dtype=torch.uint8)
    binding.pa_plan_copy_metadata(a, ia)
    binding.pa_plan_copy_metadata(b, ib)
    assert ia.any() and not torch.equal(ia, ib)
    again = torch.zeros(n, dtype=torch.uint8)
    binding.pa_plan_copy_metadata(a, again)
    assert torch.equal(ia, again)
    small = torch.zeros(n - 16, dtype=torch.uint8)
    assert binding.pa_plan_copy_metadata_status(a, small.data_ptr(), n - 16) == binding.PA_ERR_INVALID_ARGUMENT
    up = lib.pa_upload_metadata_from
    ws = 1 << 20   # a fake, 256-aligned address: never dereferenced on these paths
    assert up(None, 16, ws, 1 << 20, None) == binding.PA_ERR_INVALID_ARGUMENT
    assert up(ia.data_ptr(), 16, None, 1 << 20, None) == binding.PA_ERR_INVALID_ARGUMENT
    assert up(ia.data_ptr(), 24, ws, 1 << 20, None) == binding.PA_ERR_INVALID_ARGUMENT
    assert up(ia.data_ptr(), n, ws, 256 + n - 16, None) == binding.PA_ERR_WORKSPACE_TOO_SMALL
    assert up(None, 0, ws, 1 << 20, None) == binding.PA_OK


@pytest.mark.parametrize("shape,status", [
    (dict(max_tokens=8, max_reqs=64), binding.PA_ERR_CAPACITY),            # too many tokens
    (dict(max_tokens=64, max_reqs=4), binding.PA_ERR_CAPACITY),            # too many requests
    (dict(max_tokens=0, max_reqs=64), binding.PA_ERR_INVALID_ARGUMENT),
    (dict(max_tokens=64, max_reqs=64, max_extend_tiles=-1), binding.PA_ERR_INVALID_ARGUMENT),
    (dict(max_tokens=64, max_reqs=64, max_partial_slots=3), binding.PA_ERR_CAPACITY),
])
def test_fixed_plan_capacity_errors(lib, shape, status):
    b = workloads.decode(batch=16, lo=300, hi=900, num_blocks=4000)
    assert binding.pa_plan_fixed_status(**shape, **desc(b)) == status


def test_fixed_plan_tile_capacity(lib):
    b = workloads.mixed(n_decode=8, n_shared=0, chunk=300, chunk_b_cached=500, lo=100, hi=900)
    kw = desc(b)
    assert binding.pa_plan_fixed_status(max_tokens=1024, max_reqs=64, **kw) == binding.PA_ERR_CAPACITY
    fp8 = dict(kw, kv_cache_dtype=binding.PA_KV_FP8_E4M3, k_scale=0.1, v_scale=0.1)
    # FP8 tiles read bf16 copies: tile room without block room is malformed
    assert binding.pa_plan_fixed_status(max_tokens=1024, max_reqs=64, max_extend_tiles=128,
                                        **fp8) == binding.PA_ERR_INVALID_ARGUMENT
    assert binding.pa_plan_fixed_status(max_tokens=1024, max_reqs=64, max_extend_tiles=128,
                                        max_dequant_blocks=4, **fp8) == binding.PA_ERR_CAPACITY
    assert binding.pa_plan_fixed_status(max_tokens=1024, max_reqs=64, max_extend_tiles=128,
                                        max_dequant_blocks=4096, **fp8) == binding.PA_OK


def test_fixed_plan_decode_prefix(lib):
    """decode_prefix_tokens bounds the rows the decode stream reads: a step
    whose decode or small multi-token rows reach past it is refused; the
    chunk rows may lie anywhere."""
    make = lambda ql, sl: make_batch(name="prefix", num_heads_q=32, num_heads_kv=8, head_dim=128, q_lens=ql,
                                     seq_lens=sl, num_blocks=600, seed=5, max_blocks_per_req=64)
    shape = dict(max_tokens=512, max_reqs=8, max_extend_tiles=64)
    first = make([1, 3, 1, 200], [90, 40, 700, 260])          # decode-stream rows: tokens 0..4
    assert binding.pa_plan_fixed_status(**shape, decode_prefix_tokens=5, **desc(first)) == binding.PA_OK
    assert binding.pa_plan_fixed_status(**shape, decode_prefix_tokens=4, **desc(first)) == binding.PA_ERR_CAPACITY
    assert binding.pa_plan_fixed_status(**shape, decode_prefix_tokens=-1, **desc(first)) == \
        binding.PA_ERR_INVALID_ARGUMENT
    late = make([200, 1], [260, 90])                           # the decode row is token 200
    assert binding.pa_plan_fixed_status(**shape, decode_prefix_tokens=16, **desc(late)) == binding.PA_ERR_CAPACITY
    assert binding.pa_plan_fixed_status(**shape, decode_prefix_tokens=201, **desc(late)) == binding.PA_OK
    assert binding.pa_plan_fixed_status(**shape, **desc(late)) == binding.PA_OK


def test_fixed_plan_decode_prefix_moves_the_split(lib):
    """With staged inputs the tiles start after the late rows' copy, so the
    planner gives them more SMs (and the decode stream fewer) than for the
    same step with every input resident; the decode grid stays the shape's."""
    b = workloads.mixed()
    kw = desc(b)
    info = binding.pa_plan(**kw).info()
    shape = dict(max_tokens=b.num_tokens, max_reqs=b.num_reqs, max_extend_tiles=info["num_extend_tiles"],
                 max_partial_slots=max(info["num_partial_slots"], 1))
    plain = binding.pa_plan_fixed(**shape, **kw).info()
    staged = binding.pa_plan_fixed(**shape, decode_prefix_tokens=256, **kw).info()
    assert plain["side_by_side"] == staged["side_by_side"] == 1
    assert plain["num_extend_ctas"] == info["num_extend_ctas"]
    assert staged["num_extend_ctas"] > plain["num_extend_ctas"]
    assert staged["num_decode_ctas"] == plain["num_decode_ctas"]


def test_fixed_plan_decode_prefix_no_merged_late_rows(lib):
    """Rows from the decode prefix on must be final when the tiles finish: a
    cascade step with a chunk row (whose rows are merged from prefix and
    suffix partials) is refused when that row lies past the prefix."""
    b = make_batch(name="cascade-chunk", num_heads_q=32, num_heads_kv=8, head_dim=128, q_lens=[1, 1, 40],
                   seq_lens=[300, 300, 400], num_blocks=600, seed=6, max_blocks_per_req=64,
                   shared_prefix=[([0, 1, 2], 4)], num_common_prefix_blocks=4)
    shape = dict(max_tokens=512, max_reqs=8, max_extend_tiles=64, max_partial_slots=4096)
    assert binding.pa_plan_fixed_status(**shape, **desc(b)) == binding.PA_OK
    assert binding.pa_plan_fixed_status(**shape, decode_prefix_tokens=2, **desc(b)) == binding.PA_ERR_CAPACITY
    assert binding.pa_plan_fixed_status(**shape, decode_prefix_tokens=42, **desc(b)) == binding.PA_OK


def test_staged_launch_argument_checks(lib):
    """The staged launch needs a fixed-shape plan with a decode prefix and an
    event; both are checked before anything is enqueued."""
    b = make_batch(name="prefix", num_heads_q=32, num_heads_kv=8, head_dim=128, q_lens=[1, 200],
                   seq_lens=[90, 260], num_blocks=600, seed=5, max_blocks_per_req=64)
    shape = dict(max_tokens=512, max_reqs=8, max_extend_tiles=64)
    f = binding.load().pa_attention_with_kv_update_launch_staged
    fake = 1 << 20   # aligned, never dereferenced on these paths
    plain = binding.pa_plan_fixed(**shape, **desc(b))
    staged = binding.pa_plan_fixed(**shape, decode_prefix_tokens=1, **desc(b))
    eager = binding.pa_plan(**desc(b))
    args = lambda plan, ev: (plan.handle, fake, fake, fake, fake, fake, fake, None, fake, fake, 1 << 40, None, ev,
                             None)
    assert f(*args(plain, fake)) == binding.PA_ERR_INVALID_ARGUMENT
    assert f(*args(eager, fake)) == binding.PA_ERR_INVALID_ARGUMENT
    assert f(*args(staged, None)) == binding.PA_ERR_INVALID_ARGUMENT


def test_zero_blocks_argument_checks(lib):
    """Host-side validation of pa_zero_blocks (no kernel is enqueued)."""
    L = binding.load()
    assert L.pa_zero_blocks(None, 0, 10, 8, 128, binding.PA_KV_BF16, None, None, None, None) == binding.PA_OK
    assert L.pa_zero_blocks(None, -1, 10, 8, 128, 0, None, None, None, None) == binding.PA_ERR_INVALID_ARGUMENT
    assert L.pa_zero_blocks(None, 1, 10, 8, 128, 0, None, None, None, None) == binding.PA_ERR_INVALID_ARGUMENT
    assert L.pa_zero_blocks(None, 0, 10, 8, 128, 7, None, None, None, None) == binding.PA_ERR_INVALID_ARGUMENT


@pytest.mark.parametrize("g,q_len,units", [(4, 3, 1), (4, 4, 1), (4, 5, 2), (8, 3, 2), (8, 8, 4), (1, 8, 1),
                                           (16, 2, 2), (4, 9, 0)])
def test_small_q_units(lib, g, q_len, units):
    """Rows of 2..8 query tokens run on the decode kernel in units of 16 / G
    tokens (each unit reads its keys once); longer rows go to the tiles."""
    hkv = 2
    qsl = np.array([0, q_len], np.int32)
    seq = np.array([500], np.int32)
    kw = dict(num_heads_q=g * hkv, num_heads_kv=hkv, head_dim=128, num_blocks=64, query_start_loc=qsl,
              seq_lens=seq, num_computed_tokens=seq - q_len, max_blocks_per_req=32, softmax_scale=0.1,
              num_sms=152)
    info = binding.pa_plan(**kw).info()
    if units == 0:
        assert info["num_small_q_rows"] == 0 and info["num_extend_rows"] == 1
        return
    assert info["num_small_q_rows"] == 1 and info["num_extend_tiles"] == 0
    tg = max(1, 16 // g)
    ends = [500 - q_len + min(q_len, j + tg) for j in range(0, q_len, tg)]
    assert len(ends) == units
    assert info["decode_kv_bytes"] == sum(ends) * hkv * 128 * 4


def test_small_q_routing_by_parallelism(lib):
    """Rows needing several units go to the decode kernel only while their
    tiles would not fill the GPU; one-unit rows always do."""
    def plan(n, q_len, g=4):
        qsl = np.arange(n + 1, dtype=np.int32) * q_len
        seq = np.full(n, 1000, np.int32)
        return binding.pa_plan(num_heads_q=8 * g, num_heads_kv=8, head_dim=128, num_blocks=64 * n + 64,
                               query_start_loc=qsl, seq_lens=seq, num_computed_tokens=seq - q_len,
                               max_blocks_per_req=64, softmax_scale=0.1, num_sms=152).info()
    assert plan(64, 4)["num_small_q_rows"] == 64                      # one unit each
    assert plan(18, 8)["num_small_q_rows"] == 18                      # 18 x 8 tiles < 152 SMs
    i = plan(64, 8)                                                   # 512 tile CTAs: tiles read keys once
    assert i["num_small_q_rows"] == 0 and i["num_extend_rows"] == 64


def test_graph_executor_rejects_bad_arguments(lib):
    """pa_graph_*: NULL and partial arguments are refused before any CUDA
    call (host only)."""
    import ctypes
    b = workloads.tiny("1A")
    d, keep = binding.make_desc(**desc(b))
    fs = binding._fixed_shape(8, 4)
    bufs = binding.GraphBuffers()
    h = ctypes.c_void_p(123)
    assert lib.pa_graph_create(None, ctypes.byref(fs), ctypes.byref(bufs), ctypes.byref(h)) == binding.PA_ERR_INVALID_ARGUMENT
    assert h.value is None
    assert lib.pa_graph_create(ctypes.byref(d), ctypes.byref(fs), ctypes.byref(bufs), ctypes.byref(h)) == \
        binding.PA_ERR_INVALID_ARGUMENT   # every device buffer NULL
    for name in ("q", "key", "value", "out", "query_start_loc", "num_computed", "block_table", "key_cache",
                 "value_cache"):
        setattr(bufs, name, 4096)
    bufs.in_bytes = 64                    # host input copy given in part
    assert lib.pa_graph_create(ctypes.byref(d), ctypes.byref(fs), ctypes.byref(bufs), ctypes.byref(h)) == \
        binding.PA_ERR_INVALID_ARGUMENT
    bufs.in_bytes = 0
    bufs.q = 4097                         # misaligned
    assert lib.pa_graph_create(ctypes.byref(d), ctypes.byref(fs), ctypes.byref(bufs), ctypes.byref(h)) == \
        binding.PA_ERR_INVALID_ARGUMENT
    assert lib.pa_graph_step(None, ctypes.byref(d), None) == binding.PA_ERR_INVALID_ARGUMENT
    assert lib.pa_graph_wait(None, 0) == binding.PA_ERR_INVALID_ARGUMENT
    assert lib.pa_graph_turn(None) == 0
    assert lib.pa_graph_workspace(None) is None and lib.pa_graph_slot_mapping(None) is None
    lib.pa_graph_destroy(None)
