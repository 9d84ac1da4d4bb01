"""Fixed-shape plans and CUDA-graph replays (needs a GB300).

One graph is captured per shape (slot mapping, cache write and the attention
kernels, or the fused write + attention call); every later step of a different size only uploads its metadata and
replays.  Each replayed step is checked against the oracle (caches bit for
bit, attention within tolerance) on the cache state it started from, and
against the eager path (pa_plan + pa_attention) on the same inputs, bit for
bit: a fixed-shape plan cuts the work exactly as the eager plan does.
Also here: block zeroing against the oracle.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

from gpu_common import assert_close, cache_bits, ensure_library, run_gpu, run_oracle
from oracle.oracle import default as default_oracle
from paged_kv_cache_16_gb300 import binding, workloads
from paged_kv_cache_16_gb300.step import GraphStep
from paged_kv_cache_16_gb300.workloads import make_batch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_library()


def graph_args(b, max_blocks):
    return dict(num_heads_q=b.num_heads_q, num_heads_kv=b.num_heads_kv, head_dim=b.head_dim,
                num_blocks=b.num_blocks, max_blocks_per_req=max_blocks, softmax_scale=b.softmax_scale,
                kv_cache_dtype=b.kv_cache_dtype, k_scale=b.k_scale, v_scale=b.v_scale)


def graph_for(b, max_blocks, fused=False, **shape):
    return GraphStep(fused=fused, **graph_args(b, max_blocks), **shape)


def replay_steps(batches, fused=False, **shape):
    """Run every batch through one captured graph on one shared cache pool
    (fused: the graph holds pa_attention_with_kv_update_launch)."""
    dev = torch.device("cuda")
    mb = max(b.block_table.shape[1] for b in batches)
    gs = graph_for(batches[0], mb, fused, **shape)
    kc = batches[0].key_cache.to(dev, copy=True)
    vc = batches[0].value_cache.to(dev, copy=True)
    for b in batches:
        before = replace(b, key_cache=kc.cpu(), value_cache=vc.cpu())
        out = gs.run(b, b.q.to(dev), b.key.to(dev), b.value.to(dev), kc, vc).clone()
        torch.cuda.synchronize()
        assert gs.check_errors() == 0, b.name
        okc, ovc, oslots, oout = run_oracle(before)
        assert np.array_equal(cache_bits(kc), okc) and np.array_equal(cache_bits(vc), ovc), b.name
        if b.num_tokens:
            assert np.array_equal(gs.slots[:b.num_tokens].cpu().numpy(), oslots), b.name
            assert_close(out, oout, what=b.name)
            eager = run_gpu(before)
            assert eager.bits == 0
            assert torch.equal(eager.out, out), f"{b.name}: graph replay differs from the eager path"
    return gs


def decode_steps(kv="bf16"):
    """Three decode steps on one 3000-block pool: 40, 17 and 48 requests."""
    out = []
    for i, (n, lo, hi) in enumerate(((40, 1, 700), (17, 300, 2000), (48, 1, 64))):
        b = workloads.decode(batch=n, lo=lo, hi=hi, num_blocks=3000, seed=60 + i, kv_cache_dtype=kv)
        out.append(replace(b, name=f"decode-step{i}"))
    return out


@pytest.mark.parametrize("fused", [False, True])
def test_graph_replay_decode_steps(fused):
    replay_steps(decode_steps(), fused, max_tokens=48, max_reqs=48)


@pytest.mark.parametrize("fused", [False, True])
def test_graph_replay_decode_steps_fp8(fused):
    replay_steps(decode_steps("fp8"), fused, max_tokens=48, max_reqs=48)


def mixed_steps(kv="bf16"):
    """Decodes with chunked prefills of changing size (and a step of decodes
    only) on one 600-block pool, one shape."""
    specs = [([1, 1, 37, 1, 129, 1], [300, 77, 37, 512, 400, 19]),
             ([200, 1, 1, 3], [1000, 64, 1, 500]),
             ([1, 1, 1], [90, 1, 700]),
             ([64, 1, 300, 1, 2], [64, 33, 700, 16, 17])]
    out = []
    for i, (ql, sl) in enumerate(specs):
        out.append(make_batch(name=f"mixed-step{i}", num_heads_q=32, num_heads_kv=8, head_dim=128, q_lens=ql,
                              seq_lens=sl, num_blocks=600, seed=70 + i, max_blocks_per_req=64,
                              kv_cache_dtype=kv))
    return out


@pytest.mark.parametrize("fused", [False, True])
def test_graph_replay_mixed_steps(fused):
    replay_steps(mixed_steps(), fused, max_tokens=512, max_reqs=8, max_extend_tiles=64)


@pytest.mark.parametrize("fused", [False, True])
def test_graph_replay_mixed_steps_fp8(fused):
    replay_steps(mixed_steps("fp8"), fused, max_tokens=512, max_reqs=8, max_extend_tiles=64,
                 max_dequant_blocks=256)


@pytest.mark.parametrize("fused", [False, True])
def test_graph_replay_cascade_steps(fused):
    """Cascade steps (shared prefix, batch-wide n) of two sizes in one shape;
    prefix splits need explicit partial-slot room."""
    steps = []
    for i, (n, nb) in enumerate(((24, 16), (9, 8))):
        steps.append(replace(workloads.cascade(batch=n, prefix_tokens=16 * nb, lo=1, hi=200, num_blocks=700,
                                               seed=80 + i), name=f"cascade-step{i}"))
    replay_steps(steps, fused, max_tokens=24, max_reqs=24, max_extend_tiles=256, max_partial_slots=24 * 160)


def test_fixed_plan_eager_equals_plain_plan():
    """pa_attention with a fixed-shape plan (no graph) is the eager result bit for bit."""
    dev = torch.device("cuda")
    b = workloads.mixed(n_decode=20, n_shared=4, shared_tokens=64, lo=65, hi=700, chunk=200, chunk_b_cached=300,
                        seed=90)
    ref = run_gpu(b)
    gs = graph_for(b, b.block_table.shape[1], max_tokens=1024, max_reqs=64, max_extend_tiles=256)
    plan = gs.make_plan(b)
    kc, vc = b.key_cache.to(dev, copy=True), b.value_cache.to(dev, copy=True)
    gs.load(b, plan, b.q.to(dev), b.key.to(dev), b.value.to(dev))
    gs.enqueue(plan, kc, vc)
    torch.cuda.synchronize()
    assert gs.check_errors() == 0
    assert torch.equal(gs.out[:b.num_tokens], ref.out)


def test_upload_from_pageable_memory_refused():
    """The captured upload reads page-locked memory only."""
    dev = torch.device("cuda")
    ws = torch.zeros(1 << 16, dtype=torch.uint8, device=dev)
    pageable = torch.zeros(1024, dtype=torch.uint8)
    st = binding.load().pa_upload_metadata_from(pageable.data_ptr(), 1024, ws.data_ptr(), ws.numel(), None)
    assert st == binding.PA_ERR_INVALID_ARGUMENT
    pinned = torch.zeros(1024, dtype=torch.uint8).pin_memory()
    pinned[:] = torch.arange(1024) % 251
    binding.pa_upload_metadata_from(pinned, 1024, ws)
    torch.cuda.synchronize()
    assert torch.equal(ws[256:256 + 1024].cpu(), pinned)


def test_graph_images_alternate():
    """Consecutive steps replay the two captures in turn; a step whose image
    the host rewrote while the other graph ran still sees its own metadata."""
    steps = decode_steps() + decode_steps()
    gs = replay_steps(steps, max_tokens=48, max_reqs=48)
    assert len(gs.graphs) == 2 and gs.turn == len(steps) % 2


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_zero_blocks(kv):
    """pa_zero_blocks against the oracle: listed blocks zero, the rest
    untouched, -1 skipped, an id past the cache reported."""
    dev = torch.device("cuda")
    nb, hkv, d = 40, 8, 128
    g = torch.Generator().manual_seed(5)
    if kv == "fp8":
        kc = torch.randint(1, 256, (nb, 16, hkv, d), generator=g, dtype=torch.uint8)
        vc = torch.randint(1, 256, (nb, 16, hkv, d), generator=g, dtype=torch.uint8)
        okc, ovc = kc.numpy().copy(), vc.numpy().copy()
    else:
        kc = torch.randn(nb, 16, hkv, d, generator=g).to(torch.bfloat16)
        vc = torch.randn(nb, 16, hkv, d, generator=g).to(torch.bfloat16)
        okc, ovc = workloads.bf16_bits(kc).copy(), workloads.bf16_bits(vc).copy()
    ids = np.array([7, -1, 0, 39, 7, 12], dtype=np.int32)
    assert default_oracle().zero_blocks(ids, okc, ovc) == 0
    gkc, gvc = kc.to(dev), vc.to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    binding.pa_zero_blocks(torch.as_tensor(ids, device=dev), gkc, gvc, err)
    torch.cuda.synchronize()
    assert binding.pa_check_device_errors(err) == 0
    assert np.array_equal(cache_bits(gkc), okc) and np.array_equal(cache_bits(gvc), ovc)
    bad = torch.tensor([3, nb], dtype=torch.int32, device=dev)
    binding.pa_zero_blocks(bad, gkc, gvc, err)
    assert binding.pa_check_device_errors(err) & binding.PA_DEVERR_BLOCK_RANGE
    assert not gkc[3].any() and not gvc[3].any()


@pytest.mark.parametrize("fused", [False, True])
def test_graph_replay_host_io(fused):
    """Graphs that also copy a page-locked input image in and the output back
    (host memory to host memory): steps of changing size, each equal bit for
    bit to the device-resident graph on the same caches and to the eager path,
    and within tolerance of the oracle; the two images alternate."""
    dev = torch.device("cuda")
    batches = decode_steps()
    mb = max(b.block_table.shape[1] for b in batches)
    shape = dict(max_tokens=48, max_reqs=48)
    gh = GraphStep(host_io=True, fused=fused, **{**graph_args(batches[0], mb), **shape})
    gd = GraphStep(fused=fused, **{**graph_args(batches[0], mb), **shape})
    kc = batches[0].key_cache.to(dev, copy=True)
    vc = batches[0].value_cache.to(dev, copy=True)
    kc2, vc2 = kc.clone(), vc.clone()
    for n, b in enumerate(batches):
        before = replace(b, key_cache=kc.cpu(), value_cache=vc.cpu())
        plan = gh.make_plan(b)
        if gh.graphs is None:
            gh.load(b, plan, b.q.to(dev), b.key.to(dev), b.value.to(dev))
            gh.capture(plan, kc, vc)
        turn = gh.turn
        gh.stage_host(b, b.q, b.key, b.value)
        gh.replay(plan)
        view = gh.host_output(b.num_tokens)
        assert gh.turn != turn
        assert view.device.type == "cpu" and view.is_pinned()
        out = view.clone()
        ref = gd.run(b, b.q.to(dev), b.key.to(dev), b.value.to(dev), kc2, vc2)
        torch.cuda.synchronize()
        assert gh.check_errors() == 0 and gd.check_errors() == 0, b.name
        assert torch.equal(out, ref.cpu()), f"{b.name}: host-io replay differs from the device replay"
        assert torch.equal(kc, kc2) and torch.equal(vc, vc2), b.name
        _, _, _, oout = run_oracle(before)
        assert_close(out, oout, what=b.name)
        eager = run_gpu(before)
        assert torch.equal(eager.out.cpu(), out), f"{b.name}: host-io replay differs from the eager path"


def native_steps(batches, fused, host_io, own_pool=False, eager_exact=True, **shape):
    """Every batch through the library's graph executor (pa_graph_*) on one
    cache pool: caches and slots against the oracle bit for bit, output within
    tolerance of the oracle and equal bit for bit to the eager path.
    own_pool: each step first loads its batch's own pool contents into the
    graph's cache buffers (otherwise a step's history may land on slots an
    earlier batch filled with its +-3e4 poison, where one bf16 ulp of the
    output is 128, beyond the absolute tolerance).  eager_exact=False: the
    plan's SM split may differ from the eager plan's (staged inputs), so the
    decode cut and the merge's rounding may too; the oracle check stands."""
    from paged_kv_cache_16_gb300.step import NativeGraphStep
    dev = torch.device("cuda")
    mb = max(b.block_table.shape[1] for b in batches)
    kc = batches[0].key_cache.to(dev, copy=True)
    vc = batches[0].value_cache.to(dev, copy=True)
    ns = NativeGraphStep(fused=fused, host_io=host_io, key_cache=kc, value_cache=vc, device=dev,
                         **graph_args(batches[0], mb), **shape)
    turns = []
    for b in batches:
        if own_pool:
            kc.copy_(b.key_cache.to(dev))
            vc.copy_(b.value_cache.to(dev))
        before = replace(b, key_cache=kc.cpu(), value_cache=vc.cpu())
        turns.append(ns.graph.turn)
        out = ns.run(b, b.q, b.key, b.value) if host_io else ns.run(b, b.q.to(dev), b.key.to(dev), b.value.to(dev))
        out = out.clone()
        torch.cuda.synchronize()
        assert ns.check_errors() == 0, b.name
        assert out.device.type == ("cpu" if host_io else "cuda")
        okc, ovc, oslots, oout = run_oracle(before)
        assert np.array_equal(cache_bits(kc), okc) and np.array_equal(cache_bits(vc), ovc), b.name
        if b.num_tokens:
            assert np.array_equal(ns.slot_mapping[:b.num_tokens].cpu().numpy(), oslots), b.name
            assert_close(out, oout, what=b.name)
            eager = run_gpu(before)
            assert eager.bits == 0
            if eager_exact:
                assert torch.equal(eager.out.cpu(), out.cpu()), f"{b.name}: native graph differs from the eager path"
    assert turns == [i % 2 for i in range(len(batches))]
    ns.destroy()


@pytest.mark.parametrize("host_io", [False, True])
@pytest.mark.parametrize("fused", [False, True])
def test_native_graph_decode_steps(fused, host_io):
    native_steps(decode_steps() + decode_steps(), fused, host_io, max_tokens=48, max_reqs=48)


@pytest.mark.parametrize("host_io", [False, True])
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_native_graph_mixed_steps(kv, host_io):
    native_steps(mixed_steps(kv), True, host_io, max_tokens=512, max_reqs=8, max_extend_tiles=64,
                 max_dequant_blocks=256 if kv == "fp8" else 0)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_native_graph_host_out_copy(kv):
    """A host output buffer for fewer rows than the shape holds: the graph
    copies those rows back at its end (a whole-output buffer is stored into
    by the kernels instead); every step's rows fit in it."""
    steps = mixed_steps(kv)
    assert max(b.num_tokens for b in steps) <= 384
    native_steps(steps, True, True, out_rows=384, max_tokens=512, max_reqs=8, max_extend_tiles=64,
                 max_dequant_blocks=256 if kv == "fp8" else 0)


def test_native_graph_cascade_steps():
    steps = []
    for i, (n, nb) in enumerate(((24, 16), (9, 8))):
        steps.append(replace(workloads.cascade(batch=n, prefix_tokens=16 * nb, lo=1, hi=200, num_blocks=700,
                                               seed=80 + i), name=f"cascade-step{i}"))
    native_steps(steps, False, True, max_tokens=24, max_reqs=24, max_extend_tiles=256, max_partial_slots=24 * 160)


def staged_steps(kv="bf16"):
    """Steps whose decode-stream rows (one-token decodes and 2..8-token rows)
    lie in the first 16 token rows, chunks after them, and a step of decodes
    only, on one 600-block pool."""
    specs = [([1, 3, 1, 2, 200, 37], [300, 40, 512, 19, 400, 37]),
             ([1, 1, 4, 7, 300], [64, 90, 33, 20, 700]),
             ([1] * 8, [90, 1, 700, 16, 33, 5, 64, 200]),
             ([2, 1, 64, 129], [2, 500, 64, 200])]
    return [make_batch(name=f"staged-step{i}", num_heads_q=32, num_heads_kv=8, head_dim=128, q_lens=ql,
                       seq_lens=sl, num_blocks=600, seed=95 + i, max_blocks_per_req=64, kv_cache_dtype=kv)
            for i, (ql, sl) in enumerate(specs)]


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_native_graph_staged_host_io(kv):
    """Host I/O with a decode prefix: each graph copies the image but the
    late rows first, starts the decode stream, and the chunks' write and
    tiles wait for the late rows' copy on a second stream, whose rows of the
    output are copied back as soon as the tiles are done.  Checked against
    the oracle (caches and slots bit for bit, output within tolerance)."""
    native_steps(staged_steps(kv), True, True, own_pool=True, eager_exact=False, max_tokens=512, max_reqs=8,
                 max_extend_tiles=64, max_dequant_blocks=256 if kv == "fp8" else 0, decode_prefix_tokens=16)


def test_native_graph_staged_cascade():
    """Cascade steps (decode rows only, all below the decode prefix) through a
    staged host-I/O graph: the prefix tiles wait for the late copy on the
    library stream and the merge of prefix and suffix partials (rows below
    the prefix) runs after the join."""
    steps = []
    for i, (n, nb) in enumerate(((24, 16), (9, 8))):
        steps.append(replace(workloads.cascade(batch=n, prefix_tokens=16 * nb, lo=1, hi=200, num_blocks=700,
                                               seed=80 + i), name=f"staged-cascade-step{i}"))
    native_steps(steps, True, True, own_pool=True, eager_exact=False, max_tokens=32, max_reqs=24,
                 max_extend_tiles=256, max_partial_slots=32 * 160, decode_prefix_tokens=24)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_staged_launch_waits_for_late_rows(kv):
    """pa_attention_with_kv_update_launch_staged with rows 16.. copied in on
    another stream behind a ~25 ms busy kernel, long after the call's work has
    started: caches equal the oracle's bit for bit and the output is within
    tolerance of the oracle's, so nothing read those rows before they landed;
    the late-output event has fired once the stream is done."""
    dev = torch.device("cuda")
    b = staged_steps(kv)[0]
    P, T, M = 16, b.num_tokens, 512
    before = replace(b)
    fp8 = kv == "fp8"
    plan = binding.pa_plan_fixed(
        max_tokens=M, max_reqs=8, max_extend_tiles=64, max_dequant_blocks=256 if fp8 else 0, decode_prefix_tokens=P,
        num_heads_q=b.num_heads_q, num_heads_kv=b.num_heads_kv, head_dim=b.head_dim, num_blocks=b.num_blocks,
        max_blocks_per_req=b.block_table.shape[1], softmax_scale=b.softmax_scale,
        kv_cache_dtype=binding.PA_KV_FP8_E4M3 if fp8 else binding.PA_KV_BF16, k_scale=b.k_scale, v_scale=b.v_scale,
        query_start_loc=b.query_start_loc, seq_lens=b.seq_lens, num_computed_tokens=b.num_computed,
        block_table_host=b.block_table)
    ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    bufs = {}
    for name, src in (("q", b.q), ("key", b.key), ("value", b.value)):
        full = torch.zeros((M,) + tuple(src.shape[1:]), dtype=src.dtype, device=dev)
        full[:P] = src[:P].to(dev)
        bufs[name] = (full, src[P:T].to(dev))
    out = torch.zeros_like(bufs["q"][0])
    kc, vc = b.key_cache.to(dev, copy=True), b.value_cache.to(dev, copy=True)
    bt = torch.as_tensor(b.block_table, device=dev)
    slots = torch.zeros(M, dtype=torch.int64, device=dev)
    torch.cuda.synchronize()
    main, side = torch.cuda.current_stream(), torch.cuda.Stream()
    late, late_out = torch.cuda.Event(), torch.cuda.Event()
    binding.pa_upload_metadata(plan, ws, main)
    with torch.cuda.stream(side):
        torch.cuda._sleep(50_000_000)
        for full, rest in bufs.values():
            full[P:T].copy_(rest)
        late.record(side)
    binding.pa_attention_with_kv_update_launch_staged(plan, bufs["q"][0], bufs["key"][0], bufs["value"][0], kc, vc,
                                                      bt, out, ws, late, slot_mapping=slots, stream=main,
                                                      late_out_ready=late_out)
    torch.cuda.synchronize()
    assert late_out.query()
    assert binding.pa_check_device_errors(ws[:4].view(torch.int32)) == 0
    okc, ovc, oslots, oout = run_oracle(before)
    assert np.array_equal(cache_bits(kc), okc) and np.array_equal(cache_bits(vc), ovc)
    assert np.array_equal(slots[:T].cpu().numpy(), oslots)
    assert_close(out[:T], oout, what=f"staged launch ({kv})")


def test_native_graph_rejects_other_model_and_capacity():
    """A step whose model fields differ from the graph's, or that needs more
    than its shape holds, is refused and launches nothing."""
    from paged_kv_cache_16_gb300.step import NativeGraphStep
    dev = torch.device("cuda")
    b = mixed_steps()[0]                    # has extend rows
    kc, vc = b.key_cache.to(dev, copy=True), b.value_cache.to(dev, copy=True)
    ns = NativeGraphStep(key_cache=kc, value_cache=vc, device=dev, **graph_args(b, b.block_table.shape[1]),
                         max_tokens=512, max_reqs=8)   # no tensor-core tiles
    ns.prepare(b, b.q.to(dev), b.key.to(dev), b.value.to(dev))
    with pytest.raises(binding.PaError) as e:
        ns.launch(b.num_reqs)
    assert e.value.status == binding.PA_ERR_CAPACITY
    d = ns.graph._descs[0]
    d.num_reqs = 0
    d.softmax_scale *= 2
    with pytest.raises(binding.PaError) as e:
        ns.graph.step(0)
    assert e.value.status == binding.PA_ERR_INVALID_ARGUMENT
    d.softmax_scale /= 2
    assert ns.graph.turn == 0
    decode = replace(workloads.decode(batch=8, lo=1, hi=300, num_blocks=600, seed=91), name="decode-after")
    ns.run(decode, decode.q.to(dev), decode.key.to(dev), decode.value.to(dev))
    torch.cuda.synchronize()
    assert ns.check_errors() == 0 and ns.graph.turn == 1
    ns.destroy()


def test_native_graph_refuses_pageable_host_io():
    """Host I/O buffers must be page-locked: pageable ones are refused at
    creation, before anything is captured."""
    from paged_kv_cache_16_gb300.step import _input_layout
    dev = torch.device("cuda")
    b = decode_steps()[0]
    kc, vc = b.key_cache.to(dev, copy=True), b.value_cache.to(dev, copy=True)
    lay = _input_layout(b.num_tokens, b.num_reqs, b.num_heads_q, b.num_heads_kv, b.head_dim, b.block_table.shape[1])
    dev_in = torch.zeros(lay["bytes"], dtype=torch.uint8, device=dev)
    out = torch.zeros(b.num_tokens, b.num_heads_q, b.head_dim, dtype=torch.bfloat16, device=dev)
    meta = {"query_start_loc": np.zeros(b.num_reqs + 1, np.int32), "seq_lens": np.zeros(b.num_reqs, np.int32),
            "num_computed": np.zeros(b.num_reqs, np.int32),
            "block_table": np.zeros((b.num_reqs, b.block_table.shape[1]), np.int32)}
    bufs = {"q": dev_in, "key": dev_in, "value": dev_in, "out": out, "query_start_loc": dev_in,
            "num_computed": dev_in, "block_table": dev_in, "key_cache": kc, "value_cache": vc,
            "device_in": dev_in, "in_bytes": lay["bytes"],
            "host_in": [torch.zeros(lay["bytes"], dtype=torch.uint8), torch.zeros(lay["bytes"], dtype=torch.uint8)]}
    ga = graph_args(b, b.block_table.shape[1])
    ga.pop("max_blocks_per_req")
    ga["kv_cache_dtype"] = binding.PA_KV_BF16
    with pytest.raises(binding.PaError) as e:
        binding.NativeGraph(shape=dict(max_tokens=b.num_tokens, max_reqs=b.num_reqs), host=meta, buffers=bufs,
                            num_reqs=0, fused=True, **ga)
    assert e.value.status == binding.PA_ERR_INVALID_ARGUMENT
