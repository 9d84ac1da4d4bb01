"""One engine step on device tensors: slot mapping, cache write, attention.

Thin glue over the C ABI; torch only allocates memory and supplies streams.
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding
from .workloads import Batch


class DeviceStep:
    """Device-resident metadata, plan, workspace and output of one batch."""

    def __init__(self, batch: Batch, device="cuda", num_sms: int = 0, plan: bool = True):
        self.batch = batch
        dev = torch.device(device)
        self.device = dev
        self.qsl = torch.as_tensor(batch.query_start_loc, device=dev)
        self.seq_lens = torch.as_tensor(batch.seq_lens, device=dev)
        self.num_computed = torch.as_tensor(batch.num_computed, device=dev)
        self.block_table = torch.as_tensor(batch.block_table, device=dev)
        T = batch.num_tokens
        self.slots = torch.empty(max(T, 1), dtype=torch.int64, device=dev)
        self.out = torch.empty(max(T, 1), batch.num_heads_q, batch.head_dim, dtype=torch.bfloat16, device=dev)
        self.num_sms = num_sms
        self.plan = self.make_plan() if plan else None
        ws = self.plan.workspace_bytes if self.plan else 256
        self.workspace = torch.zeros(ws, dtype=torch.uint8, device=dev)

    def make_plan(self) -> binding.Plan:
        b = self.batch
        return binding.pa_plan(num_heads_q=b.num_heads_q, num_heads_kv=b.num_heads_kv, head_dim=b.head_dim,
                               num_blocks=b.num_blocks, query_start_loc=b.query_start_loc,
                               seq_lens=b.seq_lens, num_computed_tokens=b.num_computed,
                               block_table_host=b.block_table,
                               num_common_prefix_blocks=b.num_common_prefix_blocks,
                               softmax_scale=b.softmax_scale, num_sms=self.num_sms,
                               block_size=b.block_size,
                               kv_cache_dtype=binding.PA_KV_FP8_E4M3 if b.kv_cache_dtype == "fp8" else binding.PA_KV_BF16,
                               k_scale=b.k_scale, v_scale=b.v_scale)

    @property
    def error_word(self) -> torch.Tensor:
        return self.workspace[:4].view(torch.int32)

    def slot_mapping(self, stream=None):
        b = self.batch
        binding.pa_slot_mapping(self.qsl, self.num_computed, self.block_table, b.num_tokens, self.slots,
                                b.block_size, stream)
        return self.slots[:b.num_tokens]

    def write(self, key, value, key_cache, value_cache, stream=None):
        if self.batch.kv_cache_dtype == "fp8":
            binding.pa_write_kv_fp8(key, value, self.slots, key_cache, value_cache, self.batch.k_scale,
                                    self.batch.v_scale, self.error_word, stream)
        else:
            binding.pa_write_kv(key, value, self.slots, key_cache, value_cache, self.error_word, stream)

    def attend(self, q, key_cache, value_cache, stream=None, plan=None):
        binding.pa_attention(plan or self.plan, q, key_cache, value_cache, self.block_table, self.out,
                             self.workspace, stream)
        return self.out[:self.batch.num_tokens]

    def run(self, q, key, value, key_cache, value_cache, stream=None):
        """slot mapping -> cache write -> attention; returns out [T, Hq, D]."""
        self.slot_mapping(stream)
        self.write(key, value, key_cache, value_cache, stream)
        return self.attend(q, key_cache, value_cache, stream)

    def run_fused(self, q, key, value, key_cache, value_cache, stream=None, plan=None):
        """Cache write and attention as one call (slots land in self.slots)."""
        binding.pa_attention_with_kv_update(plan or self.plan, q, key, value, key_cache, value_cache,
                                            self.block_table, self.out, self.workspace, self.slots, stream)
        return self.out[:self.batch.num_tokens]

    def check_errors(self, stream=None) -> int:
        return binding.pa_check_device_errors(self.error_word, stream)


def _device_view(ptr: int, n: int, dtype, device) -> torch.Tensor:
    """A tensor over n elements of library-owned device memory (no copy)."""
    typestr = {torch.int64: "<i8", torch.int32: "<i4"}[dtype]

    class _Array:
        __cuda_array_interface__ = {"shape": (n,), "typestr": typestr, "data": (ptr, False), "version": 3}
    return torch.as_tensor(_Array(), device=device)


def _input_layout(max_tokens, max_reqs, hq, hkv, d, mb):
    """Byte offsets of the step's inputs in one block (256-byte aligned)."""
    sizes = [("q", max_tokens * hq * d * 2), ("key", max_tokens * hkv * d * 2), ("value", max_tokens * hkv * d * 2),
             ("qsl", (max_reqs + 1) * 4), ("num_computed", max_reqs * 4), ("block_table", max_reqs * mb * 4),
             ("seq_lens", max_reqs * 4)]
    lay, off = {}, 0
    for name, n in sizes:
        lay[name] = (off, n)
        off += (n + 255) // 256 * 256
    lay["bytes"] = off
    lay["dims"] = (max_tokens, max_reqs, hq, hkv, d, mb)
    return lay


def _input_views(block: torch.Tensor, lay) -> dict:
    """Typed views of an input block (device or page-locked host)."""
    t, r, hq, hkv, d, mb = lay["dims"]

    def view(name, dtype, shape):
        off, n = lay[name]
        return block[off:off + n].view(dtype).view(*shape)
    return {"q": view("q", torch.bfloat16, (t, hq, d)), "key": view("key", torch.bfloat16, (t, hkv, d)),
            "value": view("value", torch.bfloat16, (t, hkv, d)), "qsl": view("qsl", torch.int32, (r + 1,)),
            "num_computed": view("num_computed", torch.int32, (r,)),
            "block_table": view("block_table", torch.int32, (r, mb)), "seq_lens": view("seq_lens", torch.int32, (r,))}


def _fill(views: dict, batch: Batch, q=None, key=None, value=None):
    """Write a step's metadata (padded to the static shapes: spare requests
    get no tokens) and, if given, its new rows into a set of input views."""
    R, T = batch.num_reqs, batch.num_tokens
    mr, mb = views["num_computed"].numel(), views["block_table"].shape[1]
    qsl = np.full(mr + 1, T, dtype=np.int32)
    qsl[:R + 1] = batch.query_start_loc
    nc = np.zeros(mr, dtype=np.int32)
    nc[:R] = batch.num_computed
    bt = np.zeros((mr, mb), dtype=np.int32)
    bt[:R, :batch.block_table.shape[1]] = batch.block_table
    views["qsl"].copy_(torch.from_numpy(qsl))
    views["num_computed"].copy_(torch.from_numpy(nc))
    views["block_table"].copy_(torch.from_numpy(bt))
    if "seq_lens" in views:
        sl = np.zeros(mr, dtype=np.int32)
        sl[:R] = batch.seq_lens
        views["seq_lens"].copy_(torch.from_numpy(sl))
    for name, src in (("q", q), ("key", key), ("value", value)):
        if src is not None:
            views[name][:T].copy_(src)


class GraphStep:
    """Engine steps replayed from one CUDA graph (fixed-shape plans).

    Graph mode as the page "vLLM 源码完全拆解（十六）" (fourth walk-through)
    describes it: the execution of a stable shape is captured once; for every
    step the new data is copied to the same addresses and the graph replayed,
    with request counts rounded up to a capture size and spare rows padded.
    Static buffers hold max_tokens rows of q / key / value / out and max_reqs
    rows of metadata; padding requests have no tokens, so padding tokens get
    slot -1 and are neither written nor attended.  A graph holds the metadata
    upload from a page-locked image (pa_upload_metadata_from), the cache write
    and the attention kernels (fused: pa_attention_with_kv_update_launch; else
    slot mapping, pa_write_kv and pa_attention_launch).  Two images and two
    graphs alternate, so the host writes one step's image while the previous
    step's graph may still be reading the other.  With ``host_io`` each graph
    also brings the step's inputs in from a page-locked input image (one copy:
    q, key, value and the request metadata share one layout) and copies the
    output back to page-locked memory, so a replay goes from host memory to
    host memory.
    """

    def __init__(self, *, num_heads_q, num_heads_kv, head_dim, num_blocks, max_blocks_per_req, softmax_scale,
                 max_tokens, max_reqs, max_extend_tiles=0, max_dequant_blocks=0, max_partial_slots=0,
                 kv_cache_dtype="bf16", k_scale=1.0, v_scale=1.0, num_sms=0, device="cuda", fused=True,
                 host_io=False):
        dev = torch.device(device)
        self.device = dev
        self.fused = fused
        self.model = dict(num_heads_q=num_heads_q, num_heads_kv=num_heads_kv, head_dim=head_dim,
                          num_blocks=num_blocks, max_blocks_per_req=max_blocks_per_req,
                          softmax_scale=softmax_scale, num_sms=num_sms,
                          kv_cache_dtype=binding.PA_KV_FP8_E4M3 if kv_cache_dtype == "fp8" else binding.PA_KV_BF16,
                          k_scale=k_scale, v_scale=v_scale)
        self.shape = dict(max_tokens=max_tokens, max_reqs=max_reqs, max_extend_tiles=max_extend_tiles,
                          max_dequant_blocks=max_dequant_blocks, max_partial_slots=max_partial_slots)
        self.fp8 = kv_cache_dtype == "fp8"
        self.k_scale, self.v_scale = k_scale, v_scale
        # the step's inputs (q, key, value, query_start_loc, num_computed,
        # block_table) are views of one device block, so that one copy from a
        # page-locked image of the same layout brings a whole step in
        self._in_layout = _input_layout(max_tokens, max_reqs, num_heads_q, num_heads_kv, head_dim,
                                        max_blocks_per_req)
        self._in = torch.zeros(self._in_layout["bytes"], dtype=torch.uint8, device=dev)
        views = _input_views(self._in, self._in_layout)
        self.q, self.key, self.value = views["q"], views["key"], views["value"]
        self.qsl, self.num_computed, self.block_table = views["qsl"], views["num_computed"], views["block_table"]
        self.out = torch.zeros_like(self.q)
        self.slots = torch.zeros(max_tokens, dtype=torch.int64, device=dev)
        # host_io: each graph also copies a page-locked input image (the
        # layout above) to the device first and the output back last, so a
        # replay is a whole step from host memory to host memory
        self.host_in = None
        self.host_out = None
        if host_io:
            self.host_in = [torch.zeros(self._in_layout["bytes"], dtype=torch.uint8).pin_memory() for _ in range(2)]
            self.host_out = [torch.zeros(self.out.shape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        self.workspace = None
        self.graphs = None       # two captures, one per metadata image
        self.images = None       # page-locked metadata images
        self.done = None         # events: the last replay of graph i has run
        self.turn = 0
        self.caches = None

    def make_plan(self, batch: Batch) -> binding.Plan:
        bt = batch.block_table
        mb = self.model["max_blocks_per_req"]
        if bt.shape[1] != mb:                      # host copy with the static row stride
            padded = np.zeros((bt.shape[0], mb), dtype=np.int32)
            padded[:, :bt.shape[1]] = bt
            bt = padded
        return binding.pa_plan_fixed(**self.shape, query_start_loc=batch.query_start_loc, seq_lens=batch.seq_lens,
                                     num_computed_tokens=batch.num_computed, block_table_host=bt,
                                     num_common_prefix_blocks=batch.num_common_prefix_blocks, **self.model)

    @property
    def error_word(self) -> torch.Tensor:
        return self.workspace[:4].view(torch.int32)

    def load(self, batch: Batch, plan: binding.Plan, q=None, key=None, value=None, stream=None):
        """Copy a step's metadata (and, if given, its new q / key / value rows)
        into the static buffers and upload the plan's metadata (not captured)."""
        self.stage(batch, q, key, value)
        if self.workspace is None:
            self.workspace = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device=self.device)
        binding.pa_upload_metadata(plan, self.workspace, stream)

    def stage(self, batch: Batch, q=None, key=None, value=None):
        """Copy a step's request metadata and new rows into the static buffers."""
        _fill({"q": self.q, "key": self.key, "value": self.value, "qsl": self.qsl,
               "num_computed": self.num_computed, "block_table": self.block_table}, batch, q, key, value)

    def host_inputs(self, i=None) -> dict:
        """Views of page-locked input image i (default: the one the next
        replay copies in): q, key, value, qsl, num_computed, block_table."""
        return _input_views(self.host_in[self.turn if i is None else i], self._in_layout)

    def stage_host(self, batch: Batch, q=None, key=None, value=None, i=None):
        """Write a step's metadata and new rows into page-locked input image i."""
        if i is None and self.done is not None:
            self.done[self.turn].synchronize()   # the replay that last read it has run
        _fill(self.host_inputs(i), batch, q, key, value)

    def host_output(self, num_tokens: int) -> torch.Tensor:
        """The last replay's output in page-locked host memory (waits for it)."""
        i = 1 - self.turn
        self.done[i].synchronize()
        return self.host_out[i][:num_tokens]

    def enqueue(self, plan: binding.Plan, key_cache, value_cache, stream=None):
        """Slot mapping, cache write and attention over the static buffers
        (every launch sized by the capacities; capturable).  Fused: one
        pa_attention_with_kv_update_launch does all three."""
        if self.fused:
            binding.pa_attention_with_kv_update_launch(plan, self.q, self.key, self.value, key_cache, value_cache,
                                                       self.block_table, self.out, self.workspace, self.slots, stream)
            return
        binding.pa_slot_mapping(self.qsl, self.num_computed, self.block_table, self.slots.numel(), self.slots,
                                stream=stream)
        if self.fp8:
            binding.pa_write_kv_fp8(self.key, self.value, self.slots, key_cache, value_cache, self.k_scale,
                                    self.v_scale, self.error_word, stream)
        else:
            binding.pa_write_kv(self.key, self.value, self.slots, key_cache, value_cache, self.error_word, stream)
        binding.pa_attention_launch(plan, self.q, key_cache, value_cache, self.block_table, self.out,
                                    self.workspace, stream)

    def capture(self, plan: binding.Plan, key_cache, value_cache):
        """Capture the upload of each metadata image followed by enqueue();
        the caches are part of the graphs."""
        if self.workspace is None:
            self.workspace = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device=self.device)
        binding.pa_upload_metadata(plan, self.workspace)   # prepares the kernels (not capturable)
        nbytes = binding.pa_plan_metadata_bytes(plan)
        self.images = [torch.zeros(max(nbytes, 16), dtype=torch.uint8).pin_memory() for _ in range(2)]
        for img in self.images:
            binding.pa_plan_copy_metadata(plan, img)
        self.graphs = []
        for img in self.images:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                if self.host_in is not None:
                    self._in.copy_(self.host_in[len(self.graphs)], non_blocking=True)
                binding.pa_upload_metadata_from(img, nbytes, self.workspace)
                self.enqueue(plan, key_cache, value_cache)
                if self.host_out is not None:
                    self.host_out[len(self.graphs)].copy_(self.out, non_blocking=True)
            self.graphs.append(g)
        self.done = [torch.cuda.Event(), torch.cuda.Event()]
        self.turn = 0
        self.caches = (key_cache.data_ptr(), value_cache.data_ptr())

    def prepare_replay(self, plan: binding.Plan):
        """Write the plan's metadata image for the next replay (host work)."""
        i = self.turn
        self.done[i].synchronize()   # the replay that last read image i has run
        binding.pa_plan_copy_metadata(plan, self.images[i])

    def launch_replay(self):
        """Replay the graph that uploads the prepared image."""
        i = self.turn
        self.graphs[i].replay()
        self.done[i].record()
        self.turn = 1 - i

    def replay(self, plan: binding.Plan):
        """Write the plan's metadata image and replay the graph that uploads it."""
        self.prepare_replay(plan)
        self.launch_replay()

    def run(self, batch: Batch, q, key, value, key_cache, value_cache) -> torch.Tensor:
        """One step: plan, copy in, replay (capturing on first use)."""
        plan = self.make_plan(batch)
        self.stage(batch, q, key, value)
        if self.graphs is None:
            self.capture(plan, key_cache, value_cache)
        elif self.caches != (key_cache.data_ptr(), value_cache.data_ptr()):
            raise ValueError("a captured step replays on the caches it was captured with")
        self.replay(plan)
        return self.out[:batch.num_tokens]

    def check_errors(self, stream=None) -> int:
        return binding.pa_check_device_errors(self.error_word, stream)


class NativeGraphStep:
    """Engine steps through the library's own graph executor (pa_graph_*).

    The same graph mode as GraphStep (two graphs of one fixed shape, each
    uploading its own page-locked metadata image, alternating), but captured,
    planned and launched inside the library: a step is one C call
    (pa_graph_step: fixed plan from the host metadata, copy of its metadata
    image, graph launch).  The inputs share one layout (q, key, value,
    query_start_loc, num_computed, block_table, seq_lens).  With ``host_io``
    the graphs copy a page-locked input image in first and the output back
    last, and the planner reads the metadata from that same image; without
    it the caller stages device inputs (``prepare``) and host metadata.
    """

    def __init__(self, *, num_heads_q, num_heads_kv, head_dim, num_blocks, max_blocks_per_req, softmax_scale,
                 max_tokens, max_reqs, key_cache, value_cache, max_extend_tiles=0, max_dequant_blocks=0,
                 max_partial_slots=0, kv_cache_dtype="bf16", k_scale=1.0, v_scale=1.0, num_sms=0, device="cuda",
                 fused=True, host_io=False, out_rows=None, decode_prefix_tokens=0):
        dev = torch.device(device)
        self.device = dev
        self.host_io = host_io
        lay = _input_layout(max_tokens, max_reqs, num_heads_q, num_heads_kv, head_dim, max_blocks_per_req)
        self._lay = lay
        self._in = torch.zeros(lay["bytes"], dtype=torch.uint8, device=dev)
        self.inputs = _input_views(self._in, lay)
        self.out = torch.zeros(max_tokens, num_heads_q, head_dim, dtype=torch.bfloat16, device=dev)
        bufs = {"q": self.inputs["q"], "key": self.inputs["key"], "value": self.inputs["value"], "out": self.out,
                "query_start_loc": self.inputs["qsl"], "num_computed": self.inputs["num_computed"],
                "block_table": self.inputs["block_table"], "key_cache": key_cache, "value_cache": value_cache}
        if host_io:
            self.host_in = [torch.zeros(lay["bytes"], dtype=torch.uint8).pin_memory() for _ in range(2)]
            # out_rows < max_tokens: host buffers for the first out_rows rows
            # only, which the graph copies back at its end (a whole-output
            # buffer is stored into by the kernels instead)
            rows = max_tokens if out_rows is None else out_rows
            self.host_out = [torch.zeros((rows,) + tuple(self.out.shape[1:]), dtype=torch.bfloat16).pin_memory()
                             for _ in range(2)]
            views = [_input_views(t, lay) for t in self.host_in]
            bufs.update(host_in=self.host_in, device_in=self._in, in_bytes=lay["bytes"], host_out=self.host_out,
                        out_bytes=self.host_out[0].numel() * 2)
        else:
            self.host_in = self.host_out = None
            meta = {"qsl": np.zeros(max_reqs + 1, dtype=np.int32), "seq_lens": np.zeros(max_reqs, dtype=np.int32),
                    "num_computed": np.zeros(max_reqs, dtype=np.int32),
                    "block_table": np.zeros((max_reqs, max_blocks_per_req), dtype=np.int32)}
            views = [{k: torch.from_numpy(v) for k, v in meta.items()}] * 2
        self._host_views = views
        host = [{"query_start_loc": v["qsl"].numpy(), "seq_lens": v["seq_lens"].numpy(),
                 "num_computed": v["num_computed"].numpy(), "block_table": v["block_table"].numpy()} for v in views]
        self.graph = binding.NativeGraph(
            shape=dict(max_tokens=max_tokens, max_reqs=max_reqs, max_extend_tiles=max_extend_tiles,
                       max_dequant_blocks=max_dequant_blocks, max_partial_slots=max_partial_slots,
                       decode_prefix_tokens=decode_prefix_tokens),
            host=host, buffers=bufs, num_reqs=0, fused=fused, num_heads_q=num_heads_q, num_heads_kv=num_heads_kv,
            head_dim=head_dim, num_blocks=num_blocks, softmax_scale=softmax_scale, num_sms=num_sms,
            kv_cache_dtype=binding.PA_KV_FP8_E4M3 if kv_cache_dtype == "fp8" else binding.PA_KV_BF16,
            k_scale=k_scale, v_scale=v_scale)
        self._last = None   # graph index of the last step launched
        self._keep = (key_cache, value_cache)

    def prepare(self, batch: Batch, q=None, key=None, value=None):
        """Write the step's metadata and new rows where the next graph reads
        them: its page-locked input image (host_io; after that graph's last
        run finished) or the device inputs and host metadata (after the last
        step finished)."""
        i = self.graph.turn
        if self.host_io:
            self.graph.wait(i)
            _fill(self._host_views[i], batch, q, key, value)
            return
        if self._last is not None:
            self.graph.wait(self._last)
        _fill(self._host_views[0], batch)
        _fill(self.inputs, batch, q, key, value)

    def fill_host_image(self, i: int, batch: Batch, q=None, key=None, value=None):
        """Write a step into page-locked input image i (host_io), after graph
        i's last run finished."""
        self.graph.wait(i)
        _fill(self._host_views[i], batch, q, key, value)

    def launch(self, num_reqs: int, num_common_prefix_blocks: int = 0, stream=None):
        """One step: plan (host), metadata image, graph launch (one C call)."""
        turn = self.graph.turn
        self.graph.step(num_reqs, stream, num_common_prefix_blocks)
        self._last = turn

    def output(self, num_tokens: int) -> torch.Tensor:
        """The last step's output: page-locked host memory (host_io, after
        waiting for it) or the device buffer (stream ordered)."""
        if self.host_io:
            self.graph.wait(self._last)
            return self.host_out[self._last][:num_tokens]
        return self.out[:num_tokens]

    def run(self, batch: Batch, q, key, value) -> torch.Tensor:
        self.prepare(batch, q, key, value)
        self.launch(batch.num_reqs, batch.num_common_prefix_blocks)
        return self.output(batch.num_tokens)

    @property
    def slot_mapping(self) -> torch.Tensor:
        """Device slot buffer of the executor (int64 [max_tokens]), as a tensor view."""
        return _device_view(self.graph.slot_mapping_ptr(), self.out.shape[0], torch.int64, self.device)

    def check_errors(self, stream=None) -> int:
        return binding.pa_check_device_errors(self.graph.workspace_ptr(), stream)

    def destroy(self):
        self.graph.destroy()
