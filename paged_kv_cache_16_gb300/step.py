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
    step's graph may still be reading the other.
    """

    def __init__(self, *, num_heads_q, num_heads_kv, head_dim, num_blocks, max_blocks_per_req, softmax_scale,
                 max_tokens, max_reqs, max_extend_tiles=0, max_dequant_blocks=0, max_partial_slots=0,
                 kv_cache_dtype="bf16", k_scale=1.0, v_scale=1.0, num_sms=0, device="cuda", fused=True):
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
        self.q = torch.zeros(max_tokens, num_heads_q, head_dim, dtype=torch.bfloat16, device=dev)
        self.key = torch.zeros(max_tokens, num_heads_kv, head_dim, dtype=torch.bfloat16, device=dev)
        self.value = torch.zeros_like(self.key)
        self.out = torch.zeros_like(self.q)
        self.qsl = torch.zeros(max_reqs + 1, dtype=torch.int32, device=dev)
        self.num_computed = torch.zeros(max_reqs, dtype=torch.int32, device=dev)
        self.block_table = torch.zeros(max_reqs, max_blocks_per_req, dtype=torch.int32, device=dev)
        self.slots = torch.zeros(max_tokens, dtype=torch.int64, device=dev)
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
        R, T = batch.num_reqs, batch.num_tokens
        mr, mb = self.num_computed.numel(), self.block_table.shape[1]
        qsl = np.full(mr + 1, T, dtype=np.int32)
        qsl[:R + 1] = batch.query_start_loc
        nc = np.zeros(mr, dtype=np.int32)
        nc[:R] = batch.num_computed
        bt = np.zeros((mr, mb), dtype=np.int32)
        bt[:R, :batch.block_table.shape[1]] = batch.block_table
        self.qsl.copy_(torch.from_numpy(qsl))
        self.num_computed.copy_(torch.from_numpy(nc))
        self.block_table.copy_(torch.from_numpy(bt))
        for dst, src in ((self.q, q), (self.key, key), (self.value, value)):
            if src is not None:
                dst[:T].copy_(src)

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
                binding.pa_upload_metadata_from(img, nbytes, self.workspace)
                self.enqueue(plan, key_cache, value_cache)
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
