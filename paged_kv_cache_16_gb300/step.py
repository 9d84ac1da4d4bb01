"""One engine step on device tensors: slot mapping, cache write, attention.

Thin glue over the C ABI; torch only allocates memory and supplies streams.
"""
from __future__ import annotations

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

    def check_errors(self, stream=None) -> int:
        return binding.pa_check_device_errors(self.error_word, stream)
