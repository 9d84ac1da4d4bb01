"""ctypes binding of libpa.so: argument marshalling only.

Every function here forwards to the C ABI declared in ``include/pa.h`` with
the same name; device tensors are passed as raw pointers (``data_ptr()``)
and streams as ``cudaStream_t`` handles.  No step of the computation runs in
Python: if the compiled library is missing, loading fails with an error.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

from . import build as _build

PA_OK = 0
PA_ERR_INVALID_ARGUMENT = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_CUDA = 3
PA_ERR_DEVICE_CHECK = 4
PA_ERR_WORKSPACE_TOO_SMALL = 5
PA_ERR_CAPACITY = 6

PA_KV_BF16 = 0
PA_KV_FP8_E4M3 = 1

PA_DEVERR_SLOT_RANGE = 0x1
PA_DEVERR_BLOCK_RANGE = 0x2
PA_DEVERR_TIMEOUT = 0x4

# symbols include/pa.h declares (checked by the CPU tests)
EXPORTED = ("pa_plan", "pa_plan_destroy", "pa_plan_get_info", "pa_slot_mapping", "pa_write_kv",
            "pa_attention", "pa_check_device_errors", "pa_plan_enable_timing",
            "pa_plan_kernel_times", "pa_status_string", "pa_attention_no_alloc", "pa_write_kv_fp8",
            "pa_plan_fixed", "pa_upload_metadata", "pa_attention_launch", "pa_zero_blocks",
            "pa_attention_with_kv_update", "pa_attention_with_kv_update_launch", "pa_plan_metadata_bytes",
            "pa_plan_copy_metadata", "pa_upload_metadata_from", "pa_graph_create", "pa_graph_step",
            "pa_graph_turn", "pa_graph_wait", "pa_graph_workspace", "pa_graph_slot_mapping", "pa_graph_destroy",
            "pa_attention_with_kv_update_launch_staged")


class PaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} ({status})")
        self.status = status


class BatchDesc(ctypes.Structure):
    _fields_ = [
        ("num_reqs", ctypes.c_int32),
        ("num_heads_q", ctypes.c_int32),
        ("num_heads_kv", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32),
        ("max_blocks_per_req", ctypes.c_int32),
        ("query_start_loc", ctypes.c_void_p),      # const int32_t * (host)
        ("seq_lens", ctypes.c_void_p),
        ("num_computed_tokens", ctypes.c_void_p),
        ("block_table_host", ctypes.c_void_p),
        ("num_common_prefix_blocks", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float),
        ("num_sms", ctypes.c_int32),
        ("kv_cache_dtype", ctypes.c_int32),
        ("k_scale", ctypes.c_float),
        ("v_scale", ctypes.c_float),
    ]


class PlanInfo(ctypes.Structure):
    _fields_ = [
        ("num_tokens", ctypes.c_int32),
        ("num_decode_rows", ctypes.c_int32),
        ("num_extend_rows", ctypes.c_int32),
        ("num_decode_ctas", ctypes.c_int32),
        ("num_decode_items", ctypes.c_int32),
        ("num_extend_tiles", ctypes.c_int32),
        ("num_prefix_tiles", ctypes.c_int32),
        ("num_partial_slots", ctypes.c_int32),
        ("num_merge_rows", ctypes.c_int32),
        ("kernels_per_call", ctypes.c_int32),
        ("num_dequant_blocks", ctypes.c_int32),
        ("decode_kv_bytes", ctypes.c_int64),
        ("prefix_kv_bytes", ctypes.c_int64),
        ("extend_flops", ctypes.c_double),
        ("prefix_flops", ctypes.c_double),
        ("num_small_q_rows", ctypes.c_int32),
        ("num_extend_ctas", ctypes.c_int32),
        ("side_by_side", ctypes.c_int32),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


_LIB = None


class FixedShape(ctypes.Structure):
    _fields_ = [
        ("max_tokens", ctypes.c_int32),
        ("max_reqs", ctypes.c_int32),
        ("max_extend_tiles", ctypes.c_int32),
        ("max_dequant_blocks", ctypes.c_int32),
        ("max_partial_slots", ctypes.c_int32),
        ("decode_prefix_tokens", ctypes.c_int32),
    ]


class GraphBuffers(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p),
        ("key", ctypes.c_void_p),
        ("value", ctypes.c_void_p),
        ("out", ctypes.c_void_p),
        ("query_start_loc", ctypes.c_void_p),
        ("num_computed", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p),
        ("key_cache", ctypes.c_void_p),
        ("value_cache", ctypes.c_void_p),
        ("fused", ctypes.c_int32),
        ("host_in", ctypes.c_void_p * 2),
        ("device_in", ctypes.c_void_p),
        ("in_bytes", ctypes.c_size_t),
        ("host_out", ctypes.c_void_p * 2),
        ("out_bytes", ctypes.c_size_t),
    ]


def library_path() -> str:
    return _build.LIBRARY


def load(path: str | None = None, build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libpa.so (optionally building it first)."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or _build.LIBRARY
    if not os.path.exists(p):
        if build_if_missing:
            p = _build.build()
        else:
            raise RuntimeError(f"libpa.so not built ({p}); run paged_kv_cache_16_gb300.build.build()")
    lib = ctypes.CDLL(p)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    i32p = ctypes.POINTER(ctypes.c_int32)
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_status_string.argtypes = [ctypes.c_int]
    lib.pa_plan.restype = ctypes.c_int
    lib.pa_plan.argtypes = [ctypes.POINTER(BatchDesc), ctypes.POINTER(vp), ctypes.POINTER(sz)]
    lib.pa_plan_fixed.restype = ctypes.c_int
    lib.pa_plan_fixed.argtypes = [ctypes.POINTER(BatchDesc), ctypes.POINTER(FixedShape), ctypes.POINTER(vp),
                                  ctypes.POINTER(sz)]
    lib.pa_upload_metadata.restype = ctypes.c_int
    lib.pa_upload_metadata.argtypes = [vp, vp, sz, vp]
    lib.pa_plan_metadata_bytes.restype = sz
    lib.pa_plan_metadata_bytes.argtypes = [vp]
    lib.pa_plan_copy_metadata.restype = ctypes.c_int
    lib.pa_plan_copy_metadata.argtypes = [vp, vp, sz]
    lib.pa_upload_metadata_from.restype = ctypes.c_int
    lib.pa_upload_metadata_from.argtypes = [vp, sz, vp, sz, vp]
    lib.pa_graph_create.restype = ctypes.c_int
    lib.pa_graph_create.argtypes = [vp, vp, vp, ctypes.POINTER(vp)]
    lib.pa_graph_step.restype = ctypes.c_int
    lib.pa_graph_step.argtypes = [vp, vp, vp]
    lib.pa_graph_turn.restype = i32
    lib.pa_graph_turn.argtypes = [vp]
    lib.pa_graph_wait.restype = ctypes.c_int
    lib.pa_graph_wait.argtypes = [vp, i32]
    lib.pa_graph_workspace.restype = vp
    lib.pa_graph_workspace.argtypes = [vp]
    lib.pa_graph_slot_mapping.restype = vp
    lib.pa_graph_slot_mapping.argtypes = [vp]
    lib.pa_graph_destroy.restype = None
    lib.pa_graph_destroy.argtypes = [vp]
    lib.pa_attention_launch.restype = ctypes.c_int
    lib.pa_attention_launch.argtypes = [vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.pa_attention_with_kv_update.restype = ctypes.c_int
    lib.pa_attention_with_kv_update.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.pa_attention_with_kv_update_launch.restype = ctypes.c_int
    lib.pa_attention_with_kv_update_launch.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.pa_attention_with_kv_update_launch_staged.restype = ctypes.c_int
    lib.pa_attention_with_kv_update_launch_staged.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp, vp]
    lib.pa_zero_blocks.restype = ctypes.c_int
    lib.pa_zero_blocks.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, vp, vp]
    lib.pa_plan_destroy.restype = None
    lib.pa_plan_destroy.argtypes = [vp]
    lib.pa_plan_get_info.restype = ctypes.c_int
    lib.pa_plan_get_info.argtypes = [vp, ctypes.POINTER(PlanInfo)]
    lib.pa_slot_mapping.restype = ctypes.c_int
    lib.pa_slot_mapping.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp]
    lib.pa_write_kv.restype = ctypes.c_int
    lib.pa_write_kv.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp, i64, vp, vp]
    lib.pa_write_kv_fp8.restype = ctypes.c_int
    lib.pa_write_kv_fp8.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp, i64, ctypes.c_float, ctypes.c_float, vp, vp]
    lib.pa_attention.restype = ctypes.c_int
    lib.pa_attention.argtypes = [vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.pa_attention_no_alloc.restype = ctypes.c_int
    lib.pa_attention_no_alloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
    lib.pa_check_device_errors.restype = ctypes.c_int
    lib.pa_check_device_errors.argtypes = [vp, i32p, vp]
    lib.pa_plan_enable_timing.restype = ctypes.c_int
    lib.pa_plan_enable_timing.argtypes = [vp, i32]
    lib.pa_plan_kernel_times.restype = ctypes.c_int
    lib.pa_plan_kernel_times.argtypes = [vp, ctypes.POINTER(ctypes.c_double), i32p]
    if path is None:
        _LIB = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load().pa_status_string(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


def _check(status: int, what: str):
    if status != PA_OK:
        raise PaError(status, what)


def _ptr(t) -> int | None:
    """Raw device/host address of a tensor or an address (or None)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return int(t.data_ptr())


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


@dataclass
class Plan:
    handle: int
    workspace_bytes: int
    _keep: tuple  # host arrays referenced while pa_plan runs

    def info(self) -> dict:
        pi = PlanInfo()
        _check(load().pa_plan_get_info(self.handle, ctypes.byref(pi)), "pa_plan_get_info")
        return pi.as_dict()

    def enable_timing(self, on: bool = True):
        _check(load().pa_plan_enable_timing(self.handle, 1 if on else 0), "pa_plan_enable_timing")

    def kernel_times(self):
        ms = (ctypes.c_double * 4)()
        n = (ctypes.c_int32 * 4)()
        _check(load().pa_plan_kernel_times(self.handle, ms, n), "pa_plan_kernel_times")
        return list(ms), list(n)

    def destroy(self):
        if self.handle:
            load().pa_plan_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.destroy()
        except Exception:  # noqa: BLE001 -- interpreter shutdown
            pass


def make_desc(*, num_heads_q, num_heads_kv, head_dim, num_blocks, query_start_loc, seq_lens,
              num_computed_tokens, block_table_host=None, max_blocks_per_req=None,
              num_common_prefix_blocks=0, softmax_scale, num_sms=0, block_size=16, kv_cache_dtype=0,
              k_scale=1.0, v_scale=1.0):
    qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    nc = np.ascontiguousarray(num_computed_tokens, dtype=np.int32)
    bt = None if block_table_host is None else np.ascontiguousarray(block_table_host, dtype=np.int32)
    if max_blocks_per_req is None:
        max_blocks_per_req = bt.shape[1] if bt is not None else 1
    d = BatchDesc(len(sl), num_heads_q, num_heads_kv, head_dim, block_size, num_blocks, int(max_blocks_per_req),
                  qsl.ctypes.data, sl.ctypes.data, nc.ctypes.data, bt.ctypes.data if bt is not None else None,
                  int(num_common_prefix_blocks), float(softmax_scale), int(num_sms), int(kv_cache_dtype),
                  float(k_scale), float(v_scale))
    return d, (qsl, sl, nc, bt)


def pa_plan(**kw) -> Plan:
    """Validate the step's metadata and build its plan (see pa.h)."""
    d, keep = make_desc(**kw)
    handle = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    _check(load().pa_plan(ctypes.byref(d), ctypes.byref(handle), ctypes.byref(ws)), "pa_plan")
    return Plan(handle.value, ws.value, keep)


def _fixed_shape(max_tokens, max_reqs, max_extend_tiles=0, max_dequant_blocks=0, max_partial_slots=0,
                 decode_prefix_tokens=0):
    fs = FixedShape()
    fs.max_tokens, fs.max_reqs = int(max_tokens), int(max_reqs)
    fs.max_extend_tiles, fs.max_dequant_blocks = int(max_extend_tiles), int(max_dequant_blocks)
    fs.max_partial_slots = int(max_partial_slots)
    fs.decode_prefix_tokens = int(decode_prefix_tokens)
    return fs


def pa_plan_fixed(*, max_tokens, max_reqs, max_extend_tiles=0, max_dequant_blocks=0, max_partial_slots=0,
                  decode_prefix_tokens=0, **kw) -> Plan:
    """A fixed-shape plan (graph-capturable launches, see pa.h)."""
    d, keep = make_desc(**kw)
    fs = _fixed_shape(max_tokens, max_reqs, max_extend_tiles, max_dequant_blocks, max_partial_slots,
                      decode_prefix_tokens)
    handle = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    _check(load().pa_plan_fixed(ctypes.byref(d), ctypes.byref(fs), ctypes.byref(handle), ctypes.byref(ws)),
           "pa_plan_fixed")
    return Plan(handle.value, ws.value, keep)


def pa_plan_fixed_status(*, max_tokens, max_reqs, max_extend_tiles=0, max_dequant_blocks=0, max_partial_slots=0,
                         decode_prefix_tokens=0, **kw) -> int:
    """Status code pa_plan_fixed returns (plan discarded)."""
    d, keep = make_desc(**kw)
    fs = _fixed_shape(max_tokens, max_reqs, max_extend_tiles, max_dequant_blocks, max_partial_slots,
                      decode_prefix_tokens)
    handle = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    st = load().pa_plan_fixed(ctypes.byref(d), ctypes.byref(fs), ctypes.byref(handle), ctypes.byref(ws))
    if st == PA_OK:
        load().pa_plan_destroy(handle.value)
    return st


def pa_plan_status(**kw) -> int:
    """Status code pa_plan returns for this descriptor (plan discarded)."""
    d, keep = make_desc(**kw)
    handle = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    st = load().pa_plan(ctypes.byref(d), ctypes.byref(handle), ctypes.byref(ws))
    if st == PA_OK:
        load().pa_plan_destroy(handle.value)
    return st


def pa_slot_mapping(query_start_loc, num_computed, block_table, num_tokens: int, slot_mapping,
                    block_size: int = 16, stream=None):
    _check(load().pa_slot_mapping(_ptr(query_start_loc), _ptr(num_computed), _ptr(block_table),
                                  int(num_computed.numel()), int(num_tokens), int(block_table.shape[1]),
                                  int(block_size), _ptr(slot_mapping), _stream(stream)), "pa_slot_mapping")


def pa_write_kv(key, value, slot_mapping, key_cache, value_cache, device_error_word=None, stream=None):
    T, hkv, d = key.shape
    num_slots = key_cache.shape[0] * key_cache.shape[1]
    _check(load().pa_write_kv(_ptr(key), _ptr(value), _ptr(slot_mapping), T, hkv, d, _ptr(key_cache),
                              _ptr(value_cache), num_slots, _ptr(device_error_word), _stream(stream)),
           "pa_write_kv")


def pa_write_kv_fp8(key, value, slot_mapping, key_cache, value_cache, k_scale: float, v_scale: float,
                    device_error_word=None, stream=None):
    """Quantising cache write into E4M3 caches (uint8 tensors)."""
    T, hkv, d = key.shape
    num_slots = key_cache.shape[0] * key_cache.shape[1]
    _check(load().pa_write_kv_fp8(_ptr(key), _ptr(value), _ptr(slot_mapping), T, hkv, d, _ptr(key_cache),
                                  _ptr(value_cache), num_slots, float(k_scale), float(v_scale),
                                  _ptr(device_error_word), _stream(stream)), "pa_write_kv_fp8")


def pa_attention(plan: Plan, q, key_cache, value_cache, block_table, out, workspace, stream=None):
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().pa_attention(plan.handle, _ptr(q), _ptr(key_cache), _ptr(value_cache), _ptr(block_table),
                               _ptr(out), _ptr(workspace), nbytes, _stream(stream)), "pa_attention")


def pa_upload_metadata(plan: Plan, workspace, stream=None):
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().pa_upload_metadata(plan.handle, _ptr(workspace), nbytes, _stream(stream)), "pa_upload_metadata")


def pa_plan_metadata_bytes(plan: Plan) -> int:
    return int(load().pa_plan_metadata_bytes(plan.handle))


def pa_plan_copy_metadata_status(plan: Plan, host_dst, nbytes: int) -> int:
    """Raw status of pa_plan_copy_metadata into host memory at address host_dst."""
    return load().pa_plan_copy_metadata(plan.handle, host_dst, nbytes)


def pa_plan_copy_metadata(plan: Plan, host_dst):
    """Copy the plan's metadata image into a host tensor (uint8, at least
    pa_plan_metadata_bytes long)."""
    nbytes = host_dst.numel() * host_dst.element_size()
    _check(pa_plan_copy_metadata_status(plan, _ptr(host_dst), nbytes), "pa_plan_copy_metadata")


def pa_upload_metadata_from(host_src, nbytes: int, workspace, stream=None):
    """Enqueue the upload of a metadata image from page-locked host memory
    (capturable; see pa.h)."""
    wbytes = workspace.numel() * workspace.element_size()
    _check(load().pa_upload_metadata_from(_ptr(host_src), nbytes, _ptr(workspace), wbytes, _stream(stream)),
           "pa_upload_metadata_from")


def pa_attention_launch(plan: Plan, q, key_cache, value_cache, block_table, out, workspace, stream=None):
    """The attention kernels alone (capturable in a CUDA graph; see pa.h)."""
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().pa_attention_launch(plan.handle, _ptr(q), _ptr(key_cache), _ptr(value_cache), _ptr(block_table),
                                      _ptr(out), _ptr(workspace), nbytes, _stream(stream)), "pa_attention_launch")


def pa_attention_with_kv_update(plan: Plan, q, key, value, key_cache, value_cache, block_table, out, workspace,
                                slot_mapping=None, stream=None):
    """Cache write + attention in one call (see pa.h)."""
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().pa_attention_with_kv_update(plan.handle, _ptr(q), _ptr(key), _ptr(value), _ptr(key_cache),
                                              _ptr(value_cache), _ptr(block_table), _ptr(slot_mapping), _ptr(out),
                                              _ptr(workspace), nbytes, _stream(stream)),
           "pa_attention_with_kv_update")


def pa_attention_with_kv_update_launch(plan: Plan, q, key, value, key_cache, value_cache, block_table, out,
                                       workspace, slot_mapping=None, stream=None):
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().pa_attention_with_kv_update_launch(plan.handle, _ptr(q), _ptr(key), _ptr(value), _ptr(key_cache),
                                                     _ptr(value_cache), _ptr(block_table), _ptr(slot_mapping),
                                                     _ptr(out), _ptr(workspace), nbytes, _stream(stream)),
           "pa_attention_with_kv_update_launch")


def pa_attention_with_kv_update_launch_staged(plan: Plan, q, key, value, key_cache, value_cache, block_table, out,
                                              workspace, late_rows, slot_mapping=None, stream=None,
                                              late_out_ready=None):
    """As pa_attention_with_kv_update_launch; rows from the plan's decode
    prefix on may still be written until late_rows (a torch.cuda.Event,
    already recorded) fires.  late_out_ready (a torch.cuda.Event) is recorded
    once out's rows from the prefix on are final."""
    nbytes = workspace.numel() * workspace.element_size()
    if late_out_ready is not None and not late_out_ready.cuda_event:
        late_out_ready.record()   # torch creates the CUDA event at its first record
    _check(load().pa_attention_with_kv_update_launch_staged(
        plan.handle, _ptr(q), _ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache), _ptr(block_table),
        _ptr(slot_mapping), _ptr(out), _ptr(workspace), nbytes, _stream(stream),
        ctypes.c_void_p(late_rows.cuda_event if late_rows is not None else 0),
        ctypes.c_void_p(late_out_ready.cuda_event if late_out_ready is not None else 0)),
        "pa_attention_with_kv_update_launch_staged")


def pa_zero_blocks(block_ids, key_cache, value_cache, device_error_word=None, stream=None):
    """Zero the K and V entries of the listed blocks (ids < 0 skipped)."""
    nb, bs, hkv, d = key_cache.shape
    kv = PA_KV_FP8_E4M3 if key_cache.element_size() == 1 else PA_KV_BF16
    _check(load().pa_zero_blocks(_ptr(block_ids), int(block_ids.numel()), nb, hkv, d, kv, _ptr(key_cache),
                                 _ptr(value_cache), _ptr(device_error_word), _stream(stream)), "pa_zero_blocks")


def pa_attention_no_alloc(plan: Plan, q, key_cache, value_cache, block_table, out, device_error_word=None,
                          stream=None):
    """pa_attention with the library's fixed scratch array instead of a workspace
    (for callers that cannot allocate device memory; see pa.h)."""
    _check(load().pa_attention_no_alloc(plan.handle, _ptr(q), _ptr(key_cache), _ptr(value_cache),
                                        _ptr(block_table), _ptr(out), _ptr(device_error_word), _stream(stream)),
           "pa_attention_no_alloc")


NO_ALLOC_SCRATCH_BYTES = 16 << 20


def pa_check_device_errors(word, stream=None) -> int:
    """Read and clear a device error word; returns the PA_DEVERR_* bits seen."""
    bits = ctypes.c_int32(0)
    st = load().pa_check_device_errors(_ptr(word), ctypes.byref(bits), _stream(stream))
    if st not in (PA_OK, PA_ERR_DEVICE_CHECK):
        raise PaError(st, "pa_check_device_errors")
    return int(bits.value)


class NativeGraph:
    """pa_graph_t: the two captured step graphs of one fixed shape (see pa.h).

    ``host``: the step's metadata arrays the planner reads each step
    (query_start_loc [max_reqs+1], seq_lens [max_reqs], num_computed
    [max_reqs], block_table [max_reqs][max_blocks_per_req], int32 numpy
    arrays kept by the caller and rewritten in place), or a pair of such sets,
    one per graph (step n reads set ``turn``); ``num_reqs`` is set per step.
    ``buffers``: the device (and optional page-locked host I/O) buffers of
    pa_graph_buffers, as tensors or raw addresses.
    """

    def __init__(self, *, shape: dict, host: dict, buffers: dict, num_reqs: int, fused: bool, **model):
        sets = list(host) if isinstance(host, (list, tuple)) else [host, host]
        self._host = sets
        self._descs = []
        for hs in sets:
            for k in ("query_start_loc", "seq_lens", "num_computed", "block_table"):
                a = hs[k]
                if not (isinstance(a, np.ndarray) and a.dtype == np.int32 and a.flags.c_contiguous):
                    raise ValueError(f"host[{k!r}] must be a C-contiguous int32 numpy array")
            d, _ = make_desc(query_start_loc=hs["query_start_loc"], seq_lens=hs["seq_lens"],
                             num_computed_tokens=hs["num_computed"], block_table_host=hs["block_table"], **model)
            # the descriptor points into the caller's arrays, rewritten each step
            d.query_start_loc = hs["query_start_loc"].ctypes.data
            d.seq_lens = hs["seq_lens"].ctypes.data
            d.num_computed_tokens = hs["num_computed"].ctypes.data
            d.block_table_host = hs["block_table"].ctypes.data
            d.num_reqs = int(num_reqs)
            self._descs.append(d)
        self._shape = _fixed_shape(**shape)
        addr = lambda t: None if t is None else (t if isinstance(t, int) else int(t.data_ptr()))  # noqa: E731
        b = GraphBuffers()
        for k in ("q", "key", "value", "out", "query_start_loc", "num_computed", "block_table", "key_cache",
                  "value_cache", "device_in"):
            setattr(b, k, addr(buffers.get(k)))
        b.fused = 1 if fused else 0
        for k, n in (("host_in", "in_bytes"), ("host_out", "out_bytes")):
            pair = buffers.get(k)
            if pair is not None:
                getattr(b, k)[0] = addr(pair[0])
                getattr(b, k)[1] = addr(pair[1])
                setattr(b, n, int(buffers[n]))
        self._buffers = buffers
        h = ctypes.c_void_p()
        self.handle = None
        _check(load().pa_graph_create(ctypes.byref(self._descs[0]), ctypes.byref(self._shape), ctypes.byref(b),
                                      ctypes.byref(h)), "pa_graph_create")
        self.handle = h.value
        self._step = load().pa_graph_step
        self._turn = 0

    def step(self, num_reqs: int, stream=None, num_common_prefix_blocks: int = 0):
        """Plan the step now in the host arrays (set ``turn``) and launch the
        next graph (num_common_prefix_blocks > 0: the cascade route)."""
        d = self._descs[self._turn]
        d.num_reqs = num_reqs
        d.num_common_prefix_blocks = num_common_prefix_blocks
        _check(self._step(self.handle, ctypes.byref(d), _stream(stream)), "pa_graph_step")
        self._turn = 1 - self._turn

    @property
    def turn(self) -> int:
        """Graph (and host set / I/O buffers) the next step uses."""
        return int(load().pa_graph_turn(self.handle))

    def wait(self, turn: int):
        _check(load().pa_graph_wait(self.handle, int(turn)), "pa_graph_wait")

    def workspace_ptr(self) -> int:
        return int(load().pa_graph_workspace(self.handle))

    def slot_mapping_ptr(self) -> int:
        return int(load().pa_graph_slot_mapping(self.handle))

    def destroy(self):
        if self.handle:
            load().pa_graph_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass
