"""ctypes front end of the fp64 CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this module; the product package never
does.  The oracle shares no code with the CUDA library.

``build()`` compiles ``oracle.c`` with gcc (OpenMP, -O2) into
``oracle/_build/liboracle.so``.  ``Oracle`` wraps one compiled library; a
path to another build (for example a deliberately broken copy used by the
mutation tests) can be passed in.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIBRARY = os.path.join(BUILD_DIR, "liboracle.so")

OK = 0
BAD_METADATA = 1
BAD_BLOCK = 2
NO_MEMORY = 3


def compile_source(source: str, output: str) -> str:
    """Compile one oracle C source into a shared library at ``output``."""
    os.makedirs(os.path.dirname(output), exist_ok=True)
    tmp = output + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, source, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, output)
    return output


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    if (not force and os.path.exists(LIBRARY)
            and os.path.getmtime(LIBRARY) >= os.path.getmtime(SOURCE)):
        return LIBRARY
    return compile_source(SOURCE, LIBRARY)


_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_f64p = ctypes.POINTER(ctypes.c_double)


def _ptr(a: np.ndarray | None, ctype):
    if a is None:
        return ctypes.cast(None, ctype)
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctype)


class OracleError(RuntimeError):
    pass


@dataclass
class AttentionResult:
    out: np.ndarray   # [T, Hq, D] float64
    m: np.ndarray     # [T, Hq] float64 (natural-log running max)
    l: np.ndarray     # [T, Hq] float64 (sum of exp(s - m))


class Oracle:
    def __init__(self, library: str | None = None):
        path = library or build()
        self.lib = ctypes.CDLL(path)
        L = self.lib
        L.oracle_bf16_value.restype = ctypes.c_double
        L.oracle_bf16_value.argtypes = [ctypes.c_uint16]
        L.oracle_num_threads.restype = ctypes.c_int
        L.oracle_set_num_threads.restype = None
        L.oracle_set_num_threads.argtypes = [ctypes.c_int]
        L.oracle_slot_mapping.restype = ctypes.c_int
        L.oracle_slot_mapping.argtypes = [ctypes.c_int32, _i32p, _i32p, _i32p, ctypes.c_int32,
                                          ctypes.c_int32, _i64p]
        L.oracle_write_kv.restype = ctypes.c_int
        L.oracle_write_kv.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _u16p, _u16p,
                                      _i64p, _u16p, _u16p, ctypes.c_int64]
        L.oracle_attention_range.restype = ctypes.c_int
        L.oracle_attention_range.argtypes = [
            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
            ctypes.c_int32, ctypes.c_int32, _i32p, _i32p, _i32p, _i32p, ctypes.c_double,
            _u16p, _u16p, _u16p, _i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
            _f64p, _f64p, _f64p]
        L.oracle_merge_partials.restype = None
        L.oracle_merge_partials.argtypes = [ctypes.c_int32, ctypes.c_int32, _f64p, _f64p, _f64p,
                                            _f64p, _f64p, _f64p]
        _u8p = ctypes.POINTER(ctypes.c_uint8)
        L.oracle_zero_blocks.restype = ctypes.c_int
        L.oracle_zero_blocks.argtypes = [ctypes.c_int32, _i32p, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.POINTER(ctypes.c_uint8), ctypes.POINTER(ctypes.c_uint8)]
        L.oracle_e4m3_value.restype = ctypes.c_double
        L.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_encode.restype = ctypes.c_uint8
        L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        L.oracle_write_kv_fp8.restype = ctypes.c_int
        L.oracle_write_kv_fp8.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _u16p, _u16p, _i64p,
                                          _u8p, _u8p, ctypes.c_int64, ctypes.c_float, ctypes.c_float]
        L.oracle_attention_fp8.restype = ctypes.c_int
        L.oracle_attention_fp8.argtypes = [
            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
            ctypes.c_int32, ctypes.c_int32, _i32p, _i32p, _i32p, _i32p, ctypes.c_double,
            _u16p, _u8p, _u8p, ctypes.c_float, ctypes.c_float, _i32p, ctypes.c_int32, _f64p]
        L.oracle_check_common_prefix.restype = ctypes.c_int
        L.oracle_check_common_prefix.argtypes = [ctypes.c_int32, _i32p, _i32p, _i32p,
                                                 ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]

    # -- scalar helpers -------------------------------------------------
    def bf16_value(self, bits: int) -> float:
        return self.lib.oracle_bf16_value(int(bits) & 0xFFFF)

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def set_num_threads(self, n: int) -> None:
        """Threads the oracle's parallel loops use from now on (n >= 1)."""
        self.lib.oracle_set_num_threads(int(n))

    # -- step 1: slot mapping --------------------------------------------
    def slot_mapping(self, query_start_loc, num_computed, block_table, block_size: int):
        qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
        nc = np.ascontiguousarray(num_computed, dtype=np.int32)
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        num_reqs = len(nc)
        out = np.full(int(qsl[-1]), -1, dtype=np.int64)
        st = self.lib.oracle_slot_mapping(num_reqs, _ptr(qsl, _i32p), _ptr(nc, _i32p),
                                          _ptr(bt, _i32p), bt.shape[1], block_size,
                                          _ptr(out, _i64p))
        if st != OK:
            raise OracleError(f"slot_mapping status {st}")
        return out

    # -- step 2: cache write (in place on the given caches) ---------------
    def write_kv(self, key, value, slot_mapping, key_cache, value_cache) -> int:
        key = np.ascontiguousarray(key, dtype=np.uint16)
        value = np.ascontiguousarray(value, dtype=np.uint16)
        slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        assert key_cache.dtype == np.uint16 and key_cache.flags["C_CONTIGUOUS"]
        assert value_cache.dtype == np.uint16 and value_cache.flags["C_CONTIGUOUS"]
        T, hkv, d = key.shape
        num_slots = key_cache.shape[0] * key_cache.shape[1]
        return int(self.lib.oracle_write_kv(T, hkv, d, _ptr(key, _u16p), _ptr(value, _u16p),
                                            _ptr(slots, _i64p), _ptr(key_cache, _u16p),
                                            _ptr(value_cache, _u16p), num_slots))

    def zero_blocks(self, block_ids, key_cache, value_cache) -> int:
        """Zero the K and V entries of the listed blocks in place (any cache
        element type; ids < 0 skipped)."""
        ids = np.ascontiguousarray(block_ids, dtype=np.int32)
        assert key_cache.flags["C_CONTIGUOUS"] and value_cache.flags["C_CONTIGUOUS"]
        assert key_cache.shape == value_cache.shape and key_cache.dtype == value_cache.dtype
        nb = key_cache.shape[0]
        block_bytes = key_cache.nbytes // nb
        u8 = ctypes.POINTER(ctypes.c_uint8)
        return int(self.lib.oracle_zero_blocks(len(ids), _ptr(ids, _i32p), nb, block_bytes,
                                               key_cache.ctypes.data_as(u8), value_cache.ctypes.data_as(u8)))

    # -- step 3: attention -----------------------------------------------
    def attention_range(self, *, query_start_loc, seq_lens, num_computed, block_table, q,
                        key_cache, value_cache, softmax_scale: float, rows=None,
                        key_begin: int = -1, key_end: int = -1) -> AttentionResult:
        qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        nc = np.ascontiguousarray(num_computed, dtype=np.int32)
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        q = np.ascontiguousarray(q, dtype=np.uint16)
        kc = np.ascontiguousarray(key_cache, dtype=np.uint16)
        vc = np.ascontiguousarray(value_cache, dtype=np.uint16)
        T, hq, d = q.shape
        num_blocks, block_size, hkv, d2 = kc.shape
        assert d == d2 and vc.shape == kc.shape
        out = np.full((T, hq, d), np.nan, dtype=np.float64)
        m = np.full((T, hq), np.nan, dtype=np.float64)
        l = np.full((T, hq), np.nan, dtype=np.float64)
        rows_arr = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
        n_rows = 0 if rows_arr is None else len(rows_arr)
        st = self.lib.oracle_attention_range(
            len(sl), hq, hkv, d, block_size, num_blocks, bt.shape[1], _ptr(qsl, _i32p),
            _ptr(sl, _i32p), _ptr(nc, _i32p), _ptr(bt, _i32p), float(softmax_scale),
            _ptr(q, _u16p), _ptr(kc, _u16p), _ptr(vc, _u16p), _ptr(rows_arr, _i32p), n_rows,
            int(key_begin), int(key_end), _ptr(out, _f64p), _ptr(m, _f64p), _ptr(l, _f64p))
        if st != OK:
            raise OracleError(f"attention status {st}")
        return AttentionResult(out, m, l)

    def attention(self, **kw) -> np.ndarray:
        return self.attention_range(**kw).out

    def merge(self, m_parts, l_parts, o_parts):
        m_parts = np.ascontiguousarray(m_parts, dtype=np.float64)
        l_parts = np.ascontiguousarray(l_parts, dtype=np.float64)
        o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
        n, d = o_parts.shape
        o = np.zeros(d, dtype=np.float64)
        m = np.zeros(1, dtype=np.float64)
        l = np.zeros(1, dtype=np.float64)
        self.lib.oracle_merge_partials(n, d, _ptr(m_parts, _f64p), _ptr(l_parts, _f64p),
                                       _ptr(o_parts, _f64p), _ptr(o, _f64p), _ptr(m, _f64p),
                                       _ptr(l, _f64p))
        return o, float(m[0]), float(l[0])

    def check_common_prefix(self, query_start_loc, num_computed, block_table, block_size: int,
                            num_common_prefix_blocks: int) -> int:
        qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
        nc = np.ascontiguousarray(num_computed, dtype=np.int32)
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        return int(self.lib.oracle_check_common_prefix(
            len(nc), _ptr(qsl, _i32p), _ptr(nc, _i32p), _ptr(bt, _i32p), bt.shape[1],
            block_size, int(num_common_prefix_blocks)))

    # -- FP8 (E4M3) cache ---------------------------------------------------
    def e4m3_value(self, code: int) -> float:
        return self.lib.oracle_e4m3_value(int(code) & 0xFF)

    def e4m3_encode(self, x: float) -> int:
        return int(self.lib.oracle_e4m3_encode(float(x)))

    def write_kv_fp8(self, key, value, slot_mapping, key_cache, value_cache, k_scale: float,
                     v_scale: float) -> int:
        key = np.ascontiguousarray(key, dtype=np.uint16)
        value = np.ascontiguousarray(value, dtype=np.uint16)
        slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        assert key_cache.dtype == np.uint8 and key_cache.flags["C_CONTIGUOUS"]
        assert value_cache.dtype == np.uint8 and value_cache.flags["C_CONTIGUOUS"]
        T, hkv, d = key.shape
        num_slots = key_cache.shape[0] * key_cache.shape[1]
        u8 = ctypes.POINTER(ctypes.c_uint8)
        return int(self.lib.oracle_write_kv_fp8(T, hkv, d, _ptr(key, _u16p), _ptr(value, _u16p),
                                                _ptr(slots, _i64p), _ptr(key_cache, u8), _ptr(value_cache, u8),
                                                num_slots, float(k_scale), float(v_scale)))

    def attention_fp8(self, *, query_start_loc, seq_lens, num_computed, block_table, q, key_cache,
                      value_cache, softmax_scale: float, k_scale: float, v_scale: float, rows=None):
        qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        nc = np.ascontiguousarray(num_computed, dtype=np.int32)
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        q = np.ascontiguousarray(q, dtype=np.uint16)
        kc = np.ascontiguousarray(key_cache, dtype=np.uint8)
        vc = np.ascontiguousarray(value_cache, dtype=np.uint8)
        T, hq, d = q.shape
        num_blocks, block_size, hkv, d2 = kc.shape
        assert d == d2 and vc.shape == kc.shape
        out = np.full((T, hq, d), np.nan, dtype=np.float64)
        rows_arr = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
        n_rows = 0 if rows_arr is None else len(rows_arr)
        u8 = ctypes.POINTER(ctypes.c_uint8)
        st = self.lib.oracle_attention_fp8(
            len(sl), hq, hkv, d, block_size, num_blocks, bt.shape[1], _ptr(qsl, _i32p), _ptr(sl, _i32p),
            _ptr(nc, _i32p), _ptr(bt, _i32p), float(softmax_scale), _ptr(q, _u16p), _ptr(kc, u8),
            _ptr(vc, u8), float(k_scale), float(v_scale), _ptr(rows_arr, _i32p), n_rows, _ptr(out, _f64p))
        if st != OK:
            raise OracleError(f"attention_fp8 status {st}")
        return out

    def step_fp8(self, *, query_start_loc, seq_lens, num_computed, block_table, q, key, value,
                 key_cache, value_cache, softmax_scale: float, k_scale: float, v_scale: float, rows=None):
        """FP8 cache: write (quantising), then attend (dequantising)."""
        kc = np.array(key_cache, dtype=np.uint8, copy=True, order="C")
        vc = np.array(value_cache, dtype=np.uint8, copy=True, order="C")
        block_size = kc.shape[1]
        slots = self.slot_mapping(query_start_loc, num_computed, block_table, block_size)
        st = self.write_kv_fp8(key, value, slots, kc, vc, k_scale, v_scale)
        if st != OK:
            raise OracleError(f"write_fp8 status {st}")
        out = self.attention_fp8(query_start_loc=query_start_loc, seq_lens=seq_lens, num_computed=num_computed,
                                 block_table=block_table, q=q, key_cache=kc, value_cache=vc,
                                 softmax_scale=softmax_scale, k_scale=k_scale, v_scale=v_scale, rows=rows)
        return kc, vc, slots, out

    # -- the whole step: write, then attend ---------------------------------
    def step(self, *, query_start_loc, seq_lens, num_computed, block_table, q, key, value,
             key_cache, value_cache, softmax_scale: float, rows=None):
        """Apply the cache write to copies of the caches, then run attention.

        Returns (key_cache_after, value_cache_after, slot_mapping, out[T,Hq,D]).
        """
        kc = np.array(key_cache, dtype=np.uint16, copy=True, order="C")
        vc = np.array(value_cache, dtype=np.uint16, copy=True, order="C")
        block_size = kc.shape[1]
        slots = self.slot_mapping(query_start_loc, num_computed, block_table, block_size)
        st = self.write_kv(key, value, slots, kc, vc)
        if st != OK:
            raise OracleError(f"write status {st}")
        out = self.attention(query_start_loc=query_start_loc, seq_lens=seq_lens,
                             num_computed=num_computed, block_table=block_table, q=q,
                             key_cache=kc, value_cache=vc, softmax_scale=softmax_scale,
                             rows=rows)
        return kc, vc, slots, out


_DEFAULT: Oracle | None = None


def default() -> Oracle:
    """The oracle built from ``oracle.c`` (compiled on first use)."""
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle()
    return _DEFAULT
