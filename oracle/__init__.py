"""Oracle for the PagedAttention decode hot path (TEST INFRASTRUCTURE ONLY).

A plain, slow fp64 CPU restatement of what the path computes, written from
the PagedAttention pages (cited per function in ``oracle.c`` and
``block_manager.py``). Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package. The
product library never imports it, and the two share no code: the oracle has
its own decoders, slot arithmetic, loops and block manager.

Every function here is pinned by ``tests/test_oracle_pins.py`` (values the
pages print, closed forms, library routines, brute force) or by
``tests/test_block_manager.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

F16 = 0
BF16 = 1

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (plain -O2, IEEE semantics, no fast-math),
    with OpenMP for the row-parallel batch functions when the compiler has
    it (the results are the same either way)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", _SRC, "-o", tmp]
    try:
        subprocess.check_call(base + ["-fopenmp", "-lm"], stderr=subprocess.DEVNULL)
    except subprocess.CalledProcessError:
        subprocess.check_call(base + ["-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    c_u16p = ctypes.POINTER(ctypes.c_uint16)
    c_i32p = ctypes.POINTER(ctypes.c_int32)
    c_dp = ctypes.POINTER(ctypes.c_double)
    i, d, ll = ctypes.c_int, ctypes.c_double, ctypes.c_longlong
    lib.oracle_set_threads.argtypes = [ctypes.c_int]
    lib.oracle_set_threads.restype = None
    lib.oracle_threads.argtypes = []
    lib.oracle_threads.restype = ctypes.c_int
    lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_to_double.restype = d
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_double.restype = d
    lib.oracle_decode_elems.argtypes = [c_u16p, c_dp, ll, i]
    lib.oracle_slot.argtypes = [c_i32p, i, ll]
    lib.oracle_slot.restype = ll
    lib.oracle_reshape_and_cache.argtypes = [c_u16p, c_u16p, c_u16p, c_i32p, i, i, i, i, i]
    lib.oracle_reshape_and_cache.restype = i
    lib.oracle_copy_blocks.argtypes = [ctypes.POINTER(c_u16p), i, c_i32p, i, i, i, i, i]
    lib.oracle_copy_blocks.restype = i
    lib.oracle_attention_contiguous.argtypes = [c_dp, c_u16p, c_u16p, c_u16p, i, i, d, i]
    lib.oracle_attention_online.argtypes = [c_dp, c_u16p, c_u16p, c_u16p, i, i, d, i, i]
    lib.oracle_decode_one.argtypes = [c_dp, c_u16p, c_u16p, c_i32p, i, c_i32p, i, i, d,
                                      i, i, i, i, i, i]
    lib.oracle_decode.argtypes = [c_dp, c_u16p, c_u16p, c_i32p, i, c_i32p, i, d,
                                  i, i, i, i, i, i]
    lib.oracle_decode_sampled.argtypes = [c_dp, c_i32p, c_i32p, i, c_u16p, c_u16p, c_i32p, i,
                                          c_i32p, d, i, i, i, i, i, i]
    c_u8p = ctypes.POINTER(ctypes.c_uint8)
    f = ctypes.c_float
    lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_double.restype = d
    lib.oracle_e4m3_from_float.argtypes = [f]
    lib.oracle_e4m3_from_float.restype = ctypes.c_uint8
    lib.oracle_quantize_e4m3.argtypes = [ctypes.c_uint16, i, f]
    lib.oracle_quantize_e4m3.restype = ctypes.c_uint8
    lib.oracle_reshape_and_cache_fp8.argtypes = [c_u16p, c_u16p, c_u8p, c_i32p, i, i, i, i, i,
                                                 i, f, f]
    lib.oracle_reshape_and_cache_fp8.restype = i
    lib.oracle_decode_fp8.argtypes = [c_dp, c_u16p, c_u8p, c_i32p, i, c_i32p, i, d,
                                      i, i, i, i, i, i, d, d]
    lib.oracle_decode_fp8_sampled.argtypes = [c_dp, c_i32p, c_i32p, i, c_u16p, c_u8p, c_i32p, i,
                                              c_i32p, d, i, i, i, i, i, i, d, d]
    lib.oracle_prefill.argtypes = [c_dp, c_u16p, c_u16p, c_i32p, i, c_i32p, c_i32p, i, d,
                                   i, i, i, i, i, i]
    lib.oracle_prefill_fp8.argtypes = [c_dp, c_u16p, c_u8p, c_i32p, i, c_i32p, c_i32p, i, d,
                                       i, i, i, i, i, i, d, d]
    _lib = lib
    return lib


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    assert a.dtype == np.uint16, a.dtype
    return a


def _i32(a) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a


def _p(a, ct):
    return a.ctypes.data_as(ctypes.POINTER(ct))


def set_threads(n: int) -> None:
    """Threads for the batch-level calls (decode, decode_sampled, their FP8
    forms, prefill); each output row is still computed by one thread with the
    same arithmetic, so results do not depend on n."""
    _load().oracle_set_threads(int(n))


def threads() -> int:
    """Threads the next batch-level call will use (1 if built without OpenMP)."""
    return int(_load().oracle_threads())


def f16_to_double(bits: int) -> float:
    return _load().oracle_f16_to_double(int(bits))


def bf16_to_double(bits: int) -> float:
    return _load().oracle_bf16_to_double(int(bits))


def decode_elems(bits, dtype: int) -> np.ndarray:
    """Exact value (float64) of every 16-bit pattern in ``bits``."""
    b = _u16(bits)
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_decode_elems(_p(b, ctypes.c_uint16), _p(out, ctypes.c_double), b.size, dtype)
    return out


def slot(table, block_size: int, pos: int) -> int:
    t = _i32(table)
    return int(_load().oracle_slot(_p(t, ctypes.c_int32), block_size, pos))


def reshape_and_cache(key, value, pool, slot_mapping, num_blocks, block_size,
                      num_kv_heads, head_size) -> int:
    """Writes in place into ``pool`` (uint16 array, pool layout)."""
    assert pool.dtype == np.uint16 and pool.flags["C_CONTIGUOUS"]
    k, v, s = _u16(key), _u16(value), _i32(slot_mapping)
    return _load().oracle_reshape_and_cache(
        _p(k, ctypes.c_uint16), _p(v, ctypes.c_uint16), _p(pool, ctypes.c_uint16),
        _p(s, ctypes.c_int32), len(s), num_blocks, block_size, num_kv_heads, head_size)


def copy_blocks(pools, pairs, num_blocks, block_size, num_kv_heads, head_size) -> int:
    """Copies in place inside every pool of ``pools`` (list of uint16 arrays)."""
    for p in pools:
        assert p.dtype == np.uint16 and p.flags["C_CONTIGUOUS"]
    arr = (ctypes.POINTER(ctypes.c_uint16) * max(1, len(pools)))(
        *[_p(p, ctypes.c_uint16) for p in pools])
    pr = _i32(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    return _load().oracle_copy_blocks(arr, len(pools), _p(pr, ctypes.c_int32), pr.shape[0],
                                      num_blocks, block_size, num_kv_heads, head_size)


def attention_contiguous(q, k, v, scale: float, dtype: int) -> np.ndarray:
    """q [D], k/v [L, D] (16-bit patterns) -> out [D] float64."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    head_size = q.shape[-1]
    seq_len = k.shape[0] if k.ndim == 2 else 0
    out = np.empty(head_size, dtype=np.float64)
    _load().oracle_attention_contiguous(_p(out, ctypes.c_double), _p(q, ctypes.c_uint16),
                                        _p(k, ctypes.c_uint16), _p(v, ctypes.c_uint16),
                                        seq_len, head_size, float(scale), dtype)
    return out


def attention_online(q, k, v, scale: float, dtype: int, part_len: int) -> np.ndarray:
    """Online-softmax (partitioned, merged) form of ``attention_contiguous``."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    head_size = q.shape[-1]
    out = np.empty(head_size, dtype=np.float64)
    _load().oracle_attention_online(_p(out, ctypes.c_double), _p(q, ctypes.c_uint16),
                                    _p(k, ctypes.c_uint16), _p(v, ctypes.c_uint16),
                                    k.shape[0], head_size, float(scale), dtype, part_len)
    return out


def decode(query, pool, block_tables, seq_lens, scale, num_q_heads, num_kv_heads,
           head_size, num_blocks, block_size, dtype) -> np.ndarray:
    """Paged decode of a batch -> [num_seqs, num_q_heads, head_size] float64."""
    q, kv = _u16(query), _u16(pool)
    bt, sl = _i32(block_tables), _i32(seq_lens)
    num_seqs = sl.shape[0]
    max_blocks = bt.shape[1] if bt.ndim == 2 else 0
    out = np.zeros((num_seqs, num_q_heads, head_size), dtype=np.float64)
    _load().oracle_decode(_p(out, ctypes.c_double), _p(q, ctypes.c_uint16),
                          _p(kv, ctypes.c_uint16), _p(bt, ctypes.c_int32), max_blocks,
                          _p(sl, ctypes.c_int32), num_seqs, float(scale), num_q_heads,
                          num_kv_heads, head_size, num_blocks, block_size, dtype)
    return out


def decode_sampled(seq_ids, q_heads, query, pool, block_tables, seq_lens, scale,
                   num_q_heads, num_kv_heads, head_size, num_blocks, block_size,
                   dtype) -> np.ndarray:
    """Paged decode of sampled (seq, q_head) pairs -> [n, head_size] float64."""
    q, kv = _u16(query), _u16(pool)
    bt, sl = _i32(block_tables), _i32(seq_lens)
    si, hi = _i32(seq_ids), _i32(q_heads)
    out = np.zeros((len(si), head_size), dtype=np.float64)
    _load().oracle_decode_sampled(_p(out, ctypes.c_double), _p(si, ctypes.c_int32),
                                  _p(hi, ctypes.c_int32), len(si), _p(q, ctypes.c_uint16),
                                  _p(kv, ctypes.c_uint16), _p(bt, ctypes.c_int32), bt.shape[1],
                                  _p(sl, ctypes.c_int32), float(scale), num_q_heads,
                                  num_kv_heads, head_size, num_blocks, block_size, dtype)
    return out


# ---------------------------------------------------------------- FP8 cache

def _u8(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.int8:
        a = a.view(np.uint8)
    assert a.dtype == np.uint8, a.dtype
    return a


def e4m3_to_double(code: int) -> float:
    """Exact value of an OCP E4M3 code (NaN for 0x7F / 0xFF)."""
    return _load().oracle_e4m3_to_double(int(code))


def e4m3_from_float(x: float) -> int:
    """E4M3 code nearest to the fp32 value x (ties to even, saturating at +-448)."""
    return int(_load().oracle_e4m3_from_float(float(x)))


def quantize_e4m3(bits: int, dtype: int, scale: float) -> int:
    """Cache code of one 16-bit element: e4m3(fp32(element) / fp32(scale))."""
    return int(_load().oracle_quantize_e4m3(int(bits), dtype, float(scale)))


def reshape_and_cache_fp8(key, value, pool, slot_mapping, num_blocks, block_size,
                          num_kv_heads, head_size, dtype, k_scale, v_scale) -> int:
    """Writes E4M3 codes in place into ``pool`` (uint8 array, pool layout)."""
    assert pool.dtype == np.uint8 and pool.flags["C_CONTIGUOUS"]
    k, v, s = _u16(key), _u16(value), _i32(slot_mapping)
    return _load().oracle_reshape_and_cache_fp8(
        _p(k, ctypes.c_uint16), _p(v, ctypes.c_uint16), _p(pool, ctypes.c_uint8),
        _p(s, ctypes.c_int32), len(s), num_blocks, block_size, num_kv_heads, head_size,
        dtype, float(k_scale), float(v_scale))


def decode_fp8(query, pool, block_tables, seq_lens, scale, num_q_heads, num_kv_heads,
               head_size, num_blocks, block_size, dtype, k_scale, v_scale) -> np.ndarray:
    """Paged decode over an E4M3 pool -> [num_seqs, num_q_heads, head_size] float64."""
    q, kv = _u16(query), _u8(pool)
    bt, sl = _i32(block_tables), _i32(seq_lens)
    num_seqs = sl.shape[0]
    max_blocks = bt.shape[1] if bt.ndim == 2 else 0
    out = np.zeros((num_seqs, num_q_heads, head_size), dtype=np.float64)
    _load().oracle_decode_fp8(_p(out, ctypes.c_double), _p(q, ctypes.c_uint16),
                              _p(kv, ctypes.c_uint8), _p(bt, ctypes.c_int32), max_blocks,
                              _p(sl, ctypes.c_int32), num_seqs, float(scale), num_q_heads,
                              num_kv_heads, head_size, num_blocks, block_size, dtype,
                              float(k_scale), float(v_scale))
    return out


def decode_fp8_sampled(seq_ids, q_heads, query, pool, block_tables, seq_lens, scale,
                       num_q_heads, num_kv_heads, head_size, num_blocks, block_size,
                       dtype, k_scale, v_scale) -> np.ndarray:
    """FP8-cache decode of sampled (seq, q_head) pairs -> [n, head_size] float64."""
    q, kv = _u16(query), _u8(pool)
    bt, sl = _i32(block_tables), _i32(seq_lens)
    si, hi = _i32(seq_ids), _i32(q_heads)
    out = np.zeros((len(si), head_size), dtype=np.float64)
    _load().oracle_decode_fp8_sampled(_p(out, ctypes.c_double), _p(si, ctypes.c_int32),
                                      _p(hi, ctypes.c_int32), len(si), _p(q, ctypes.c_uint16),
                                      _p(kv, ctypes.c_uint8), _p(bt, ctypes.c_int32),
                                      bt.shape[1], _p(sl, ctypes.c_int32), float(scale),
                                      num_q_heads, num_kv_heads, head_size, num_blocks,
                                      block_size, dtype, float(k_scale), float(v_scale))
    return out


# ------------------------------------------------------------------ prefill

def prefill(query, pool, block_tables, cu_seqlens_q, seq_lens, scale, num_q_heads,
            num_kv_heads, head_size, num_blocks, block_size, dtype) -> np.ndarray:
    """Causal chunked prefill over a 16-bit pool -> [total_q, num_q_heads, head_size]
    float64 (query row cu_seqlens_q[s] + i sits at position seq_lens[s] - q_len + i)."""
    q, kv = _u16(query), _u16(pool)
    bt, cu, sl = _i32(block_tables), _i32(cu_seqlens_q), _i32(seq_lens)
    num_seqs = sl.shape[0]
    assert cu.shape[0] == num_seqs + 1
    total_q = int(cu[-1])
    max_blocks = bt.shape[1] if bt.ndim == 2 else 0
    out = np.zeros((total_q, num_q_heads, head_size), dtype=np.float64)
    _load().oracle_prefill(_p(out, ctypes.c_double), _p(q, ctypes.c_uint16),
                           _p(kv, ctypes.c_uint16), _p(bt, ctypes.c_int32), max_blocks,
                           _p(cu, ctypes.c_int32), _p(sl, ctypes.c_int32), num_seqs,
                           float(scale), num_q_heads, num_kv_heads, head_size, num_blocks,
                           block_size, dtype)
    return out


def prefill_fp8(query, pool, block_tables, cu_seqlens_q, seq_lens, scale, num_q_heads,
                num_kv_heads, head_size, num_blocks, block_size, dtype, k_scale, v_scale) -> np.ndarray:
    """Causal chunked prefill over an E4M3 pool -> [total_q, num_q_heads, head_size]
    float64 (rows as in prefill, each the FP8 decode over its causal prefix)."""
    q, kv = _u16(query), _u8(pool)
    bt, cu, sl = _i32(block_tables), _i32(cu_seqlens_q), _i32(seq_lens)
    num_seqs = sl.shape[0]
    assert cu.shape[0] == num_seqs + 1
    total_q = int(cu[-1])
    max_blocks = bt.shape[1] if bt.ndim == 2 else 0
    out = np.zeros((total_q, num_q_heads, head_size), dtype=np.float64)
    _load().oracle_prefill_fp8(_p(out, ctypes.c_double), _p(q, ctypes.c_uint16),
                               _p(kv, ctypes.c_uint8), _p(bt, ctypes.c_int32), max_blocks,
                               _p(cu, ctypes.c_int32), _p(sl, ctypes.c_int32), num_seqs,
                               float(scale), num_q_heads, num_kv_heads, head_size, num_blocks,
                               block_size, dtype, float(k_scale), float(v_scale))
    return out
