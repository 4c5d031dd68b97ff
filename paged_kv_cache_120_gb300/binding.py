"""Thin ctypes binding of libpa (``include/pa.h``), with the same names.

Argument marshalling only: tensors are turned into pointers and sizes, the
current torch CUDA stream is passed as ``stream``, and a negative status is
raised as :class:`PAError` with the library's message. Every step of the
hot path runs in libpa's kernels; there is no fallback. If the library is
not built this module raises on first use.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpa.so")

PA_OK = 0
PA_ERR_INVALID_ARG = -1
PA_ERR_UNSUPPORTED = -2
PA_ERR_CUDA = -3
PA_ERR_WORKSPACE = -4
PA_ERR_OUT_OF_BLOCKS = -5
PA_ERR_NOT_FOUND = -6
PA_F16 = 0
PA_BF16 = 1
PA_FP8_E4M3 = 2
PA_DECODE_SHARED_BLOCKS = 1
PA_DECODE_LENS_READY = 2
PA_PCACHE_NO_CACHE = 1
PA_DEVERR_BLOCK_ID = 1
PA_DEVERR_SLOT = 2
PA_DEVERR_SEQ_LEN = 4
PA_DEVERR_PAIR = 8
PA_DEVERR_TIMEOUT = 16

# (name, restype, argtypes) of every exported function, in header order.
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_u = ctypes.c_uint
_i32p = ctypes.POINTER(ctypes.c_int32)
_ip = ctypes.POINTER(ctypes.c_int)
SIGNATURES = [
    ("pa_version", _i, []),
    ("pa_last_error", ctypes.c_char_p, []),
    ("pa_reshape_and_cache", _i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp]),
    ("pa_decode_workspace_size", _i, [_i, _i, _i, _i, _i, _i, ctypes.POINTER(_sz)]),
    ("pa_decode", _i, [_vp, _vp, _vp, _vp, _i, _vp, _i, _f, _i, _i, _i, _i, _i, _i, _vp, _sz, _u, _vp]),
    ("pa_decode_static_scratch", _i, [_vp, _vp, _vp, _vp, _i, _vp, _i, _f, _i, _i, _i, _i, _i, _i, _u, _vp]),
    ("pa_reshape_and_cache_fp8", _i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _f, _vp]),
    ("pa_decode_fp8_workspace_size", _i, [_i, _i, _i, _i, _i, _i, ctypes.POINTER(_sz)]),
    ("pa_decode_fp8", _i, [_vp, _vp, _vp, _vp, _i, _vp, _i, _f, _i, _i, _i, _i, _i, _i, _f, _f,
                           _vp, _sz, _u, _vp]),
    ("pa_prefill", _i, [_vp, _vp, _vp, _vp, _i, _vp, _vp, _i, _i, _i, _f, _i, _i, _i, _i, _i, _i,
                        _vp, _sz, _vp]),
    ("pa_prefill_workspace_size", _i, [_i, _i, _i, _i, _i, ctypes.POINTER(_sz)]),
    ("pa_prefill_fp8", _i, [_vp, _vp, _vp, _vp, _i, _vp, _vp, _i, _i, _i, _f, _i, _i, _i, _i, _i, _i, _f, _f,
                            _vp, _sz, _vp]),
    ("pa_copy_blocks", _i, [ctypes.POINTER(_vp), _i, _vp, _i, _i, _i, _i, _i, _i, _vp]),
    ("pa_get_device_error", _i, [_ip]),
    ("pa_alloc_create", _vp, [_i, _i, _i32p]),
    ("pa_alloc_destroy", None, [_vp]),
    ("pa_alloc_num_free", _i, [_vp]),
    ("pa_alloc_ref_count", _i, [_vp, _i]),
    ("pa_alloc_add_seq", _i, [_vp, _i, _ip]),
    ("pa_alloc_fork", _i, [_vp, _i, _ip]),
    ("pa_alloc_append_token", _i, [_vp, _i, _i32p, _i32p, _i32p]),
    ("pa_alloc_free_seq", _i, [_vp, _i]),
    ("pa_alloc_seq_len", _i, [_vp, _i]),
    ("pa_alloc_seq_num_blocks", _i, [_vp, _i]),
    ("pa_alloc_block_tables", _i, [_vp, _ip, _i, _i, _i32p]),
    ("pa_alloc_seq_lens", _i, [_vp, _ip, _i, _i32p]),
    ("pa_pcache_create", _vp, [_i, _i]),
    ("pa_pcache_destroy", None, [_vp]),
    ("pa_pcache_num_free", _i, [_vp]),
    ("pa_pcache_add_seq", _i, [_vp, _i32p, _i, _ip, _ip]),
    ("pa_pcache_admit", _i, [_vp, _vp, _vp, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, ctypes.c_int64, _vp]),
    ("pa_pcache_append_token", _i, [_vp, _i, ctypes.c_int32, _i32p]),
    ("pa_pcache_free_seq", _i, [_vp, _i]),
    ("pa_pcache_free_seqs", _i, [_vp, _vp, _i]),
    ("pa_pcache_seq_len", _i, [_vp, _i]),
    ("pa_pcache_block_tables", _i, [_vp, _ip, _i, _i, _i32p]),
    ("pa_pcache_slots", _i, [_vp, _i, _i, _i, _i32p]),
    ("pa_pcache_free_queue", _i, [_vp, _i32p, _i]),
    ("pa_pcache_ref_count", _i, [_vp, _i]),
    ("pa_pcache_block_hash", _i, [_vp, _i, ctypes.POINTER(ctypes.c_uint8)]),
]

_lib = None


class PAError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"libpa error {code}: {message}")
        self.code = code


def lib() -> ctypes.CDLL:
    """Load libpa.so (built by paged_kv_cache_120_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libpa.so is not built ({LIB_PATH}); run "
                               "`python -m paged_kv_cache_120_gb300.build`")
        l = ctypes.CDLL(LIB_PATH)
        for name, res, args in SIGNATURES:
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _lib = l
    return _lib


def _check(rc: int) -> int:
    if rc < 0:
        raise PAError(rc, lib().pa_last_error().decode())
    return rc


def _stream(stream):
    import torch
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return PA_F16
    if t.dtype == torch.bfloat16:
        return PA_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _pool_code(t) -> int:
    """Element type of a pool: 16-bit, or E4M3 held as uint8 / float8_e4m3fn."""
    import torch
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return PA_FP8_E4M3
    return _dtype_code(t)


def _fp8_pool(t, name):
    import torch
    if t.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise TypeError(f"{name} must hold E4M3 codes (uint8 or float8_e4m3fn), not {t.dtype}")
    return _dev(t, name)


def _dev(t, name):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def _host_array(a, dtype, name):
    """A contiguous host array of the given dtype (numpy, or a CPU tensor viewed as numpy)."""
    if hasattr(a, "is_cuda"):
        if a.is_cuda or not a.is_contiguous():
            raise PAError(PA_ERR_INVALID_ARG, f"{name}: needs a contiguous host tensor")
        a = a.numpy()
    if not isinstance(a, np.ndarray) or a.dtype != dtype or not a.flags.c_contiguous:
        raise PAError(PA_ERR_INVALID_ARG, f"{name}: needs a contiguous {np.dtype(dtype).name} array")
    return a


def _host_addr(a) -> int:
    return a.data_ptr() if hasattr(a, "data_ptr") else a.ctypes.data


_TORCH_DTYPE_NAMES = {np.dtype(np.int32): "torch.int32", np.dtype(np.int64): "torch.int64"}


def _host_ptr_size(a, dtype, name):
    """(address, element count) of a contiguous host array of the given dtype:
    numpy, or a CPU tensor checked and addressed directly (no numpy view)."""
    if hasattr(a, "is_cuda"):
        if a.is_cuda or not a.is_contiguous() or str(a.dtype) != _TORCH_DTYPE_NAMES.get(np.dtype(dtype)):
            raise PAError(PA_ERR_INVALID_ARG, f"{name}: needs a contiguous host {np.dtype(dtype).name} tensor")
        return a.data_ptr(), a.numel()
    if not isinstance(a, np.ndarray) or a.dtype != dtype or not a.flags.c_contiguous:
        raise PAError(PA_ERR_INVALID_ARG, f"{name}: needs a contiguous {np.dtype(dtype).name} array")
    return a.ctypes.data, a.size


def pa_version() -> int:
    return lib().pa_version()


def pa_last_error() -> str:
    return lib().pa_last_error().decode()


def pa_reshape_and_cache(key, value, kv_cache, slot_mapping, stream=None) -> None:
    """key/value [T, Hkv, D], kv_cache (2, NB, B, Hkv, D), slot_mapping [T] int32."""
    _, nb, bs, hkv, d = kv_cache.shape
    _check(lib().pa_reshape_and_cache(
        _dev(key, "key"), _dev(value, "value"), _dev(kv_cache, "kv_cache"),
        _dev(slot_mapping, "slot_mapping"), int(slot_mapping.shape[0]), nb, bs, hkv, d,
        _dtype_code(kv_cache), _stream(stream)))


def pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
                             dtype) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_size,
                                          block_size, dtype, ctypes.byref(out)))
    return out.value


def decode_workspace(query, kv_cache):
    """A correctly sized uint8 workspace tensor for pa_decode on this batch shape."""
    import torch
    s, hq, d = query.shape
    _, _, bs, hkv, _ = kv_cache.shape
    n = pa_decode_workspace_size(s, hq, hkv, d, bs, _dtype_code(kv_cache))
    return torch.empty(max(n, 256), dtype=torch.uint8, device=query.device)


def pa_decode(out, query, kv_cache, block_tables, seq_lens, scale, workspace,
              flags=0, stream=None) -> None:
    """out/query [S, Hq, D]; kv_cache (2, NB, B, Hkv, D); block_tables [S, maxblk] int32;
    seq_lens [S] int32; workspace: uint8 CUDA tensor (see decode_workspace);
    flags: an OR of PA_DECODE_SHARED_BLOCKS and PA_DECODE_LENS_READY (0 = none)."""
    s, hq, d = query.shape
    _, nb, bs, hkv, _ = kv_cache.shape
    _check(lib().pa_decode(
        _dev(out, "out"), _dev(query, "query"), _dev(kv_cache, "kv_cache"),
        _dev(block_tables, "block_tables"), int(block_tables.shape[1]),
        _dev(seq_lens, "seq_lens"), s, float(scale), hq, hkv, d, nb, bs,
        _dtype_code(kv_cache), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), int(flags), _stream(stream)))


def pa_decode_static_scratch(out, query, kv_cache, block_tables, seq_lens, scale,
                             flags=0, stream=None) -> None:
    """pa_decode without a workspace: the scratch is the library's static
    device array (for callers that cannot allocate device memory)."""
    s, hq, d = query.shape
    _, nb, bs, hkv, _ = kv_cache.shape
    _check(lib().pa_decode_static_scratch(
        _dev(out, "out"), _dev(query, "query"), _dev(kv_cache, "kv_cache"),
        _dev(block_tables, "block_tables"), int(block_tables.shape[1]),
        _dev(seq_lens, "seq_lens"), s, float(scale), hq, hkv, d, nb, bs,
        _dtype_code(kv_cache), int(flags), _stream(stream)))


def pa_reshape_and_cache_fp8(key, value, kv_cache, slot_mapping, k_scale, v_scale,
                             stream=None) -> None:
    """key/value [T, Hkv, D] fp16/bf16; kv_cache (2, NB, B, Hkv, D) of E4M3 codes
    (uint8 or float8_e4m3fn); slot_mapping [T] int32."""
    _, nb, bs, hkv, d = kv_cache.shape
    _check(lib().pa_reshape_and_cache_fp8(
        _dev(key, "key"), _dev(value, "value"), _fp8_pool(kv_cache, "kv_cache"),
        _dev(slot_mapping, "slot_mapping"), int(slot_mapping.shape[0]), nb, bs, hkv, d,
        _dtype_code(key), float(k_scale), float(v_scale), _stream(stream)))


def pa_decode_fp8_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
                                 dtype) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().pa_decode_fp8_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_size,
                                              block_size, dtype, ctypes.byref(out)))
    return out.value


def decode_fp8_workspace(query, kv_cache):
    """A correctly sized uint8 workspace tensor for pa_decode_fp8 on this batch shape."""
    import torch
    s, hq, d = query.shape
    _, _, bs, hkv, _ = kv_cache.shape
    n = pa_decode_fp8_workspace_size(s, hq, hkv, d, bs, _dtype_code(query))
    return torch.empty(max(n, 256), dtype=torch.uint8, device=query.device)


def pa_decode_fp8(out, query, kv_cache, block_tables, seq_lens, scale, k_scale, v_scale,
                  workspace, flags=0, stream=None) -> None:
    """pa_decode over an E4M3 pool; out/query fp16 or bf16 [S, Hq, D]."""
    s, hq, d = query.shape
    _, nb, bs, hkv, _ = kv_cache.shape
    _check(lib().pa_decode_fp8(
        _dev(out, "out"), _dev(query, "query"), _fp8_pool(kv_cache, "kv_cache"),
        _dev(block_tables, "block_tables"), int(block_tables.shape[1]),
        _dev(seq_lens, "seq_lens"), s, float(scale), hq, hkv, d, nb, bs,
        _dtype_code(query), float(k_scale), float(v_scale), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), int(flags), _stream(stream)))


def _workspace_args(workspace):
    if workspace is None:
        return ctypes.c_void_p(None), 0
    return _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()


def pa_prefill_workspace_size(num_seqs, max_seqlen_q, num_q_heads, num_kv_heads, head_size) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().pa_prefill_workspace_size(int(num_seqs), int(max_seqlen_q), num_q_heads, num_kv_heads,
                                           head_size, ctypes.byref(out)))
    return out.value


def prefill_workspace(query, kv_cache, num_seqs, max_seqlen_q):
    """A uint8 workspace tensor with which pa_prefill / pa_prefill_fp8 split
    the K/V ranges of this shape, or None when they would not split."""
    import torch
    _, hq, d = query.shape
    hkv = kv_cache.shape[3]
    n = pa_prefill_workspace_size(num_seqs, max_seqlen_q, hq, hkv, d)
    return torch.empty(n, dtype=torch.uint8, device=query.device) if n else None


def pa_prefill(out, query, kv_cache, block_tables, cu_seqlens_q, seq_lens, scale, max_seqlen_q,
               workspace=None, stream=None) -> None:
    """out/query [total_q, Hq, D]; kv_cache (2, NB, B, Hkv, D); block_tables [S, maxblk] int32;
    cu_seqlens_q [S + 1] int32; seq_lens [S] int32 (chunk included); max_seqlen_q: host int;
    workspace: None (no K/V split) or a uint8 CUDA tensor (see prefill_workspace)."""
    total_q, hq, d = query.shape
    _, nb, bs, hkv, _ = kv_cache.shape
    ws, ws_bytes = _workspace_args(workspace)
    _check(lib().pa_prefill(
        _dev(out, "out"), _dev(query, "query"), _dev(kv_cache, "kv_cache"),
        _dev(block_tables, "block_tables"), int(block_tables.shape[1]),
        _dev(cu_seqlens_q, "cu_seqlens_q"), _dev(seq_lens, "seq_lens"), int(seq_lens.shape[0]),
        total_q, int(max_seqlen_q), float(scale), hq, hkv, d, nb, bs, _dtype_code(kv_cache),
        ws, ws_bytes, _stream(stream)))


def pa_prefill_fp8(out, query, kv_cache, block_tables, cu_seqlens_q, seq_lens, scale, max_seqlen_q,
                   k_scale, v_scale, workspace=None, stream=None) -> None:
    """pa_prefill over an E4M3 byte pool (2, NB, B, Hkv, D) uint8; out/query 16-bit."""
    _fp8_pool(kv_cache, "kv_cache")
    total_q, hq, d = query.shape
    _, nb, bs, hkv, _ = kv_cache.shape
    ws, ws_bytes = _workspace_args(workspace)
    _check(lib().pa_prefill_fp8(
        _dev(out, "out"), _dev(query, "query"), _dev(kv_cache, "kv_cache"),
        _dev(block_tables, "block_tables"), int(block_tables.shape[1]),
        _dev(cu_seqlens_q, "cu_seqlens_q"), _dev(seq_lens, "seq_lens"), int(seq_lens.shape[0]),
        total_q, int(max_seqlen_q), float(scale), hq, hkv, d, nb, bs, _dtype_code(query),
        float(k_scale), float(v_scale), ws, ws_bytes, _stream(stream)))


def pa_copy_blocks(kv_caches, src_dst_pairs, stream=None) -> None:
    """kv_caches: list of per-layer pools (fp16, bf16, or E4M3 codes as uint8 /
    float8_e4m3fn); src_dst_pairs [N, 2] int32 CUDA tensor."""
    _, nb, bs, hkv, d = kv_caches[0].shape
    ptrs = (ctypes.c_void_p * len(kv_caches))(*[_dev(c, "kv_cache").value for c in kv_caches])
    _check(lib().pa_copy_blocks(ptrs, len(kv_caches), _dev(src_dst_pairs, "src_dst_pairs"),
                                int(src_dst_pairs.shape[0]), nb, bs, hkv, d,
                                _pool_code(kv_caches[0]), _stream(stream)))


def pa_get_device_error() -> int:
    bits = ctypes.c_int(0)
    _check(lib().pa_get_device_error(ctypes.byref(bits)))
    return bits.value


class BlockAllocator:
    """Host block allocator (pa_alloc_*): free list, ref counts, copy-on-write."""

    def __init__(self, num_blocks: int, block_size: int, order=None):
        self.num_blocks, self.block_size = num_blocks, block_size
        if order is not None:
            self._order = np.ascontiguousarray(order, dtype=np.int32)
            optr = self._order.ctypes.data_as(_i32p)
        else:
            optr = None
        h = lib().pa_alloc_create(num_blocks, block_size, optr)
        if not h:
            raise PAError(PA_ERR_INVALID_ARG, pa_last_error())
        self._h = ctypes.c_void_p(h)

    def close(self):
        if getattr(self, "_h", None):
            lib().pa_alloc_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def num_free(self) -> int:
        return _check(lib().pa_alloc_num_free(self._h))

    def ref_count(self, block: int) -> int:
        return _check(lib().pa_alloc_ref_count(self._h, block))

    def add_seq(self, num_tokens: int) -> int:
        sid = ctypes.c_int(0)
        _check(lib().pa_alloc_add_seq(self._h, num_tokens, ctypes.byref(sid)))
        return sid.value

    def fork(self, parent: int) -> int:
        sid = ctypes.c_int(0)
        _check(lib().pa_alloc_fork(self._h, parent, ctypes.byref(sid)))
        return sid.value

    def append_token(self, seq: int):
        """-> (slot, (cow_src, cow_dst) or None)."""
        slot, src, dst = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int32(0)
        _check(lib().pa_alloc_append_token(self._h, seq, ctypes.byref(slot), ctypes.byref(src),
                                           ctypes.byref(dst)))
        return slot.value, (None if src.value < 0 else (src.value, dst.value))

    def free_seq(self, seq: int) -> None:
        _check(lib().pa_alloc_free_seq(self._h, seq))

    def seq_len(self, seq: int) -> int:
        return _check(lib().pa_alloc_seq_len(self._h, seq))

    def num_blocks_of(self, seq: int) -> int:
        return _check(lib().pa_alloc_seq_num_blocks(self._h, seq))

    def table(self, seq: int):
        n = self.num_blocks_of(seq)
        return self.block_tables([seq], max(n, 1))[0, :n].tolist()

    def block_tables(self, seqs, max_blocks_per_seq: int) -> np.ndarray:
        ids = np.ascontiguousarray(seqs, dtype=np.int32)
        out = np.empty((len(ids), max_blocks_per_seq), dtype=np.int32)
        _check(lib().pa_alloc_block_tables(self._h, ids.ctypes.data_as(_ip), len(ids),
                                           max_blocks_per_seq, out.ctypes.data_as(_i32p)))
        return out

    def seq_lens(self, seqs) -> np.ndarray:
        ids = np.ascontiguousarray(seqs, dtype=np.int32)
        out = np.empty(len(ids), dtype=np.int32)
        _check(lib().pa_alloc_seq_lens(self._h, ids.ctypes.data_as(_ip), len(ids),
                                       out.ctypes.data_as(_i32p)))
        return out


class PrefixCache:
    """Host prefix-cache block pool (pa_pcache_*): chained block hashes, a
    free queue with lazy eviction, prompts that reuse cached prefixes."""

    def __init__(self, num_blocks: int, block_size: int):
        self.num_blocks, self.block_size = num_blocks, block_size
        h = lib().pa_pcache_create(num_blocks, block_size)
        if not h:
            raise PAError(PA_ERR_INVALID_ARG, pa_last_error())
        self._h = ctypes.c_void_p(h)

    def close(self):
        if getattr(self, "_h", None):
            lib().pa_pcache_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def num_free(self) -> int:
        return _check(lib().pa_pcache_num_free(self._h))

    def add_seq(self, tokens):
        """-> (seq_id, tokens found in the cache)."""
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        sid, hit = ctypes.c_int(0), ctypes.c_int(0)
        _check(lib().pa_pcache_add_seq(self._h, t.ctypes.data_as(_i32p), len(t), ctypes.byref(sid),
                                       ctypes.byref(hit)))
        return sid.value, hit.value

    _ADMIT_OUT = ("seq_ids", "num_cached", "cu_seqlens_q", "seq_lens", "slot_mapping", "block_tables")

    def admit(self, tokens, cu_tokens, max_blocks_per_seq: int, flags: int = 0, out=None):
        """pa_pcache_admit: -> (number admitted, out). tokens is int32 and
        cu_tokens int64 (numpy or CPU tensors); out maps the six output names
        to int32 host buffers (numpy or CPU tensors, e.g. pinned), allocated
        here when not given."""
        tok_ptr, _ = _host_ptr_size(tokens, np.int32, "tokens")
        cu = _host_array(cu_tokens, np.int64, "cu_tokens")
        n = len(cu) - 1
        total = int(cu[-1]) if n > 0 else 0
        sizes = {"seq_ids": n, "num_cached": n, "cu_seqlens_q": n + 1, "seq_lens": n,
                 "slot_mapping": total, "block_tables": n * max_blocks_per_seq}
        if out is None:
            out = {k: np.empty(v, np.int32) for k, v in sizes.items()}
            out["block_tables"] = out["block_tables"].reshape(n, max_blocks_per_seq)
        ptrs = []
        for k in self._ADMIT_OUT:
            ptr, size = _host_ptr_size(out[k], np.int32, k)
            if size < sizes[k]:
                raise PAError(PA_ERR_INVALID_ARG, f"admit: {k} holds {size} < {sizes[k]}")
            ptrs.append(ptr)
            if k == "slot_mapping":
                slot_cap = size
        count = _check(lib().pa_pcache_admit(self._h, tok_ptr, _host_addr(cu), n, flags,
                                             max_blocks_per_seq, *ptrs[:5], slot_cap, ptrs[5]))
        return count, out

    def free_seqs(self, seqs) -> None:
        ptr, n = _host_ptr_size(seqs, np.int32, "seqs")
        _check(lib().pa_pcache_free_seqs(self._h, ptr, n))

    def append_token(self, seq: int, token: int) -> int:
        slot = ctypes.c_int32(0)
        _check(lib().pa_pcache_append_token(self._h, seq, int(token), ctypes.byref(slot)))
        return slot.value

    def free_seq(self, seq: int) -> None:
        _check(lib().pa_pcache_free_seq(self._h, seq))

    def seq_len(self, seq: int) -> int:
        return _check(lib().pa_pcache_seq_len(self._h, seq))

    def block_tables(self, seqs, max_blocks_per_seq: int) -> np.ndarray:
        ids = np.ascontiguousarray(seqs, dtype=np.int32)
        out = np.empty((len(ids), max_blocks_per_seq), dtype=np.int32)
        _check(lib().pa_pcache_block_tables(self._h, ids.ctypes.data_as(_ip), len(ids), max_blocks_per_seq,
                                            out.ctypes.data_as(_i32p)))
        return out

    def table(self, seq: int):
        n = -(-self.seq_len(seq) // self.block_size)
        return self.block_tables([seq], max(n, 1))[0, :n].tolist()

    def slots(self, seq: int, first_pos: int, n: int) -> np.ndarray:
        out = np.empty(n, dtype=np.int32)
        _check(lib().pa_pcache_slots(self._h, seq, first_pos, n, out.ctypes.data_as(_i32p)))
        return out

    def free_queue(self):
        cap = self.num_blocks
        out = np.empty(cap, dtype=np.int32)
        n = _check(lib().pa_pcache_free_queue(self._h, out.ctypes.data_as(_i32p), cap))
        return out[:n].tolist()

    def ref_count(self, block: int) -> int:
        return _check(lib().pa_pcache_ref_count(self._h, block))

    def block_hash(self, block: int):
        buf = (ctypes.c_uint8 * 32)()
        r = _check(lib().pa_pcache_block_hash(self._h, block, buf))
        return bytes(buf) if r == 1 else None
