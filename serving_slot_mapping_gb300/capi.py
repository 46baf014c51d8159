"""Thin ctypes binding of libpagedattn.so (see include/paged_attn.h).

Argument marshalling only: every step of the computation runs in the CUDA
library.  Tensors are torch tensors that already live on the current CUDA
device; the stream defaults to torch's current stream.  A missing library
raises immediately: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from .build import LIB_PATH

PA_OK = 0
PA_ERR_NULL = 1
PA_ERR_SHAPE = 2
PA_ERR_DTYPE = 3
PA_ERR_RANGE = 4
PA_ERR_UNSUPPORTED = 5
PA_ERR_CUDA = 6
PA_ERR_WORKSPACE = 7
PA_ERR_ALIGN = 8

PA_DTYPE_F32 = 0
PA_DTYPE_BF16 = 1
PA_DTYPE_FP8_E4M3 = 2

# Every symbol include/paged_attn.h declares, with (restype, argtypes).
_c_void_p = ctypes.c_void_p
_i32, _i64, _sz, _f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float


class PaKvPool(ctypes.Structure):
    _fields_ = [("key_pool", _c_void_p), ("value_pool", _c_void_p), ("num_pages", _i64),
                ("page_size", _i32), ("num_kv_heads", _i32), ("head_dim", _i32), ("dtype", _i32),
                ("k_scale", _f32), ("v_scale", _f32)]


_PPOOL = ctypes.POINTER(PaKvPool)

SIGNATURES = {
    "paged_kv_append": (_i32, [_PPOOL, _c_void_p, _c_void_p, _c_void_p, _i64, _c_void_p]),
    "paged_attention_decode_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32]),
    "paged_attention_decode": (_i32, [_PPOOL, _c_void_p, _c_void_p, _i32, _i32, _c_void_p, _i32,
                                      _c_void_p, _i32, _f32, _c_void_p, _sz, _c_void_p]),
    "paged_attention_decode_append": (_i32, [_PPOOL, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                             _c_void_p, _i32, _i32, _c_void_p, _i32, _c_void_p, _i32,
                                             _f32, _c_void_p, _sz, _c_void_p]),
    "paged_attention_decode_static_scratch": (_i32, [_PPOOL, _c_void_p, _c_void_p, _i32, _i32,
                                                     _c_void_p, _i32, _c_void_p, _i32, _f32,
                                                     _c_void_p]),
    "paged_attention_decode_cascade_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32]),
    "paged_attention_decode_cascade": (_i32, [_PPOOL, _c_void_p, _c_void_p, _i32, _i32, _c_void_p,
                                              _i32, _c_void_p, _i32, _c_void_p, _i32, _f32,
                                              _c_void_p, _sz, _c_void_p]),
    "paged_attention_decode_csr": (_i32, [_PPOOL, _c_void_p, _c_void_p, _i32, _i32, _c_void_p,
                                          _c_void_p, _i64, _c_void_p, _i32, _f32, _c_void_p, _sz,
                                          _c_void_p]),
    "paged_attention_prefill_csr": (_i32, [_PPOOL, _c_void_p, _c_void_p, _i32, _i32, _c_void_p, _i64,
                                           _i32, _c_void_p, _c_void_p, _i64, _c_void_p, _i32, _f32,
                                           _c_void_p]),
    "paged_attention_prefill": (_i32, [_PPOOL, _c_void_p, _c_void_p, _i32, _i32, _c_void_p, _i64,
                                       _i32, _c_void_p, _i32, _c_void_p, _i32, _f32, _c_void_p]),
    "pa_testing_decode_part_wait": (_i32, [_PPOOL, _c_void_p, _c_void_p, _i32, _i32, _c_void_p, _i32,
                                           _c_void_p, _i32, _f32, _c_void_p, _sz, ctypes.c_uint64, _i32,
                                           _c_void_p]),
    "paged_device_error": (_i32, [ctypes.POINTER(_i64), ctypes.POINTER(_i64)]),
    "pa_status_string": (ctypes.c_char_p, [_i32]),
    "pa_abi_version": (_i32, []),
}

_LIB = None


class PagedAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = lib().pa_status_string(status).decode()
        super().__init__(f"{where}: {msg} (status {status})")
        self.status = status


def lib(path: Optional[str] = None):
    """Load the shared library once; raise if it has not been built."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or os.environ.get("PAGEDATTN_LIB", LIB_PATH)
    if not os.path.exists(p):
        raise RuntimeError(f"libpagedattn.so not found at {p}: build it with "
                           "`python -m serving_slot_mapping_gb300.build`")
    handle = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(handle, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _LIB = handle
    return handle


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.bfloat16:
        return PA_DTYPE_BF16
    if t == torch.float32:
        return PA_DTYPE_F32
    if t == torch.float8_e4m3fn:
        return PA_DTYPE_FP8_E4M3
    raise TypeError(f"unsupported pool dtype {t}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(status: int, where: str):
    if status != PA_OK:
        raise PagedAttnError(status, where)


def _contig(t: torch.Tensor, name: str):
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def make_pool(key_pool: torch.Tensor, value_pool: torch.Tensor, k_scale: float = 1.0,
              v_scale: float = 1.0) -> PaKvPool:
    """Describe a [num_pages, page_size, num_kv_heads, head_dim] K/V pool pair
    (float32, bfloat16, or float8_e4m3fn with per-tensor k_scale / v_scale)."""
    if key_pool.shape != value_pool.shape or key_pool.dtype != value_pool.dtype:
        raise ValueError("key_pool and value_pool must match in shape and dtype")
    if key_pool.dim() != 4:
        raise ValueError("pools are [num_pages, page_size, num_kv_heads, head_dim]")
    _contig(key_pool, "key_pool")
    _contig(value_pool, "value_pool")
    P, ps, hkv, d = key_pool.shape
    return PaKvPool(key_pool.data_ptr(), value_pool.data_ptr(), P, ps, hkv, d,
                    _dtype_code(key_pool.dtype), float(k_scale), float(v_scale))


def _q_out(q, out, key_pool):
    """Check ``q [rows, Hq, D]`` against the pool (bf16 for bf16 and e4m3
    pools, f32 for f32 pools) and return ``out`` of the same shape and dtype
    (allocated when None)."""
    want = torch.bfloat16 if key_pool.dtype in (torch.bfloat16, torch.float8_e4m3fn) else key_pool.dtype
    _contig(q, "q")
    if q.dim() != 3 or q.dtype != want or q.shape[2] != key_pool.shape[3]:
        raise ValueError(f"q must be [rows, num_q_heads, {key_pool.shape[3]}] of {want}")
    if out is None:
        return torch.empty_like(q)
    _contig(out, "out")
    if out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("out must match q in shape and dtype")
    return out


def paged_kv_append(key_pool, value_pool, key, value, slot_mapping, stream=None, k_scale=1.0,
                    v_scale=1.0):
    """Scatter ``key/value [T, Hkv, D]`` into the pools at ``slot_mapping`` (int64 [T]).

    e4m3 pools take bf16 rows and store their codes with the given scales."""
    pool = make_pool(key_pool, value_pool, k_scale, v_scale)
    row_dtype = torch.bfloat16 if key_pool.dtype == torch.float8_e4m3fn else key_pool.dtype
    T = slot_mapping.numel()
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    for n, t in (("key", key), ("value", value)):
        _contig(t, n)
        if t.dtype != row_dtype or t.numel() != T * pool.num_kv_heads * pool.head_dim:
            raise ValueError(f"{n} must be [T, num_kv_heads, head_dim] of {row_dtype}")
    st = lib().paged_kv_append(ctypes.byref(pool), _ptr(key), _ptr(value), _ptr(slot_mapping), T,
                               _stream(stream))
    _check(st, "paged_kv_append")


def decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, dtype=torch.bfloat16) -> int:
    return int(lib().paged_attention_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                                          _dtype_code(dtype)))


def decode_workspace(batch, num_q_heads, key_pool, device=None) -> Optional[torch.Tensor]:
    """Allocate (with torch) the scratch buffer paged_attention_decode needs."""
    n = decode_workspace_size(batch, num_q_heads, key_pool.shape[2], key_pool.shape[3],
                              key_pool.dtype)
    if n == 0:
        return None
    return torch.empty(n, dtype=torch.uint8, device=device or key_pool.device)


def paged_attention_decode(key_pool, value_pool, q, block_table, seq_lens, scale,
                           max_seq_len=None, out=None, workspace=None, stream=None, k_scale=1.0,
                           v_scale=1.0):
    """Decode attention: ``q [B, Hq, D]`` -> ``out [B, Hq, D]``.

    ``block_table`` int32 [B, max_blocks]; ``seq_lens`` int32 [B] (after the
    append).  ``max_seq_len`` defaults to max_blocks * page_size (an upper
    bound needs no device read).  ``k_scale`` / ``v_scale`` apply to e4m3 pools.
    """
    pool = make_pool(key_pool, value_pool, k_scale, v_scale)
    _contig(q, "q")
    _contig(block_table, "block_table")
    B, hq, d = q.shape
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_table and seq_lens must be int32")
    mb = block_table.shape[1]
    if max_seq_len is None:
        max_seq_len = mb * pool.page_size
    out = _q_out(q, out, key_pool)
    if workspace is None:
        workspace = decode_workspace(B, hq, key_pool)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().paged_attention_decode(ctypes.byref(pool), _ptr(q), _ptr(out), B, hq,
                                      _ptr(block_table), mb, _ptr(seq_lens), int(max_seq_len),
                                      float(scale), _ptr(workspace), wbytes, _stream(stream))
    _check(st, "paged_attention_decode")
    return out


def paged_attention_decode_append(key_pool, value_pool, key, value, slot_mapping, q, block_table,
                                  seq_lens, scale, max_seq_len=None, out=None, workspace=None,
                                  stream=None, k_scale=1.0, v_scale=1.0):
    """One decode step in one launch: append ``key/value [B, Hkv, D]`` at
    ``slot_mapping`` int64 [B] (each the slot of its sequence's last key, or
    < 0 for none), then decode ``q [B, Hq, D]`` over the updated pools
    (``seq_lens`` count the new token).  Returns ``out``; the pools are
    updated in place."""
    pool = make_pool(key_pool, value_pool, k_scale, v_scale)
    for t, nm in ((q, "q"), (block_table, "block_table"), (key, "key"), (value, "value"),
                  (slot_mapping, "slot_mapping")):
        _contig(t, nm)
    B, hq, d = q.shape
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_table and seq_lens must be int32")
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    row_dtype = torch.bfloat16 if key_pool.dtype == torch.float8_e4m3fn else key_pool.dtype
    for n, t in (("key", key), ("value", value)):
        if t.dtype != row_dtype or t.numel() != B * pool.num_kv_heads * pool.head_dim:
            raise ValueError(f"{n} must be [B, num_kv_heads, head_dim] of {row_dtype}")
    if slot_mapping.numel() != B:
        raise ValueError("one new token per sequence: slot_mapping [B]")
    mb = block_table.shape[1]
    if max_seq_len is None:
        max_seq_len = mb * pool.page_size
    out = _q_out(q, out, key_pool)
    if workspace is None:
        workspace = decode_workspace(B, hq, key_pool)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().paged_attention_decode_append(ctypes.byref(pool), _ptr(key), _ptr(value),
                                             _ptr(slot_mapping), _ptr(q), _ptr(out), B, hq,
                                             _ptr(block_table), mb, _ptr(seq_lens),
                                             int(max_seq_len), float(scale), _ptr(workspace), wbytes,
                                             _stream(stream))
    _check(st, "paged_attention_decode_append")
    return out


def paged_attention_decode_static_scratch(key_pool, value_pool, q, block_table, seq_lens, scale,
                                          max_seq_len=None, out=None, stream=None, k_scale=1.0,
                                          v_scale=1.0):
    """Decode attention whose scratch is the library's own static device array.

    For callers that may not allocate device memory; see the header for the
    size limit and the sharing rules of that array.
    """
    pool = make_pool(key_pool, value_pool, k_scale, v_scale)
    _contig(q, "q")
    _contig(block_table, "block_table")
    B, hq, d = q.shape
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_table and seq_lens must be int32")
    mb = block_table.shape[1]
    if max_seq_len is None:
        max_seq_len = mb * pool.page_size
    out = _q_out(q, out, key_pool)
    st = lib().paged_attention_decode_static_scratch(ctypes.byref(pool), _ptr(q), _ptr(out), B, hq,
                                                     _ptr(block_table), mb, _ptr(seq_lens),
                                                     int(max_seq_len), float(scale),
                                                     _stream(stream))
    _check(st, "paged_attention_decode_static_scratch")
    return out


def cascade_workspace(batch, num_q_heads, key_pool, device=None) -> Optional[torch.Tensor]:
    """Allocate (with torch) the scratch buffer paged_attention_decode_cascade needs."""
    n = int(lib().paged_attention_decode_cascade_workspace_size(
        batch, num_q_heads, key_pool.shape[2], key_pool.shape[3], _dtype_code(key_pool.dtype)))
    if n == 0:
        return None
    return torch.empty(n, dtype=torch.uint8, device=device or key_pool.device)


def paged_attention_decode_cascade(key_pool, value_pool, q, prefix_block_ids, prefix_len,
                                   block_table, seq_lens, scale, max_seq_len=None, out=None,
                                   workspace=None, stream=None):
    """Decode over a prefix shared by the whole batch, then each sequence's own pages.

    ``prefix_block_ids`` int32 [ceil(prefix_len / page_size)]; ``block_table``
    int32 [B, max_blocks] and ``seq_lens`` int32 [B] describe each sequence's
    own tokens only.
    """
    pool = make_pool(key_pool, value_pool)
    _contig(q, "q")
    _contig(block_table, "block_table")
    _contig(prefix_block_ids, "prefix_block_ids")
    B, hq, d = q.shape
    if (block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32
            or prefix_block_ids.dtype != torch.int32):
        raise TypeError("prefix_block_ids, block_table and seq_lens must be int32")
    mb = block_table.shape[1]
    if max_seq_len is None:
        max_seq_len = mb * pool.page_size
    out = _q_out(q, out, key_pool)
    if workspace is None:
        workspace = cascade_workspace(B, hq, key_pool)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().paged_attention_decode_cascade(ctypes.byref(pool), _ptr(q), _ptr(out), B, hq,
                                              _ptr(prefix_block_ids), int(prefix_len),
                                              _ptr(block_table), mb, _ptr(seq_lens), int(max_seq_len),
                                              float(scale), _ptr(workspace), wbytes, _stream(stream))
    _check(st, "paged_attention_decode_cascade")
    return out


def paged_attention_prefill(key_pool, value_pool, q, query_start_loc, block_table, seq_lens,
                            scale, max_q_len, max_seq_len=None, out=None, stream=None, k_scale=1.0,
                            v_scale=1.0):
    """Varlen causal prefill: ``q [T, Hq, D]`` packed by ``query_start_loc`` int32 [B+1].

    ``max_q_len`` is a host upper bound of the per-sequence new-token counts.
    ``k_scale`` / ``v_scale`` apply to e4m3 pools.
    """
    pool = make_pool(key_pool, value_pool, k_scale, v_scale)
    _contig(q, "q")
    _contig(block_table, "block_table")
    T, hq, d = q.shape
    B = query_start_loc.numel() - 1
    if query_start_loc.dtype != torch.int32 or block_table.dtype != torch.int32 \
            or seq_lens.dtype != torch.int32:
        raise TypeError("query_start_loc, block_table and seq_lens must be int32")
    mb = block_table.shape[1]
    if max_seq_len is None:
        max_seq_len = mb * pool.page_size
    out = _q_out(q, out, key_pool)
    st = lib().paged_attention_prefill(ctypes.byref(pool), _ptr(q), _ptr(out), B, hq,
                                       _ptr(query_start_loc), T, int(max_q_len),
                                       _ptr(block_table), mb, _ptr(seq_lens), int(max_seq_len),
                                       float(scale), _stream(stream))
    _check(st, "paged_attention_prefill")
    return out


def device_error():
    """Read and clear the device error word: (code, detail); (0, 0) if clean."""
    code, detail = _i64(0), _i64(0)
    _check(lib().paged_device_error(ctypes.byref(code), ctypes.byref(detail)), "paged_device_error")
    return int(code.value), int(detail.value)


def _csr_args(kv_indptr, kv_indices, kv_last_page_len):
    for name, t in (("kv_indptr", kv_indptr), ("kv_indices", kv_indices),
                    ("kv_last_page_len", kv_last_page_len)):
        _contig(t, name)
        if t.dtype != torch.int32:
            raise TypeError(f"{name} must be int32")
    return _ptr(kv_indptr), _ptr(kv_indices), int(kv_indices.numel()), _ptr(kv_last_page_len)


def paged_attention_decode_csr(key_pool, value_pool, q, kv_indptr, kv_indices, kv_last_page_len,
                               scale, max_seq_len, out=None, workspace=None, stream=None, k_scale=1.0,
                               v_scale=1.0):
    """Decode with the page table in CSR form: sequence b's pages are
    ``kv_indices[kv_indptr[b]:kv_indptr[b+1]]``, its last page holds
    ``kv_last_page_len[b]`` tokens (all int32 device tensors)."""
    pool = make_pool(key_pool, value_pool, k_scale, v_scale)
    _contig(q, "q")
    B, hq, d = q.shape
    ip, ix, nix, last = _csr_args(kv_indptr, kv_indices, kv_last_page_len)
    out = _q_out(q, out, key_pool)
    if workspace is None:
        workspace = decode_workspace(B, hq, key_pool)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().paged_attention_decode_csr(ctypes.byref(pool), _ptr(q), _ptr(out), B, hq, ip, ix, nix, last,
                                          int(max_seq_len), float(scale), _ptr(workspace), wbytes,
                                          _stream(stream))
    _check(st, "paged_attention_decode_csr")
    return out


def paged_attention_prefill_csr(key_pool, value_pool, q, query_start_loc, kv_indptr, kv_indices,
                                kv_last_page_len, scale, max_q_len, max_seq_len, out=None, stream=None,
                                k_scale=1.0, v_scale=1.0):
    """Varlen causal prefill with the page table in CSR form (``k_scale`` /
    ``v_scale`` for e4m3 pools)."""
    pool = make_pool(key_pool, value_pool, k_scale, v_scale)
    _contig(q, "q")
    _contig(query_start_loc, "query_start_loc")
    T, hq, d = q.shape
    B = query_start_loc.numel() - 1
    ip, ix, nix, last = _csr_args(kv_indptr, kv_indices, kv_last_page_len)
    out = _q_out(q, out, key_pool)
    st = lib().paged_attention_prefill_csr(ctypes.byref(pool), _ptr(q), _ptr(out), B, hq,
                                           _ptr(query_start_loc), T, int(max_q_len), ip, ix, nix, last,
                                           int(max_seq_len), float(scale), _stream(stream))
    _check(st, "paged_attention_prefill_csr")
    return out
