"""ctypes binding of libpaged_kv.so (C ABI: include/paged_kv.h).

Argument marshalling only: tensors become device pointers and sizes, the
current torch stream becomes the call's stream, and a non-zero status becomes
a PagedKVError. Every step of the computation runs in the library's kernels;
there is no fallback of any kind, so a missing library raises on first use.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpaged_kv.so")

PKV_F16, PKV_BF16, PKV_FP8_E4M3 = 0, 1, 2
_DTYPE = {torch.float16: PKV_F16, torch.bfloat16: PKV_BF16}
_FP8_DTYPES = (torch.uint8, torch.float8_e4m3fn)  # an FP8 cache: E4M3 codes
DEVERR_BITS = {1: "BLOCK_ID", 2: "CONTEXT", 4: "SLOT", 8: "TIMEOUT", 16: "QUERY", 32: "LAYOUT"}

_lib = None


class PagedKVError(RuntimeError):
    def __init__(self, status, message):
        self.status = status
        super().__init__(message)


def load():
    """Load the library (once). Raises PagedKVError if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise PagedKVError(None, f"{LIB_PATH} is missing: build it with "
                                 "`python -m paged_kv_cache_91_gb300.build` (or __graft_entry__.build())")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.paged_kv_write.restype = i32
    lib.paged_kv_write.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, P]
    lib.paged_attention_workspace_size.restype = sz
    lib.paged_attention_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    lib.paged_attention_decode.restype = i32
    lib.paged_attention_decode.argtypes = [P, P, P, P, P, i32, P, i32, i32, f32, i32, i32, i32, i32, i32, i32,
                                           i32, P, sz, P]
    lib.paged_kv_device_errors.restype = i32
    lib.paged_kv_device_errors.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32]
    lib.pkv_status_string.restype = ctypes.c_char_p
    lib.pkv_status_string.argtypes = [i32]
    lib.pkv_last_error_message.restype = ctypes.c_char_p
    lib.pkv_last_error_message.argtypes = []
    lib.paged_kv_copy_blocks.restype = i32
    lib.paged_kv_copy_blocks.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, P]
    lib.pkv_selftest_wait_timeout.restype = i32
    lib.pkv_selftest_wait_timeout.argtypes = [i64, P]
    lib.paged_kv_write_fp8.restype = i32
    lib.paged_kv_write_fp8.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, f32, f32, P]
    lib.paged_attention_workspace_size_fp8.restype = sz
    lib.paged_attention_workspace_size_fp8.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    lib.paged_attention_multi_query_workspace_size.restype = sz
    lib.paged_attention_multi_query_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    lib.pkv_set_multi_query_tile.restype = i32
    lib.pkv_set_multi_query_tile.argtypes = [i32]
    lib.paged_attention_shared_prefix_workspace_size.restype = sz
    lib.paged_attention_shared_prefix_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    lib.paged_attention_decode_shared_prefix.restype = i32
    lib.paged_attention_decode_shared_prefix.argtypes = [P, P, P, P, P, i32, P, i32, P, i32, i32, f32, i32, i32, i32,
                                                         i32, i32, i32, P, sz, P]
    lib.paged_attention_decode_shared_prefix_fp8.restype = i32
    lib.paged_attention_decode_shared_prefix_fp8.argtypes = [P, P, P, P, P, i32, P, i32, P, i32, i32, f32, i32, i32,
                                                             i32, i32, i32, i32, f32, f32, P, sz, P]
    lib.paged_attention_multi_query.restype = i32
    lib.paged_attention_multi_query.argtypes = [P, P, P, P, P, i32, P, P, i32, i32, i32, i32, f32, i32, i32, i32,
                                                i32, i32, i32, i32, P, sz, P]
    lib.paged_attention_multi_query_fp8.restype = i32
    lib.paged_attention_multi_query_fp8.argtypes = [P, P, P, P, P, i32, P, P, i32, i32, i32, i32, f32, i32, i32,
                                                    i32, i32, i32, i32, f32, f32, i32, P, sz, P]
    lib.paged_attention_decode_fp8.restype = i32
    lib.paged_attention_decode_fp8.argtypes = [P, P, P, P, P, i32, P, i32, i32, f32, i32, i32, i32, i32, i32, i32,
                                               f32, f32, i32, P, sz, P]
    _lib = lib
    return lib


def _check(lib, status: int) -> None:
    if status != 0:
        name = lib.pkv_status_string(status).decode()
        msg = lib.pkv_last_error_message().decode()
        raise PagedKVError(status, f"{name}: {msg}")


def _ptr(t: Optional[torch.Tensor]):
    # the argtypes are c_void_p: a Python int (or None) converts without a wrapper object
    return t.data_ptr() if t is not None else None


# The current stream's handle as an int, without building a torch Stream object (about 2 us per call);
# torch.cuda.current_stream where that accessor is missing.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(t: torch.Tensor, stream):
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(t.get_device())
        stream = torch.cuda.current_stream(t.device)
    return stream.cuda_stream


def _cuda16(name: str, t: torch.Tensor) -> int:
    dt = _DTYPE.get(t.dtype)
    if dt is None or not t.is_cuda or not t.is_contiguous():
        if not t.is_cuda:
            raise PagedKVError(-1, f"{name} must be a CUDA tensor")
        if dt is None:
            raise PagedKVError(-1, f"{name} must be float16 or bfloat16, got {t.dtype}")
        raise PagedKVError(-1, f"{name} must be contiguous")
    return dt


def _cuda_i32(name: str, t: torch.Tensor) -> None:
    if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
        raise PagedKVError(-1, f"{name} must be a contiguous CUDA int32 tensor")


def _cuda_fp8(name: str, t: torch.Tensor) -> None:
    if not t.is_cuda or t.dtype not in _FP8_DTYPES or not t.is_contiguous():
        raise PagedKVError(-1, f"{name} must be a contiguous CUDA uint8 or float8_e4m3fn tensor (E4M3 codes)")


def _cache_dtype(name: str, t: torch.Tensor) -> int:
    if t.dtype in _FP8_DTYPES:
        _cuda_fp8(name, t)
        return PKV_FP8_E4M3
    return _cuda16(name, t)


def paged_kv_write(key: torch.Tensor, value: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                   slot_mapping: torch.Tensor, stream=None) -> None:
    """Scatter key/value [T][Hkv][D] into the pool [NB][Hkv][B][D] at slot_mapping [T] (int64)."""
    lib = load()
    dt = _cuda16("key_cache", key_cache)
    for n, t in (("key", key), ("value", value), ("value_cache", value_cache)):
        if _cuda16(n, t) != dt:
            raise PagedKVError(-1, f"{n} dtype differs from key_cache")
    if slot_mapping.dtype != torch.int64 or not slot_mapping.is_cuda or not slot_mapping.is_contiguous():
        raise PagedKVError(-1, "slot_mapping must be a contiguous CUDA int64 tensor")
    NB, Hkv, B, D = key_cache.shape
    T = slot_mapping.numel()
    if key.shape != (T, Hkv, D) or value.shape != (T, Hkv, D) or value_cache.shape != key_cache.shape:
        raise PagedKVError(-1, "shape mismatch between key/value, caches and slot_mapping")
    _check(lib, lib.paged_kv_write(_ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache), _ptr(slot_mapping),
                                   T, Hkv, D, B, NB, dt, _stream(key_cache, stream)))


def paged_kv_copy_blocks(key_cache: torch.Tensor, value_cache: torch.Tensor, block_mapping: torch.Tensor,
                         stream=None) -> None:
    """Copy whole physical blocks: block_mapping [num_pairs][2] int64 (src, dst) on the device."""
    lib = load()
    dt = _cache_dtype("key_cache", key_cache)
    if _cache_dtype("value_cache", value_cache) != dt or value_cache.shape != key_cache.shape:
        raise PagedKVError(-1, "value_cache must match key_cache")
    if block_mapping.dtype != torch.int64 or not block_mapping.is_cuda or not block_mapping.is_contiguous():
        raise PagedKVError(-1, "block_mapping must be a contiguous CUDA int64 tensor")
    if block_mapping.numel() % 2:
        raise PagedKVError(-1, "block_mapping must hold (src, dst) pairs")
    NB, Hkv, B, D = key_cache.shape
    _check(lib, lib.paged_kv_copy_blocks(_ptr(key_cache), _ptr(value_cache), _ptr(block_mapping),
                                         block_mapping.numel() // 2, Hkv, D, B, NB, dt, _stream(key_cache, stream)))


def paged_attention_workspace_size(num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int,
                                   block_size: int, max_context_len: int, partition_size: int = 0) -> int:
    return int(load().paged_attention_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                                     max_context_len, partition_size))


def paged_attention_decode(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                           value_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                           scale: float, block_size: Optional[int] = None, num_kv_heads: Optional[int] = None,
                           max_context_len: Optional[int] = None, partition_size: int = 0,
                           workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Decode attention: out[s][h] = softmax(scale q.K^T) V over the first context_lens[s] tokens.

    ``max_context_len`` bounds every context length on the host; when omitted it
    is max_blocks_per_seq * block_size (always safe, possibly more partitions).
    ``workspace`` (uint8, >= paged_attention_workspace_size bytes) is allocated
    here through torch when omitted and a split is needed.
    """
    lib = load()
    dt = _cuda16("query", query)
    for n, t in (("out", out), ("key_cache", key_cache), ("value_cache", value_cache)):
        if _cuda16(n, t) != dt:
            raise PagedKVError(-1, f"{n} dtype differs from query")
    _cuda_i32("block_tables", block_tables)
    _cuda_i32("context_lens", context_lens)
    NB, Hkv, B, D = key_cache.shape
    if block_size is not None and block_size != B:
        raise PagedKVError(-1, f"block_size {block_size} != key_cache.shape[2] {B}")
    if num_kv_heads is not None and num_kv_heads != Hkv:
        raise PagedKVError(-1, f"num_kv_heads {num_kv_heads} != key_cache.shape[1] {Hkv}")
    S, H, D2 = query.shape
    if D2 != D or out.shape != query.shape or value_cache.shape != key_cache.shape:
        raise PagedKVError(-1, "shape mismatch between query, out and caches")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise PagedKVError(-1, "block_tables must be [S][max_blocks] and context_lens [S]")
    maxb = block_tables.shape[1]
    if max_context_len is None:
        max_context_len = maxb * B
    if workspace is None:  # (a workspace passed in is checked against the size by the library)
        need = int(lib.paged_attention_workspace_size(S, H, Hkv, D, B, max_context_len, partition_size))
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=query.device)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib, lib.paged_attention_decode(
        _ptr(out), _ptr(query), _ptr(key_cache), _ptr(value_cache), _ptr(block_tables), maxb,
        _ptr(context_lens), S, int(max_context_len), float(scale), B, H, Hkv, D, NB, dt, int(partition_size),
        _ptr(workspace), wbytes, _stream(query, stream)))
    return out


def paged_kv_write_fp8(key: torch.Tensor, value: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                       slot_mapping: torch.Tensor, k_scale: float, v_scale: float, stream=None) -> None:
    """Quantizing scatter: key/value [T][Hkv][D] (f16/bf16) into an E4M3 pool [NB][Hkv][B][D]
    (uint8 or float8_e4m3fn): code = E4M3(x / k_scale), likewise for values with v_scale."""
    lib = load()
    dt = _cuda16("key", key)
    if _cuda16("value", value) != dt:
        raise PagedKVError(-1, "value dtype differs from key")
    _cuda_fp8("key_cache", key_cache)
    _cuda_fp8("value_cache", value_cache)
    if slot_mapping.dtype != torch.int64 or not slot_mapping.is_cuda or not slot_mapping.is_contiguous():
        raise PagedKVError(-1, "slot_mapping must be a contiguous CUDA int64 tensor")
    NB, Hkv, B, D = key_cache.shape
    T = slot_mapping.numel()
    if key.shape != (T, Hkv, D) or value.shape != (T, Hkv, D) or value_cache.shape != key_cache.shape:
        raise PagedKVError(-1, "shape mismatch between key/value, caches and slot_mapping")
    _check(lib, lib.paged_kv_write_fp8(_ptr(key), _ptr(value), _ptr(key_cache), _ptr(value_cache),
                                       _ptr(slot_mapping), T, Hkv, D, B, NB, dt, float(k_scale), float(v_scale),
                                       _stream(key_cache, stream)))


def paged_attention_workspace_size_fp8(num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int,
                                       block_size: int, max_context_len: int, partition_size: int = 0) -> int:
    return int(load().paged_attention_workspace_size_fp8(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                                         max_context_len, partition_size))


def paged_attention_decode_fp8(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                               value_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                               scale: float, k_scale: float, v_scale: float, max_context_len: Optional[int] = None,
                               partition_size: int = 0, workspace: Optional[torch.Tensor] = None,
                               stream=None) -> torch.Tensor:
    """paged_attention_decode over an E4M3 pool whose elements are code * k_scale (K) and code * v_scale (V)."""
    lib = load()
    dt = _cuda16("query", query)
    if _cuda16("out", out) != dt:
        raise PagedKVError(-1, "out dtype differs from query")
    _cuda_fp8("key_cache", key_cache)
    _cuda_fp8("value_cache", value_cache)
    _cuda_i32("block_tables", block_tables)
    _cuda_i32("context_lens", context_lens)
    NB, Hkv, B, D = key_cache.shape
    S, H, D2 = query.shape
    if D2 != D or out.shape != query.shape or value_cache.shape != key_cache.shape:
        raise PagedKVError(-1, "shape mismatch between query, out and caches")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise PagedKVError(-1, "block_tables must be [S][max_blocks] and context_lens [S]")
    maxb = block_tables.shape[1]
    if max_context_len is None:
        max_context_len = maxb * B
    if workspace is None:
        need = int(lib.paged_attention_workspace_size_fp8(S, H, Hkv, D, B, max_context_len, partition_size))
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=query.device)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib, lib.paged_attention_decode_fp8(
        _ptr(out), _ptr(query), _ptr(key_cache), _ptr(value_cache), _ptr(block_tables), maxb,
        _ptr(context_lens), S, int(max_context_len), float(scale), B, H, Hkv, D, NB, dt, float(k_scale),
        float(v_scale), int(partition_size), _ptr(workspace), wbytes, _stream(query, stream)))
    return out


MQ_TILE_AUTO, MQ_TILE_COLUMNS, MQ_TILE_ROWS, MQ_TILE_TENSOR, MQ_TILE_PAIRS = 0, 1, 2, 3, 4


def set_multi_query_tile(tile: int) -> int:
    """Choose the multi-query tile for later calls (MQ_TILE_*); returns the previous choice."""
    prev = int(load().pkv_set_multi_query_tile(int(tile)))
    if prev < 0:
        raise PagedKVError(-1, f"unknown multi-query tile {tile}")
    return prev


def paged_attention_multi_query_workspace_size(num_query_tokens: int, num_heads: int, num_kv_heads: int,
                                               head_dim: int, block_size: int, max_context_len: int,
                                               partition_size: int = 0) -> int:
    return int(load().paged_attention_multi_query_workspace_size(num_query_tokens, num_heads, num_kv_heads,
                                                                 head_dim, block_size, max_context_len,
                                                                 partition_size))


def _multi_query(out, query, key_cache, value_cache, block_tables, context_lens, query_start_loc, scale,
                 max_query_len, max_context_len, partition_size, workspace, stream, fp8, k_scale, v_scale):
    lib = load()
    dt = _cuda16("query", query)
    if _cuda16("out", out) != dt:
        raise PagedKVError(-1, "out dtype differs from query")
    for n, t in (("key_cache", key_cache), ("value_cache", value_cache)):
        if fp8:
            _cuda_fp8(n, t)
        elif _cuda16(n, t) != dt:
            raise PagedKVError(-1, f"{n} dtype differs from query")
    _cuda_i32("block_tables", block_tables)
    _cuda_i32("context_lens", context_lens)
    _cuda_i32("query_start_loc", query_start_loc)
    NB, Hkv, B, D = key_cache.shape
    T, H, D2 = query.shape
    S = context_lens.shape[0]
    if D2 != D or out.shape != query.shape or value_cache.shape != key_cache.shape:
        raise PagedKVError(-1, "shape mismatch between query, out and caches")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or query_start_loc.shape != (S + 1,):
        raise PagedKVError(-1, "block_tables must be [S][max_blocks] and query_start_loc [S + 1]")
    maxb = block_tables.shape[1]
    if max_context_len is None:
        max_context_len = maxb * B
    if max_query_len is None:
        max_query_len = int((query_start_loc[1:] - query_start_loc[:-1]).max().item()) if S else 0
    if workspace is None:
        need = int(lib.paged_attention_multi_query_workspace_size(T, H, Hkv, D, B, max_context_len,
                                                                  partition_size))
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=query.device)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    head = (_ptr(out), _ptr(query), _ptr(key_cache), _ptr(value_cache), _ptr(block_tables), maxb,
            _ptr(context_lens), _ptr(query_start_loc), S, T, int(max_query_len), int(max_context_len), float(scale),
            B, H, Hkv, D, NB, dt)
    tail = (int(partition_size), _ptr(workspace), wbytes, _stream(query, stream))
    if fp8:
        _check(lib, lib.paged_attention_multi_query_fp8(*head, float(k_scale), float(v_scale), *tail))
    else:
        _check(lib, lib.paged_attention_multi_query(*head, *tail))
    return out


def paged_attention_multi_query(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                                value_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                                query_start_loc: torch.Tensor, scale: float, max_query_len: Optional[int] = None,
                                max_context_len: Optional[int] = None, partition_size: int = 0,
                                workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Causal attention of several query tokens per sequence (query/out [T][H][D], packed by
    query_start_loc [S+1] int32): sequence s's q_len tokens are its last q_len context positions.

    ``max_query_len`` bounds every q_len on the host; when omitted it is read from
    query_start_loc, which synchronises the stream.
    """
    return _multi_query(out, query, key_cache, value_cache, block_tables, context_lens, query_start_loc, scale,
                        max_query_len, max_context_len, partition_size, workspace, stream, False, 1.0, 1.0)


def paged_attention_multi_query_fp8(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                                    value_cache: torch.Tensor, block_tables: torch.Tensor,
                                    context_lens: torch.Tensor, query_start_loc: torch.Tensor, scale: float,
                                    k_scale: float, v_scale: float, max_query_len: Optional[int] = None,
                                    max_context_len: Optional[int] = None, partition_size: int = 0,
                                    workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """paged_attention_multi_query over an E4M3 pool whose elements are code * k_scale (K) and
    code * v_scale (V); head_dim 128."""
    return _multi_query(out, query, key_cache, value_cache, block_tables, context_lens, query_start_loc, scale,
                        max_query_len, max_context_len, partition_size, workspace, stream, True, k_scale, v_scale)


def paged_attention_shared_prefix_workspace_size(num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int,
                                                 block_size: int, prefix_len: int, max_tail_len: int) -> int:
    return int(load().paged_attention_shared_prefix_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim,
                                                                   block_size, prefix_len, max_tail_len))


def _shared_prefix(out, query, key_cache, value_cache, prefix_blocks, prefix_len, block_tables, tail_lens, scale,
                   max_tail_len, workspace, stream, fp8, k_scale, v_scale):
    lib = load()
    dt = _cuda16("query", query)
    if _cuda16("out", out) != dt:
        raise PagedKVError(-1, "out dtype differs from query")
    for n, t in (("key_cache", key_cache), ("value_cache", value_cache)):
        if fp8:
            _cuda_fp8(n, t)
        elif _cuda16(n, t) != dt:
            raise PagedKVError(-1, f"{n} dtype differs from query")
    _cuda_i32("prefix_blocks", prefix_blocks)
    _cuda_i32("block_tables", block_tables)
    _cuda_i32("tail_lens", tail_lens)
    NB, Hkv, B, D = key_cache.shape
    S, H, D2 = query.shape
    if D2 != D or out.shape != query.shape or value_cache.shape != key_cache.shape:
        raise PagedKVError(-1, "shape mismatch between query, out and caches")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or tail_lens.shape != (S,):
        raise PagedKVError(-1, "block_tables must be [S][max_blocks] and tail_lens [S]")
    maxb = block_tables.shape[1]
    if max_tail_len is None:
        max_tail_len = maxb * B
    if workspace is None:
        need = paged_attention_shared_prefix_workspace_size(S, H, Hkv, D, B, int(prefix_len), int(max_tail_len))
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=query.device)
    wbytes = workspace.numel() * workspace.element_size()
    head = (_ptr(out), _ptr(query), _ptr(key_cache), _ptr(value_cache), _ptr(prefix_blocks), int(prefix_len),
            _ptr(block_tables), maxb, _ptr(tail_lens), S, int(max_tail_len), float(scale), B, H, Hkv, D, NB, dt)
    tail = (_ptr(workspace), wbytes, _stream(query, stream))
    if fp8:
        _check(lib, lib.paged_attention_decode_shared_prefix_fp8(*head, float(k_scale), float(v_scale), *tail))
    else:
        _check(lib, lib.paged_attention_decode_shared_prefix(*head, *tail))
    return out


def paged_attention_decode_shared_prefix(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                                         value_cache: torch.Tensor, prefix_blocks: torch.Tensor, prefix_len: int,
                                         block_tables: torch.Tensor, tail_lens: torch.Tensor, scale: float,
                                         max_tail_len: Optional[int] = None,
                                         workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Decode for sequences that share their first prefix_len tokens (prefix_blocks [prefix_len / B] int32);
    block_tables [S][max] and tail_lens [S] describe each sequence's tokens after the prefix. Same result as
    paged_attention_decode over prefix_blocks ++ block_tables[s], with the prefix read once."""
    return _shared_prefix(out, query, key_cache, value_cache, prefix_blocks, prefix_len, block_tables, tail_lens,
                          scale, max_tail_len, workspace, stream, False, 1.0, 1.0)


def paged_attention_decode_shared_prefix_fp8(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                                             value_cache: torch.Tensor, prefix_blocks: torch.Tensor,
                                             prefix_len: int, block_tables: torch.Tensor, tail_lens: torch.Tensor,
                                             scale: float, k_scale: float, v_scale: float,
                                             max_tail_len: Optional[int] = None,
                                             workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """paged_attention_decode_shared_prefix over an E4M3 pool (elements code * k_scale, code * v_scale)."""
    return _shared_prefix(out, query, key_cache, value_cache, prefix_blocks, prefix_len, block_tables, tail_lens,
                          scale, max_tail_len, workspace, stream, True, k_scale, v_scale)


def device_errors(clear: bool = True) -> int:
    """The current device's error word (PKV_DEVERR_* bits); synchronises the device."""
    lib = load()
    v = ctypes.c_uint32(0)
    _check(lib, lib.paged_kv_device_errors(ctypes.byref(v), 1 if clear else 0))
    return int(v.value)


def paged_attention_decode_static_workspace(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                                            value_cache: torch.Tensor, block_tables: torch.Tensor,
                                            context_lens: torch.Tensor, scale: float,
                                            max_context_len: Optional[int] = None, partition_size: int = 0,
                                            stream=None) -> torch.Tensor:
    """paged_attention_decode without a caller workspace, for callers that cannot allocate device memory.

    The split-K scratch is the library's own PKV_STATIC_WORKSPACE_BYTES (32 MiB)
    array on each device, so nothing is allocated here or in the library.
    Calls on one device share that array: calls that overlap on the GPU race.
    """
    lib = load()
    fn = lib.paged_attention_decode_static_workspace
    if fn.argtypes is None:
        P, i32, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
        fn.restype = i32
        fn.argtypes = [P, P, P, P, P, i32, P, i32, i32, f32, i32, i32, i32, i32, i32, i32, i32, P]
    dt = _cuda16("query", query)
    for n, t in (("out", out), ("key_cache", key_cache), ("value_cache", value_cache)):
        if _cuda16(n, t) != dt:
            raise PagedKVError(-1, f"{n} dtype differs from query")
    _cuda_i32("block_tables", block_tables)
    _cuda_i32("context_lens", context_lens)
    NB, Hkv, B, D = key_cache.shape
    S, H, _ = query.shape
    if out.shape != query.shape or value_cache.shape != key_cache.shape:
        raise PagedKVError(-1, "shape mismatch between query, out and caches")
    maxb = block_tables.shape[1]
    if max_context_len is None:
        max_context_len = maxb * B
    _check(lib, fn(_ptr(out), _ptr(query), _ptr(key_cache), _ptr(value_cache), _ptr(block_tables), maxb,
                   _ptr(context_lens), S, int(max_context_len), float(scale), B, H, Hkv, D, NB, dt,
                   int(partition_size), _stream(query, stream)))
    return out


def read_chunks(buffer: torch.Tensor, order: torch.Tensor, chunk_bytes: int, stream=None) -> None:
    """Read the chunks order[i] (int32, on the device) of chunk_bytes from buffer (uint8), one bulk copy each
    into shared memory: the read ceiling of an access pattern (a measurement helper, not a step of the method)."""
    lib = load()
    fn = lib.pkv_read_chunks
    if fn.argtypes is None:
        fn.restype = ctypes.c_int32
        fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                       ctypes.c_void_p]
    if buffer.dtype != torch.uint8 or not buffer.is_cuda or not buffer.is_contiguous():
        raise PagedKVError(-1, "buffer must be a contiguous CUDA uint8 tensor")
    _cuda_i32("order", order)
    _check(lib, fn(_ptr(buffer), buffer.numel(), _ptr(order), order.numel(), int(chunk_bytes),
                   _stream(buffer, stream)))


def selftest_wait_timeout(limit_cycles: int = 2_000_000) -> int:
    """Run the bounded-wait self-test; returns the error word it leaves (PKV_DEVERR_TIMEOUT expected)."""
    lib = load()
    _check(lib, lib.pkv_selftest_wait_timeout(int(limit_cycles), _stream(torch.empty(0, device="cuda"), None)))
    return device_errors(clear=True)
