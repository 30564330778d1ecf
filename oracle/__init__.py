"""CPU oracle for the paged KV cache hot path (fp64).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may use this package; the CUDA library and its
Python binding never import it. It shares no code with the CUDA path.

Two independent implementations of the same definitions:

* ``write_c`` / ``decode_c`` -- plain C (``pkv_oracle.c``), fp64, OpenMP over
  (sequence, head) pairs; fast enough for the full-size workloads.
* ``write_np`` / ``decode_np`` -- numpy, fp64, gather-then-attend; plus
  ``attention_np``, unpaged attention over contiguous K/V arrays.

Decode computes, for each sequence s and query head h with kv head
g = h // (H / Hkv) and the first ctx_s cached tokens gathered through the
block table (token j lives in block block_tables[s][j // B] at offset j % B):

    x_j = scale * q . K_j ;  w = softmax(x) ;  o = sum_j w_j V_j

("KV Cache와 PagedAttention 완전 해부", 부록; "vLLM: LLM 서빙 메모리 최적화의
교과서", 01 Problem Definition and eq. (4)). Write copies each new token's
rows bit for bit into block slot // B, offset slot % B ("[vLLM] PagedAttention:
OS 페이징 기법으로 KV 캐시를 관리하는 방법", write_to_paged_cache /
reshape_and_cache).

Pins: tests/test_oracle.py checks both implementations against closed forms,
brute force, invariants and the values the pages print (tests/golden/).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

DTYPE_CODE = {"f16": 0, "bf16": 1}


def build(force: bool = False) -> str:
    """Compile pkv_oracle.c into oracle/liboracle.so with gcc (OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int, ctypes.c_longlong, ctypes.c_double
        lib.oracle_write.restype = i64
        lib.oracle_write.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i64]
        lib.oracle_decode.restype = i32
        lib.oracle_decode.argtypes = [P, P, P, P, P, i32, P, i32, f64, i32, i32, i32, i32, i64, i32,
                                      P, i64, i32]
        lib.oracle_copy_blocks.restype = i64
        lib.oracle_copy_blocks.argtypes = [P, P, P, i32, i32, i32, i32, i64]
        lib.oracle_widen.restype = f64
        lib.oracle_widen.argtypes = [ctypes.c_uint16, i32]
        lib.oracle_max_threads.restype = i32
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


# ----------------------------------------------------------------------------
# C implementation


def write_c(key_cache, value_cache, new_key, new_value, slot_mapping, block_size):
    """Scatter new tokens into copies of the pools; returns (key_cache', value_cache')."""
    kc = np.ascontiguousarray(key_cache, dtype=np.uint16).copy()
    vc = np.ascontiguousarray(value_cache, dtype=np.uint16).copy()
    k = np.ascontiguousarray(new_key, dtype=np.uint16)
    v = np.ascontiguousarray(new_value, dtype=np.uint16)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T, Hkv, D = k.shape
    rc = _load().oracle_write(_ptr(k), _ptr(v), _ptr(kc), _ptr(vc), _ptr(sm), T, Hkv, D,
                              block_size, kc.shape[0])
    if rc < 0:
        raise ValueError(f"slot of token {-rc - 1} lies outside the pool")
    return kc, vc


def copy_blocks_c(key_cache, value_cache, block_mapping):
    """Copy whole physical blocks (src -> dst pairs) in copies of the pools."""
    kc = np.ascontiguousarray(key_cache, dtype=np.uint16).copy()
    vc = np.ascontiguousarray(value_cache, dtype=np.uint16).copy()
    bm = np.ascontiguousarray(block_mapping, dtype=np.int64).reshape(-1, 2)
    NB, Hkv, B, D = kc.shape
    rc = _load().oracle_copy_blocks(_ptr(kc), _ptr(vc), _ptr(bm), bm.shape[0], Hkv, D, B, NB)
    if rc < 0:
        raise ValueError(f"pair {-rc - 1} names a block outside the pool")
    return kc, vc


def decode_c(query, key_cache, value_cache, block_tables, context_lens, scale, dtype,
             pairs=None, num_threads: int = 0):
    """fp64 decode attention; returns out [S][H][D] (rows of unselected pairs are 0)."""
    q = np.ascontiguousarray(query, dtype=np.uint16)
    kc = np.ascontiguousarray(key_cache, dtype=np.uint16)
    vc = np.ascontiguousarray(value_cache, dtype=np.uint16)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    S, H, D = q.shape
    NB, Hkv, B, D2 = kc.shape
    assert D == D2 and vc.shape == kc.shape and bt.shape[0] == S and cl.shape == (S,)
    out = np.zeros((S, H, D), dtype=np.float64)
    if pairs is None:
        pp, npairs = None, 0
    else:
        pp = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
        npairs = pp.shape[0]
    rc = _load().oracle_decode(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1],
                               _ptr(cl), S, float(scale), B, H, Hkv, D, NB, DTYPE_CODE[dtype],
                               _ptr(pp) if pp is not None else None, npairs, int(num_threads))
    if rc:
        raise ValueError("block table entry outside the pool")
    return out


def widen_c(bits: int, dtype: str) -> float:
    return float(_load().oracle_widen(int(bits), DTYPE_CODE[dtype]))


# ----------------------------------------------------------------------------
# numpy implementation


def widen_np(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact fp64 value of fp16/bf16 bit patterns."""
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def write_np(key_cache, value_cache, new_key, new_value, slot_mapping, block_size):
    """The cache write as numpy indexing on copies of the pools."""
    kc = np.array(key_cache, dtype=np.uint16, copy=True)
    vc = np.array(value_cache, dtype=np.uint16, copy=True)
    NB = kc.shape[0]
    for t, slot in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if slot < 0:
            continue
        if slot >= NB * block_size:
            raise ValueError(f"slot of token {t} lies outside the pool")
        blk, off = divmod(int(slot), block_size)
        kc[blk, :, off, :] = new_key[t]
        vc[blk, :, off, :] = new_value[t]
    return kc, vc


def copy_blocks_np(key_cache, value_cache, block_mapping):
    """The copy-on-write block copy as numpy indexing on copies of the pools."""
    kc = np.array(key_cache, dtype=np.uint16, copy=True)
    vc = np.array(value_cache, dtype=np.uint16, copy=True)
    bm = np.asarray(block_mapping, dtype=np.int64).reshape(-1, 2)
    NB = kc.shape[0]
    if bm.size and ((bm < 0).any() or (bm >= NB).any()):
        raise ValueError("block outside the pool")
    kc[bm[:, 1]] = np.asarray(key_cache)[bm[:, 0]]
    vc[bm[:, 1]] = np.asarray(value_cache)[bm[:, 0]]
    return kc, vc


def gather_np(cache, table_row, ctx: int, kv_head: int, block_size: int) -> np.ndarray:
    """Rows 0..ctx-1 of one sequence's kv head, gathered through its block table ([ctx][D] bits)."""
    j = np.arange(ctx)
    phys = np.asarray(table_row, dtype=np.int64)[j // block_size]
    if ctx and ((phys < 0).any() or (phys >= cache.shape[0]).any()):
        raise ValueError("block table entry outside the pool")
    return cache[phys, kv_head, j % block_size, :]


def attention_np(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """softmax(scale * K q) . V for one query vector over contiguous fp64 K/V [n][D]."""
    if K.shape[0] == 0:
        return np.zeros(V.shape[1], dtype=np.float64)
    x = scale * (K @ q)
    w = np.exp(x - x.max())
    w /= w.sum()
    return w @ V


def decode_np(query, key_cache, value_cache, block_tables, context_lens, scale, dtype):
    """fp64 decode attention, gather then attend; returns out [S][H][D]."""
    query = np.asarray(query, dtype=np.uint16)
    S, H, D = query.shape
    Hkv, B = key_cache.shape[1], key_cache.shape[2]
    group = H // Hkv
    out = np.zeros((S, H, D), dtype=np.float64)
    for s in range(S):
        ctx = int(context_lens[s])
        for h in range(H):
            g = h // group
            K = widen_np(gather_np(key_cache, block_tables[s], ctx, g, B), dtype)
            V = widen_np(gather_np(value_cache, block_tables[s], ctx, g, B), dtype)
            out[s, h] = attention_np(widen_np(query[s, h], dtype), K, V, scale)
    return out
