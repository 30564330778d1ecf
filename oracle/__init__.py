"""CPU oracle for the paged KV cache hot path (fp64).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may use this package; the CUDA library and its
Python binding never import it. It shares no code with the CUDA path.

Two independent implementations of the same definitions:

* ``write_c`` / ``decode_c`` / ``copy_blocks_c`` / ``write_fp8_c`` -- plain C
  (``pkv_oracle.c``), fp64, OpenMP over (sequence, head) pairs; fast enough for
  the full-size workloads. E4M3 (FP8) codes: ``e4m3_encode_c`` / ``e4m3_decode_c``.
* ``write_np`` / ``decode_np`` -- numpy, fp64, gather-then-attend; plus
  ``attention_np``, unpaged attention over contiguous K/V arrays.
* ``multi_query_c`` / ``multi_query_np`` -- several query tokens per sequence
  (packed by ``query_start_loc``): query token i of a sequence with q_len
  query tokens sits at position ctx - q_len + i and attends positions up to
  its own (a_ij over j <= i: "vLLM: LLM 서빙 메모리 최적화의 교과서", 01 Problem
  Definition; chunked prefill and speculative verification: "Sparse
  Computation and Memory Management for Efficient LLM Inference").

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
                                      i32, f64, f64, P, i64, i32]
        lib.oracle_write_fp8.restype = i64
        lib.oracle_write_fp8.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i64, i32, ctypes.c_float,
                                         ctypes.c_float]
        lib.oracle_e4m3_encode_array.restype = None
        lib.oracle_e4m3_encode_array.argtypes = [P, P, i64]
        lib.oracle_e4m3_decode_array.restype = None
        lib.oracle_e4m3_decode_array.argtypes = [P, P, i64]
        lib.oracle_copy_blocks.restype = i64
        lib.oracle_copy_blocks.argtypes = [P, P, P, i32, i32, i32, i32, i64]
        lib.oracle_widen.restype = f64
        lib.oracle_widen.argtypes = [ctypes.c_uint16, i32]
        lib.oracle_max_threads.restype = i32
        lib.oracle_multi_query.restype = i32
        lib.oracle_multi_query.argtypes = [P, P, P, P, P, i32, P, P, i32, f64, i32, i32, i32, i32, i64, i32,
                                           i32, f64, f64, i32]
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


def e4m3_encode_c(x) -> np.ndarray:
    """E4M3 codes of float32 values (nearest, ties to even, saturating to +-448)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().oracle_e4m3_encode_array(_ptr(x), _ptr(out), x.size)
    return out


def e4m3_decode_c(codes) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _load().oracle_e4m3_decode_array(_ptr(c), _ptr(out), c.size)
    return out


def write_fp8_c(key_cache, value_cache, new_key, new_value, slot_mapping, block_size, src_dtype,
                k_scale: float, v_scale: float):
    """The quantizing write into copies of E4M3 pools (uint8 codes)."""
    kc = np.ascontiguousarray(key_cache, dtype=np.uint8).copy()
    vc = np.ascontiguousarray(value_cache, dtype=np.uint8).copy()
    k = np.ascontiguousarray(new_key, dtype=np.uint16)
    v = np.ascontiguousarray(new_value, dtype=np.uint16)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T, Hkv, D = k.shape
    rc = _load().oracle_write_fp8(_ptr(k), _ptr(v), _ptr(kc), _ptr(vc), _ptr(sm), T, Hkv, D, block_size,
                                  kc.shape[0], DTYPE_CODE[src_dtype], float(k_scale), float(v_scale))
    if rc < 0:
        raise ValueError(f"slot of token {-rc - 1} lies outside the pool")
    return kc, vc


def decode_c(query, key_cache, value_cache, block_tables, context_lens, scale, dtype,
             pairs=None, num_threads: int = 0, k_scale: float = 1.0, v_scale: float = 1.0):
    """fp64 decode attention; returns out [S][H][D] (rows of unselected pairs are 0).

    A uint8 pool is an E4M3 cache whose elements are code * k_scale (keys) and
    code * v_scale (values); 16-bit pools hold dtype bit patterns.
    """
    q = np.ascontiguousarray(query, dtype=np.uint16)
    fp8 = np.asarray(key_cache).dtype == np.uint8
    cdt = np.uint8 if fp8 else np.uint16
    kc = np.ascontiguousarray(key_cache, dtype=cdt)
    vc = np.ascontiguousarray(value_cache, dtype=cdt)
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
                               2 if fp8 else DTYPE_CODE[dtype], float(k_scale), float(v_scale),
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


def e4m3_decode_np(codes) -> np.ndarray:
    """Exact values of E4M3 codes: 1 sign, 4 exponent (bias 7), 3 mantissa bits; S.1111.111 is NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 15
    m = c & 7
    v = np.where(e == 0, np.ldexp(m.astype(np.float64), -9), np.ldexp((8 + m).astype(np.float64), e - 10))
    v = np.where((e == 15) & (m == 7), np.nan, v)
    return s * v


_E4M3_POS = None


def e4m3_encode_np(x) -> np.ndarray:
    """Nearest E4M3 code of float32 values, ties to the even mantissa, saturating to +-448."""
    global _E4M3_POS
    if _E4M3_POS is None:
        _E4M3_POS = e4m3_decode_np(np.arange(0x7F, dtype=np.uint8))  # codes 0..126, increasing values
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    a = np.minimum(np.abs(x), 448.0)
    hi = np.clip(np.searchsorted(_E4M3_POS, a, side="left"), 0, 0x7E)
    lo = np.maximum(hi - 1, 0)
    dlo, dhi = a - _E4M3_POS[lo], _E4M3_POS[hi] - a
    pick = np.where(dhi < dlo, hi, np.where(dlo < dhi, lo, np.where(hi % 2 == 0, hi, lo)))
    code = pick.astype(np.uint8) | np.where(np.signbit(x), 0x80, 0).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)


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
    kc = np.array(key_cache, copy=True)  # 16-bit patterns or 8-bit codes, kept as they are
    vc = np.array(value_cache, copy=True)
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


def decode_np(query, key_cache, value_cache, block_tables, context_lens, scale, dtype,
              k_scale: float = 1.0, v_scale: float = 1.0):
    """fp64 decode attention, gather then attend; returns out [S][H][D] (uint8 pools: E4M3 codes)."""
    query = np.asarray(query, dtype=np.uint16)
    S, H, D = query.shape
    Hkv, B = key_cache.shape[1], key_cache.shape[2]
    group = H // Hkv
    out = np.zeros((S, H, D), dtype=np.float64)
    for s in range(S):
        ctx = int(context_lens[s])
        for h in range(H):
            g = h // group
            Kc = gather_np(key_cache, block_tables[s], ctx, g, B)
            Vc = gather_np(value_cache, block_tables[s], ctx, g, B)
            if np.asarray(key_cache).dtype == np.uint8:
                K, V = e4m3_decode_np(Kc) * k_scale, e4m3_decode_np(Vc) * v_scale
            else:
                K, V = widen_np(Kc, dtype), widen_np(Vc, dtype)
            out[s, h] = attention_np(widen_np(query[s, h], dtype), K, V, scale)
    return out


def multi_query_c(query, key_cache, value_cache, block_tables, context_lens, query_start_loc, scale, dtype,
                  num_threads: int = 0, k_scale: float = 1.0, v_scale: float = 1.0):
    """fp64 multi-query attention; query [T][H][D] bits packed by query_start_loc [S+1]; returns out [T][H][D]."""
    q = np.ascontiguousarray(query, dtype=np.uint16)
    fp8 = np.asarray(key_cache).dtype == np.uint8
    cdt = np.uint8 if fp8 else np.uint16
    kc = np.ascontiguousarray(key_cache, dtype=cdt)
    vc = np.ascontiguousarray(value_cache, dtype=cdt)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
    T, H, D = q.shape
    NB, Hkv, B, D2 = kc.shape
    S = cl.shape[0]
    assert D == D2 and vc.shape == kc.shape and bt.shape[0] == S and qsl.shape == (S + 1,)
    assert qsl[0] == 0 and qsl[-1] == T and (np.diff(qsl) >= 0).all()
    out = np.zeros((T, H, D), dtype=np.float64)
    rc = _load().oracle_multi_query(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], _ptr(cl),
                                    _ptr(qsl), S, float(scale), B, H, Hkv, D, NB, DTYPE_CODE[dtype],
                                    2 if fp8 else DTYPE_CODE[dtype], float(k_scale), float(v_scale),
                                    int(num_threads))
    if rc == -1:
        raise ValueError("block table entry outside the pool")
    if rc == -2:
        raise ValueError("a sequence has more query tokens than context tokens")
    return out


def multi_query_np(query, key_cache, value_cache, block_tables, context_lens, query_start_loc, scale, dtype):
    """fp64 multi-query attention, gather then attend per query token over its causal prefix."""
    query = np.asarray(query, dtype=np.uint16)
    T, H, D = query.shape
    Hkv, B = key_cache.shape[1], key_cache.shape[2]
    group = H // Hkv
    out = np.zeros((T, H, D), dtype=np.float64)
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    for s in range(len(context_lens)):
        ctx = int(context_lens[s])
        q0, q_len = int(qsl[s]), int(qsl[s + 1] - qsl[s])
        if q_len > ctx:
            raise ValueError("a sequence has more query tokens than context tokens")
        for h in range(H):
            g = h // group
            K = widen_np(gather_np(key_cache, block_tables[s], ctx, g, B), dtype)
            V = widen_np(gather_np(value_cache, block_tables[s], ctx, g, B), dtype)
            for i in range(q_len):
                n = ctx - q_len + i + 1
                out[q0 + i, h] = attention_np(widen_np(query[q0 + i, h], dtype), K[:n], V[:n], scale)
    return out
