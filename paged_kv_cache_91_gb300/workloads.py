"""Seeded synthetic decode batches for the paged KV cache.

This module only builds inputs: context lengths, a physical block pool filled
with N(0,1) keys and values, per-sequence block tables popped from a shuffled
free list, the decode queries, and the one new token per sequence that the
cache write stores. It holds none of the attention arithmetic; both the CUDA
path and the CPU oracle consume what it returns.

Shapes follow the pages' vocabulary ("KV Cache와 PagedAttention 완전 해부",
§5단계; "Sparse Computation and Memory Management ...", Block-level Attention
Formulation):

  query        [S][H][D]            16-bit bit patterns (uint16); with several
                                    query tokens per sequence [T][H][D], packed
                                    by query_start_loc [S+1] int32
  key_cache    [NB][Hkv][B][D]      one contiguous B*D tile per (block, kv head)
  value_cache  [NB][Hkv][B][D]
  block_tables [S][max_blocks]      int32, logical block -> physical block, -1 past the end
  context_lens [S]                  int32, tokens attended by each sequence
  slot_mapping [T]                  int64, physical slot = block * B + offset, -1 = skip

Every slot of the pool that no sequence's context covers holds a NaN canary,
so any read past a context or into a free block shows up in the output.

Values are drawn in float32 from numpy's PCG64 and rounded to nearest-even to
fp16 or bf16. Large pools are drawn in fixed chunks of CHUNK_BLOCKS blocks,
each chunk seeded by (seed, stream, chunk index), so the result does not depend
on the number of threads used.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

F16 = "f16"
BF16 = "bf16"
DTYPES = (F16, BF16)

# NaN canaries (quiet NaN with a payload) written into every unused slot.
CANARY = {F16: np.uint16(0x7E5A), BF16: np.uint16(0x7FDA)}

CHUNK_BLOCKS = 64  # pool blocks per independently seeded chunk (fixed: part of the recipe)

# seed streams
_S_META, _S_QUERY, _S_KEY, _S_VALUE, _S_OUTLIER = 0, 1, 2, 3, 4


def round_f32_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to nearest-even fp16/bf16; return the uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == F16:
        return x.astype(np.float16).view(np.uint16)
    if dtype == BF16:
        u = x.view(np.uint32)
        r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
        return r.astype(np.uint16)
    raise ValueError(f"unknown dtype {dtype!r}")


def bits_to_f32(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of fp16/bf16 bit patterns to float32 (used only to build inputs)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == F16:
        return bits.view(np.float16).astype(np.float32)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class DecodeBatch:
    """One decode step's inputs for one attention layer."""

    name: str
    dtype: str
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    scale: float
    query: np.ndarray
    key_cache: np.ndarray
    value_cache: np.ndarray
    block_tables: np.ndarray
    context_lens: np.ndarray
    slot_mapping: np.ndarray
    new_key: np.ndarray
    new_value: np.ndarray
    partition_size: int = 512
    meta: dict = field(default_factory=dict)
    query_start_loc: np.ndarray | None = None  # [S+1] int32 when sequences have several query tokens

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def num_blocks(self) -> int:
        return int(self.key_cache.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def elem_bytes(self) -> int:
        return 2

    def new_token_slots(self) -> np.ndarray:
        """Physical (block, offset) pairs the step's new tokens are written to ([T, 2])."""
        s = self.slot_mapping
        keep = s >= 0
        return np.stack([s[keep] // self.block_size, s[keep] % self.block_size], axis=1)

    def pool_before_write(self):
        """Copies of the pools with the new tokens' slots reset to the canary."""
        kc = self.key_cache.copy()
        vc = self.value_cache.copy()
        slots = self.new_token_slots()
        kc[slots[:, 0], :, slots[:, 1], :] = CANARY[self.dtype]
        vc[slots[:, 0], :, slots[:, 1], :] = CANARY[self.dtype]
        return kc, vc


# ----------------------------------------------------------------------------
# pool construction


def _fill_pool(seed: int, stream: int, shape, dtype: str, outlier_frac: float,
               outlier_scale: float, threads: int) -> np.ndarray:
    nb = shape[0]
    out = np.empty(shape, dtype=np.uint16)
    nchunks = (nb + CHUNK_BLOCKS - 1) // CHUNK_BLOCKS

    def work(ci: int) -> None:
        b0 = ci * CHUNK_BLOCKS
        b1 = min(nb, b0 + CHUNK_BLOCKS)
        rng = np.random.default_rng([seed, stream, ci])
        x = rng.standard_normal((b1 - b0,) + tuple(shape[1:]), dtype=np.float32)
        if outlier_frac > 0.0:
            mrng = np.random.default_rng([seed, _S_OUTLIER, ci])
            mask = mrng.random((b1 - b0,) + tuple(shape[1:3])) < outlier_frac
            x[mask] *= np.float32(outlier_scale)
        out[b0:b1] = round_f32_to(x, dtype)

    if nchunks <= 1 or threads <= 1:
        for ci in range(nchunks):
            work(ci)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def split_shared_prefix(batch: "DecodeBatch", prefix_tokens: int):
    """The arguments of the shared-prefix decode for a batch built with
    ``shared_prefix_tokens=prefix_tokens``: (prefix_blocks [prefix_tokens / B]
    int32, tail_tables [S][max tail blocks] int32, tail_lens [S] int32). Sequence
    s's full table is prefix_blocks followed by tail_tables[s]."""
    B = batch.block_size
    if prefix_tokens % B or (batch.context_lens < prefix_tokens).any():
        raise ValueError("prefix must be block aligned and within every context")
    n = prefix_tokens // B
    if n and (batch.block_tables[:, :n] != batch.block_tables[0, :n]).any():
        raise ValueError("the sequences do not share their first blocks")
    prefix = np.ascontiguousarray(batch.block_tables[0, :n], dtype=np.int32)
    tails = np.ascontiguousarray(batch.block_tables[:, n:], dtype=np.int32)
    if tails.shape[1] == 0:
        tails = np.full((batch.num_seqs, 1), -1, dtype=np.int32)
    tail_lens = (batch.context_lens - prefix_tokens).astype(np.int32)
    return prefix, tails, tail_lens


def _draw_queries(seed: int, ctx: np.ndarray, query_lens, H: int, D: int, dtype: str):
    """The step's query rows: one per sequence with a context (decode), or q_s per sequence packed by
    query_start_loc. Returns (q_len per sequence, query_start_loc or None, query bits)."""
    S = int(ctx.shape[0])
    qrng = np.random.default_rng([seed, _S_QUERY])
    if query_lens is None:
        qlen = (ctx > 0).astype(np.int64)
        return qlen, None, round_f32_to(qrng.standard_normal((S, H, D), dtype=np.float32), dtype)
    qlen = np.asarray(query_lens, dtype=np.int64)
    if qlen.shape != ctx.shape or (qlen < 0).any() or (qlen > ctx).any():
        raise ValueError("query_lens must give 0 <= q_s <= ctx_s per sequence")
    qsl = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    return qlen, qsl, round_f32_to(qrng.standard_normal((int(qsl[-1]), H, D), dtype=np.float32), dtype)


def _new_tokens(ctx, qlen, qsl, tables, kc, vc, B: int):
    """One row per new token: sequence s's last qlen[s] context positions (decode: row s, or slot -1 when
    ctx = 0). Their K/V are copied from the pool. Returns (slot_mapping, new_key, new_value)."""
    S = int(ctx.shape[0])
    Hkv, D = kc.shape[1], kc.shape[3]
    rows = S if qsl is None else int(qsl[-1])
    slot_mapping = np.full(rows, -1, dtype=np.int64)
    new_key = np.zeros((rows, Hkv, D), dtype=np.uint16)
    new_value = np.zeros((rows, Hkv, D), dtype=np.uint16)
    for s in range(S):
        c, n = int(ctx[s]), int(qlen[s])
        r0 = s if qsl is None else int(qsl[s])
        for i in range(n):
            p = c - n + i
            phys = int(tables[s, p // B])
            off = p % B
            slot_mapping[r0 + i] = phys * B + off
            new_key[r0 + i] = kc[phys, :, off, :]
            new_value[r0 + i] = vc[phys, :, off, :]
    live = slot_mapping[slot_mapping >= 0]
    if len(np.unique(live)) != len(live):
        raise ValueError("two sequences write the same slot")
    return slot_mapping, new_key, new_value


def with_query_lens(batch: "DecodeBatch", query_lens) -> "DecodeBatch":
    """The same pool, tables and contexts with q_s query tokens per sequence (None: one decode token).
    Equal to building the batch again with ``query_lens``: the queries come from the same seeded stream."""
    ctx = batch.context_lens.astype(np.int64)
    seed = batch.meta["seed"]
    qlen, qsl, query = _draw_queries(seed, ctx, query_lens, batch.num_heads, batch.head_dim, batch.dtype)
    sm, nk, nv = _new_tokens(ctx, qlen, qsl, batch.block_tables, batch.key_cache, batch.value_cache,
                             batch.block_size)
    return DecodeBatch(
        name=batch.name, dtype=batch.dtype, num_heads=batch.num_heads, num_kv_heads=batch.num_kv_heads,
        head_dim=batch.head_dim, block_size=batch.block_size, scale=batch.scale, query=query,
        key_cache=batch.key_cache, value_cache=batch.value_cache, block_tables=batch.block_tables,
        context_lens=batch.context_lens, slot_mapping=sm, new_key=nk, new_value=nv,
        partition_size=batch.partition_size, meta=dict(batch.meta), query_start_loc=qsl)


def sub_batch(batch: "DecodeBatch", seqs) -> "DecodeBatch":
    """Sequences ``seqs`` of a batch over a compact pool that holds only their blocks (renumbered in order
    of first use), with their query rows and new tokens. Used to time the CPU oracle on a bounded sample."""
    seqs = [int(s) for s in seqs]
    B = batch.block_size
    ctx = batch.context_lens[seqs].astype(np.int64)
    nblk = (ctx + B - 1) // B
    old = []
    index = {}
    for s, n in zip(seqs, nblk):
        for j in range(int(n)):
            b = int(batch.block_tables[s, j])
            if b not in index:
                index[b] = len(old)
                old.append(b)
    old = np.asarray(old if old else [0], dtype=np.int64)
    tables = np.full((len(seqs), max(1, int(nblk.max()) if len(seqs) else 1)), -1, dtype=np.int32)
    for i, (s, n) in enumerate(zip(seqs, nblk)):
        tables[i, :n] = [index[int(b)] for b in batch.block_tables[s, :n]]
    qsl = batch.query_start_loc
    if qsl is None:
        rows = np.asarray(seqs, dtype=np.int64)
        new_qsl = None
    else:
        rows = np.concatenate([np.arange(qsl[s], qsl[s + 1]) for s in seqs]).astype(np.int64) if seqs else \
            np.zeros(0, np.int64)
        new_qsl = np.concatenate([[0], np.cumsum([qsl[s + 1] - qsl[s] for s in seqs])]).astype(np.int32)
    slots = batch.slot_mapping[rows]
    blk = np.where(slots >= 0, slots // B, 0)
    remap = np.array([index.get(int(b), -1) for b in blk], dtype=np.int64)
    new_slots = np.where((slots >= 0) & (remap >= 0), remap * B + np.where(slots >= 0, slots % B, 0), -1)
    return DecodeBatch(
        name=batch.name + "-sample", dtype=batch.dtype, num_heads=batch.num_heads, num_kv_heads=batch.num_kv_heads,
        head_dim=batch.head_dim, block_size=B, scale=batch.scale, query=batch.query[rows],
        key_cache=batch.key_cache[old], value_cache=batch.value_cache[old], block_tables=tables,
        context_lens=ctx.astype(np.int32), slot_mapping=new_slots.astype(np.int64),
        new_key=batch.new_key[rows], new_value=batch.new_value[rows], partition_size=batch.partition_size,
        meta=dict(batch.meta, sample_of=batch.name, sample_seqs=seqs), query_start_loc=new_qsl)


def build_batch(*, seed: int, context_lens, num_heads: int, num_kv_heads: int,
                head_dim: int, block_size: int, dtype: str, num_blocks: int | None = None,
                pool_factor: float = 1.0, shared_prefix_tokens: int = 0,
                key_outlier_frac: float = 0.0, key_outlier_scale: float = 8.0,
                partition_size: int = 512, name: str = "custom",
                threads: int | None = None, query_lens=None) -> DecodeBatch:
    """Build a seeded decode batch.

    Physical blocks come from a free list that is a seeded permutation of the
    pool; each sequence pops its blocks in logical order, the way blocks are
    handed out on demand ("Sparse Computation and Memory Management ...",
    Memory Allocation Pseudocode). With ``shared_prefix_tokens`` > 0 every
    sequence's first blocks point at the same physical blocks ("KV Cache와
    PagedAttention 완전 해부", §9단계 Prefix Caching).

    The step's new token of sequence s is its last context position ctx_s - 1;
    its K/V are already in the pool, and ``new_key``/``new_value`` hold a copy
    so a test can clear the slot and have the cache write restore it.

    With ``query_lens`` (q_s <= ctx_s tokens per sequence) the step's new
    tokens are each sequence's last q_s context positions, in order: a
    chunked-prefill chunk or the tokens a speculative step verifies. Then
    ``query`` is [sum q_s][H][D], packed by ``query_start_loc``, and
    ``slot_mapping`` / ``new_key`` / ``new_value`` have one row per new token.
    """
    if dtype not in DTYPES:
        raise ValueError(dtype)
    if num_heads % num_kv_heads:
        raise ValueError("num_heads must be a multiple of num_kv_heads")
    B = block_size
    ctx = np.asarray(context_lens, dtype=np.int64)
    S = int(ctx.shape[0])
    if (ctx < 0).any():
        raise ValueError("negative context length")
    if shared_prefix_tokens % B:
        raise ValueError("shared prefix must be block aligned")
    prefix_blocks = shared_prefix_tokens // B
    if shared_prefix_tokens and (ctx < shared_prefix_tokens).any():
        raise ValueError("every sequence must hold the whole shared prefix")
    nblk = (ctx + B - 1) // B
    private = nblk - prefix_blocks if prefix_blocks else nblk
    needed = int(prefix_blocks + private.sum())
    if num_blocks is None:
        num_blocks = max(1, int(math.ceil(pool_factor * needed)))
    if num_blocks < needed:
        raise ValueError(f"pool of {num_blocks} blocks < {needed} needed")
    meta_rng = np.random.default_rng([seed, _S_META])
    free_list = meta_rng.permutation(num_blocks).astype(np.int64)
    max_blocks = max(1, int(nblk.max()) if S else 1)
    tables = np.full((S, max_blocks), -1, dtype=np.int32)
    pos = 0
    prefix = free_list[pos:pos + prefix_blocks]
    pos += prefix_blocks
    for s in range(S):
        tables[s, :prefix_blocks] = prefix
        n = int(private[s])
        tables[s, prefix_blocks:prefix_blocks + n] = free_list[pos:pos + n]
        pos += n

    H, Hkv, D = num_heads, num_kv_heads, head_dim
    qlen, qsl, query = _draw_queries(seed, ctx, query_lens, H, D, dtype)

    threads = threads or max(1, min(32, os.cpu_count() or 1))
    shape = (num_blocks, Hkv, B, D)
    kc = _fill_pool(seed, _S_KEY, shape, dtype, key_outlier_frac, key_outlier_scale, threads)
    vc = _fill_pool(seed, _S_VALUE, shape, dtype, 0.0, 1.0, threads)

    # canary every slot no context covers
    used = np.zeros((num_blocks, B), dtype=bool)
    for s in range(S):
        c = int(ctx[s])
        for j in range(int(nblk[s])):
            used[tables[s, j], :min(B, c - j * B)] = True
    bi, oi = np.nonzero(~used)
    kc[bi, :, oi, :] = CANARY[dtype]
    vc[bi, :, oi, :] = CANARY[dtype]

    slot_mapping, new_key, new_value = _new_tokens(ctx, qlen, qsl, tables, kc, vc, B)

    return DecodeBatch(
        name=name, dtype=dtype, num_heads=H, num_kv_heads=Hkv, head_dim=D, block_size=B,
        scale=1.0 / math.sqrt(D), query=query, key_cache=kc, value_cache=vc,
        block_tables=tables, context_lens=ctx.astype(np.int32), slot_mapping=slot_mapping,
        new_key=new_key, new_value=new_value, partition_size=partition_size,
        meta=dict(seed=seed, pool_factor=pool_factor, shared_prefix_tokens=shared_prefix_tokens,
                  key_outlier_frac=key_outlier_frac, needed_blocks=needed),
        query_start_loc=qsl)


# ----------------------------------------------------------------------------
# the five workloads


CONFIG_NAMES = {
    1: "tiny paged decode (2 seqs, ctx 7/33, MHA 4x64, fp16)",
    2: "LLaMA-2-13B-shaped decode (batch 64, MHA 40x128, fp16, ctx U[128,2048])",
    3: "Qwen3-4B-shaped GQA decode (batch 256, 32q/8kv x128, bf16, geometric ctx)",
    4: "shared-prefix decode (128 seqs, 1024-token shared prefix + U[64,512] tails, 32q/8kv, fp16)",
    5: "long-context split-K decode (batch 16, ctx 32768, MHA 40x128, fp16, 1% keys x8)",
}


def config_context_lens(n: int) -> np.ndarray:
    """Context lengths of workload n (drawn from the workload's own seed)."""
    rng = np.random.default_rng(1000 + n)
    if n == 1:
        return np.array([7, 33], dtype=np.int64)
    if n == 2:
        return rng.integers(128, 2048, size=64, endpoint=True)
    if n == 3:
        return np.clip(15 + rng.geometric(1.0 / 985.0, size=256), 16, 8192)
    if n == 4:
        return 1024 + rng.integers(64, 512, size=128, endpoint=True)
    if n == 5:
        return np.full(16, 32768, dtype=np.int64)
    raise ValueError(n)


def make_config(n: int, threads: int | None = None, max_seqs: int | None = None,
                block_size: int = 16, query_len: int | None = None) -> DecodeBatch:
    """Workload n (1..5) at full size, or its first ``max_seqs`` sequences.

    ``block_size`` other than 16 gives the same contexts paged in blocks of 8 or
    32 tokens (the pages' block-size ablation; 16 is the default they report best).
    ``query_len`` makes each sequence's last min(query_len, ctx) tokens the step's
    query tokens (the multi-query form) instead of one decode token.
    """
    ctx = config_context_lens(n)
    if max_seqs is not None:
        ctx = ctx[:max_seqs]
    seed = 1000 + n
    common = dict(seed=seed, context_lens=ctx, block_size=block_size, name=f"cfg{n}", threads=threads,
                  query_lens=None if query_len is None else np.minimum(ctx, query_len))
    if n == 1:
        return build_batch(num_heads=4, num_kv_heads=4, head_dim=64, dtype=F16, num_blocks=16, **common)
    if n == 2:
        return build_batch(num_heads=40, num_kv_heads=40, head_dim=128, dtype=F16, pool_factor=1.2, **common)
    if n == 3:
        return build_batch(num_heads=32, num_kv_heads=8, head_dim=128, dtype=BF16, pool_factor=1.2, **common)
    if n == 4:
        return build_batch(num_heads=32, num_kv_heads=8, head_dim=128, dtype=F16, pool_factor=1.2,
                           shared_prefix_tokens=1024, **common)
    if n == 5:
        return build_batch(num_heads=40, num_kv_heads=40, head_dim=128, dtype=F16, pool_factor=1.0,
                           key_outlier_frac=0.01, key_outlier_scale=8.0, **common)
    raise ValueError(n)


# ----------------------------------------------------------------------------
# byte accounting (what a decode step must read, by definition)


def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    """K and V bytes one token occupies across all layers: 2 * L * Hkv * D * bytes.

    "KV Cache와 PagedAttention 완전 해부", §3단계 (KV Cache는 GPU 메모리에 얼마나 차지하나).
    """
    return 2 * num_layers * num_kv_heads * head_dim * elem_bytes


def algorithmic_kv_bytes(batch: DecodeBatch) -> int:
    """K+V bytes one decode step reads: every context token of every kv head, once."""
    return int(batch.context_lens.astype(np.int64).sum()) * batch.num_kv_heads * batch.head_dim * 2 * batch.elem_bytes


def unique_kv_bytes(batch: DecodeBatch) -> int:
    """K+V bytes of the distinct physical slots read (shared prefix blocks counted once)."""
    B = batch.block_size
    seen = set()
    n = 0
    for s in range(batch.num_seqs):
        c = int(batch.context_lens[s])
        for j in range((c + B - 1) // B):
            phys = int(batch.block_tables[s, j])
            valid = min(B, c - j * B)
            if phys in seen:
                continue
            seen.add(phys)
            n += valid
    return n * batch.num_kv_heads * batch.head_dim * 2 * batch.elem_bytes


def as_torch(batch: DecodeBatch, device):
    """The batch's arrays as torch tensors on ``device`` (bit patterns kept)."""
    import torch

    tdt = torch.float16 if batch.dtype == F16 else torch.bfloat16

    def half(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(tdt).to(device)

    return dict(
        query=half(batch.query), key_cache=half(batch.key_cache), value_cache=half(batch.value_cache),
        new_key=half(batch.new_key), new_value=half(batch.new_value),
        block_tables=torch.from_numpy(batch.block_tables).to(device),
        context_lens=torch.from_numpy(batch.context_lens).to(device),
        slot_mapping=torch.from_numpy(batch.slot_mapping).to(device),
        **({} if batch.query_start_loc is None
           else {"query_start_loc": torch.from_numpy(batch.query_start_loc).to(device)}),
    )
