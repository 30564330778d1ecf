"""Host-side bookkeeping of the paged KV pool: physical blocks, reference counts,
per-sequence block tables, and copy-on-write.

This is the allocation side the pages describe around the kernels:

* blocks are handed out only when a sequence's last block is full, and each
  sequence wastes at most one partly filled block ("Sparse Computation and
  Memory Management for Efficient LLM Inference", Memory Allocation
  Pseudocode; "KV Cache와 PagedAttention 완전 해부", §5단계 and §6단계);
* a sequence forked from another shares all its physical blocks, and each
  block's reference count records how many sequences use it (§9단계);
* before a token is appended into a shared last block, that block is copied to
  a fresh block for the appending sequence only, and the copy is recorded as a
  (src, dst) pair for paged_kv_copy_blocks (the same page, Copy-on-Write,
  append_kv_with_cow);
* running out of blocks is reported, not raised, so a scheduler can preempt
  ("[vLLM] PagedAttention: ...", allocate_slots returning None).

Only host integers live here; the pool's data is moved on the GPU by
paged_kv_copy_blocks (the copies) and paged_kv_write (the new tokens).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import numpy as np


@dataclass
class SequenceBlocks:
    """One sequence's block table and token count."""

    blocks: List[int] = field(default_factory=list)
    num_tokens: int = 0


class BlockPool:
    def __init__(self, num_blocks: int, block_size: int, seed: Optional[int] = None):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        self.num_blocks = num_blocks
        self.block_size = block_size
        order = np.arange(num_blocks) if seed is None else np.random.default_rng(seed).permutation(num_blocks)
        self._free: List[int] = [int(b) for b in order[::-1]]  # pop() hands out order[0] first
        self.ref_count = np.zeros(num_blocks, dtype=np.int64)

    @property
    def num_free(self) -> int:
        return len(self._free)

    def allocate(self) -> Optional[int]:
        """A free physical block with reference count 1, or None when the pool is exhausted."""
        if not self._free:
            return None
        b = self._free.pop()
        self.ref_count[b] = 1
        return b

    def release(self, block: int) -> None:
        if self.ref_count[block] <= 0:
            raise ValueError(f"block {block} is not in use")
        self.ref_count[block] -= 1
        if self.ref_count[block] == 0:
            self._free.append(block)

    # ---- sequence operations

    def new_sequence(self) -> SequenceBlocks:
        return SequenceBlocks()

    def fork(self, seq: SequenceBlocks) -> SequenceBlocks:
        """A sequence sharing every physical block of `seq` (parallel sampling, beam search)."""
        for b in seq.blocks:
            self.ref_count[b] += 1
        return SequenceBlocks(list(seq.blocks), seq.num_tokens)

    def free_sequence(self, seq: SequenceBlocks) -> None:
        for b in seq.blocks:
            self.release(b)
        seq.blocks.clear()
        seq.num_tokens = 0

    def blocks_needed(self, seq: SequenceBlocks, num_new_tokens: int) -> int:
        """Blocks `append_tokens` would take from the pool for num_new_tokens more tokens."""
        B = self.block_size
        used = seq.num_tokens % B
        need = -(-(seq.num_tokens + num_new_tokens) // B) - len(seq.blocks)
        if used and self.ref_count[seq.blocks[-1]] > 1 and num_new_tokens > 0:
            need += 1  # the shared last block is copied
        return max(0, need)

    def append_tokens(self, seq: SequenceBlocks, num_new_tokens: int
                      ) -> Optional[Tuple[List[int], List[Tuple[int, int]]]]:
        """Reserve slots for num_new_tokens tokens appended to `seq`.

        Returns (slots, copies): the physical slot (block * B + offset) of each
        new token, and the (src, dst) block copies that must run before those
        tokens are written. Returns None, changing nothing, if the pool lacks
        the blocks.
        """
        if self.blocks_needed(seq, num_new_tokens) > self.num_free:
            return None
        B = self.block_size
        slots: List[int] = []
        copies: List[Tuple[int, int]] = []
        for _ in range(num_new_tokens):
            off = seq.num_tokens % B
            if off == 0:  # the last block is full (or there is none): take a new one
                seq.blocks.append(self.allocate())
            else:
                last = seq.blocks[-1]
                if self.ref_count[last] > 1:  # shared: copy it before writing into it
                    dst = self.allocate()
                    copies.append((last, dst))
                    self.ref_count[last] -= 1
                    seq.blocks[-1] = dst
            slots.append(seq.blocks[-1] * B + off)
            seq.num_tokens += 1
        return slots, copies

    @staticmethod
    def tables(seqs: List[SequenceBlocks], width: Optional[int] = None) -> np.ndarray:
        """Block tables [S][width] (int32, -1 past each sequence's blocks)."""
        width = width or max(1, max((len(s.blocks) for s in seqs), default=1))
        t = np.full((len(seqs), width), -1, dtype=np.int32)
        for i, s in enumerate(seqs):
            t[i, :len(s.blocks)] = s.blocks
        return t
