"""Host block pool (reference counts, copy-on-write) and the block-copy oracle."""
import numpy as np
import pytest

import oracle
from paged_kv_cache_91_gb300.block_pool import BlockPool


def test_blocks_fill_left_to_right_and_waste_at_most_one_block():
    """New blocks are taken only when the last one is full ("Memory Allocation Pseudocode")."""
    pool = BlockPool(num_blocks=10, block_size=4)
    seq = pool.new_sequence()
    slots, copies = pool.append_tokens(seq, 6)
    assert copies == [] and len(seq.blocks) == 2 and pool.num_free == 8
    b0, b1 = seq.blocks
    assert slots == [b0 * 4 + 0, b0 * 4 + 1, b0 * 4 + 2, b0 * 4 + 3, b1 * 4 + 0, b1 * 4 + 1]
    slots, _ = pool.append_tokens(seq, 2)  # fills block b1 exactly
    assert len(seq.blocks) == 2 and slots == [b1 * 4 + 2, b1 * 4 + 3]
    slots, _ = pool.append_tokens(seq, 1)  # the ninth token opens a third block
    assert len(seq.blocks) == 3 and slots == [seq.blocks[2] * 4]


def test_block_counts_match_the_pages(golden):
    g = golden["block_counts"]
    for case in g["cases"]:
        pool = BlockPool(num_blocks=8, block_size=g["block_size"])
        seq = pool.new_sequence()
        pool.append_tokens(seq, case["tokens"])
        assert len(seq.blocks) == case["blocks"]
        assert len(seq.blocks) * g["block_size"] - case["tokens"] == case["empty_slots_in_last_block"]


def test_shared_prompt_copy_on_write(golden):
    """A prompt block shared by three requests (reference count 3): each write into it by a
    request that still shares it copies the block first; the last holder writes in place."""
    ref = golden["shared_prefix_tables"]["ref_count"]
    pool = BlockPool(num_blocks=16, block_size=16, seed=3)
    a = pool.new_sequence()
    pool.append_tokens(a, 8)  # the system prompt: 8 tokens in one block
    shared = a.blocks[0]
    b, c = pool.fork(a), pool.fork(a)
    assert pool.ref_count[shared] == ref == 3
    slots_a, copies_a = pool.append_tokens(a, 1)
    assert len(copies_a) == 1 and copies_a[0][0] == shared and a.blocks[0] == copies_a[0][1] != shared
    assert slots_a == [a.blocks[0] * 16 + 8] and pool.ref_count[shared] == 2
    _, copies_b = pool.append_tokens(b, 1)
    assert len(copies_b) == 1 and pool.ref_count[shared] == 1
    slots_c, copies_c = pool.append_tokens(c, 1)
    assert copies_c == [] and c.blocks == [shared] and slots_c == [shared * 16 + 8]
    assert len({a.blocks[0], b.blocks[0], c.blocks[0]}) == 3


def test_full_shared_block_is_not_copied():
    """Appending after a full shared block opens a new private block; the shared one stays shared."""
    pool = BlockPool(num_blocks=8, block_size=4)
    a = pool.new_sequence()
    pool.append_tokens(a, 4)
    b = pool.fork(a)
    _, copies = pool.append_tokens(b, 1)
    assert copies == [] and b.blocks[0] == a.blocks[0] and pool.ref_count[a.blocks[0]] == 2
    assert len(b.blocks) == 2


def test_out_of_blocks_returns_none_and_changes_nothing():
    pool = BlockPool(num_blocks=3, block_size=4)
    a = pool.new_sequence()
    pool.append_tokens(a, 10)  # 3 blocks
    before = (list(a.blocks), a.num_tokens, pool.ref_count.copy(), pool.num_free)
    assert pool.append_tokens(a, 3) is None
    assert (list(a.blocks), a.num_tokens, pool.num_free) == (before[0], before[1], before[3])
    np.testing.assert_array_equal(pool.ref_count, before[2])
    b = pool.fork(a)
    assert pool.append_tokens(b, 1) is None  # the copy-on-write copy needs a block too


def test_free_returns_blocks_when_no_sequence_uses_them():
    pool = BlockPool(num_blocks=6, block_size=4)
    a = pool.new_sequence()
    pool.append_tokens(a, 7)
    b = pool.fork(a)
    pool.free_sequence(a)
    assert pool.num_free == 4 and (pool.ref_count[b.blocks] == 1).all()
    pool.free_sequence(b)
    assert pool.num_free == 6 and (pool.ref_count == 0).all()
    with pytest.raises(ValueError):
        pool.release(0)


def test_blocks_needed_is_exact():
    rng = np.random.default_rng(5)
    for _ in range(200):
        pool = BlockPool(num_blocks=64, block_size=int(rng.choice([4, 8, 16])))
        a = pool.new_sequence()
        pool.append_tokens(a, int(rng.integers(0, 40)))
        b = pool.fork(a) if rng.random() < 0.5 else a
        k = int(rng.integers(0, 30))
        need = pool.blocks_needed(b, k)
        free = pool.num_free
        pool.append_tokens(b, k)
        assert free - pool.num_free == need


def test_copy_blocks_oracles_agree_and_copy_exactly():
    rng = np.random.default_rng(6)
    kc = rng.integers(0, 65536, size=(12, 3, 8, 64), dtype=np.uint16)
    vc = rng.integers(0, 65536, size=(12, 3, 8, 64), dtype=np.uint16)
    pairs = np.array([[2, 7], [9, 0], [5, 11]], dtype=np.int64)
    a = oracle.copy_blocks_c(kc, vc, pairs)
    b = oracle.copy_blocks_np(kc, vc, pairs)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    for s, d in pairs:
        np.testing.assert_array_equal(a[0][d], kc[s])
        np.testing.assert_array_equal(a[1][d], vc[s])
    untouched = [i for i in range(12) if i not in pairs[:, 1]]
    np.testing.assert_array_equal(a[0][untouched], kc[untouched])
    with pytest.raises(ValueError):
        oracle.copy_blocks_c(kc, vc, np.array([[1, 12]]))
    with pytest.raises(ValueError):
        oracle.copy_blocks_np(kc, vc, np.array([[-1, 3]]))
