"""The seeded input builder: determinism, pool invariants and the pages' byte accounting."""
import numpy as np
import pytest

from paged_kv_cache_91_gb300 import workloads as W
from paged_kv_cache_91_gb300.workloads import BF16, CANARY, F16


def test_kv_bytes_llama2_13b(golden):
    g = golden["kv_bytes_llama2_13b"]
    per_tok = W.kv_bytes_per_token(g["num_layers"], g["num_kv_heads"], g["head_dim"], g["elem_bytes"])
    assert per_tok == g["bytes_per_token"] == 819200
    assert abs(per_tok / 2**20 - g["approx_mb_per_token"]) < 0.01
    total = per_tok * g["max_model_len"]
    assert abs(total / 2**30 - g["approx_gb_at_max_model_len"]) < 0.1 or abs(total / 1e9 - 3.2) < 0.2


def test_kv_bytes_mixtral_32k(golden):
    g = golden["kv_bytes_mixtral_32k"]
    per_req = W.kv_bytes_per_token(g["num_layers"], g["num_kv_heads"], g["head_dim"], g["elem_bytes"]) * g["context_len"]
    assert per_req == 4 * 2**30
    assert abs(per_req / 2**30 - g["approx_gb_per_request"]) < 0.01


def test_block_counts_and_waste(golden):
    """ceil(n / B) blocks per sequence; only the last block has empty slots, at most B - 1."""
    g = golden["block_counts"]
    B = g["block_size"]
    ctxs = [c["tokens"] for c in g["cases"]]
    b = W.build_batch(seed=1, context_lens=ctxs, num_heads=2, num_kv_heads=2, head_dim=64,
                      block_size=B, dtype=F16)
    for s, case in enumerate(g["cases"]):
        used = int((b.block_tables[s] >= 0).sum())
        assert used == case["blocks"] == -(-case["tokens"] // B)
        last = b.block_tables[s, used - 1]
        empty = int((b.key_cache[last, 0, :, 0] == CANARY[F16]).sum())
        assert empty == case["empty_slots_in_last_block"] <= g["max_waste_slots"] == B - 1


def test_determinism_and_thread_independence():
    kw = dict(seed=77, context_lens=[300, 5, 1000], num_heads=8, num_kv_heads=2, head_dim=64,
              block_size=16, dtype=BF16, pool_factor=1.5)
    a = W.build_batch(threads=1, **kw)
    b = W.build_batch(threads=5, **kw)
    for f in ("query", "key_cache", "value_cache", "block_tables", "context_lens", "slot_mapping",
              "new_key", "new_value"):
        np.testing.assert_array_equal(getattr(a, f), getattr(b, f))
    c = W.build_batch(threads=2, **{**kw, "seed": 78})
    assert not np.array_equal(a.key_cache, c.key_cache)


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_pool_invariants(dtype):
    b = W.build_batch(seed=3, context_lens=[1, 16, 17, 250, 0], num_heads=4, num_kv_heads=2,
                      head_dim=128, block_size=16, dtype=dtype, pool_factor=1.2)
    B = b.block_size
    tables = b.block_tables
    live = tables[tables >= 0]
    assert len(np.unique(live)) == len(live)  # no block shared without a shared prefix
    assert live.max() < b.num_blocks
    used = np.zeros((b.num_blocks, B), dtype=bool)
    for s, c in enumerate(b.context_lens):
        nb = -(-int(c) // B)
        assert (tables[s, nb:] == -1).all()
        for j in range(int(c)):
            used[tables[s, j // B], j % B] = True
    kc = b.key_cache.transpose(0, 2, 1, 3)  # [NB][B][Hkv][D]
    assert (kc[~used] == CANARY[dtype]).all()
    vals = W.bits_to_f32(kc[used], dtype)
    assert np.isfinite(vals).all() and abs(vals.mean()) < 0.05 and abs(vals.std() - 1) < 0.05
    # the new token of each sequence sits at position ctx - 1
    for s, c in enumerate(b.context_lens):
        if c == 0:
            assert b.slot_mapping[s] == -1
            continue
        slot = int(b.slot_mapping[s])
        assert slot // B == tables[s, (c - 1) // B] and slot % B == (c - 1) % B
        np.testing.assert_array_equal(b.new_key[s], b.key_cache[slot // B, :, slot % B, :])
    kc0, vc0 = b.pool_before_write()
    slots = b.new_token_slots()
    assert (kc0[slots[:, 0], :, slots[:, 1], :] == CANARY[dtype]).all()


def test_round_to_nearest_even():
    x = np.array([1.0, 1.0 + 2**-11, 1.0 + 3 * 2**-11, -2.5, 65504.0, 1e-8], dtype=np.float32)
    f = W.round_f32_to(x, F16).view(np.float16).astype(np.float64)
    np.testing.assert_array_equal(f, x.astype(np.float16).astype(np.float64))
    y = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, 1.0 + 2**-8 + 2**-20, -3.0], dtype=np.float32)
    bf = W.bits_to_f32(W.round_f32_to(y, BF16), BF16)
    np.testing.assert_array_equal(bf, np.array([1.0, 1.0, 1.0 + 4 * 2**-8, 1.0 + 2**-7, -3.0], dtype=np.float32))


def test_config1_shape():
    b = W.make_config(1)
    assert list(b.context_lens) == [7, 33] and b.num_blocks == 16
    assert b.num_heads == b.num_kv_heads == 4 and b.head_dim == 64 and b.dtype == F16
    assert abs(b.scale - 1 / 8) < 1e-15
    assert (b.block_tables[0] >= 0).sum() == 1 and (b.block_tables[1] >= 0).sum() == 3
    perm = np.random.default_rng([1001, 0]).permutation(16)
    assert list(b.block_tables[0, :1]) == list(perm[:1]) and list(b.block_tables[1, :3]) == list(perm[1:4])


def test_config_context_distributions():
    c2 = W.config_context_lens(2)
    assert len(c2) == 64 and c2.min() >= 128 and c2.max() <= 2048
    c3 = W.config_context_lens(3)
    assert len(c3) == 256 and c3.min() >= 16 and c3.max() <= 8192 and 700 < c3.mean() < 1300
    c4 = W.config_context_lens(4)
    assert len(c4) == 128 and c4.min() >= 1024 + 64 and c4.max() <= 1024 + 512
    assert (W.config_context_lens(5) == 32768).all()


def test_shared_prefix_tables():
    b = W.build_batch(seed=4, context_lens=[1024 + 70, 1024 + 300, 1024 + 64], num_heads=8,
                      num_kv_heads=2, head_dim=64, block_size=16, dtype=F16,
                      shared_prefix_tokens=1024, pool_factor=1.2)
    t = b.block_tables
    assert (t[:, :64] == t[0, :64]).all()
    tails = np.concatenate([t[s, 64:][t[s, 64:] >= 0] for s in range(3)])
    assert len(np.unique(tails)) == len(tails) and not np.isin(tails, t[0, :64]).any()
    assert W.unique_kv_bytes(b) < W.algorithmic_kv_bytes(b)


def test_split_shared_prefix():
    """The prefix / tail split concatenates back to every sequence's table; a context equal to the
    prefix has an empty tail."""
    b = W.build_batch(seed=6, context_lens=[64 + 20, 64, 64 + 33], num_heads=4, num_kv_heads=2, head_dim=64,
                      block_size=16, dtype=F16, shared_prefix_tokens=64, pool_factor=1.2)
    prefix, tails, lens = W.split_shared_prefix(b, 64)
    assert prefix.dtype == tails.dtype == lens.dtype == np.int32
    assert list(lens) == [20, 0, 33]
    for s in range(3):
        nb = (b.context_lens[s] + 15) // 16
        full = np.concatenate([prefix, tails[s]])[:nb]
        assert (full == b.block_tables[s, :nb]).all()
    with pytest.raises(ValueError):
        W.split_shared_prefix(b, 80)  # not block aligned
    with pytest.raises(ValueError):
        W.split_shared_prefix(b, 128)  # longer than a context


def test_key_outliers():
    b = W.build_batch(seed=5, context_lens=[4096] * 4, num_heads=4, num_kv_heads=4, head_dim=64,
                      block_size=16, dtype=F16, key_outlier_frac=0.01, key_outlier_scale=8.0)
    k = W.bits_to_f32(b.key_cache, F16)
    norms = np.sqrt((k.astype(np.float64) ** 2).sum(-1))  # [NB][Hkv][B]
    frac = (norms > 3 * np.sqrt(64)).mean()
    assert 0.007 < frac < 0.013
    v = W.bits_to_f32(b.value_cache, F16)
    assert (np.sqrt((v.astype(np.float64) ** 2).sum(-1)) < 3 * np.sqrt(64)).all()


def test_algorithmic_bytes():
    b = W.build_batch(seed=6, context_lens=[10, 20], num_heads=4, num_kv_heads=2, head_dim=64,
                      block_size=16, dtype=F16)
    assert W.algorithmic_kv_bytes(b) == 30 * 2 * 64 * 2 * 2


@pytest.mark.parametrize("q", [None, 1, 3, 40])
def test_with_query_lens_equals_a_rebuilt_batch(q):
    """The bench derives multi-query batches from an already built pool; they must be the batches that
    building with query_len gives."""
    base = W.make_config(4, max_seqs=6)
    rebuilt = W.make_config(4, max_seqs=6, query_len=q)
    derived = W.with_query_lens(base, None if q is None else np.minimum(base.context_lens, q))
    for f in ("query", "key_cache", "value_cache", "block_tables", "context_lens", "slot_mapping", "new_key",
              "new_value"):
        assert np.array_equal(getattr(rebuilt, f), getattr(derived, f)), f
    if q is None:
        assert derived.query_start_loc is None
    else:
        assert np.array_equal(rebuilt.query_start_loc, derived.query_start_loc)


def test_sub_batch_keeps_each_sequence_and_compacts_the_pool():
    b = W.make_config(4, max_seqs=5, query_len=3)  # shared prefix: blocks used by several sequences
    sb = W.sub_batch(b, [4, 1])
    B = b.block_size
    assert sb.num_seqs == 2 and list(sb.context_lens) == [b.context_lens[4], b.context_lens[1]]
    used = sb.block_tables[sb.block_tables >= 0]
    assert sorted(set(used.tolist())) == list(range(sb.num_blocks))  # every compact block is used
    for i, s in enumerate([4, 1]):
        n = -(-int(b.context_lens[s]) // B)
        for j in range(n):  # same bits behind every logical block
            assert np.array_equal(sb.key_cache[sb.block_tables[i, j]], b.key_cache[b.block_tables[s, j]])
            assert np.array_equal(sb.value_cache[sb.block_tables[i, j]], b.value_cache[b.block_tables[s, j]])
        rows = np.arange(b.query_start_loc[s], b.query_start_loc[s + 1])
        got = np.arange(sb.query_start_loc[i], sb.query_start_loc[i + 1])
        assert np.array_equal(sb.query[got], b.query[rows])
        # the new tokens' slots point at the same (logical) positions
        for r_new, r_old in zip(got, rows):
            so, sn = int(b.slot_mapping[r_old]), int(sb.slot_mapping[r_new])
            assert np.array_equal(sb.key_cache[sn // B, :, sn % B], b.key_cache[so // B, :, so % B])
