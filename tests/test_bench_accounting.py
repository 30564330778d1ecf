"""The bench's byte and flop accounting, which the roofline fractions divide by, checked on tiny batches
against counts written out by hand."""
import numpy as np

import bench
from paged_kv_cache_91_gb300 import workloads as W
from paged_kv_cache_91_gb300.workloads import F16


def tiny(ctx, H=4, Hkv=2, D=64, B=16, query_lens=None, prefix=0):
    return W.build_batch(seed=3, context_lens=ctx, num_heads=H, num_kv_heads=Hkv, head_dim=D, block_size=B,
                         dtype=F16, pool_factor=1.5, query_lens=query_lens, shared_prefix_tokens=prefix)


def test_decode_step_bytes_by_hand():
    b = tiny([10, 40])  # one partition each (512 or 1024 tokens): no partials
    kv, call = bench.step_bytes(b, 512)
    assert kv == (10 + 40) * 2 * 64 * 2 * 2  # tokens x kv heads x D x (K, V) x 2 bytes
    q_out = 2 * 2 * 4 * 64 * 2  # q and out: S x H x D x 2 bytes
    tables = (1 + 3) * 4 + 2 * 4  # the blocks' entries and the context lengths
    assert call == kv + q_out + tables


def test_decode_step_bytes_with_partials():
    b = tiny([10, 40])
    kv, call = bench.step_bytes(b, 16)  # partitions of 16 tokens: 1 and 3 of them
    partials = 3 * 1 * 4 * (64 + 2) * 4 * 2  # only the split sequence: parts x rows x (D + 2) floats, written and read
    assert call == kv + 2 * 2 * 4 * 64 * 2 + (1 + 3) * 4 + 2 * 4 + partials


def test_fp8_cache_halves_the_kv_bytes():
    b = tiny([10, 40, 300])
    kv16, _ = bench.step_bytes(b, 512, cache_bytes=2)
    kv8, _ = bench.step_bytes(b, 512, cache_bytes=1)
    assert kv8 * 2 == kv16


def test_multi_query_step_bytes_count_every_query_row():
    b = tiny([10, 40], query_lens=[3, 5])
    kv, call = bench.step_bytes(b, 2048)
    q_out = 2 * (3 + 5) * 4 * 64 * 2
    assert call == kv + q_out + (1 + 3) * 4 + 2 * 4


def test_shared_prefix_bytes_read_the_prefix_once():
    b = tiny([64 + 5, 64 + 20, 64 + 33], prefix=64)
    unique = W.unique_kv_bytes(b)
    per_token = 2 * 64 * 2 * 2
    assert unique == (64 + 5 + 20 + 33) * per_token  # the 64 prefix tokens once
    ws = 1000
    got = bench.shared_prefix_call_bytes(b, 64, ws)
    tail_blocks = 1 + 2 + 3
    assert got == unique + 2 * 3 * 4 * 64 * 2 + (64 // 16 + tail_blocks) * 4 + 3 * 4 + 2 * ws
    assert bench.shared_prefix_call_bytes(b, 64, ws, cache_bytes=1) == got - unique // 2


def test_multi_query_flops_and_tile_labels():
    b = tiny([10, 40], H=8, Hkv=2, query_lens=[3, 5])  # G = 4: 20 rows per kv head
    m = bench.mq_summary(b, "auto", 1.0)
    visible = (3 * 7 + 3 * 4 // 2) + (5 * 35 + 5 * 6 // 2)  # per query token: its causal prefix
    assert m["attention_gflop_per_call"] == round(4.0 * 64 * 8 * visible / 1e9, 2)
    assert m["rows_per_kv_head"] == 20 and m["tile"] == "tensor"  # above 16 rows
    assert bench.mq_summary(b, "auto", 1.0, fp8=True)["tile"] == "pairs"  # FP8: 16-row pairs from 9 to 32 rows
    assert bench.mq_summary(b, "rows", 1.0, fp8=True)["tile"] == "columns"
    assert bench.mq_summary(b, "tensor", 1.0, fp8=True)["tile"] == "tensor"
    assert bench.mq_summary(b, "pairs", 1.0)["tile"] == "columns"  # no 16-bit form of the pairs
    few = tiny([10, 40], H=8, Hkv=4, query_lens=[3, 4])  # G = 2: 8 rows per kv head
    assert bench.mq_summary(few, "auto", 1.0, fp8=True)["tile"] == "columns"


def test_kernel_hashes_cover_existing_sources():
    for kind in bench.KERNEL_SOURCES:
        h = bench.kernel_hash(kind)
        assert len(h) == 16 and int(h, 16) >= 0
