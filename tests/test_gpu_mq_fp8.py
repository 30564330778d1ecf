"""GPU parity of multi-query paged attention over an FP8 (E4M3) pool.

The pools are the 16-bit pools encoded by the oracle's E4M3 encoder (value / scale in fp32, then rounded),
so the oracle and the library read the same codes; every output row must satisfy
|gpu - ref| <= 1e-2 + 1e-2 |ref| against the oracle's fp64 multi-query attention over the values
code * scale. Unused slots hold NaN codes, so a read past a context shows as a NaN.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_91_gb300 import binding
from paged_kv_cache_91_gb300 import workloads as W
from paged_kv_cache_91_gb300.workloads import BF16, F16
from test_gpu_fp8 import as_bits, check_close, fp8_pools, to_dev_u8

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def run_mq_fp8(batch, t, kc8, vc8, ks, vs, partition_size=0):
    out = torch.empty_like(t["query"])
    ql = np.diff(batch.query_start_loc)
    binding.paged_attention_multi_query_fp8(out, t["query"], kc8, vc8, t["block_tables"], t["context_lens"],
                                            t["query_start_loc"], batch.scale, ks, vs,
                                            max_query_len=int(ql.max()), max_context_len=batch.max_context_len,
                                            partition_size=partition_size)
    torch.cuda.synchronize()
    return out


def reference(batch, kc8, vc8, ks, vs):
    return oracle.multi_query_c(batch.query, kc8, vc8, batch.block_tables, batch.context_lens,
                                batch.query_start_loc, batch.scale, batch.dtype, k_scale=ks, v_scale=vs)


CASES = [
    # H, Hkv, dtype, block, contexts, query lens, k_scale, v_scale, partition
    (8, 8, F16, 16, [1, 17, 300, 1000, 2100], [1, 5, 8, 3, 7], 2 ** -6, 2 ** -6, 0),     # MHA, split past 2048
    (16, 4, BF16, 8, [40, 129, 700, 1500], [4, 4, 4, 4], 2 ** -5, 2 ** -7, 0),            # GQA 4: 16 rows
    (32, 4, BF16, 32, [64, 333, 1024, 2050], [6, 2, 6, 1], 0.013, 0.021, 256),           # GQA 8: 48 rows, split
    (4, 4, F16, 16, [9, 33, 64], [9, 33, 64], 2 ** -6, 2 ** -6, 0),                      # the whole prompt, causal
    (16, 2, F16, 16, [2048, 4000], [16, 3], 2 ** -6, 2 ** -6, 1024),                     # 128 rows, long contexts
    (12, 4, F16, 16, [50, 700, 2100], [3, 1, 3], 2 ** -6, 2 ** -6, 0),                    # GQA 3: 9 rows, pairs
    (16, 4, BF16, 32, [300, 1000, 2500], [6, 5, 2], 0.013, 0.021, 0),                     # 24 rows: a ragged pair
    (16, 4, F16, 16, [0, 5, 90, 600], [0, 4, 0, 4], 2 ** -6, 2 ** -6, 0),                 # empty context, q_len 0
]


@pytest.mark.parametrize("H,Hkv,dtype,B,ctx,ql,ks,vs,P", CASES)
def test_multi_query_fp8_matches_oracle(cuda_lib, H, Hkv, dtype, B, ctx, ql, ks, vs, P):
    batch = W.build_batch(seed=820 + H + B + len(ctx), context_lens=ctx, num_heads=H, num_kv_heads=Hkv,
                          head_dim=128, block_size=B, dtype=dtype, pool_factor=1.3, query_lens=ql)
    kc8, vc8 = fp8_pools(batch, ks, vs)
    t = W.as_torch(batch, DEV)
    binding.device_errors(clear=True)
    out = run_mq_fp8(batch, t, to_dev_u8(kc8), to_dev_u8(vc8), ks, vs, partition_size=P)
    err = check_close(as_bits(out), reference(batch, kc8, vc8, ks, vs), dtype, f"H {H} Hkv {Hkv} P {P}")
    assert binding.device_errors() == 0
    print(f"max abs err {err:.3e}")


def test_one_query_token_each_equals_fp8_decode(cuda_lib):
    """q_len 1 everywhere is the FP8 decode step: both calls match the decode oracle."""
    ctx = [1, 16, 17, 511, 1025, 3000]
    batch = W.build_batch(seed=830, context_lens=ctx, num_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                          dtype=BF16, pool_factor=1.3, query_lens=[1] * len(ctx))
    ks, vs = 2 ** -6, 2 ** -6
    kc8, vc8 = fp8_pools(batch, ks, vs)
    t = W.as_torch(batch, DEV)
    K, V = to_dev_u8(kc8), to_dev_u8(vc8)
    out_mq = run_mq_fp8(batch, t, K, V, ks, vs)
    out_dec = torch.empty_like(out_mq)
    binding.paged_attention_decode_fp8(out_dec, t["query"], K, V, t["block_tables"], t["context_lens"], batch.scale,
                                       ks, vs, max_context_len=batch.max_context_len)
    torch.cuda.synchronize()
    ref = oracle.decode_c(batch.query, kc8, vc8, batch.block_tables, batch.context_lens, batch.scale, BF16,
                          k_scale=ks, v_scale=vs)
    check_close(as_bits(out_mq), ref, BF16, "multi-query")
    check_close(as_bits(out_dec), ref, BF16, "decode")
    assert binding.device_errors() == 0


def test_bad_block_id_is_reported(cuda_lib):
    """An out-of-range block id sets PKV_DEVERR_BLOCK_ID; its tokens are skipped, nothing faults."""
    batch = W.build_batch(seed=831, context_lens=[100, 300], num_heads=8, num_kv_heads=2, head_dim=128,
                          block_size=16, dtype=F16, pool_factor=1.5, query_lens=[4, 4])
    ks, vs = 2 ** -6, 2 ** -6
    kc8, vc8 = fp8_pools(batch, ks, vs)
    t = W.as_torch(batch, DEV)
    t["block_tables"][1, 3] = batch.num_blocks + 5
    binding.device_errors(clear=True)
    out = run_mq_fp8(batch, t, to_dev_u8(kc8), to_dev_u8(vc8), ks, vs)
    assert binding.device_errors() & 1
    assert torch.isfinite(out.float()).all()


TILES = {"columns": binding.MQ_TILE_COLUMNS, "tensor": binding.MQ_TILE_TENSOR, "pairs": binding.MQ_TILE_PAIRS}


@pytest.mark.parametrize("tile", ["columns", "tensor", "pairs"])
@pytest.mark.parametrize("H,Hkv,dtype,B,ctx,ql,ks,vs,P", [CASES[0], CASES[2], CASES[3], CASES[4], CASES[6]])
def test_both_tiles_match_oracle(cuda_lib, tile, H, Hkv, dtype, B, ctx, ql, ks, vs, P):
    """The 8-column tile (E4M3 contraction), the 16-row pairs of 8-column groups (each widened K/V fragment
    shared by both groups) and the tensor-memory tile (codes widened to f16 in shared memory; a bf16 query
    scaled per row into f16) on the same FP8 inputs, each against the oracle."""
    batch = W.build_batch(seed=840 + H + B + len(ctx), context_lens=ctx, num_heads=H, num_kv_heads=Hkv,
                          head_dim=128, block_size=B, dtype=dtype, pool_factor=1.3, query_lens=ql)
    kc8, vc8 = fp8_pools(batch, ks, vs)
    t = W.as_torch(batch, DEV)
    prev = binding.set_multi_query_tile(TILES[tile])
    try:
        binding.device_errors(clear=True)
        out = run_mq_fp8(batch, t, to_dev_u8(kc8), to_dev_u8(vc8), ks, vs, partition_size=P)
    finally:
        binding.set_multi_query_tile(prev)
    check_close(as_bits(out), reference(batch, kc8, vc8, ks, vs), dtype, f"{tile}: H {H} Hkv {Hkv} P {P}")
    assert binding.device_errors() == 0
