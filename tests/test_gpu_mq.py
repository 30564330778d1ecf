"""GPU parity of multi-query paged attention (chunked-prefill chunks, speculative verification).

Every output row must satisfy |gpu - ref| <= 1e-2 + 1e-2 |ref| against the
oracle's fp64 multi-query attention on the same inputs. Unused pool slots hold
NaN canaries, so a read past a query token's causal limit inside the context
would not show (those tokens are finite), but one past the context would.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_91_gb300 import binding
from paged_kv_cache_91_gb300 import workloads as W
from paged_kv_cache_91_gb300.workloads import BF16, CANARY, F16

pytestmark = pytest.mark.gpu

ATOL = 1e-2
RTOL = 1e-2
DEV = "cuda:0"


TILES = {"columns": binding.MQ_TILE_COLUMNS, "rows": binding.MQ_TILE_ROWS, "tensor": binding.MQ_TILE_TENSOR}


@pytest.fixture(autouse=True, params=list(TILES))
def mq_tile(request, cuda_lib):
    """Every test runs on each multi-query tile (they must give the same results)."""
    prev = binding.set_multi_query_tile(TILES[request.param])
    binding.device_errors(clear=True)
    yield request.param
    binding.set_multi_query_tile(prev)


def as_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def check_close(gpu_bits, ref, dtype, what=""):
    got = oracle.widen_np(gpu_bits, dtype)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), (f"{what}: {bad.sum()} elements out of tolerance; max abs err "
                           f"{err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")
    return float(err.max())


def run_mq(batch, t, partition_size=0, max_query_len=None, out=None):
    out = torch.empty_like(t["query"]) if out is None else out
    ql = np.diff(batch.query_start_loc)
    mql = int(ql.max()) if max_query_len is None else max_query_len
    binding.paged_attention_multi_query(out, t["query"], t["key_cache"], t["value_cache"], t["block_tables"],
                                        t["context_lens"], t["query_start_loc"], batch.scale, max_query_len=mql,
                                        max_context_len=batch.max_context_len, partition_size=partition_size)
    return out


def reference(batch):
    return oracle.multi_query_c(batch.query, batch.key_cache, batch.value_cache, batch.block_tables,
                                batch.context_lens, batch.query_start_loc, batch.scale, batch.dtype)


def test_one_query_token_each_matches_decode():
    """q_len = 1 for every sequence is the decode step: both calls agree with the decode oracle."""
    ctx = [1, 17, 300, 513, 1000, 2048]
    batch = W.build_batch(seed=91, context_lens=ctx, num_heads=16, num_kv_heads=4, head_dim=128, block_size=16,
                          dtype=BF16, pool_factor=1.3, query_lens=[1] * len(ctx))
    t = W.as_torch(batch, DEV)
    out_mq = run_mq(batch, t)
    out_dec = torch.empty_like(out_mq)
    binding.paged_attention_decode(out_dec, t["query"], t["key_cache"], t["value_cache"], t["block_tables"],
                                   t["context_lens"], batch.scale, max_context_len=batch.max_context_len)
    torch.cuda.synchronize()
    ref = oracle.decode_c(batch.query, batch.key_cache, batch.value_cache, batch.block_tables,
                          batch.context_lens, batch.scale, BF16)
    check_close(as_bits(out_mq), ref, BF16, "multi-query")
    check_close(as_bits(out_dec), ref, BF16, "decode")
    assert binding.device_errors() == 0


CASES = [
    # H, Hkv, D, B, dtype, contexts, query lengths
    (8, 8, 128, 16, F16, [40, 300, 700, 16, 5], [4, 4, 64, 16, 5]),          # MHA: verify, chunk, whole prompts
    (32, 8, 128, 16, BF16, [200, 1100, 33, 600], [4, 100, 33, 1]),            # GQA 4
    (16, 8, 128, 8, F16, [513, 96, 1500], [7, 96, 20]),                        # GQA 2, block 8
    (64, 8, 128, 32, BF16, [64, 900, 257], [3, 9, 2]),                         # GQA 8, block 32
    (16, 1, 64, 16, F16, [300, 45, 1024], [5, 45, 17]),                        # GQA 16 (rows span tiles)
    (12, 4, 64, 8, BF16, [129, 700, 7, 2048], [0, 50, 7, 128]),                # GQA 3, D 64, an empty query
]


@pytest.mark.parametrize("H,Hkv,D,B,dtype,ctx,qlens", CASES)
@pytest.mark.parametrize("P", [0, 64])
def test_multi_query_matches_oracle(H, Hkv, D, B, dtype, ctx, qlens, P):
    if P and P % B:
        pytest.skip("partition size must be a multiple of the block size")
    batch = W.build_batch(seed=92 + H + D + B, context_lens=ctx, num_heads=H, num_kv_heads=Hkv, head_dim=D,
                          block_size=B, dtype=dtype, pool_factor=1.3, query_lens=qlens)
    ref = reference(batch)
    t = W.as_torch(batch, DEV)
    out = run_mq(batch, t, partition_size=P)
    torch.cuda.synchronize()
    check_close(as_bits(out), ref, dtype, f"P={P}")
    assert binding.device_errors() == 0


def test_write_then_multi_query_step():
    """The step: paged_kv_write stores each sequence's q_len new tokens (their slots start as canaries),
    then the multi-query call attends them causally. The write is bit-exact over the whole pool."""
    batch = W.build_batch(seed=93, context_lens=[100, 37, 520, 64], num_heads=32, num_kv_heads=8, head_dim=128,
                          block_size=16, dtype=F16, pool_factor=1.25, query_lens=[4, 37, 64, 1])
    t = W.as_torch(batch, DEV)
    expect_k, expect_v = t["key_cache"].clone(), t["value_cache"].clone()
    slots = torch.from_numpy(batch.new_token_slots()).to(DEV)
    c = int(np.array(CANARY[F16]).view(np.int16))
    for name in ("key_cache", "value_cache"):
        t[name].view(torch.int16)[slots[:, 0], :, slots[:, 1], :] = c
    binding.paged_kv_write(t["new_key"], t["new_value"], t["key_cache"], t["value_cache"], t["slot_mapping"])
    out = run_mq(batch, t)
    torch.cuda.synchronize()
    assert torch.equal(t["key_cache"].view(torch.int16), expect_k.view(torch.int16))
    assert torch.equal(t["value_cache"].view(torch.int16), expect_v.view(torch.int16))
    check_close(as_bits(out), reference(batch), F16)
    assert binding.device_errors() == 0


def test_long_chunk_many_row_tiles_and_split():
    """A 600-token chunk of a 3000-token context with GQA 4: 300 row tiles, six 512-token partitions."""
    batch = W.build_batch(seed=94, context_lens=[3000, 800], num_heads=8, num_kv_heads=2, head_dim=128,
                          block_size=16, dtype=BF16, pool_factor=1.2, query_lens=[600, 3])
    t = W.as_torch(batch, DEV)
    out = run_mq(batch, t)
    torch.cuda.synchronize()
    check_close(as_bits(out), reference(batch), BF16)


def test_bad_query_start_loc_is_reported_and_skipped():
    batch = W.build_batch(seed=95, context_lens=[50, 60, 70], num_heads=4, num_kv_heads=4, head_dim=64,
                          block_size=16, dtype=F16, pool_factor=1.5, query_lens=[3, 4, 5])
    ref = reference(batch)
    t = W.as_torch(batch, DEV)
    out = torch.zeros_like(t["query"])
    # sequence 1 claims 4 query tokens but max_query_len says at most 3 -> it is skipped
    run_mq(batch, t, max_query_len=3, out=out)
    torch.cuda.synchronize()
    assert binding.device_errors() & 16
    q = batch.query_start_loc
    got = as_bits(out)
    check_close(got[q[0]:q[1]], ref[q[0]:q[1]], F16, "seq 0")
    assert (got[q[1]:q[2]] == 0).all()  # not written
    # sequence 2 (5 tokens > 3) is skipped as well
    assert (got[q[2]:q[3]] == 0).all()


def test_query_count_above_context_is_reported():
    batch = W.build_batch(seed=96, context_lens=[20, 30], num_heads=4, num_kv_heads=2, head_dim=64,
                          block_size=16, dtype=F16, pool_factor=1.5, query_lens=[2, 2])
    t = W.as_torch(batch, DEV)
    t["query_start_loc"].copy_(torch.tensor([0, 2, 2], dtype=torch.int32))  # fine: seq 1 has no query
    run_mq(batch, t, max_query_len=2)
    torch.cuda.synchronize()
    assert binding.device_errors() == 0
    t["context_lens"][0] = 1  # seq 0 now has 2 query tokens but 1 context token
    run_mq(batch, t, max_query_len=2)
    torch.cuda.synchronize()
    assert binding.device_errors() & 16


def test_sequence_order_changes_nothing(mq_tile):
    """With room for it in the workspace, the 128-row tile runs the sequences longest context first; with a
    workspace of only the partials' size it runs them in index order. The outputs are bit-identical (the
    order moves whole items between CTAs, never the arithmetic of one) and match the oracle."""
    rng = np.random.default_rng(95)
    S = 24
    ctx = rng.integers(64, 3000, size=S)  # some past 2048 tokens: split into two partitions
    ql = np.minimum(rng.integers(20, 65, size=S), ctx)
    batch = W.build_batch(seed=96, context_lens=ctx, num_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                          dtype=F16, pool_factor=1.2, query_lens=ql)
    t = W.as_torch(batch, DEV)
    T, H, Hkv, D, B = int(batch.query_start_loc[-1]), batch.num_heads, batch.num_kv_heads, batch.head_dim, 16
    full = binding.paged_attention_multi_query_workspace_size(T, H, Hkv, D, B, batch.max_context_len)
    order_room = (T * 4 + 255) // 256 * 256
    partials = full - order_room
    assert partials > 0
    outs = []
    for nbytes in (full, partials):
        ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
        out = torch.empty_like(t["query"])
        binding.paged_attention_multi_query(out, t["query"], t["key_cache"], t["value_cache"], t["block_tables"],
                                            t["context_lens"], t["query_start_loc"], batch.scale,
                                            max_query_len=int(ql.max()), max_context_len=batch.max_context_len,
                                            workspace=ws)
        outs.append(as_bits(out))
    torch.cuda.synchronize()
    assert np.array_equal(outs[0], outs[1])
    check_close(outs[0], reference(batch), F16, f"{mq_tile}, sequence order")
    assert binding.device_errors() == 0


def test_many_short_sequences(mq_tile):
    """2500 sequences (the length sort loops over more sequences than it has threads), contexts of 1 to 40
    tokens, up to 4 query tokens each, GQA 8: up to 32 rows per kv head."""
    rng = np.random.default_rng(97)
    S = 2500
    ctx = rng.integers(1, 41, size=S)
    ql = np.minimum(rng.integers(1, 5, size=S), ctx)
    batch = W.build_batch(seed=98, context_lens=ctx, num_heads=16, num_kv_heads=2, head_dim=64, block_size=16,
                          dtype=BF16, pool_factor=1.1, query_lens=ql)
    t = W.as_torch(batch, DEV)
    out = run_mq(batch, t)
    torch.cuda.synchronize()
    check_close(as_bits(out), reference(batch), BF16, f"{mq_tile}, {S} sequences")
    assert binding.device_errors() == 0


def test_graph_capture_and_replay(mq_tile):
    """The call is stream-ordered (length sort, tile, reduce): a CUDA graph captured around it replays
    correctly, contexts long enough to be split into partitions."""
    rng = np.random.default_rng(99)
    ctx = rng.integers(100, 2600, size=12)
    ql = np.minimum(rng.integers(1, 24, size=12), ctx)
    batch = W.build_batch(seed=100, context_lens=ctx, num_heads=16, num_kv_heads=4, head_dim=128, block_size=16,
                          dtype=F16, pool_factor=1.2, query_lens=ql)
    t = W.as_torch(batch, DEV)
    T, H, Hkv, D = int(batch.query_start_loc[-1]), batch.num_heads, batch.num_kv_heads, batch.head_dim
    ws = torch.empty(binding.paged_attention_multi_query_workspace_size(T, H, Hkv, D, 16, batch.max_context_len),
                     dtype=torch.uint8, device=DEV)
    out = torch.zeros_like(t["query"])
    mql = int(ql.max())

    def call():
        binding.paged_attention_multi_query(out, t["query"], t["key_cache"], t["value_cache"], t["block_tables"],
                                            t["context_lens"], t["query_start_loc"], batch.scale, max_query_len=mql,
                                            max_context_len=batch.max_context_len, workspace=ws)

    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream(DEV))
    with torch.cuda.stream(side):
        call()  # warm up outside the capture
    torch.cuda.current_stream(DEV).wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    check_close(as_bits(out), reference(batch), F16, f"{mq_tile}, graph replay")
    assert binding.device_errors() == 0
