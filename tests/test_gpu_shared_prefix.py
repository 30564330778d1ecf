"""GPU parity of the shared-prefix decode (prefix once for all sequences, then each tail, then a merge).

Its result is defined as decode attention over prefix_blocks ++ block_tables[s] with context
prefix_len + tail_lens[s], so the reference is the oracle's decode of the full batch. Every
output row must satisfy |gpu - ref| <= 1e-2 + 1e-2 |ref|. Unused pool slots hold NaN canaries.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_91_gb300 import binding
from paged_kv_cache_91_gb300 import workloads as W
from paged_kv_cache_91_gb300.workloads import BF16, F16

pytestmark = pytest.mark.gpu

ATOL = 1e-2
RTOL = 1e-2
DEV = "cuda:0"


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


def run_shared(batch, prefix, workspace=None):
    t = W.as_torch(batch, DEV)
    pb, tails, lens = W.split_shared_prefix(batch, prefix)
    pb_d = torch.from_numpy(pb).to(DEV) if len(pb) else torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.empty_like(t["query"])
    binding.paged_attention_decode_shared_prefix(out, t["query"], t["key_cache"], t["value_cache"], pb_d, prefix,
                                                 torch.from_numpy(tails).to(DEV), torch.from_numpy(lens).to(DEV),
                                                 batch.scale, max_tail_len=int(lens.max()), workspace=workspace)
    torch.cuda.synchronize()
    return out, t


def reference(batch):
    return oracle.decode_c(batch.query, batch.key_cache, batch.value_cache, batch.block_tables, batch.context_lens,
                           batch.scale, batch.dtype)


CASES = [
    # H, Hkv, D, B, dtype, num_seqs, prefix tokens, tail range
    (32, 8, 128, 16, F16, 16, 256, (1, 200)),      # 64 rows per kv head: prefix on the tensor-memory tile
    (8, 8, 128, 16, BF16, 8, 512, (0, 300)),       # MHA, 8 rows: prefix on the 8-column tile; empty tails
    (16, 8, 64, 8, F16, 40, 128, (1, 90)),         # GQA 2, head_dim 64, block 8: 80 rows, tensor tile
    (16, 4, 128, 32, BF16, 4, 1024, (2100, 2300)),  # block 32, split prefix, tails past one 2048-token partition
    (64, 8, 128, 16, BF16, 40, 2048, (1, 64)),     # GQA 8, 320 rows (3 row tiles), long prefix in partitions
    (12, 4, 64, 16, F16, 30, 0, (1, 700)),         # no prefix at all: the tails are the whole contexts
    (24, 8, 128, 16, BF16, 8, 512, (1, 300)),      # GQA 3, 24 rows (above 16): tensor tile, group not a power of 2
    (8, 1, 128, 16, F16, 2, 4096, (1, 100)),       # one kv head: 64 prefix partitions, more than 32 partials a row
]


@pytest.mark.parametrize("H,Hkv,D,B,dtype,S,prefix,tails", CASES)
def test_shared_prefix_matches_decode_oracle(cuda_lib, H, Hkv, D, B, dtype, S, prefix, tails):
    rng = np.random.default_rng(500 + H + D + B + S)
    ctx = prefix + rng.integers(tails[0], tails[1] + 1, size=S)
    batch = W.build_batch(seed=501 + S, context_lens=ctx, num_heads=H, num_kv_heads=Hkv, head_dim=D,
                          block_size=B, dtype=dtype, pool_factor=1.3, shared_prefix_tokens=prefix)
    binding.device_errors(clear=True)
    out, _ = run_shared(batch, prefix)
    check_close(as_bits(out), reference(batch), dtype, f"prefix {prefix}")
    assert binding.device_errors() == 0


def test_shared_prefix_equals_plain_decode(cuda_lib):
    """Both calls on the same batch agree with each other as well as with the oracle."""
    ctx = 1024 + np.arange(64, 64 + 24 * 17, 17)
    batch = W.build_batch(seed=510, context_lens=ctx, num_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                          dtype=F16, pool_factor=1.2, shared_prefix_tokens=1024)
    out, t = run_shared(batch, 1024)
    dec = torch.empty_like(out)
    binding.paged_attention_decode(dec, t["query"], t["key_cache"], t["value_cache"], t["block_tables"],
                                   t["context_lens"], batch.scale, max_context_len=batch.max_context_len)
    torch.cuda.synchronize()
    ref = reference(batch)
    check_close(as_bits(out), ref, F16, "shared prefix")
    check_close(as_bits(dec), ref, F16, "decode")
    a = oracle.widen_np(as_bits(out), F16)
    b = oracle.widen_np(as_bits(dec), F16)
    assert np.abs(a - b).max() < 2e-2


def test_bad_prefix_block_is_reported(cuda_lib):
    """An out-of-range prefix block id sets PKV_DEVERR_BLOCK_ID; its tokens are skipped, nothing faults."""
    batch = W.build_batch(seed=511, context_lens=[128 + 10, 128 + 40], num_heads=8, num_kv_heads=2, head_dim=64,
                          block_size=16, dtype=F16, pool_factor=1.5, shared_prefix_tokens=128)
    t = W.as_torch(batch, DEV)
    pb, tails, lens = W.split_shared_prefix(batch, 128)
    pb[3] = batch.num_blocks + 7
    out = torch.empty_like(t["query"])
    binding.device_errors(clear=True)
    binding.paged_attention_decode_shared_prefix(out, t["query"], t["key_cache"], t["value_cache"],
                                                 torch.from_numpy(pb).to(DEV), 128, torch.from_numpy(tails).to(DEV),
                                                 torch.from_numpy(lens).to(DEV), batch.scale)
    torch.cuda.synchronize()
    assert binding.device_errors() & 1
    assert torch.isfinite(out.float()).all()


def test_rejections(cuda_lib):
    batch = W.build_batch(seed=512, context_lens=[64 + 5], num_heads=4, num_kv_heads=2, head_dim=64,
                          block_size=16, dtype=F16, pool_factor=1.5, shared_prefix_tokens=64)
    t = W.as_torch(batch, DEV)
    pb, tails, lens = W.split_shared_prefix(batch, 64)
    args = (torch.empty_like(t["query"]), t["query"], t["key_cache"], t["value_cache"],
            torch.from_numpy(pb).to(DEV))
    with pytest.raises(binding.PagedKVError):  # prefix not a whole number of blocks
        binding.paged_attention_decode_shared_prefix(*args, 40, torch.from_numpy(tails).to(DEV),
                                                     torch.from_numpy(lens).to(DEV), batch.scale)
    with pytest.raises(binding.PagedKVError):  # workspace too small
        binding.paged_attention_decode_shared_prefix(*args, 64, torch.from_numpy(tails).to(DEV),
                                                     torch.from_numpy(lens).to(DEV), batch.scale,
                                                     workspace=torch.empty(16, dtype=torch.uint8, device=DEV))


def test_graph_capture_and_replay(cuda_lib):
    """The calls are stream-ordered (the shared-prefix call forks to a side stream and joins back), so a
    CUDA graph captured around a write + shared-prefix decode + plain decode replays them correctly."""
    batch = W.build_batch(seed=513, context_lens=256 + np.arange(40, 40 + 12 * 23, 23), num_heads=16,
                          num_kv_heads=4, head_dim=128, block_size=16, dtype=BF16, pool_factor=1.3,
                          shared_prefix_tokens=256)
    t = W.as_torch(batch, DEV)
    pb, tails, lens = W.split_shared_prefix(batch, 256)
    max_tail = int(lens.max())  # host values only inside the capture: no device-to-host read there
    pb, tails, lens = (torch.from_numpy(x).to(DEV) for x in (pb, tails, lens))
    H, Hkv, D, B = batch.num_heads, batch.num_kv_heads, batch.head_dim, batch.block_size
    ws_sp = torch.empty(binding.paged_attention_shared_prefix_workspace_size(batch.num_seqs, H, Hkv, D, B, 256,
                                                                             max_tail),
                        dtype=torch.uint8, device=DEV)
    ws_dec = torch.empty(max(16, binding.paged_attention_workspace_size(batch.num_seqs, H, Hkv, D, B,
                                                                        batch.max_context_len)),
                         dtype=torch.uint8, device=DEV)
    out_sp = torch.zeros_like(t["query"])
    out_dec = torch.zeros_like(t["query"])

    def step():
        binding.paged_kv_write(t["new_key"], t["new_value"], t["key_cache"], t["value_cache"], t["slot_mapping"])
        binding.paged_attention_decode_shared_prefix(out_sp, t["query"], t["key_cache"], t["value_cache"], pb, 256,
                                                     tails, lens, batch.scale, max_tail_len=max_tail, workspace=ws_sp)
        binding.paged_attention_decode(out_dec, t["query"], t["key_cache"], t["value_cache"], t["block_tables"],
                                       t["context_lens"], batch.scale, max_context_len=batch.max_context_len,
                                       workspace=ws_dec)

    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream(DEV))
    with torch.cuda.stream(side):
        step()  # warm up (library first-use setup) outside the capture
    torch.cuda.current_stream(DEV).wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    out_sp.zero_()
    out_dec.zero_()
    graph.replay()
    torch.cuda.synchronize()
    ref = reference(batch)
    check_close(as_bits(out_sp), ref, BF16, "shared prefix, graph replay")
    check_close(as_bits(out_dec), ref, BF16, "decode, graph replay")
    assert binding.device_errors() == 0


FP8_CASES = [
    # H, Hkv, dtype, B, num_seqs, prefix tokens, tail range, k_scale, v_scale
    (32, 8, F16, 16, 16, 256, (1, 200), 2 ** -6, 2 ** -6),        # 64 rows: the prefix on the tensor tile
    (8, 8, BF16, 16, 8, 512, (0, 300), 2 ** -5, 2 ** -7),         # MHA, 8 rows: prefix on the 8-column tile
    (16, 4, BF16, 32, 12, 1024, (1, 700), 0.013, 0.021),          # bf16 query scaled per row, block 32
    (64, 8, BF16, 16, 40, 2048, (1, 64), 2 ** -6, 2 ** -6),       # 320 rows, long prefix in partitions
]


@pytest.mark.parametrize("H,Hkv,dtype,B,S,prefix,tails,ks,vs", FP8_CASES)
def test_shared_prefix_fp8_matches_decode_oracle(cuda_lib, H, Hkv, dtype, B, S, prefix, tails, ks, vs):
    """paged_attention_decode_shared_prefix_fp8 against the oracle's decode of the full tables over the same
    E4M3 codes (the pools are the 16-bit pools encoded by the oracle)."""
    from test_gpu_fp8 import fp8_pools, to_dev_u8
    rng = np.random.default_rng(900 + H + B + S)
    ctx = prefix + rng.integers(tails[0], tails[1] + 1, size=S)
    batch = W.build_batch(seed=901 + S, context_lens=ctx, num_heads=H, num_kv_heads=Hkv, head_dim=128,
                          block_size=B, dtype=dtype, pool_factor=1.3, shared_prefix_tokens=prefix)
    kc8, vc8 = fp8_pools(batch, ks, vs)
    t = W.as_torch(batch, DEV)
    pb, tails_t, lens = W.split_shared_prefix(batch, prefix)
    out = torch.empty_like(t["query"])
    binding.device_errors(clear=True)
    binding.paged_attention_decode_shared_prefix_fp8(out, t["query"], to_dev_u8(kc8), to_dev_u8(vc8),
                                                     torch.from_numpy(pb).to(DEV), prefix,
                                                     torch.from_numpy(tails_t).to(DEV), torch.from_numpy(lens).to(DEV),
                                                     batch.scale, ks, vs, max_tail_len=int(lens.max()))
    torch.cuda.synchronize()
    ref = oracle.decode_c(batch.query, kc8, vc8, batch.block_tables, batch.context_lens, batch.scale, dtype,
                          k_scale=ks, v_scale=vs)
    check_close(as_bits(out), ref, dtype, f"fp8, prefix {prefix}")
    assert binding.device_errors() == 0


def test_shared_prefix_fp8_rejects_head_dim_64(cuda_lib):
    batch = W.build_batch(seed=910, context_lens=[64 + 5], num_heads=4, num_kv_heads=2, head_dim=64,
                          block_size=16, dtype=F16, pool_factor=1.5, shared_prefix_tokens=64)
    t = W.as_torch(batch, DEV)
    pb, tails, lens = W.split_shared_prefix(batch, 64)
    k8 = torch.zeros(t["key_cache"].shape, dtype=torch.uint8, device=DEV)
    with pytest.raises(binding.PagedKVError):
        binding.paged_attention_decode_shared_prefix_fp8(torch.empty_like(t["query"]), t["query"], k8, k8.clone(),
                                                         torch.from_numpy(pb).to(DEV), 64,
                                                         torch.from_numpy(tails).to(DEV),
                                                         torch.from_numpy(lens).to(DEV), batch.scale, 1.0, 1.0)
