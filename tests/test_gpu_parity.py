"""GPU parity: the CUDA library against the CPU oracle on the same seeded inputs.

Cache writes must match bit for bit (the whole pool, canaries included).
Attention output must satisfy |gpu - ref| <= 1e-2 + 1e-2 |ref| elementwise,
with ref the oracle's fp64 result. Every unused pool slot holds a NaN canary,
so a read outside a context shows up as a NaN in the output.
"""
import math

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


@pytest.fixture(autouse=True)
def clear_device_errors(cuda_lib):
    binding.device_errors(clear=True)
    yield


def as_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    return oracle.widen_np(bits, dtype)


def check_close(gpu_bits, ref, dtype, what=""):
    got = to_f64(gpu_bits, dtype)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), (f"{what}: {bad.sum()} elements out of tolerance; max abs err "
                           f"{err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")
    return float(err.max())


def canary_slots(t, batch):
    """Reset the new tokens' slots on the device to the canary, as before the step's write."""
    slots = torch.from_numpy(batch.new_token_slots()).to(DEV)
    c = int(np.array(CANARY[batch.dtype]).view(np.int16))
    for name in ("key_cache", "value_cache"):
        t[name].view(torch.int16)[slots[:, 0], :, slots[:, 1], :] = c


def run_step(batch, t, partition_size=0, write=True, max_context_len=None, stream=None):
    if write:
        binding.paged_kv_write(t["new_key"], t["new_value"], t["key_cache"], t["value_cache"],
                               t["slot_mapping"], stream=stream)
    out = torch.empty_like(t["query"])
    mcl = batch.max_context_len if max_context_len is None else max_context_len
    binding.paged_attention_decode(out, t["query"], t["key_cache"], t["value_cache"], t["block_tables"],
                                   t["context_lens"], batch.scale, max_context_len=mcl,
                                   partition_size=partition_size, stream=stream)
    return out


def reference(batch):
    return oracle.decode_c(batch.query, batch.key_cache, batch.value_cache, batch.block_tables,
                           batch.context_lens, batch.scale, batch.dtype)


# ----------------------------------------------------------------------------
# the five workloads at full size: write + decode, the launch configuration the bench times


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_workload_full_size(n):
    batch = W.make_config(n)
    t = W.as_torch(batch, DEV)
    expect_k = t["key_cache"].clone()
    expect_v = t["value_cache"].clone()
    canary_slots(t, batch)
    out = run_step(batch, t)
    torch.cuda.synchronize()
    # the write restored exactly the slots it names and touched nothing else
    assert torch.equal(t["key_cache"].view(torch.int16), expect_k.view(torch.int16))
    assert torch.equal(t["value_cache"].view(torch.int16), expect_v.view(torch.int16))
    del expect_k, expect_v
    ref = reference(batch)
    err = check_close(as_np(out), ref, batch.dtype, f"cfg{n}")
    assert binding.device_errors() == 0
    print(f"cfg{n}: max abs err {err:.3e}")


def test_config1_write_matches_oracle_write():
    """On the tiny workload the step's write equals the oracle's write of the same tokens."""
    batch = W.make_config(1)
    kc0, vc0 = batch.pool_before_write()
    ek, ev = oracle.write_c(kc0, vc0, batch.new_key, batch.new_value, batch.slot_mapping, batch.block_size)
    t = W.as_torch(batch, DEV)
    canary_slots(t, batch)
    run_step(batch, t)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(as_np(t["key_cache"]), ek)
    np.testing.assert_array_equal(as_np(t["value_cache"]), ev)


# ----------------------------------------------------------------------------
# split-K partitions


@pytest.mark.parametrize("H,Hkv,dtype", [(8, 8, F16), (16, 4, BF16), (24, 8, F16), (32, 2, BF16)])
def test_split_k_partitions(H, Hkv, dtype):
    ctx = [1, 15, 16, 17, 300, 511, 512, 513, 1500, 2048]
    batch = W.build_batch(seed=21, context_lens=ctx, num_heads=H, num_kv_heads=Hkv, head_dim=128,
                          block_size=16, dtype=dtype, pool_factor=1.3)
    ref = reference(batch)
    t = W.as_torch(batch, DEV)
    outs = []
    for P in (16, 32, 64, 128, 512, 2048):
        out = run_step(batch, t, partition_size=P, write=False)
        torch.cuda.synchronize()
        check_close(as_np(out), ref, dtype, f"P={P}")
        outs.append(to_f64(as_np(out), dtype))
    for o in outs[1:]:
        assert np.abs(o - outs[0]).max() <= 2 * (ATOL + RTOL)
    assert binding.device_errors() == 0


@pytest.mark.parametrize("H,Hkv,D,B,dtype", [(8, 8, 128, 16, F16), (16, 4, 128, 16, BF16), (8, 8, 64, 8, BF16),
                                               (16, 2, 64, 32, F16)])
@pytest.mark.parametrize("ctx", [[1023, 1024, 1025, 2047, 2048, 2049, 3073],
                                 [2047, 2048, 2049, 4097, 9000]])
def test_default_partition_boundary(H, Hkv, D, B, dtype, ctx):
    """partition_size 0: 1024 tokens, or 2048 when the longest context passes 8192 (second set; 1024 for blocks
    of 8, whose partitions hold 128 blocks at most). Contexts just below, at and above one and two
    partitions: the direct and the split path side by side."""
    batch = W.build_batch(seed=23 + H + D + len(ctx), context_lens=ctx, num_heads=H, num_kv_heads=Hkv, head_dim=D,
                          block_size=B, dtype=dtype, pool_factor=1.2)
    t = W.as_torch(batch, DEV)
    out = run_step(batch, t, write=False)
    torch.cuda.synchronize()
    check_close(as_np(out), reference(batch), dtype, "default partition")
    assert binding.device_errors() == 0


def test_long_context_with_outliers_split():
    """1% of keys scaled by 8 (wide score range), 16 partitions of 2048 merged by log-sum-exp."""
    batch = W.build_batch(seed=22, context_lens=[32768, 20000, 513], num_heads=8, num_kv_heads=8,
                          head_dim=128, block_size=16, dtype=F16, key_outlier_frac=0.01)
    t = W.as_torch(batch, DEV)
    out = run_step(batch, t)
    torch.cuda.synchronize()
    check_close(as_np(out), reference(batch), F16, "outliers")


# ----------------------------------------------------------------------------
# random shapes


def fuzz_cases():
    rng = np.random.default_rng(2024)
    cases = []
    for i in range(48):
        D = int(rng.choice([64, 128]))
        B = int(rng.choice([8, 16, 32]))
        G = int(rng.choice([1, 2, 3, 4, 8, 16]))
        Hkv = int(rng.choice([1, 2, 3]))
        S = int(rng.integers(1, 7))
        special = [0, 1, B - 1, B, B + 1, 2 * B + 3]
        ctx = [int(rng.choice(special)) if rng.random() < 0.4 else int(rng.integers(1, 900)) for _ in range(S)]
        P = int(B * rng.integers(1, 128 // max(1, B // 8) + 1)) if rng.random() < 0.5 else 0
        P = min(P, 128 * B)
        cases.append((i, D, B, G, Hkv, ctx, P, F16 if rng.random() < 0.5 else BF16))
    return cases


@pytest.mark.parametrize("case", fuzz_cases(), ids=lambda c: f"c{c[0]}")
def test_fuzz(case):
    i, D, B, G, Hkv, ctx, P, dtype = case
    batch = W.build_batch(seed=3000 + i, context_lens=ctx, num_heads=G * Hkv, num_kv_heads=Hkv, head_dim=D,
                          block_size=B, dtype=dtype, pool_factor=1.5)
    t = W.as_torch(batch, DEV)
    canary_slots(t, batch)
    out = run_step(batch, t, partition_size=P, max_context_len=max(ctx))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(as_np(t["key_cache"]), batch.key_cache)
    np.testing.assert_array_equal(as_np(t["value_cache"]), batch.value_cache)
    check_close(as_np(out), reference(batch), dtype, str(case))
    assert binding.device_errors() == 0


# ----------------------------------------------------------------------------
# behaviour


def test_deterministic_and_stream_ordered():
    batch = W.build_batch(seed=31, context_lens=[700, 33, 2000], num_heads=32, num_kv_heads=8, head_dim=128,
                          block_size=16, dtype=BF16, pool_factor=1.2)
    t = W.as_torch(batch, DEV)
    a = run_step(batch, t, write=False)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        b = run_step(batch, t, write=False, stream=s)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_empty_contexts_and_batch():
    batch = W.build_batch(seed=32, context_lens=[0, 5, 0, 1200], num_heads=8, num_kv_heads=2, head_dim=64,
                          block_size=16, dtype=F16, pool_factor=1.2)
    t = W.as_torch(batch, DEV)
    out = torch.full_like(t["query"], float("nan"))
    binding.paged_attention_decode(out, t["query"], t["key_cache"], t["value_cache"], t["block_tables"],
                                   t["context_lens"], batch.scale, max_context_len=1200)
    torch.cuda.synchronize()
    got = to_f64(as_np(out), F16)
    assert (got[0] == 0).all() and (got[2] == 0).all()
    check_close(as_np(out), reference(batch), F16, "empty")
    e = torch.empty(0, 8, 64, dtype=torch.float16, device=DEV)
    binding.paged_attention_decode(e, e, t["key_cache"], t["value_cache"],
                                   torch.zeros(0, 1, dtype=torch.int32, device=DEV),
                                   torch.zeros(0, dtype=torch.int32, device=DEV), 0.125)


def test_bad_block_table_entry_is_reported_not_read():
    batch = W.build_batch(seed=33, context_lens=[40, 40], num_heads=4, num_kv_heads=4, head_dim=128,
                          block_size=16, dtype=F16)
    t = W.as_torch(batch, DEV)
    t["block_tables"][0, 1] = batch.num_blocks + 1000  # outside the pool
    out = run_step(batch, t, write=False)
    torch.cuda.synchronize()
    assert binding.device_errors() & 1
    ref = reference(batch)
    check_close(as_np(out)[1:], ref[1:], F16, "untouched sequence")


def test_context_above_bound_is_clamped_and_reported():
    batch = W.build_batch(seed=34, context_lens=[100, 64], num_heads=2, num_kv_heads=2, head_dim=64,
                          block_size=16, dtype=F16)
    t = W.as_torch(batch, DEV)
    out = run_step(batch, t, write=False, max_context_len=64)  # seq 0 claims 100 > 64
    torch.cuda.synchronize()
    assert binding.device_errors() & 2
    clamped = W.DecodeBatch(**{**batch.__dict__, "context_lens": np.array([64, 64], dtype=np.int32)})
    check_close(as_np(out), reference(clamped), F16, "clamped")


def test_bad_slot_is_reported_and_skipped():
    batch = W.build_batch(seed=35, context_lens=[20, 30], num_heads=4, num_kv_heads=2, head_dim=128,
                          block_size=16, dtype=BF16)
    t = W.as_torch(batch, DEV)
    before_k = t["key_cache"].clone()
    t["slot_mapping"][0] = batch.num_blocks * batch.block_size  # one past the pool
    t["slot_mapping"][1] = -1
    binding.paged_kv_write(t["new_key"], t["new_value"], t["key_cache"], t["value_cache"], t["slot_mapping"])
    torch.cuda.synchronize()
    assert binding.device_errors() & 4
    assert torch.equal(t["key_cache"].view(torch.int16), before_k.view(torch.int16))


@pytest.mark.parametrize("D,B", [(64, 8), (64, 32), (128, 8), (128, 16), (128, 32)])
def test_write_copies_arbitrary_bits(D, B):
    rng = np.random.default_rng(36)
    NB, Hkv, T = 60, 3, 333
    kc = rng.integers(0, 65536, size=(NB, Hkv, B, D), dtype=np.uint16)
    vc = rng.integers(0, 65536, size=(NB, Hkv, B, D), dtype=np.uint16)
    slots = rng.choice(NB * B, size=T, replace=False).astype(np.int64)
    slots[rng.random(T) < 0.1] = -1
    nk = rng.integers(0, 65536, size=(T, Hkv, D), dtype=np.uint16)
    nv = rng.integers(0, 65536, size=(T, Hkv, D), dtype=np.uint16)
    ek, ev = oracle.write_c(kc, vc, nk, nv, slots, B)

    def dev(a):
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(DEV)

    tk, tv = dev(kc), dev(vc)
    binding.paged_kv_write(dev(nk), dev(nv), tk, tv, torch.from_numpy(slots).to(DEV))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(as_np(tk), ek)
    np.testing.assert_array_equal(as_np(tv), ev)


def test_largest_partition_and_group():
    """A partition of 128 blocks (the kernel's limit) and the largest tensor-core group (8)."""
    batch = W.build_batch(seed=37, context_lens=[2048, 2047, 4096], num_heads=64, num_kv_heads=8, head_dim=128,
                          block_size=16, dtype=BF16)
    t = W.as_torch(batch, DEV)
    out = run_step(batch, t, partition_size=2048)
    torch.cuda.synchronize()
    check_close(as_np(out), reference(batch), BF16, "P=2048 G=8")


# ----------------------------------------------------------------------------
# edge shapes: thousands of tiny sequences, one very long sequence


@pytest.mark.parametrize("Hkv", [8, 2])
def test_many_tiny_sequences(Hkv):
    """2000 sequences of 0..40 tokens, empty ones among them."""
    rng = np.random.default_rng(41)
    ctx = rng.integers(0, 41, size=2000)
    ctx[::97] = 0
    batch = W.build_batch(seed=41, context_lens=ctx, num_heads=8, num_kv_heads=Hkv, head_dim=64, block_size=16,
                          dtype=BF16, pool_factor=1.1)
    t = W.as_torch(batch, DEV)
    out = run_step(batch, t)
    torch.cuda.synchronize()
    check_close(as_np(out), reference(batch), BF16, "tiny")
    assert binding.device_errors() == 0


@pytest.mark.parametrize("H,Hkv", [(2, 2), (8, 2)])
def test_one_long_sequence_across_all_warps(H, Hkv):
    """A single 32768-token sequence with 1% of its keys x8: 64 partitions merged by the reduce."""
    batch = W.build_batch(seed=42, context_lens=[32768], num_heads=H, num_kv_heads=Hkv, head_dim=128,
                          block_size=16, dtype=F16, key_outlier_frac=0.01)
    t = W.as_torch(batch, DEV)
    out = run_step(batch, t)
    torch.cuda.synchronize()
    check_close(as_np(out), reference(batch), F16, "long")


def test_2100_short_sequences_in_blocks_of_8():
    """2100 sequences of 1..59 tokens in 8-token blocks."""
    rng = np.random.default_rng(43)
    batch = W.build_batch(seed=43, context_lens=rng.integers(1, 60, size=2100), num_heads=4, num_kv_heads=4,
                          head_dim=64, block_size=8, dtype=F16)
    t = W.as_torch(batch, DEV)
    out = run_step(batch, t)
    torch.cuda.synchronize()
    check_close(as_np(out), reference(batch), F16, "fallback")


def test_bounded_wait_reports_timeout_and_context_survives():
    """A barrier wait that nothing completes gives up, sets PKV_DEVERR_TIMEOUT, and the GPU stays usable."""
    assert binding.device_errors() == 0
    assert binding.selftest_wait_timeout(2_000_000) & 8
    batch = W.make_config(1)
    t = W.as_torch(batch, DEV)
    out = run_step(batch, t, write=False)
    torch.cuda.synchronize()
    check_close(as_np(out), reference(batch), F16, "after timeout")
    assert binding.device_errors() == 0


# ----------------------------------------------------------------------------
# copy-on-write: block copies and writes driven by the host block pool


def test_copy_on_write_step_matches_oracle():
    """Fork sequences, append tokens (copying shared blocks first), then decode each sequence."""
    from paged_kv_cache_91_gb300.block_pool import BlockPool

    rng = np.random.default_rng(61)
    B, Hkv, H, D, dtype = 16, 4, 8, 128, F16
    pool = BlockPool(num_blocks=96, block_size=B, seed=61)
    seqs = []
    for n in (23, 40, 16, 5):
        s = pool.new_sequence()
        pool.append_tokens(s, n)
        seqs.append(s)
    seqs += [pool.fork(seqs[0]), pool.fork(seqs[0]), pool.fork(seqs[1]), pool.fork(seqs[2])]
    kc = W.round_f32_to(rng.standard_normal((96, Hkv, B, D), dtype=np.float32), dtype)
    vc = W.round_f32_to(rng.standard_normal((96, Hkv, B, D), dtype=np.float32), dtype)
    # one decode step: every sequence appends 1-3 tokens
    slots, copies = [], []
    for s in seqs:
        sl, cp = pool.append_tokens(s, int(rng.integers(1, 4)))
        slots += sl
        copies += cp
    assert len(copies) >= 3  # the forks' shared last blocks were copied
    slots = np.array(slots, dtype=np.int64)
    mapping = np.array(copies, dtype=np.int64).reshape(-1, 2)
    new_k = W.round_f32_to(rng.standard_normal((len(slots), Hkv, D), dtype=np.float32), dtype)
    new_v = W.round_f32_to(rng.standard_normal((len(slots), Hkv, D), dtype=np.float32), dtype)
    ek, ev = oracle.copy_blocks_c(kc, vc, mapping)
    ek, ev = oracle.write_c(ek, ev, new_k, new_v, slots, B)

    def dev16(a):
        return torch.from_numpy(a.view(np.int16)).view(torch.float16).to(DEV)

    tk, tv = dev16(kc), dev16(vc)
    binding.paged_kv_copy_blocks(tk, tv, torch.from_numpy(mapping).to(DEV))
    binding.paged_kv_write(dev16(new_k), dev16(new_v), tk, tv, torch.from_numpy(slots).to(DEV))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(as_np(tk), ek)
    np.testing.assert_array_equal(as_np(tv), ev)

    tables = BlockPool.tables(seqs)
    ctx = np.array([s.num_tokens for s in seqs], dtype=np.int32)
    q = W.round_f32_to(rng.standard_normal((len(seqs), H, D), dtype=np.float32), dtype)
    out = torch.empty(len(seqs), H, D, dtype=torch.float16, device=DEV)
    binding.paged_attention_decode(out, dev16(q), tk, tv, torch.from_numpy(tables).to(DEV),
                                   torch.from_numpy(ctx).to(DEV), 1 / np.sqrt(D), max_context_len=int(ctx.max()))
    torch.cuda.synchronize()
    ref = oracle.decode_c(q, ek, ev, tables, ctx, 1 / np.sqrt(D), dtype)
    check_close(as_np(out), ref, dtype, "after copy-on-write")
    assert binding.device_errors() == 0


@pytest.mark.parametrize("D,B", [(64, 8), (128, 32)])
def test_copy_blocks_many_pairs_and_bad_pair(D, B):
    rng = np.random.default_rng(62)
    NB, Hkv = 300, 2
    kc = rng.integers(0, 65536, size=(NB, Hkv, B, D), dtype=np.uint16)
    vc = rng.integers(0, 65536, size=(NB, Hkv, B, D), dtype=np.uint16)
    perm = rng.permutation(NB)
    pairs = np.stack([perm[:100], perm[100:200]], axis=1).astype(np.int64)
    ek, ev = oracle.copy_blocks_c(kc, vc, pairs)

    def dev(a):
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(DEV)

    tk, tv = dev(kc), dev(vc)
    bad = np.concatenate([pairs, [[NB + 5, perm[250]]]]).astype(np.int64)  # last pair names no block
    binding.paged_kv_copy_blocks(tk, tv, torch.from_numpy(bad).to(DEV))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(as_np(tk), ek)
    np.testing.assert_array_equal(as_np(tv), ev)
    assert binding.device_errors() & 1


def test_read_chunks_helper_reads_in_bounds_and_reports_bad_indices():
    """The bench's read-ceiling helper: valid orders leave no error; an index past the buffer is skipped and
    reported, and the context stays usable."""
    buf = torch.empty(64 << 20, dtype=torch.uint8, device=DEV)
    for ch in (1024, 2048, 4096, 8192):
        n = buf.numel() // ch
        order = torch.randperm(n, device=DEV, dtype=torch.int32, generator=torch.Generator(DEV).manual_seed(ch))
        binding.read_chunks(buf, order, ch)
        binding.read_chunks(buf, order[: 1000], ch)  # a partial last warp
    assert binding.device_errors() == 0
    bad = torch.tensor([0, 1, buf.numel() // 2048, -5, 3], dtype=torch.int32, device=DEV)
    binding.read_chunks(buf, bad, 2048)
    assert binding.device_errors() == 1  # PKV_DEVERR_BLOCK_ID
    batch = W.make_config(1)
    t = W.as_torch(batch, DEV)
    out = run_step(batch, t, write=False)
    torch.cuda.synchronize()
    check_close(as_np(out), reference(batch), F16, "after the read helper")
