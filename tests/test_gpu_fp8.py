"""GPU parity of the FP8 (E4M3) KV cache: quantizing write and decode over an FP8 pool.

The write must match the oracle's quantizing write code for code. The decode
reads pools of E4M3 codes made by the oracle's encoder (each 16-bit pool value
divided by the scale in fp32, then rounded to E4M3), so the oracle and the
library see the same codes; the output must satisfy
|gpu - ref| <= 1e-2 + 1e-2 |ref| against the oracle's fp64 result over the
values code * scale. Unused slots hold NaN codes (the encoded NaN canaries), so
a read outside a context shows up as a NaN in the output.
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
NAN_CODES = (0x7F, 0xFF)


@pytest.fixture(autouse=True)
def clean_errors(cuda_lib):
    binding.device_errors(clear=True)
    yield


def as_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def fp8_lut(dtype: str, scale: float) -> np.ndarray:
    """Oracle code of every 16-bit pattern x: E4M3(fp32(x) / fp32(scale)), as a 65536-entry table."""
    vals = oracle.widen_np(np.arange(65536, dtype=np.uint32).astype(np.uint16), dtype).astype(np.float32)
    with np.errstate(invalid="ignore", over="ignore"):
        return oracle.e4m3_encode_np(vals / np.float32(scale))


def fp8_pools(batch, k_scale, v_scale):
    """The batch's pools as E4M3 codes (what the quantizing write would have stored)."""
    return fp8_lut(batch.dtype, k_scale)[batch.key_cache], fp8_lut(batch.dtype, v_scale)[batch.value_cache]


def check_close(gpu_bits, ref, dtype, what=""):
    got = oracle.widen_np(gpu_bits, dtype)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), (f"{what}: {bad.sum()} elements out of tolerance; max abs err "
                           f"{err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")
    return float(err.max())


def to_dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def decode_fp8(batch, t, kc8, vc8, k_scale, v_scale, partition_size=0, max_context_len=None):
    out = torch.empty_like(t["query"])
    mcl = batch.max_context_len if max_context_len is None else max_context_len
    binding.paged_attention_decode_fp8(out, t["query"], kc8, vc8, t["block_tables"], t["context_lens"],
                                       batch.scale, k_scale, v_scale, max_context_len=mcl,
                                       partition_size=partition_size)
    return out


def reference(batch, kc8, vc8, k_scale, v_scale):
    return oracle.decode_c(batch.query, kc8, vc8, batch.block_tables, batch.context_lens, batch.scale,
                           batch.dtype, k_scale=k_scale, v_scale=v_scale)


# ----------------------------------------------------------------------------
# quantizing write


@pytest.mark.parametrize("dtype,D,B", [(F16, 128, 16), (BF16, 128, 16), (F16, 64, 8), (BF16, 64, 32)])
@pytest.mark.parametrize("k_scale,v_scale", [(2.0 ** -6, 2.0 ** -5), (0.0137, 0.0211), (1.0, 3.7)])
def test_write_fp8_matches_oracle(dtype, D, B, k_scale, v_scale):
    rng = np.random.default_rng(81)
    T, Hkv, NB = 300, 4, 40
    # N(0,1) values, a few large ones (saturation at 448 * scale) and signed zeros
    k = rng.standard_normal((T, Hkv, D), dtype=np.float32) * 2
    v = rng.standard_normal((T, Hkv, D), dtype=np.float32)
    k.flat[rng.choice(k.size, 500, replace=False)] *= 1e4
    v.flat[:64] = -0.0
    kb, vb = W.round_f32_to(k, dtype), W.round_f32_to(v, dtype)
    slots = rng.choice(NB * B, size=T, replace=False).astype(np.int64)
    slots[::37] = -1  # padding tokens
    kc0 = rng.integers(0, 256, size=(NB, Hkv, B, D), dtype=np.uint8)
    vc0 = rng.integers(0, 256, size=(NB, Hkv, B, D), dtype=np.uint8)
    ek, ev = oracle.write_fp8_c(kc0, vc0, kb, vb, slots, B, dtype, k_scale, v_scale)
    tdt = torch.float16 if dtype == F16 else torch.bfloat16
    half = lambda a: torch.from_numpy(a.view(np.int16)).view(tdt).to(DEV)  # noqa: E731
    kc, vc = to_dev_u8(kc0), to_dev_u8(vc0)
    binding.paged_kv_write_fp8(half(kb), half(vb), kc, vc, torch.from_numpy(slots).to(DEV), k_scale, v_scale)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(kc.cpu().numpy(), ek)
    np.testing.assert_array_equal(vc.cpu().numpy(), ev)
    assert binding.device_errors() == 0


def test_write_fp8_arbitrary_bits_and_float8_tensors():
    """Every 16-bit pattern (NaN and infinities included) through the write; caches as float8_e4m3fn."""
    T, Hkv, D, B = 512, 1, 128, 16
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(T, Hkv, D)
    vbits = bits[::-1].copy()
    slots = np.arange(T, dtype=np.int64)
    for dtype in (F16, BF16):
        kc0 = np.zeros((T // B, Hkv, B, D), dtype=np.uint8)
        ek, ev = oracle.write_fp8_c(kc0, kc0, bits, vbits, slots, B, dtype, 0.5, 3.0)
        tdt = torch.float16 if dtype == F16 else torch.bfloat16
        kc = torch.zeros(kc0.shape, dtype=torch.float8_e4m3fn, device=DEV)
        vc = torch.zeros(kc0.shape, dtype=torch.float8_e4m3fn, device=DEV)
        binding.paged_kv_write_fp8(torch.from_numpy(bits.view(np.int16)).view(tdt).to(DEV),
                                   torch.from_numpy(vbits.view(np.int16)).view(tdt).to(DEV), kc, vc,
                                   torch.from_numpy(slots).to(DEV), 0.5, 3.0)
        torch.cuda.synchronize()
        for got, exp in ((kc.view(torch.uint8).cpu().numpy(), ek), (vc.view(torch.uint8).cpu().numpy(), ev)):
            nan = np.isin(exp, NAN_CODES)
            assert np.isin(got[nan], NAN_CODES).all()  # a NaN gives a NaN code; its sign is not specified
            np.testing.assert_array_equal(got[~nan], exp[~nan])


def test_write_fp8_bad_slot_is_skipped_and_reported():
    T, Hkv, D, B, NB = 3, 2, 64, 16, 4
    kb = W.round_f32_to(np.ones((T, Hkv, D), np.float32), F16)
    kc = torch.zeros((NB, Hkv, B, D), dtype=torch.uint8, device=DEV)
    vc = torch.zeros_like(kc)
    slots = torch.tensor([0, NB * B, 5], dtype=torch.int64, device=DEV)
    t = torch.from_numpy(kb.view(np.int16)).view(torch.float16).to(DEV)
    binding.paged_kv_write_fp8(t, t, kc, vc, slots, 1.0, 1.0)
    assert binding.device_errors() & 4
    got = kc.cpu().numpy()
    assert (got[0, :, 0] == 0x38).all() and (got[0, :, 5] == 0x38).all()
    assert (got[0, :, 1:5] == 0).all() and (got[1:] == 0).all()


# ----------------------------------------------------------------------------
# decode over an FP8 pool


@pytest.mark.parametrize("H,Hkv,D,B,dtype", [
    (8, 8, 128, 16, F16), (8, 8, 128, 16, BF16), (16, 4, 128, 16, BF16), (12, 4, 64, 16, F16),
    (8, 8, 128, 8, F16), (8, 2, 128, 32, BF16), (6, 6, 64, 8, BF16), (4, 4, 64, 32, F16),
    (32, 2, 128, 16, F16), (9, 1, 64, 16, BF16),
    # an odd number of kv heads: no kv-head pairs, the one-head tile
    (6, 3, 128, 16, F16), (5, 5, 128, 8, BF16), (8, 1, 128, 16, F16),
])
def test_decode_fp8_shapes(H, Hkv, D, B, dtype):
    ctx = [1, 2, 7, B, B + 1, 100, 511, 512, 513, 1300]
    batch = W.build_batch(seed=82 + H + D + B, context_lens=ctx, num_heads=H, num_kv_heads=Hkv, head_dim=D,
                          block_size=B, dtype=dtype, pool_factor=1.3)
    ks, vs = 0.0137, 0.0093
    kc8, vc8 = fp8_pools(batch, ks, vs)
    ref = reference(batch, kc8, vc8, ks, vs)
    t = W.as_torch(batch, DEV)
    K, V = to_dev_u8(kc8), to_dev_u8(vc8)
    for P in (0, B, 4 * B):
        out = decode_fp8(batch, t, K, V, ks, vs, partition_size=P)
        torch.cuda.synchronize()
        check_close(as_bits(out), ref, dtype, f"P={P}")
    assert binding.device_errors() == 0


@pytest.mark.parametrize("H,Hkv,D,dtype", [(8, 8, 128, F16), (16, 4, 128, BF16), (12, 4, 64, F16)])
def test_decode_fp8_default_partition_boundary(H, Hkv, D, dtype):
    """partition_size 0 (1024 tokens): contexts just below, at and above one and two partitions."""
    ctx = [1023, 1024, 1025, 2048, 2049]
    batch = W.build_batch(seed=91 + H + D, context_lens=ctx, num_heads=H, num_kv_heads=Hkv, head_dim=D,
                          block_size=16, dtype=dtype, pool_factor=1.2)
    ks, vs = 0.0137, 0.0093
    kc8, vc8 = fp8_pools(batch, ks, vs)
    t = W.as_torch(batch, DEV)
    out = decode_fp8(batch, t, to_dev_u8(kc8), to_dev_u8(vc8), ks, vs)
    torch.cuda.synchronize()
    check_close(as_bits(out), reference(batch, kc8, vc8, ks, vs), dtype, "default partition")
    assert binding.device_errors() == 0


@pytest.mark.parametrize("H,Hkv,B,dtype", [(16, 8, 16, F16), (24, 8, 8, BF16), (64, 8, 32, F16), (8, 8, 16, BF16)])
def test_decode_fp8_group_sizes(H, Hkv, B, dtype):
    """Group sizes 2, 3, 8 and 1 on the tensor-core tile (head_dim 128)."""
    ctx = [3, 16, 33, 250, 512, 700, 2047]
    batch = W.build_batch(seed=87 + H + B, context_lens=ctx, num_heads=H, num_kv_heads=Hkv, head_dim=128,
                          block_size=B, dtype=dtype, pool_factor=1.2)
    ks, vs = 0.011, 0.017
    kc8, vc8 = fp8_pools(batch, ks, vs)
    ref = reference(batch, kc8, vc8, ks, vs)
    t = W.as_torch(batch, DEV)
    out = decode_fp8(batch, t, to_dev_u8(kc8), to_dev_u8(vc8), ks, vs, partition_size=128)
    torch.cuda.synchronize()
    check_close(as_bits(out), ref, dtype)
    assert binding.device_errors() == 0


@pytest.mark.parametrize("dtype,factors", [
    (BF16, (2.0 ** 40, 2.0 ** -40, 1e4, 3e-5)),   # beyond f16 range: per-head power-of-two rescaling
    (F16, (300.0, 2.0 ** -10, 1.0, 40.0)),
])
def test_decode_fp8_query_magnitudes(dtype, factors):
    """Query heads of very different magnitudes (one factor per kv-head group) over one FP8 pool."""
    H, Hkv = 16, 4
    batch = W.build_batch(seed=88, context_lens=[64, 700, 9], num_heads=H, num_kv_heads=Hkv, head_dim=128,
                          block_size=16, dtype=dtype, pool_factor=1.3)
    q = W.bits_to_f32(batch.query, dtype)
    for g, f in enumerate(factors):
        q[:, g * 4:(g + 1) * 4, :] *= np.float32(f)
    q[:, 1, :5] = 0.0  # exact zeros next to large values
    batch.query = W.round_f32_to(q, dtype)
    scale = 1.0 / max(factors)  # keeps the scores finite for the largest factor
    batch.scale = scale
    ks, vs = 0.02, 0.02
    kc8, vc8 = fp8_pools(batch, ks, vs)
    ref = reference(batch, kc8, vc8, ks, vs)
    t = W.as_torch(batch, DEV)
    out = decode_fp8(batch, t, to_dev_u8(kc8), to_dev_u8(vc8), ks, vs)
    torch.cuda.synchronize()
    check_close(as_bits(out), ref, dtype)


@pytest.mark.parametrize("H,Hkv,D", [(8, 8, 128), (16, 4, 128), (4, 4, 64)])
def test_decode_fp8_subnormal_codes(H, Hkv, D):
    """Pools of E4M3 subnormal codes only (exponent field 0), scaled up so that a widening or an
    MMA that flushed them to zero would miss the output by far more than the tolerance."""
    rng = np.random.default_rng(89)
    batch = W.build_batch(seed=89, context_lens=[5, 100, 37], num_heads=H, num_kv_heads=Hkv, head_dim=D,
                          block_size=16, dtype=F16, pool_factor=1.5)
    shape = batch.key_cache.shape
    kc8 = (rng.integers(1, 8, size=shape) | (rng.integers(0, 2, size=shape) << 7)).astype(np.uint8)
    vc8 = rng.integers(1, 8, size=shape).astype(np.uint8)  # positive: the mean does not cancel
    ks, vs = 64.0, 64.0  # values up to 7 * 2^-9 * 64 = 0.875
    ref = reference(batch, kc8, vc8, ks, vs)
    assert np.abs(ref).max() > 0.3
    t = W.as_torch(batch, DEV)
    out = decode_fp8(batch, t, to_dev_u8(kc8), to_dev_u8(vc8), ks, vs)
    torch.cuda.synchronize()
    check_close(as_bits(out), ref, F16)


def test_decode_fp8_full_range_codes_and_outliers():
    """Keys with 1% outliers scaled by 8 and a scale that spreads values over the whole E4M3 range."""
    batch = W.build_batch(seed=83, context_lens=[4096, 3000, 17, 900], num_heads=8, num_kv_heads=8,
                          head_dim=128, block_size=16, dtype=F16, key_outlier_frac=0.01)
    ks, vs = 16.0 / 448, 5.0 / 448
    kc8, vc8 = fp8_pools(batch, ks, vs)
    used = np.unique(kc8)
    assert 0x7E in used and 0xFE in used and 0x01 in used  # saturated and subnormal codes occur
    ref = reference(batch, kc8, vc8, ks, vs)
    t = W.as_torch(batch, DEV)
    out = decode_fp8(batch, t, to_dev_u8(kc8), to_dev_u8(vc8), ks, vs)
    torch.cuda.synchronize()
    check_close(as_bits(out), ref, F16, "outliers")
    assert binding.device_errors() == 0


def test_decode_fp8_empty_contexts_and_repeat_calls():
    batch = W.build_batch(seed=84, context_lens=[0, 5, 0, 700], num_heads=4, num_kv_heads=4, head_dim=64,
                          block_size=16, dtype=BF16, pool_factor=1.5)
    kc8, vc8 = fp8_pools(batch, 0.02, 0.02)
    ref = reference(batch, kc8, vc8, 0.02, 0.02)
    t = W.as_torch(batch, DEV)
    K, V = to_dev_u8(kc8), to_dev_u8(vc8)
    outs = [decode_fp8(batch, t, K, V, 0.02, 0.02) for _ in range(2)]
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])
    check_close(as_bits(outs[0]), ref, BF16)
    assert (as_bits(outs[0])[[0, 2]] == 0).all()


def test_decode_fp8_bad_block_id_is_reported():
    batch = W.build_batch(seed=85, context_lens=[40, 40], num_heads=4, num_kv_heads=4, head_dim=64,
                          block_size=16, dtype=F16, pool_factor=1.5)
    kc8, vc8 = fp8_pools(batch, 0.05, 0.05)
    t = W.as_torch(batch, DEV)
    t["block_tables"][1, 1] = batch.num_blocks + 3
    out = decode_fp8(batch, t, to_dev_u8(kc8), to_dev_u8(vc8), 0.05, 0.05)
    torch.cuda.synchronize()
    assert binding.device_errors() & 1
    # the untouched sequence is still right
    ref = reference(batch, kc8, vc8, 0.05, 0.05)
    check_close(as_bits(out)[:1], ref[:1], F16)


# ----------------------------------------------------------------------------
# the full-size step: the LLaMA-2-13B-shaped batch with an FP8 pool


def test_fp8_step_llama13b_shape():
    """Workload 2's shapes (64 sequences, 40 heads, D 128, contexts 128-2048) with an E4M3 pool:
    the quantizing write of the step's new tokens, then the decode, in the bench's configuration."""
    batch = W.make_config(2)
    ks, vs = 2.0 ** -6, 2.0 ** -6
    kc8, vc8 = fp8_pools(batch, ks, vs)
    t = W.as_torch(batch, DEV)
    K, V = to_dev_u8(kc8), to_dev_u8(vc8)
    slots = batch.new_token_slots()
    sb, so = torch.from_numpy(slots[:, 0]).to(DEV), torch.from_numpy(slots[:, 1]).to(DEV)
    K[sb, :, so, :] = 0x7F  # the new tokens' slots start as NaN codes
    V[sb, :, so, :] = 0x7F
    binding.paged_kv_write_fp8(t["new_key"], t["new_value"], K, V, t["slot_mapping"], ks, vs)
    out = decode_fp8(batch, t, K, V, ks, vs)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(K.cpu().numpy(), kc8)  # the write stored exactly the oracle's codes
    np.testing.assert_array_equal(V.cpu().numpy(), vc8)
    ref = reference(batch, kc8, vc8, ks, vs)
    err = check_close(as_bits(out), ref, F16, "fp8 step")
    assert binding.device_errors() == 0
    print(f"fp8 step: max abs err {err:.3e}")


def test_copy_blocks_fp8_pool():
    rng = np.random.default_rng(86)
    kc0 = rng.integers(0, 256, size=(30, 4, 16, 128), dtype=np.uint8)
    vc0 = rng.integers(0, 256, size=(30, 4, 16, 128), dtype=np.uint8)
    pairs = np.array([[3, 9], [17, 0], [29, 28]], dtype=np.int64)
    ek, ev = oracle.copy_blocks_np(kc0, vc0, pairs)
    kc, vc = to_dev_u8(kc0), to_dev_u8(vc0)
    binding.paged_kv_copy_blocks(kc, vc, torch.from_numpy(pairs).to(DEV))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(kc.cpu().numpy(), ek)
    np.testing.assert_array_equal(vc.cpu().numpy(), ev)
