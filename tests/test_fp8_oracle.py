"""Pins for the oracle's FP8 (E4M3) codec, quantizing write and fp8-cache decode."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_91_gb300.workloads import F16, round_f32_to

ALL = np.arange(256, dtype=np.uint8)


def torch_decode(codes):
    return torch.from_numpy(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def torch_encode(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_decode_matches_library_for_every_code():
    ref = torch_decode(ALL)
    for impl in (oracle.e4m3_decode_c, oracle.e4m3_decode_np):
        got = impl(ALL)
        assert (np.isnan(got) == np.isnan(ref)).all()
        np.testing.assert_array_equal(got[~np.isnan(ref)], ref[~np.isnan(ref)])


def test_format_landmarks():
    d = oracle.e4m3_decode_np
    assert d(0x38) == 1.0 and d(0xB8) == -1.0 and d(0x7E) == 448.0 and np.isnan(d(0x7F))
    assert d(0x01) == 2.0 ** -9 and d(0x08) == 2.0 ** -6 and d(0x07) == 7 * 2.0 ** -9


def test_encode_hand_cases():
    x = np.array([1.0625, 1.1875, 500.0, -1000.0, 2.0 ** -10, 3 * 2.0 ** -10, 464.0, -0.0], dtype=np.float32)
    #            tie->1.0 tie->1.25 sat   sat     tie->0      tie->2^-8   ->448   -0
    want = np.array([0x38, 0x3A, 0x7E, 0xFE, 0x00, 0x02, 0x7E, 0x80], dtype=np.uint8)
    for impl in (oracle.e4m3_encode_c, oracle.e4m3_encode_np):
        np.testing.assert_array_equal(impl(x), want)


def test_encode_matches_library_in_range_including_ties():
    rng = np.random.default_rng(71)
    vals = torch_decode(np.arange(0x7F, dtype=np.uint8))  # 0 .. 448, increasing
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)  # exact ties (representable in fp32)
    x = np.concatenate([rng.standard_normal(200000).astype(np.float32) * 30,
                        (rng.random(20000) * 2.0 ** -6).astype(np.float32), mids, -mids])
    ref = torch_encode(x)
    np.testing.assert_array_equal(oracle.e4m3_encode_np(x), ref)
    np.testing.assert_array_equal(oracle.e4m3_encode_c(x), ref)


def test_round_trip_of_every_finite_code():
    finite = ALL[~np.isnan(torch_decode(ALL))]
    vals = oracle.e4m3_decode_np(finite).astype(np.float32)
    np.testing.assert_array_equal(oracle.e4m3_encode_np(vals), finite)
    np.testing.assert_array_equal(oracle.e4m3_encode_c(vals), finite)


def test_write_fp8_is_divide_then_round():
    rng = np.random.default_rng(72)
    T, Hkv, D, B, NB = 5, 2, 64, 16, 4
    k = round_f32_to(rng.standard_normal((T, Hkv, D), dtype=np.float32) * 3, F16)
    v = round_f32_to(rng.standard_normal((T, Hkv, D), dtype=np.float32), F16)
    slots = np.array([0, 17, -1, 63, 40], dtype=np.int64)
    kc0 = np.zeros((NB, Hkv, B, D), dtype=np.uint8)
    ks, vs = np.float32(0.03125), np.float32(0.0117)
    kc, vc = oracle.write_fp8_c(kc0, kc0, k, v, slots, B, F16, ks, vs)
    kf = k.view(np.float16).astype(np.float32)
    vf = v.view(np.float16).astype(np.float32)
    for t, slot in enumerate(slots):
        if slot < 0:
            continue
        b, o = divmod(int(slot), B)
        np.testing.assert_array_equal(kc[b, :, o, :], oracle.e4m3_encode_np(kf[t] / ks))
        np.testing.assert_array_equal(vc[b, :, o, :], oracle.e4m3_encode_np(vf[t] / vs))
    assert (kc[0, :, 1:16] == 0).all()  # untouched slots


def test_fp8_decode_equals_fp16_decode_of_the_same_values():
    """With a power-of-two scale every E4M3 value times the scale is an fp16 value, so a decode
    over the fp8 cache must equal a decode over the fp16 cache holding those values."""
    rng = np.random.default_rng(73)
    NB, Hkv, B, D, S, H = 10, 2, 16, 64, 3, 4
    codes_k = rng.integers(0, 0x7F, size=(NB, Hkv, B, D), dtype=np.uint8) | (rng.integers(0, 2, (NB, Hkv, B, D)) << 7).astype(np.uint8)
    codes_v = rng.integers(0, 0x7F, size=(NB, Hkv, B, D), dtype=np.uint8)
    codes_k[codes_k == 0xFF] = 0x7E
    ks, vs = 2.0 ** -6, 2.0 ** -5
    kc16 = round_f32_to((oracle.e4m3_decode_np(codes_k) * ks).astype(np.float32), F16)
    vc16 = round_f32_to((oracle.e4m3_decode_np(codes_v) * vs).astype(np.float32), F16)
    np.testing.assert_array_equal(kc16.view(np.float16).astype(np.float64), oracle.e4m3_decode_np(codes_k) * ks)
    q = round_f32_to(rng.standard_normal((S, H, D), dtype=np.float32), F16)
    bt = np.array([[3, 1, 7], [0, -1, -1], [9, 2, -1]], dtype=np.int32)
    cl = np.array([40, 3, 20], dtype=np.int32)
    a = oracle.decode_c(q, codes_k, codes_v, bt, cl, 0.125, F16, k_scale=ks, v_scale=vs)
    b = oracle.decode_c(q, kc16, vc16, bt, cl, 0.125, F16)
    c = oracle.decode_np(q, codes_k, codes_v, bt, cl, 0.125, F16, k_scale=ks, v_scale=vs)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_allclose(a, c, rtol=0, atol=1e-12)
