"""Pins for the CPU oracle (both the C and the numpy implementation).

Each pin checks the oracle against something other than itself: a closed form,
an invariant of the definition, a pure-Python brute force over contiguous
K/V, or a value printed on the pages (tests/golden/pages_examples.json). The
mutation test at the end plants plausible mistakes in a copy of the numpy
oracle and checks that every one of them fails at least one pin.
"""
import math
import struct

import numpy as np
import pytest

import oracle
from paged_kv_cache_91_gb300.workloads import BF16, CANARY, F16, round_f32_to

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ----------------------------------------------------------------------------
# helpers (test-side construction of paged inputs from contiguous sequences)


def widen_py(bits: int, dtype: str) -> float:
    if dtype == F16:
        return struct.unpack("<e", struct.pack("<H", int(bits)))[0]
    return struct.unpack("<f", struct.pack("<I", int(bits) << 16))[0]


def bruteforce(q_bits, K_bits, V_bits, scale, dtype, g):
    """Pure-Python unpaged attention for one query head over contiguous K/V [n][Hkv][D] bits."""
    q = [widen_py(b, dtype) for b in q_bits]
    D = len(q)
    n = len(K_bits)
    if n == 0:
        return [0.0] * D
    x = []
    for j in range(n):
        acc = 0.0
        for d in range(D):
            acc += q[d] * widen_py(K_bits[j][g][d], dtype)
        x.append(scale * acc)
    m = max(x)
    e = [math.exp(v - m) for v in x]
    z = sum(e)
    return [sum(e[j] * widen_py(V_bits[j][g][d], dtype) for j in range(n)) / z for d in range(D)]


class Paged:
    """Small paged batch built from contiguous per-sequence K/V."""

    def __init__(self, rng, ctxs, H, Hkv, D, B, dtype, NB=None, tables=None):
        S = len(ctxs)
        nblk = [(c + B - 1) // B for c in ctxs]
        if tables is None:
            need = sum(nblk)
            NB = NB or need + 3
            perm = rng.permutation(NB)
            tables, p = [], 0
            for n in nblk:
                tables.append(list(perm[p:p + n]))
                p += n
        maxb = max(1, max(len(t) for t in tables))
        self.bt = np.full((S, maxb), -1, dtype=np.int32)
        for s, t in enumerate(tables):
            self.bt[s, :len(t)] = t
        self.NB = NB
        self.q = round_f32_to(rng.standard_normal((S, H, D), dtype=np.float32), dtype)
        self.K = [round_f32_to(rng.standard_normal((c, Hkv, D), dtype=np.float32), dtype) for c in ctxs]
        self.V = [round_f32_to(rng.standard_normal((c, Hkv, D), dtype=np.float32), dtype) for c in ctxs]
        self.cl = np.array(ctxs, dtype=np.int32)
        self.H, self.Hkv, self.D, self.B, self.dtype = H, Hkv, D, B, dtype
        self.scale = 1.0 / math.sqrt(D)
        self.build_pool()

    def build_pool(self):
        B = self.B
        self.kc = np.full((self.NB, self.Hkv, B, self.D), CANARY[self.dtype], dtype=np.uint16)
        self.vc = self.kc.copy()
        for s, c in enumerate(self.cl):
            for j in range(int(c)):
                phys = self.bt[s, j // B]
                self.kc[phys, :, j % B, :] = self.K[s][j]
                self.vc[phys, :, j % B, :] = self.V[s][j]

    def args(self):
        return (self.q, self.kc, self.vc, self.bt, self.cl, self.scale, self.dtype)

    def brute(self):
        S, H, D = self.q.shape
        G = H // self.Hkv
        out = np.zeros((S, H, D))
        for s in range(S):
            for h in range(H):
                out[s, h] = bruteforce(self.q[s, h], self.K[s], self.V[s], self.scale, self.dtype, h // G)
        return out


def w(bits, dtype):
    return oracle.widen_np(bits, dtype)


# ----------------------------------------------------------------------------
# pins: each takes decode(query, key_cache, value_cache, block_tables, context_lens, scale, dtype)


def pin_single_token(decode):
    """ctx = 1: the only weight is exp(0)/exp(0) = 1, so o = v exactly."""
    rng = np.random.default_rng(1)
    for dtype in (F16, BF16):
        P = Paged(rng, [1, 1, 1], H=4, Hkv=2, D=64, B=16, dtype=dtype)
        out = decode(*P.args())
        for s in range(3):
            for h in range(4):
                np.testing.assert_array_equal(out[s, h], w(P.V[s][0, h // 2], dtype))


def pin_identical_keys(decode):
    """All keys equal: the weights are uniform and o is the mean of the values."""
    rng = np.random.default_rng(2)
    P = Paged(rng, [37, 5], H=2, Hkv=1, D=32, B=16, dtype=F16)
    for s in range(2):
        P.K[s][:] = P.K[s][0]
    P.build_pool()
    out = decode(*P.args())
    for s in range(2):
        mean = w(P.V[s][:, 0], F16).mean(axis=0)
        for h in range(2):
            np.testing.assert_allclose(out[s, h], mean, rtol=0, atol=1e-12)


def pin_two_tokens(decode):
    """ctx = 2: o = sigmoid(D) v1 + sigmoid(-D) v2 with D = scale * q . (k1 - k2)."""
    rng = np.random.default_rng(3)
    P = Paged(rng, [2, 2], H=2, Hkv=2, D=16, B=16, dtype=F16)
    out = decode(*P.args())
    for s in range(2):
        for h in range(2):
            q = w(P.q[s, h], F16)
            k1, k2 = w(P.K[s][0, h], F16), w(P.K[s][1, h], F16)
            v1, v2 = w(P.V[s][0, h], F16), w(P.V[s][1, h], F16)
            delta = P.scale * float(q @ (k1 - k2))
            a = 1.0 / (1.0 + math.exp(-delta))
            np.testing.assert_allclose(out[s, h], a * v1 + (1 - a) * v2, rtol=0, atol=1e-12)


def pin_dominant_key(decode):
    """A key far more aligned with q than the rest takes all the weight: o = v at that position.

    The first position, a middle one, the last one (ctx - 1) and the slot just
    past the context (which must be ignored) are each tried.
    """
    rng = np.random.default_rng(4)
    ctx = 40
    for pos in (0, 17, ctx - 1, ctx):
        P = Paged(rng, [ctx + 1], H=1, Hkv=1, D=64, B=16, dtype=F16)
        q = w(P.q[0, 0], F16)
        P.K[0][pos, 0] = round_f32_to((6.0 * q).astype(np.float32), F16)
        P.build_pool()
        P.cl[0] = ctx  # the slot at position ctx stays in the pool but is past the context
        out = decode(*P.args())[0, 0]
        if pos < ctx:
            np.testing.assert_allclose(out, w(P.V[0][pos, 0], F16), rtol=0, atol=1e-9)
        else:
            ref = w(P.V[0][:ctx, 0], F16)
            x = P.scale * (w(P.K[0][:ctx, 0], F16) @ q)
            e = np.exp(x - x.max())
            np.testing.assert_allclose(out, (e / e.sum()) @ ref, rtol=0, atol=1e-12)


def pin_constant_values(decode):
    """Every value row equal to c: the weights sum to 1, so o = c."""
    rng = np.random.default_rng(5)
    P = Paged(rng, [29, 64, 3], H=4, Hkv=4, D=16, B=8, dtype=BF16)
    for s in range(3):
        P.V[s][:] = P.V[s][0]
    P.build_pool()
    out = decode(*P.args())
    for s in range(3):
        for h in range(4):
            np.testing.assert_allclose(out[s, h], w(P.V[s][0, h], BF16), rtol=1e-14, atol=1e-14)


def pin_block_permutation(decode):
    """Relabelling physical blocks (pool and tables together) leaves every output unchanged."""
    rng = np.random.default_rng(6)
    P = Paged(rng, [33, 7, 50], H=4, Hkv=2, D=32, B=16, dtype=F16)
    base = decode(*P.args())
    perm = rng.permutation(P.NB)
    kc = np.empty_like(P.kc)
    vc = np.empty_like(P.vc)
    kc[perm] = P.kc
    vc[perm] = P.vc
    bt = np.where(P.bt >= 0, perm[np.maximum(P.bt, 0)], -1).astype(np.int32)
    moved = decode(P.q, kc, vc, bt, P.cl, P.scale, P.dtype)
    np.testing.assert_array_equal(base, moved)


def pin_gqa_is_repeated_mha(decode):
    """GQA with group G equals MHA whose kv heads are each kv head repeated G times."""
    rng = np.random.default_rng(7)
    P = Paged(rng, [21, 40], H=8, Hkv=2, D=16, B=16, dtype=F16)
    gqa = decode(*P.args())
    kc = np.repeat(P.kc, 4, axis=1)
    vc = np.repeat(P.vc, 4, axis=1)
    mha = decode(P.q, kc, vc, P.bt, P.cl, P.scale, P.dtype)
    np.testing.assert_array_equal(gqa, mha)


def pin_paged_equals_bruteforce(decode):
    """Paged decode equals pure-Python attention over the contiguous sequences (block sizes 4, 8, 16)."""
    rng = np.random.default_rng(8)
    for B in (4, 8, 16):
        for dtype in (F16, BF16):
            P = Paged(rng, [1, 16, 45, 0], H=4, Hkv=2, D=8, B=B, dtype=dtype)
            np.testing.assert_allclose(decode(*P.args()), P.brute(), rtol=0, atol=1e-12)


def pin_page_tables(decode, golden):
    """The pages' block tables: request B -> [7, 23, 61], and the shared-prefix tables [5, x]."""
    rng = np.random.default_rng(9)
    tb = golden["request_b_block_table"]["block_table"]
    P = Paged(rng, [40], H=2, Hkv=2, D=8, B=16, dtype=F16, NB=64, tables=[tb])
    np.testing.assert_allclose(decode(*P.args()), P.brute(), rtol=0, atol=1e-12)

    t = golden["shared_prefix_tables"]["tables"]
    tables = [t["A"], t["B"], t["C"]]
    P = Paged(rng, [21, 21, 21], H=2, Hkv=1, D=8, B=16, dtype=F16, NB=64, tables=tables)
    for s in (1, 2):  # one shared prefix block: tokens 0..15 equal in all three
        P.K[s][:16] = P.K[0][:16]
        P.V[s][:16] = P.V[0][:16]
    P.K[1][:] = P.K[0]  # A and B also have equal private tails
    P.V[1][:] = P.V[0]
    P.q[1:] = P.q[0]
    P.build_pool()
    assert (P.kc[golden["shared_prefix_tables"]["shared_block"]] != CANARY[F16]).any()
    out = decode(*P.args())
    np.testing.assert_array_equal(out[0], out[1])
    assert np.abs(out[0] - out[2]).max() > 1e-3
    np.testing.assert_allclose(out, P.brute(), rtol=0, atol=1e-12)


def pin_block_grouping_b4(decode, golden):
    """B = 4: token 5 (1-based) is the first row of logical block 2 (k5 in K2)."""
    rng = np.random.default_rng(10)
    g = golden["block_grouping_b4"]
    assert g["tokens_1_based_by_logical_block"][1][0] == 5
    P = Paged(rng, [8], H=1, Hkv=1, D=64, B=4, dtype=F16, NB=6, tables=[[3, 1]])
    q = w(P.q[0, 0], F16)
    P.K[0][4, 0] = round_f32_to((6.0 * q).astype(np.float32), F16)
    P.build_pool()
    np.testing.assert_array_equal(P.kc[1, 0, 0], P.K[0][4, 0])
    np.testing.assert_allclose(decode(*P.args())[0, 0], w(P.V[0][4, 0], F16), rtol=0, atol=1e-9)


def pin_softmax_example(decode, golden):
    """The worked example's scores: the weights sum to 1 and follow the scores' order."""
    ex = golden["softmax_worked_example"]
    scores = np.array(ex["scores"])
    printed = np.array(ex["printed_weights"])
    n = len(scores)
    # q = e0, K[j] = (score_j, 0, ...), scale 1, V = identity rows: o is the weight vector
    q = np.zeros((1, 1, 8), dtype=np.uint16)
    q[0, 0, 0] = round_f32_to(np.float32([1.0]), F16)[0]
    kc = np.zeros((1, 1, 8, 8), dtype=np.uint16)
    vc = np.zeros((1, 1, 8, 8), dtype=np.uint16)
    kc[0, 0, :n, 0] = round_f32_to(scores.astype(np.float32), F16)
    for j in range(n):
        vc[0, 0, j, j] = round_f32_to(np.float32([1.0]), F16)[0]
    bt = np.zeros((1, 1), dtype=np.int32)
    cl = np.array([n], dtype=np.int32)
    wts = decode(q, kc, vc, bt, cl, 1.0, F16)[0, 0, :n]
    assert abs(wts.sum() - 1.0) < 1e-12 and abs(printed.sum() - 1.0) < 1e-9
    assert (np.argsort(wts) == np.argsort(scores)).all()
    assert (np.argsort(printed) == np.argsort(scores)).all()
    s16 = w(kc[0, 0, :n, 0], F16)
    e = [math.exp(x) for x in s16]
    np.testing.assert_allclose(wts, np.array(e) / sum(e), rtol=0, atol=1e-14)


def pin_empty_context(decode):
    """A context of 0 tokens gives an all-zero output; other sequences are unaffected."""
    rng = np.random.default_rng(11)
    P = Paged(rng, [0, 9], H=2, Hkv=1, D=16, B=16, dtype=F16)
    out = decode(*P.args())
    assert (out[0] == 0).all()
    np.testing.assert_allclose(out[1], P.brute()[1], rtol=0, atol=1e-12)


PINS = [pin_single_token, pin_identical_keys, pin_two_tokens, pin_dominant_key, pin_constant_values,
        pin_block_permutation, pin_gqa_is_repeated_mha, pin_paged_equals_bruteforce, pin_page_tables,
        pin_block_grouping_b4, pin_softmax_example, pin_empty_context]


def run_pin(pin, decode, golden):
    if pin.__code__.co_argcount == 2:
        pin(decode, golden)
    else:
        pin(decode)


def decode_c(q, kc, vc, bt, cl, scale, dtype):
    return oracle.decode_c(q, kc, vc, bt, cl, scale, dtype)


IMPLS = {"c": decode_c, "numpy": oracle.decode_np}


@pytest.mark.parametrize("impl", sorted(IMPLS))
@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_decode_pin(pin, impl, golden):
    run_pin(pin, IMPLS[impl], golden)


def test_c_and_numpy_agree_on_random_batches():
    """The two implementations agree on random batches (GQA, both dtypes, ragged contexts)."""
    rng = np.random.default_rng(12)
    for B, H, Hkv, D, dtype in [(16, 8, 2, 64, F16), (8, 6, 3, 128, BF16), (32, 4, 4, 64, BF16)]:
        P = Paged(rng, [0, 1, 31, 32, 33, 100], H=H, Hkv=Hkv, D=D, B=B, dtype=dtype)
        a = oracle.decode_c(*P.args())
        b = oracle.decode_np(*P.args())
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_c_pairs_and_threads():
    """Selected (seq, head) pairs and thread counts give the same rows as the full run."""
    rng = np.random.default_rng(13)
    P = Paged(rng, [5, 70, 18], H=4, Hkv=2, D=64, B=16, dtype=F16)
    full = oracle.decode_c(*P.args(), num_threads=1)
    pairs = [(2, 3), (0, 1), (1, 0)]
    part = oracle.decode_c(*P.args(), pairs=pairs, num_threads=3)
    for s, h in pairs:
        np.testing.assert_array_equal(part[s, h], full[s, h])
    assert (part[0, 0] == 0).all()


def test_widen_exact():
    """fp16/bf16 widening: C, numpy and struct agree on every fp16 pattern and a sweep of bf16 ones."""
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f16 = oracle.widen_np(allbits, F16)
    ref = np.array([widen_py(b, F16) for b in allbits])
    finite = np.isfinite(ref)
    np.testing.assert_array_equal(f16[finite], ref[finite])
    for b in (0x0001, 0x03FF, 0x0400, 0x3C00, 0x7BFF, 0x8001, 0xC000):
        assert oracle.widen_c(b, F16) == widen_py(b, F16)
    assert oracle.widen_c(0x0001, F16) == 2.0 ** -24
    assert oracle.widen_c(0x3C00, F16) == 1.0
    bf = oracle.widen_np(allbits[::97], BF16)
    refb = np.array([widen_py(b, BF16) for b in allbits[::97]])
    fin = np.isfinite(refb)
    np.testing.assert_array_equal(bf[fin], refb[fin])
    assert oracle.widen_c(0x3F80, BF16) == 1.0 and oracle.widen_c(0xC040, BF16) == -3.0


# ----------------------------------------------------------------------------
# the cache write


def test_write_block_42_example(golden):
    """The pages' example: a 6-token prompt fills slots 0..5 of physical block 42; the next token lands in slot 6."""
    ex = golden["block_42_example"]
    B, blk = ex["block_size"], ex["physical_block"]
    rng = np.random.default_rng(14)
    kc = np.full((64, 2, B, 8), CANARY[F16], dtype=np.uint16)
    vc = kc.copy()
    toks = round_f32_to(rng.standard_normal((7, 2, 8), dtype=np.float32), F16)
    vals = round_f32_to(rng.standard_normal((7, 2, 8), dtype=np.float32), F16)
    prompt = np.array([blk * B + s for s in ex["prompt_slots"]], dtype=np.int64)
    assert (len(prompt) + B - 1) // B == ex["blocks_for_prompt"]
    for impl in (oracle.write_c, oracle.write_np):
        k1, v1 = impl(kc, vc, toks[:6], vals[:6], prompt, B)
        nxt = np.array([blk * B + ex["next_token_offset"]], dtype=np.int64)
        assert nxt[0] == 678
        k2, v2 = impl(k1, v1, toks[6:], vals[6:], nxt, B)
        for j in range(7):
            np.testing.assert_array_equal(k2[blk, :, j, :], toks[j])
            np.testing.assert_array_equal(v2[blk, :, j, :], vals[j])
        touched = np.zeros(kc.shape, dtype=bool)
        touched[blk, :, :7, :] = True
        assert (k2[~touched] == CANARY[F16]).all() and (v2[~touched] == CANARY[F16]).all()


def test_write_skips_negative_and_rejects_out_of_range():
    rng = np.random.default_rng(15)
    kc = np.zeros((4, 1, 16, 8), dtype=np.uint16)
    vc = kc.copy()
    t = round_f32_to(rng.standard_normal((3, 1, 8), dtype=np.float32), F16)
    k, v = oracle.write_c(kc, vc, t, t, np.array([-1, 5, -7], dtype=np.int64), 16)
    assert (k[0, 0, 5] == t[1, 0]).all() and np.count_nonzero(k) == np.count_nonzero(t[1])
    for impl in (oracle.write_c, oracle.write_np):
        with pytest.raises(ValueError):
            impl(kc, vc, t, t, np.array([0, 64, 1], dtype=np.int64), 16)


def test_write_c_equals_numpy_random():
    rng = np.random.default_rng(16)
    for B, Hkv, D in [(16, 8, 128), (8, 3, 64), (32, 1, 64)]:
        NB = 20
        kc = rng.integers(0, 65536, size=(NB, Hkv, B, D), dtype=np.uint16)
        vc = rng.integers(0, 65536, size=(NB, Hkv, B, D), dtype=np.uint16)
        T = 25
        slots = rng.choice(NB * B, size=T, replace=False).astype(np.int64)
        slots[::7] = -1
        nk = rng.integers(0, 65536, size=(T, Hkv, D), dtype=np.uint16)
        nv = rng.integers(0, 65536, size=(T, Hkv, D), dtype=np.uint16)
        a = oracle.write_c(kc, vc, nk, nv, slots, B)
        b = oracle.write_np(kc, vc, nk, nv, slots, B)
        np.testing.assert_array_equal(a[0], b[0])
        np.testing.assert_array_equal(a[1], b[1])


# ----------------------------------------------------------------------------
# mutation check: plausible mistakes planted in a copy of the numpy oracle


def _mutant(kind):
    def decode(query, key_cache, value_cache, block_tables, context_lens, scale, dtype):
        S, H, D = query.shape
        Hkv, B = key_cache.shape[1], key_cache.shape[2]
        G = H // Hkv
        out = np.zeros((S, H, D))
        for s in range(S):
            ctx = int(context_lens[s])
            if kind == "ctx_off_by_one":
                ctx = max(ctx - 1, 0)
            for h in range(H):
                g = h % Hkv if kind == "gqa_modulo" else h // G
                j = np.arange(ctx)
                if kind == "ignore_table":
                    phys = j // B
                elif kind == "swap_block_offset":
                    phys = block_tables[s][np.minimum(j % B, block_tables.shape[1] - 1)]
                else:
                    phys = block_tables[s][j // B]
                off = j // B if kind == "swap_block_offset" else j % B
                phys = np.clip(phys, 0, key_cache.shape[0] - 1)
                K = oracle.widen_np(key_cache[phys, g, off % B, :], dtype)
                V = oracle.widen_np(value_cache[phys, g, off % B, :], dtype)
                if kind == "k_for_v":
                    V = K
                q = oracle.widen_np(query[s, h], dtype)
                if ctx == 0:
                    continue
                x = (1.0 if kind == "no_scale" else scale) * (K @ q)
                if kind == "wrong_sign":
                    x = -x
                e = np.exp(x - x.max())
                o = e @ V
                out[s, h] = o if kind == "no_normalise" else o / e.sum()
        return out

    return decode


MUTANTS = ["no_scale", "gqa_modulo", "k_for_v", "ctx_off_by_one", "no_normalise", "wrong_sign",
           "swap_block_offset", "ignore_table"]


@pytest.mark.parametrize("kind", MUTANTS)
def test_pins_catch_planted_mistake(kind, golden):
    dec = _mutant(kind)
    caught = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                run_pin(pin, dec, golden)
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {kind!r}"
