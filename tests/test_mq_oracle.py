"""Pins for the multi-query oracle (several query tokens per sequence, causal)."""
import math

import numpy as np
import pytest

import oracle
from paged_kv_cache_91_gb300 import workloads as W
from paged_kv_cache_91_gb300.workloads import BF16, F16


def mq_case(seed, ctx, q_lens, H=4, Hkv=2, D=32, B=8, dtype=F16):
    batch = W.build_batch(seed=seed, context_lens=ctx, num_heads=H, num_kv_heads=Hkv, head_dim=D,
                          block_size=B, dtype=dtype, pool_factor=1.5)
    rng = np.random.default_rng(seed + 1)
    qsl = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q = W.round_f32_to(rng.standard_normal((int(qsl[-1]), H, D), dtype=np.float32), dtype)
    return batch, q, qsl


def test_single_query_token_is_decode():
    batch, _, _ = mq_case(11, [1, 9, 40, 17], [1, 1, 1, 1])
    qsl = np.arange(5, dtype=np.int32)
    want = oracle.decode_c(batch.query, batch.key_cache, batch.value_cache, batch.block_tables,
                           batch.context_lens, batch.scale, batch.dtype)
    for impl in (oracle.multi_query_c, oracle.multi_query_np):
        got = impl(batch.query, batch.key_cache, batch.value_cache, batch.block_tables, batch.context_lens,
                   qsl, batch.scale, batch.dtype)
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_each_query_token_is_decode_over_its_causal_prefix(dtype):
    """Query token i of a sequence with q_len tokens equals a decode whose context ends at its own
    position ctx - q_len + i (the decode oracle is pinned separately)."""
    ctx, q_lens = [5, 23, 40, 8, 16], [5, 3, 7, 0, 1]
    batch, q, qsl = mq_case(12, ctx, q_lens, dtype=dtype)
    got_c = oracle.multi_query_c(q, batch.key_cache, batch.value_cache, batch.block_tables, batch.context_lens,
                                 qsl, batch.scale, dtype)
    got_np = oracle.multi_query_np(q, batch.key_cache, batch.value_cache, batch.block_tables,
                                   batch.context_lens, qsl, batch.scale, dtype)
    np.testing.assert_allclose(got_c, got_np, rtol=0, atol=1e-12)
    for s, (c, n) in enumerate(zip(ctx, q_lens)):
        for i in range(n):
            row = qsl[s] + i
            want = oracle.decode_c(q[row:row + 1], batch.key_cache, batch.value_cache, batch.block_tables[s:s + 1],
                                   np.array([c - n + i + 1], np.int32), batch.scale, dtype)
            np.testing.assert_allclose(got_c[row], want[0], rtol=0, atol=1e-12)


def causal_bruteforce(qf, Kf, Vf, scale):
    """o_i = sum_{j <= i} softmax_j(scale q_i . k_j) v_j with plain loops (whole prefix as queries)."""
    n, D = Kf.shape
    out = np.zeros((n, D))
    for i in range(n):
        xs = [scale * sum(qf[i][d] * Kf[j][d] for d in range(D)) for j in range(i + 1)]
        m = max(xs)
        ws = [math.exp(x - m) for x in xs]
        tot = sum(ws)
        for j in range(i + 1):
            for d in range(D):
                out[i][d] += ws[j] / tot * Vf[j][d]
    return out


def test_whole_prompt_as_queries_is_causal_self_attention():
    """q_len = ctx (a prefill of the whole prompt) gives causal attention over the contiguous sequence."""
    ctx = [11, 6]
    batch, q, qsl = mq_case(13, ctx, ctx, H=2, Hkv=1, D=8, B=4)
    got = oracle.multi_query_c(q, batch.key_cache, batch.value_cache, batch.block_tables, batch.context_lens,
                               qsl, batch.scale, F16)
    for s, c in enumerate(ctx):
        for h in range(2):
            Kf = oracle.widen_np(oracle.gather_np(batch.key_cache, batch.block_tables[s], c, 0, 4), F16)
            Vf = oracle.widen_np(oracle.gather_np(batch.value_cache, batch.block_tables[s], c, 0, 4), F16)
            qf = oracle.widen_np(q[qsl[s]:qsl[s + 1], h], F16)
            np.testing.assert_allclose(got[qsl[s]:qsl[s + 1], h], causal_bruteforce(qf, Kf, Vf, batch.scale),
                                       rtol=1e-12, atol=1e-13)
    # the first token attends only itself: o_0 = v_0
    v0 = oracle.widen_np(oracle.gather_np(batch.value_cache, batch.block_tables[0], 1, 0, 4), F16)[0]
    np.testing.assert_array_equal(got[0, 0], v0)


def test_bad_query_count_is_rejected():
    batch, q, _ = mq_case(14, [4, 4], [2, 2])
    for impl in (oracle.multi_query_c, oracle.multi_query_np):
        with pytest.raises((ValueError, AssertionError)):
            impl(np.zeros((7, 4, 32), np.uint16), batch.key_cache, batch.value_cache, batch.block_tables,
                 batch.context_lens, np.array([0, 5, 7], np.int32), batch.scale, F16)


def test_pins_catch_planted_mistakes():
    """Plausible slips in a copy of the numpy oracle each fail the causal-prefix pin."""
    ctx, q_lens = [9, 30], [4, 6]
    batch, q, qsl = mq_case(15, ctx, q_lens)
    ref = oracle.multi_query_c(q, batch.key_cache, batch.value_cache, batch.block_tables, batch.context_lens,
                               qsl, batch.scale, F16)
    B, group = batch.block_size, batch.num_heads // batch.num_kv_heads

    def mutant(limit):
        out = np.zeros_like(ref)
        for s, c in enumerate(ctx):
            for h in range(batch.num_heads):
                K = oracle.widen_np(oracle.gather_np(batch.key_cache, batch.block_tables[s], c, h // group, B), F16)
                V = oracle.widen_np(oracle.gather_np(batch.value_cache, batch.block_tables[s], c, h // group, B), F16)
                for i in range(q_lens[s]):
                    n = limit(c, q_lens[s], i)
                    out[qsl[s] + i, h] = oracle.attention_np(oracle.widen_np(q[qsl[s] + i, h], F16), K[:n], V[:n],
                                                             batch.scale)
        return out

    for name, limit in [("not causal", lambda c, n, i: c),
                        ("excludes itself", lambda c, n, i: c - n + i),
                        ("counts from the start", lambda c, n, i: i + 1),
                        ("one too many", lambda c, n, i: min(c, c - n + i + 2))]:
        assert np.abs(mutant(limit) - ref).max() > 1e-6, name
