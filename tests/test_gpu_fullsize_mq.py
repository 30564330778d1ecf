"""The multi-query and shared-prefix calls at the bench's full sizes, in its launch configuration (the
library's automatic tile choice, the workspace from the size function, so the 128-row and 8-column tiles run
their sequences longest context first).

A sequence's output rows depend only on its own query rows, block-table row and context length, so the
oracle computes a few sampled sequences alone, over the same pool, and the GPU rows of those sequences, taken
from the full-batch call, must match them: |gpu - ref| <= 1e-2 + 1e-2 |ref|. The sample is the longest and
the shortest context and two seeded picks. The shared-prefix call is checked against the oracle's decode of
the whole batch (that oracle is fast at this size).

The FP8 lines run the same calls over E4M3 pools (k_scale = v_scale = 2^-6), the 16-bit pools encoded by
the oracle's encoder, so both sides read the same codes.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_91_gb300 import binding
from paged_kv_cache_91_gb300 import workloads as W
from test_gpu_fp8 import fp8_pools, to_dev_u8

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


def sample_seqs(ctx: np.ndarray, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    picks = {int(np.argmax(ctx)), int(np.argmin(ctx))} | set(rng.choice(len(ctx), size=2, replace=False).tolist())
    return np.array(sorted(picks))


# (workload, query tokens per sequence): the multi-query bench lines
CASES = [(2, 128), (3, 32), (2, 4), (3, 4)]
FP8_SCALE = 2.0 ** -6


@pytest.mark.parametrize("fp8", [False, True], ids=["16bit", "fp8"])
@pytest.mark.parametrize("cfg,ql", CASES)
def test_multi_query_bench_workload_sampled(cuda_lib, cfg, ql, fp8):
    batch = W.make_config(cfg, query_len=ql)
    t = W.as_torch(batch, DEV)
    qsl = batch.query_start_loc
    qlens = np.diff(qsl)
    binding.device_errors(clear=True)
    out = torch.empty_like(t["query"])
    if fp8:
        kc, vc = fp8_pools(batch, FP8_SCALE, FP8_SCALE)
        scales = {"k_scale": FP8_SCALE, "v_scale": FP8_SCALE}
        K, V = to_dev_u8(kc), to_dev_u8(vc)
        del t["key_cache"], t["value_cache"]
        binding.paged_attention_multi_query_fp8(out, t["query"], K, V, t["block_tables"], t["context_lens"],
                                                t["query_start_loc"], batch.scale, FP8_SCALE, FP8_SCALE,
                                                max_query_len=int(qlens.max()), max_context_len=batch.max_context_len)
        del K, V
    else:
        kc, vc, scales = batch.key_cache, batch.value_cache, {}
        binding.paged_attention_multi_query(out, t["query"], t["key_cache"], t["value_cache"], t["block_tables"],
                                            t["context_lens"], t["query_start_loc"], batch.scale,
                                            max_query_len=int(qlens.max()), max_context_len=batch.max_context_len)
    torch.cuda.synchronize()
    got = as_bits(out)
    del out, t
    sel = sample_seqs(batch.context_lens, 700 + cfg * 1000 + ql)
    rows = np.concatenate([np.arange(qsl[s], qsl[s + 1]) for s in sel])
    sub_qsl = np.concatenate([[0], np.cumsum(qlens[sel])]).astype(np.int32)
    ref = oracle.multi_query_c(batch.query[rows], kc, vc, batch.block_tables[sel], batch.context_lens[sel],
                               sub_qsl, batch.scale, batch.dtype, num_threads=os.cpu_count() or 1, **scales)
    what = f"workload {cfg}, q_len {ql}, {'fp8' if fp8 else '16-bit'}, sequences {sel.tolist()}"
    err = check_close(got[rows], ref, batch.dtype, what)
    assert binding.device_errors() == 0
    print(f"{what}: max abs err {err:.3e}")


@pytest.mark.parametrize("fp8", [False, True], ids=["16bit", "fp8"])
def test_shared_prefix_bench_workload(cuda_lib, fp8):
    """Workload 4 (128 sequences sharing a 1024-token prefix) through the shared-prefix call."""
    batch = W.make_config(4)
    t = W.as_torch(batch, DEV)
    pb, tails, lens = W.split_shared_prefix(batch, 1024)
    args = (torch.from_numpy(pb).to(DEV), 1024, torch.from_numpy(tails).to(DEV), torch.from_numpy(lens).to(DEV),
            batch.scale)
    binding.device_errors(clear=True)
    out = torch.empty_like(t["query"])
    if fp8:
        kc, vc = fp8_pools(batch, FP8_SCALE, FP8_SCALE)
        scales = {"k_scale": FP8_SCALE, "v_scale": FP8_SCALE}
        binding.paged_attention_decode_shared_prefix_fp8(out, t["query"], to_dev_u8(kc), to_dev_u8(vc), *args,
                                                         FP8_SCALE, FP8_SCALE, max_tail_len=int(lens.max()))
    else:
        kc, vc, scales = batch.key_cache, batch.value_cache, {}
        binding.paged_attention_decode_shared_prefix(out, t["query"], t["key_cache"], t["value_cache"], *args,
                                                     max_tail_len=int(lens.max()))
    torch.cuda.synchronize()
    ref = oracle.decode_c(batch.query, kc, vc, batch.block_tables, batch.context_lens, batch.scale, batch.dtype,
                          **scales)
    what = f"shared prefix, workload 4, {'fp8' if fp8 else '16-bit'}"
    err = check_close(as_bits(out), ref, batch.dtype, what)
    assert binding.device_errors() == 0
    print(f"{what}: max abs err {err:.3e}")
