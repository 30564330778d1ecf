"""paged_attention_decode_static_workspace, the decode call that allocates nothing.

Callers that cannot allocate device memory at call time (a plain C host with
no device allocator, a process whose device memory another allocator holds in
full, a decode loop that must not call cudaMalloc) use this entry point; its
split-K scratch is a fixed array inside the library. These tests call it
through the C ABI with ctypes and compare each output both with the fp64 CPU
oracle and with paged_attention_decode given an ordinary workspace, on two
calls in a row with different inputs, so a call that picked up the previous
call's scratch would show. Both decode paths are covered, since they lay the
scratch out differently.

The file name sorts last, so a run that stops at the first failure has run
every other test first.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_91_gb300 import binding
from paged_kv_cache_91_gb300 import workloads as W
from paged_kv_cache_91_gb300.workloads import BF16, F16

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
ATOL = RTOL = 1e-2
STATIC_BYTES = 32 * 1024 * 1024


def static_entry(lib):
    fn = lib.paged_attention_decode_static_workspace
    P, i32, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
    fn.restype = i32
    fn.argtypes = [P, P, P, P, P, i32, P, i32, i32, f32, i32, i32, i32, i32, i32, i32, i32, P]
    return fn


def call_static(fn, out, t, batch, max_context_len, partition_size):
    NB, Hkv, B, D = t["key_cache"].shape
    S, H, _ = t["query"].shape
    dt = 0 if batch.dtype == F16 else 1
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ptr = lambda x: ctypes.c_void_p(x.data_ptr())  # noqa: E731
    return fn(ptr(out), ptr(t["query"]), ptr(t["key_cache"]), ptr(t["value_cache"]), ptr(t["block_tables"]),
              t["block_tables"].shape[1], ptr(t["context_lens"]), S, max_context_len, batch.scale, B, H, Hkv, D, NB,
              dt, partition_size, stream)


def as_f64(x: torch.Tensor) -> np.ndarray:
    return x.detach().to(torch.float64).cpu().numpy()


CASES = [
    dict(seed=51, context_lens=[3000, 100, 1700, 513], num_heads=40, num_kv_heads=40, dtype=F16, P=512),
    dict(seed=52, context_lens=[2049, 4096, 7, 1200, 900], num_heads=32, num_kv_heads=8, dtype=BF16, P=256),
]


def run_two_calls(fn):
    """Two back-to-back calls with different shapes; each compared with the oracle and with the decode call
    on a workspace of its own."""
    for c in CASES:
        batch = W.build_batch(seed=c["seed"], context_lens=c["context_lens"], num_heads=c["num_heads"],
                              num_kv_heads=c["num_kv_heads"], head_dim=128, block_size=16, dtype=c["dtype"],
                              pool_factor=1.2)
        mcl = batch.max_context_len
        need = binding.paged_attention_workspace_size(batch.num_seqs, batch.num_heads, batch.num_kv_heads, 128, 16,
                                                      mcl, c["P"])
        assert 0 < need <= STATIC_BYTES  # the case exercises the split-K scratch
        t = W.as_torch(batch, DEV)
        ref = torch.empty_like(t["query"])
        binding.paged_attention_decode(ref, t["query"], t["key_cache"], t["value_cache"], t["block_tables"],
                                       t["context_lens"], batch.scale, max_context_len=mcl,
                                       partition_size=c["P"])
        got = torch.full_like(t["query"], float("nan"))
        assert call_static(fn, got, t, batch, mcl, c["P"]) == 0
        torch.cuda.synchronize()
        r, g = as_f64(ref), as_f64(got)
        assert np.isfinite(g).all()
        assert (np.abs(g - r) <= ATOL + RTOL * np.abs(r)).all(), np.abs(g - r).max()
        want = oracle.decode_c(batch.query, batch.key_cache, batch.value_cache, batch.block_tables,
                               batch.context_lens, batch.scale, batch.dtype)
        err = np.abs(g - want)
        assert (err <= ATOL + RTOL * np.abs(want)).all(), err.max()
    assert binding.device_errors() == 0


def test_static_workspace_matches_oracle_and_decode_on_two_calls(cuda_lib):
    run_two_calls(static_entry(binding.load()))


def test_static_workspace_reports_bad_arguments_before_the_size(cuda_lib):
    """An oversize call with a bad argument gets that argument's error, not PKV_ERR_WORKSPACE."""
    lib = binding.load()
    fn = static_entry(lib)
    S, H, D, mcl, P = 3000, 64, 128, 32768, 512
    fake = ctypes.c_void_p(0x10000)
    assert fn(fake, fake, fake, fake, fake, mcl // 16, fake, S, mcl, 0.1, 16, H, H, D, 2048, 7, P, None) == -1
    assert "dtype" in lib.pkv_last_error_message().decode()
    assert fn(fake, fake, fake, fake, fake, mcl // 16, fake, S, mcl, 0.1, 16, H, H, 96, 2048, 0, P, None) == -2
    assert "head_dim" in lib.pkv_last_error_message().decode()
    assert fn(fake, fake, fake, fake, fake, mcl // 16, fake, S, mcl, 0.1, 16, H, H, D, 2048, 0, 24, None) == -2
    assert "partition_size" in lib.pkv_last_error_message().decode()


def test_static_workspace_rejects_oversize_requests(cuda_lib):
    lib = binding.load()
    fn = static_entry(lib)
    S, H, D, mcl, P = 3000, 64, 128, 32768, 512  # 3000 x 64 heads x 64 partitions of partials
    need = binding.paged_attention_workspace_size(S, H, H, D, 16, mcl, P)
    assert need > STATIC_BYTES
    fake = ctypes.c_void_p(0x10000)
    st = fn(fake, fake, fake, fake, fake, mcl // 16, fake, S, mcl, 0.1, 16, H, H, D, 2048, 0, P, None)
    assert st == -3  # PKV_ERR_WORKSPACE, before any CUDA call
    msg = lib.pkv_last_error_message().decode()
    assert str(need) in msg and str(STATIC_BYTES) in msg
