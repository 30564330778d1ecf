"""The C ABI without a GPU: the library builds, loads, exports every symbol the
header declares, sizes workspaces, and rejects bad arguments on the host
before any CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "paged_kv.h")

OK, INVALID, UNSUPPORTED, WORKSPACE = 0, -1, -2, -3


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_91_gb300 import build as b
    from paged_kv_cache_91_gb300 import binding

    b.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:pkv_status_t|size_t|int32_t|const char\s*\*)\s*(\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("paged_kv_write", "paged_attention_decode", "paged_attention_workspace_size",
              "paged_kv_device_errors", "pkv_status_string", "pkv_last_error_message",
              "pkv_selftest_wait_timeout", "paged_attention_decode_static_workspace", "paged_kv_copy_blocks",
              "paged_kv_write_fp8", "paged_attention_decode_fp8", "paged_attention_workspace_size_fp8",
              "paged_attention_multi_query", "paged_attention_multi_query_workspace_size",
              "paged_attention_multi_query_fp8", "paged_attention_decode_shared_prefix_fp8",
              "pkv_set_multi_query_tile", "pkv_read_chunks"):
        assert n in names


def test_exports_every_declared_symbol(lib):
    from paged_kv_cache_91_gb300 import binding

    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for n in declared_functions():
        assert n in exported, n
        assert hasattr(lib, n)


def test_status_strings(lib):
    assert lib.pkv_status_string(0) == b"PKV_OK"
    assert lib.pkv_status_string(-3) == b"PKV_ERR_WORKSPACE"
    assert lib.pkv_status_string(7) == b"PKV_UNKNOWN_STATUS"


def test_workspace_size(lib):
    ws = lib.paged_attention_workspace_size
    assert ws(64, 40, 40, 128, 16, 512, 512) == 0  # one partition: no workspace
    assert ws(64, 40, 40, 128, 16, 513, 512) == 64 * 40 * 2 * 130 * 4
    assert ws(16, 40, 40, 128, 16, 32768, 0) == 16 * 40 * 16 * 130 * 4  # 0 selects 2048 above 8192 tokens
    assert ws(16, 40, 40, 128, 8, 32768, 0) == 16 * 40 * 32 * 130 * 4  # at most 128 blocks: 1024 for blocks of 8
    assert ws(16, 40, 40, 128, 16, 8192, 0) == 16 * 40 * 8 * 130 * 4  # 8192 and below: 1024
    assert ws(256, 32, 8, 128, 16, 8192, 0) == 256 * 32 * 8 * 130 * 4
    assert ws(3000, 8, 8, 64, 16, 4096, 0) == 3000 * 8 * 4 * 66 * 4
    assert ws(64, 40, 40, 128, 16, 1024, 0) == 0 and ws(64, 40, 40, 128, 16, 1025, 0) == 64 * 40 * 2 * 130 * 4
    assert ws(0, 40, 40, 128, 16, 4096, 0) == 0 and ws(4, 40, 40, 128, 16, -1, 0) == 0


P = ctypes.c_void_p


def fake(n=1):
    """A non-null, 256-byte aligned address that is never dereferenced on the host path."""
    return P(0x10000 * n)


def decode(lib, **kw):
    a = dict(out=fake(1), query=fake(2), key_cache=fake(3), value_cache=fake(4), block_tables=fake(5),
             max_blocks_per_seq=8, context_lens=fake(6), num_seqs=2, max_context_len=128, scale=0.125,
             block_size=16, num_heads=4, num_kv_heads=4, head_dim=64, num_blocks=16, dtype=0,
             partition_size=0, workspace=None, workspace_bytes=0, stream=None)
    a.update(kw)
    return lib.paged_attention_decode(*a.values())


@pytest.mark.parametrize("kw,status", [
    (dict(out=None), INVALID),
    (dict(num_seqs=-1), INVALID),
    (dict(num_heads=6, num_kv_heads=4), INVALID),
    (dict(num_kv_heads=0), INVALID),
    (dict(head_dim=96), UNSUPPORTED),
    (dict(block_size=12), UNSUPPORTED),
    (dict(dtype=5), INVALID),
    (dict(scale=float("nan")), INVALID),
    (dict(max_context_len=129), INVALID),           # > max_blocks_per_seq * block_size
    (dict(partition_size=24), UNSUPPORTED),          # not a multiple of block_size
    (dict(partition_size=16 * 129), UNSUPPORTED),    # more blocks than the kernel keeps per partition
    (dict(query=P(0x10008)), INVALID),               # misaligned
    (dict(max_blocks_per_seq=128, max_context_len=2048), WORKSPACE),   # split needs a workspace
    (dict(max_blocks_per_seq=128, max_context_len=2048, workspace=fake(9), workspace_bytes=100), WORKSPACE),
    (dict(max_blocks_per_seq=64, max_context_len=1024, partition_size=512), WORKSPACE),
    (dict(num_seqs=70000), UNSUPPORTED),
])
def test_decode_rejects_on_host(lib, kw, status):
    assert decode(lib, **kw) == status
    assert lib.pkv_last_error_message() != b""


def test_decode_empty_batch_is_a_noop(lib):
    assert decode(lib, num_seqs=0, out=None, query=None) == OK


def write(lib, **kw):
    a = dict(key=fake(1), value=fake(2), key_cache=fake(3), value_cache=fake(4), slot_mapping=fake(5),
             num_tokens=4, num_kv_heads=2, head_dim=128, block_size=16, num_blocks=8, dtype=1, stream=None)
    a.update(kw)
    return lib.paged_kv_write(*a.values())


@pytest.mark.parametrize("kw,status", [
    (dict(key=None), INVALID),
    (dict(slot_mapping=None), INVALID),
    (dict(num_tokens=-2), INVALID),
    (dict(head_dim=80), UNSUPPORTED),
    (dict(block_size=64), UNSUPPORTED),
    (dict(num_blocks=0), INVALID),
    (dict(key_cache=P(0x30004)), INVALID),
    (dict(dtype=2), INVALID),
])
def test_write_rejects_on_host(lib, kw, status):
    assert write(lib, **kw) == status


def test_write_zero_tokens_is_a_noop(lib):
    assert write(lib, num_tokens=0, key=None) == OK


def test_binding_refuses_cpu_tensors(lib):
    import torch

    from paged_kv_cache_91_gb300 import binding

    x = torch.zeros(2, 4, 64, dtype=torch.float16)
    kc = torch.zeros(4, 4, 16, 64, dtype=torch.float16)
    with pytest.raises(binding.PagedKVError):
        binding.paged_attention_decode(x, x, kc, kc, torch.zeros(2, 1, dtype=torch.int32),
                                       torch.zeros(2, dtype=torch.int32), 0.125)


def test_package_does_not_import_the_oracle():
    """The product package and its sources never reference the oracle."""
    pkg = os.path.join(ROOT, "paged_kv_cache_91_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", src, flags=re.M), f
                assert "liboracle" not in src and "pkv_oracle" not in src, f


def test_fp8_workspace_size(lib):
    ws8 = lib.paged_attention_workspace_size_fp8
    assert ws8(64, 40, 40, 128, 16, 513, 512) == 64 * 40 * 2 * 130 * 4
    assert ws8(256, 32, 8, 128, 16, 8192, 0) == 256 * 32 * 8 * 130 * 4  # 0 selects 1024 for FP8
    assert ws8(256, 32, 8, 128, 16, 1024, 0) == 0
    assert ws8(64, 40, 40, 128, 16, 512, 512) == 0
    assert ws8(0, 40, 40, 128, 16, 4096, 0) == 0


def decode_fp8(lib, **kw):
    a = dict(out=fake(1), query=fake(2), key_cache=fake(3), value_cache=fake(4), block_tables=fake(5),
             max_blocks_per_seq=8, context_lens=fake(6), num_seqs=2, max_context_len=128, scale=0.125,
             block_size=16, num_heads=4, num_kv_heads=4, head_dim=64, num_blocks=16, dtype=0,
             k_scale=0.5, v_scale=0.25, partition_size=0, workspace=None, workspace_bytes=0, stream=None)
    a.update(kw)
    return lib.paged_attention_decode_fp8(*a.values())


@pytest.mark.parametrize("kw,status", [
    (dict(k_scale=0.0), INVALID),
    (dict(v_scale=-1.0), INVALID),
    (dict(k_scale=float("inf")), INVALID),
    (dict(v_scale=float("nan")), INVALID),
    (dict(dtype=2), INVALID),                        # the query cannot be FP8
    (dict(head_dim=96), UNSUPPORTED),
    (dict(out=None), INVALID),
    (dict(max_blocks_per_seq=65, max_context_len=1025), WORKSPACE),  # > 1024 (the FP8 default partition)
])
def test_decode_fp8_rejects_on_host(lib, kw, status):
    assert decode_fp8(lib, **kw) == status
    assert lib.pkv_last_error_message() != b""


def write_fp8(lib, **kw):
    a = dict(key=fake(1), value=fake(2), key_cache=fake(3), value_cache=fake(4), slot_mapping=fake(5),
             num_tokens=4, num_kv_heads=2, head_dim=128, block_size=16, num_blocks=8, dtype=1, k_scale=1.0,
             v_scale=1.0, stream=None)
    a.update(kw)
    return lib.paged_kv_write_fp8(*a.values())


@pytest.mark.parametrize("kw,status", [
    (dict(k_scale=0.0), INVALID),
    (dict(v_scale=float("inf")), INVALID),
    (dict(dtype=2), INVALID),
    (dict(key=None), INVALID),
    (dict(block_size=4), UNSUPPORTED),
    (dict(value_cache=P(0x40001)), INVALID),
])
def test_write_fp8_rejects_on_host(lib, kw, status):
    assert write_fp8(lib, **kw) == status


def test_fp8_zero_work_is_a_noop(lib):
    assert write_fp8(lib, num_tokens=0, key=None) == OK
    assert decode_fp8(lib, num_seqs=0, out=None) == OK


def test_multi_query_workspace_size(lib):
    ws = lib.paged_attention_multi_query_workspace_size
    order = 512  # room for the sequence order: 100 int32, rounded up to 256 bytes
    assert ws(100, 32, 8, 128, 16, 512, 512) == order  # one partition: no partials
    assert ws(100, 32, 8, 128, 16, 513, 512) == 100 * 32 * 2 * 130 * 4 + order
    assert ws(100, 32, 8, 128, 16, 2048, 0) == order  # 0 selects 2048 tokens
    assert ws(100, 32, 8, 128, 8, 2048, 0) == 100 * 32 * 2 * 130 * 4 + order  # capped at 128 blocks of 8
    assert ws(7, 4, 4, 64, 16, 2048, 256) == 7 * 4 * 8 * 66 * 4 + 256
    assert ws(0, 4, 4, 64, 16, 2048, 256) == 0
    assert ws(-1, 4, 4, 64, 16, 2048, 256) == 0


def multi_query(lib, **kw):
    a = dict(out=fake(1), query=fake(2), key_cache=fake(3), value_cache=fake(4), block_tables=fake(5),
             max_blocks_per_seq=8, context_lens=fake(6), query_start_loc=fake(7), num_seqs=2, num_query_tokens=5,
             max_query_len=4, max_context_len=128, scale=0.125, block_size=16, num_heads=8, num_kv_heads=2,
             head_dim=64, num_blocks=16, dtype=0, partition_size=0, workspace=None, workspace_bytes=0, stream=None)
    a.update(kw)
    return lib.paged_attention_multi_query(*a.values())


@pytest.mark.parametrize("kw,status", [
    (dict(query_start_loc=None), INVALID),
    (dict(num_query_tokens=-1), INVALID),
    (dict(max_query_len=-3), INVALID),
    (dict(max_query_len=129), INVALID),                # more query tokens than the context can hold
    (dict(num_heads=7), INVALID),
    (dict(head_dim=80), UNSUPPORTED),
    (dict(dtype=2), INVALID),
    (dict(max_context_len=129), INVALID),
    (dict(partition_size=20), UNSUPPORTED),
    (dict(num_kv_heads=1, num_heads=64, max_query_len=128, max_blocks_per_seq=64, max_context_len=1024,
          num_query_tokens=1 << 26), UNSUPPORTED),  # too many rows
    (dict(max_blocks_per_seq=200, max_context_len=3000), WORKSPACE),
])
def test_multi_query_rejects_on_host(lib, kw, status):
    assert multi_query(lib, **kw) == status
    assert lib.pkv_last_error_message() != b""


def test_multi_query_nothing_to_do_is_a_noop(lib):
    assert multi_query(lib, num_seqs=0, out=None) == OK
    assert multi_query(lib, num_query_tokens=0, out=None) == OK
    assert multi_query(lib, max_query_len=0, out=None) == OK


def multi_query_fp8(lib, **kw):
    a = dict(out=fake(1), query=fake(2), key_cache=fake(3), value_cache=fake(4), block_tables=fake(5),
             max_blocks_per_seq=8, context_lens=fake(6), query_start_loc=fake(7), num_seqs=2, num_query_tokens=5,
             max_query_len=4, max_context_len=128, scale=0.125, block_size=16, num_heads=8, num_kv_heads=2,
             head_dim=128, num_blocks=16, dtype=0, k_scale=0.5, v_scale=0.25, partition_size=0, workspace=None,
             workspace_bytes=0, stream=None)
    a.update(kw)
    return lib.paged_attention_multi_query_fp8(*a.values())


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=64), UNSUPPORTED),                  # the E4M3 tile is head_dim 128
    (dict(k_scale=0.0), INVALID),
    (dict(v_scale=-1.0), INVALID),
    (dict(k_scale=float("inf")), INVALID),
    (dict(dtype=2), INVALID),                          # the query dtype: f16 or bf16
    (dict(query_start_loc=None), INVALID),
    (dict(max_query_len=129), INVALID),
    (dict(max_blocks_per_seq=200, max_context_len=3000), WORKSPACE),
])
def test_multi_query_fp8_rejects_on_host(lib, kw, status):
    assert multi_query_fp8(lib, **kw) == status
    assert lib.pkv_last_error_message() != b""


def test_multi_query_fp8_nothing_to_do_is_a_noop(lib):
    assert multi_query_fp8(lib, num_seqs=0, out=None) == OK
    assert multi_query_fp8(lib, num_query_tokens=0, out=None) == OK


def test_multi_query_tile_switch(lib):
    prev = lib.pkv_set_multi_query_tile(2)
    try:
        assert lib.pkv_set_multi_query_tile(1) == 2
        assert lib.pkv_set_multi_query_tile(9) == -1
        assert lib.pkv_set_multi_query_tile(3) == 1  # the tensor-memory tile
        assert lib.pkv_set_multi_query_tile(4) == 3  # the FP8 16-row pairs
        assert lib.pkv_set_multi_query_tile(0) == 4
    finally:
        lib.pkv_set_multi_query_tile(prev)


def test_binding_constants_match_the_header():
    """The binding's dtype, decode-path, tile and device-error constants are the header's values."""
    from paged_kv_cache_91_gb300 import binding

    with open(HEADER) as f:
        text = f.read()
    defines = {m[0]: int(m[1]) for m in re.findall(r"^#define PKV_(\w+) (\d+)u?\b", text, flags=re.M)}
    enum = {m[0]: int(m[1]) for m in re.findall(r"PKV_(F16|BF16|FP8_E4M3) = (\d+)", text)}
    assert enum == {"F16": binding.PKV_F16, "BF16": binding.PKV_BF16, "FP8_E4M3": binding.PKV_FP8_E4M3}
    for name in ("AUTO", "COLUMNS", "ROWS", "TENSOR", "PAIRS"):
        assert defines[f"MQ_TILE_{name}"] == getattr(binding, f"MQ_TILE_{name}")
    header_bits = {v: k[len("DEVERR_"):] for k, v in defines.items() if k.startswith("DEVERR_")}
    assert header_bits == binding.DEVERR_BITS


def test_read_chunks_host_checks(lib):
    """The read helper rejects bad chunk sizes and null or unaligned pointers before any CUDA call."""
    import ctypes

    fn = lib.pkv_read_chunks
    fn.restype = ctypes.c_int32
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p]
    fake = 0x10000
    assert fn(fake, 1 << 20, fake, 16, 3000, None) == -2
    assert fn(None, 1 << 20, fake, 16, 2048, None) == -1
    assert fn(fake + 8, 1 << 20, fake, 16, 2048, None) == -1
    assert fn(fake, 1 << 20, fake, -1, 2048, None) == -1
    assert fn(fake, 1 << 20, fake, 0, 2048, None) == 0  # nothing to read
