"""Paged KV cache decode attention for GB300 (sm_103a).

The CUDA library (``libpaged_kv.so``, C ABI in ``include/paged_kv.h``) does the
work; ``binding`` marshals torch tensors into its calls. Importing this package
does not load the library; the first call does, and fails loudly if it is
missing.
"""
from .binding import (  # noqa: F401
    PagedKVError,
    paged_attention_decode,
    paged_attention_decode_fp8,
    paged_attention_decode_shared_prefix,
    paged_attention_decode_shared_prefix_fp8,
    paged_attention_multi_query,
    paged_attention_multi_query_fp8,
    paged_attention_multi_query_workspace_size,
    paged_attention_shared_prefix_workspace_size,
    paged_attention_workspace_size,
    paged_attention_workspace_size_fp8,
    paged_kv_copy_blocks,
    paged_kv_write,
    paged_kv_write_fp8,
)
