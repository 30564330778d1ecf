// paged_attention_decode_static_workspace: the decode call for callers that
// cannot allocate device memory at call time.
//
// Who needs it: a plain C host that has no device allocator of its own; a
// process whose device memory another allocator has already reserved in full
// (a fresh cudaMalloc would fail); a latency-bound decode loop that must not
// call cudaMalloc (it can synchronise the device). paged_attention_decode asks
// such callers for a split-K workspace they cannot provide; this entry point
// uses a fixed scratch array that lives in the library instead.
//
// The scratch is a file-scope __device__ array of PKV_STATIC_WORKSPACE_BYTES.
// Every GPU that loads the library holds it until the process exits. In host
// code the array's name is only a host-side stand-in, so the device address is
// looked up once per device with cudaGetSymbolAddress, with that device current,
// on the first call made on that device, and kept for the life of the process.
#include <stdio.h>

#include <atomic>

#include "paged_kv.h"
#include "pkv_internal.h"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_workspace[PKV_STATIC_WORKSPACE_BYTES];

}  // namespace

extern "C" pkv_status_t paged_attention_decode_static_workspace(
    void* out, const void* query, const void* key_cache, const void* value_cache, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs, int32_t max_context_len,
    float scale, int32_t block_size, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t num_blocks, pkv_dtype_t dtype, int32_t partition_size, cudaStream_t stream) {
  // Device addresses of the scratch array, one per device ordinal, looked up once and kept for the life of
  // the process. Atomic: two host threads may make their first calls at the same time (both store the
  // same address).
  static std::atomic<void*> device_ptr[kMaxDevices];
  char msg[256];
  const size_t need =
      paged_attention_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_context_len,
                                     partition_size);
  if (need > PKV_STATIC_WORKSPACE_BYTES) {
    // The arguments are validated first, so that a bad dtype, head_dim or partition size reports its own
    // error: paged_attention_decode checks every argument before it looks at the workspace, and with no
    // workspace for a call that needs one it returns PKV_ERR_WORKSPACE without launching anything.
    const pkv_status_t st =
        paged_attention_decode(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq, context_lens,
                               num_seqs, max_context_len, scale, block_size, num_heads, num_kv_heads, head_dim,
                               num_blocks, dtype, partition_size, nullptr, 0, stream);
    if (st != PKV_ERR_WORKSPACE) return st;
    snprintf(msg, sizeof msg,
             "split-K scratch of %zu bytes exceeds the static workspace of %u bytes; "
             "use paged_attention_decode with a caller workspace",
             need, (unsigned)PKV_STATIC_WORKSPACE_BYTES);
    pkv::set_last_error_message(msg);
    return PKV_ERR_WORKSPACE;
  }
  // set-up, once per device: the scratch array's device address on the current device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    snprintf(msg, sizeof msg, "cudaGetDevice: %s", cudaGetErrorString(e));
    pkv::set_last_error_message(msg);
    return PKV_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    pkv::set_last_error_message("device ordinal outside the supported range");
    return PKV_ERR_UNSUPPORTED;
  }
  void* scratch = device_ptr[dev].load(std::memory_order_relaxed);
  if (!scratch) {
    e = cudaGetSymbolAddress(&scratch, g_static_workspace);
    if (e != cudaSuccess || !scratch) {
      snprintf(msg, sizeof msg, "cudaGetSymbolAddress of the static workspace: %s", cudaGetErrorString(e));
      pkv::set_last_error_message(msg);
      return PKV_ERR_CUDA;
    }
    device_ptr[dev].store(scratch, std::memory_order_relaxed);
  }
  // Nothing in the scratch needs clearing: the decode kernel writes every
  // partition's (m, l, o) before the reduce kernel reads it.
  return paged_attention_decode(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                                context_lens, num_seqs, max_context_len, scale, block_size, num_heads,
                                num_kv_heads, head_dim, num_blocks, dtype, partition_size, scratch,
                                (size_t)PKV_STATIC_WORKSPACE_BYTES, stream);
}
