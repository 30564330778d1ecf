// CUDA-core decode over an FP8 (E4M3) KV cache: f16 and bf16 queries.
#include "pkv_decode_simt.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

template <typename T>
cudaError_t dispatch(const DecodeParams& p, int head_dim, int block_size, int num_seqs, cudaStream_t stream) {
  using C = __nv_fp8_e4m3;
  if (head_dim == 128) {
    if (block_size == 16) return launch_decode_simt<T, 128, 16, C>(p, num_seqs, stream);
    if (block_size == 8) return launch_decode_simt<T, 128, 8, C>(p, num_seqs, stream);
    if (block_size == 32) return launch_decode_simt<T, 128, 32, C>(p, num_seqs, stream);
  } else if (head_dim == 64) {
    if (block_size == 16) return launch_decode_simt<T, 64, 16, C>(p, num_seqs, stream);
    if (block_size == 8) return launch_decode_simt<T, 64, 8, C>(p, num_seqs, stream);
    if (block_size == 32) return launch_decode_simt<T, 64, 32, C>(p, num_seqs, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t decode_simt_fp8_f16(const DecodeParams& p, int head_dim, int block_size, int num_seqs,
                                cudaStream_t stream) {
  return dispatch<__half>(p, head_dim, block_size, num_seqs, stream);
}

cudaError_t decode_simt_fp8_bf16(const DecodeParams& p, int head_dim, int block_size, int num_seqs,
                                 cudaStream_t stream) {
  return dispatch<__nv_bfloat16>(p, head_dim, block_size, num_seqs, stream);
}

}  // namespace pkv
