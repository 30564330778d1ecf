// Tensor-core decode over an FP8 (E4M3) KV cache: f16 and bf16 queries, head_dim 128.
#include "pkv_decode_mma_fp8.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

template <typename T>
cudaError_t dispatch(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap, int head_dim,
                     int block_size, int num_seqs, cudaStream_t stream) {
  constexpr int R = PKV_MMA_FP8_RING_BYTES;
  if (head_dim == 128) {
    if (block_size == 16) return launch_decode_gqa_mma<MmaTileE4M3<T, 128, 16>, R>(p, kmap, vmap, num_seqs, stream);
    if (block_size == 8) return launch_decode_gqa_mma<MmaTileE4M3<T, 128, 8>, R>(p, kmap, vmap, num_seqs, stream);
    if (block_size == 32) return launch_decode_gqa_mma<MmaTileE4M3<T, 128, 32>, R>(p, kmap, vmap, num_seqs, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t decode_mma_fp8_f16(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                               int head_dim, int block_size, int num_seqs, cudaStream_t stream) {
  return dispatch<__half>(p, kmap, vmap, head_dim, block_size, num_seqs, stream);
}

cudaError_t decode_mma_fp8_bf16(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                int head_dim, int block_size, int num_seqs, cudaStream_t stream) {
  return dispatch<__nv_bfloat16>(p, kmap, vmap, head_dim, block_size, num_seqs, stream);
}

}  // namespace pkv
