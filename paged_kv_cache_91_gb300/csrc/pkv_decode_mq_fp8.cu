// Multi-query paged attention over an FP8 (E4M3) KV pool, f16 and bf16 queries, head_dim 128: the
// 8-column tile with the E4M3 tensor-core contraction (pkv_decode_mma_fp8.cuh), or the tensor-memory
// tile widening each K/V tile's codes to f16 in shared memory (pkv_mq_tc.cuh).
#include "pkv_decode_mma_fp8.cuh"
#include "pkv_decode_mq.cuh"
#include "pkv_internal.h"
#include "pkv_mq_tc.cuh"

namespace pkv {

namespace {

template <typename T>
cudaError_t dispatch(const DecodeParams& p, const MqParams& mq, const CUtensorMap& kmap, const CUtensorMap& vmap,
                     int head_dim, int block_size, int num_seqs, int tile, cudaStream_t stream) {
  constexpr int R = PKV_MMA_FP8_RING_BYTES;
  if (head_dim == 128 && tile == PKV_MQ_TILE_TENSOR) {
    if (block_size == 16) return launch_mq_tc<T, 128, 16, true>(p, mq, kmap, vmap, num_seqs, stream);
    if (block_size == 8) return launch_mq_tc<T, 128, 8, true>(p, mq, kmap, vmap, num_seqs, stream);
    if (block_size == 32) return launch_mq_tc<T, 128, 32, true>(p, mq, kmap, vmap, num_seqs, stream);
    return cudaErrorInvalidValue;
  }
  if (head_dim == 128) {
    if (block_size == 16) return launch_mq_mma<MmaTileE4M3<T, 128, 16>, R>(p, mq, kmap, vmap, num_seqs, stream);
    if (block_size == 8) return launch_mq_mma<MmaTileE4M3<T, 128, 8>, R>(p, mq, kmap, vmap, num_seqs, stream);
    if (block_size == 32) return launch_mq_mma<MmaTileE4M3<T, 128, 32>, R>(p, mq, kmap, vmap, num_seqs, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t decode_mq_fp8_f16(const DecodeParams& p, const MqParams& mq, const CUtensorMap& kmap,
                              const CUtensorMap& vmap, int head_dim, int block_size, int num_seqs, int tile,
                              cudaStream_t stream) {
  return dispatch<__half>(p, mq, kmap, vmap, head_dim, block_size, num_seqs, tile, stream);
}

cudaError_t decode_mq_fp8_bf16(const DecodeParams& p, const MqParams& mq, const CUtensorMap& kmap,
                               const CUtensorMap& vmap, int head_dim, int block_size, int num_seqs, int tile,
                               cudaStream_t stream) {
  return dispatch<__nv_bfloat16>(p, mq, kmap, vmap, head_dim, block_size, num_seqs, tile, stream);
}

}  // namespace pkv
