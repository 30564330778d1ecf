// Multi-query paged attention (the 8-column tile, the 64-row tile and the 128-row
// tensor-memory tile), f16 and bf16 instantiations.
#include "pkv_decode_mq.cuh"
#include "pkv_internal.h"
#include "pkv_mq_tc.cuh"
#include "pkv_mq_wide.cuh"

namespace pkv {

namespace {

template <typename T>
cudaError_t dispatch(const DecodeParams& p, const MqParams& mq, const CUtensorMap& kmap, const CUtensorMap& vmap,
                     int head_dim, int block_size, int num_seqs, int tile, cudaStream_t stream) {
  if (tile == PKV_MQ_TILE_TENSOR) {
    if (head_dim == 128) {
      if (block_size == 16) return launch_mq_tc<T, 128, 16>(p, mq, kmap, vmap, num_seqs, stream);
      if (block_size == 8) return launch_mq_tc<T, 128, 8>(p, mq, kmap, vmap, num_seqs, stream);
      if (block_size == 32) return launch_mq_tc<T, 128, 32>(p, mq, kmap, vmap, num_seqs, stream);
    } else if (head_dim == 64) {
      if (block_size == 16) return launch_mq_tc<T, 64, 16>(p, mq, kmap, vmap, num_seqs, stream);
      if (block_size == 8) return launch_mq_tc<T, 64, 8>(p, mq, kmap, vmap, num_seqs, stream);
      if (block_size == 32) return launch_mq_tc<T, 64, 32>(p, mq, kmap, vmap, num_seqs, stream);
    }
    return cudaErrorInvalidValue;
  }
  if (tile == PKV_MQ_TILE_ROWS) {
    if (head_dim == 128) {
      if (block_size == 16) return launch_mq_wide<T, 128, 16>(p, mq, kmap, vmap, num_seqs, stream);
      if (block_size == 8) return launch_mq_wide<T, 128, 8>(p, mq, kmap, vmap, num_seqs, stream);
      if (block_size == 32) return launch_mq_wide<T, 128, 32>(p, mq, kmap, vmap, num_seqs, stream);
    } else if (head_dim == 64) {
      if (block_size == 16) return launch_mq_wide<T, 64, 16>(p, mq, kmap, vmap, num_seqs, stream);
      if (block_size == 8) return launch_mq_wide<T, 64, 8>(p, mq, kmap, vmap, num_seqs, stream);
      if (block_size == 32) return launch_mq_wide<T, 64, 32>(p, mq, kmap, vmap, num_seqs, stream);
    }
    return cudaErrorInvalidValue;
  }
  if (head_dim == 128) {
    if (block_size == 16) return launch_mq_mma<MmaTile<T, 128, 16>>(p, mq, kmap, vmap, num_seqs, stream);
    if (block_size == 8) return launch_mq_mma<MmaTile<T, 128, 8>>(p, mq, kmap, vmap, num_seqs, stream);
    if (block_size == 32) return launch_mq_mma<MmaTile<T, 128, 32>>(p, mq, kmap, vmap, num_seqs, stream);
  } else if (head_dim == 64) {
    if (block_size == 16) return launch_mq_mma<MmaTile<T, 64, 16>>(p, mq, kmap, vmap, num_seqs, stream);
    if (block_size == 8) return launch_mq_mma<MmaTile<T, 64, 8>>(p, mq, kmap, vmap, num_seqs, stream);
    if (block_size == 32) return launch_mq_mma<MmaTile<T, 64, 32>>(p, mq, kmap, vmap, num_seqs, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t decode_mq_f16(const DecodeParams& p, const MqParams& mq, const CUtensorMap& kmap,
                          const CUtensorMap& vmap, int head_dim, int block_size, int num_seqs, int tile,
                          cudaStream_t stream) {
  return dispatch<__half>(p, mq, kmap, vmap, head_dim, block_size, num_seqs, tile, stream);
}

cudaError_t decode_mq_bf16(const DecodeParams& p, const MqParams& mq, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, int head_dim, int block_size, int num_seqs, int tile,
                           cudaStream_t stream) {
  return dispatch<__nv_bfloat16>(p, mq, kmap, vmap, head_dim, block_size, num_seqs, tile, stream);
}

}  // namespace pkv
