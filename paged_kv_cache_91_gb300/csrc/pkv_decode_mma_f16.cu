// Tensor-core grouped-query decode kernels, f16 instantiations.
#include "pkv_decode_mma.cuh"
#include "pkv_internal.h"

namespace pkv {

cudaError_t decode_mma_f16(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                           int head_dim, int block_size, int num_seqs, cudaStream_t stream) {
  using T = __half;
  if (head_dim == 128) {
    if (block_size == 16) return launch_decode_gqa_mma<MmaTile<T, 128, 16>>(p, kmap, vmap, num_seqs, stream);
    if (block_size == 8) return launch_decode_gqa_mma<MmaTile<T, 128, 8>>(p, kmap, vmap, num_seqs, stream);
    if (block_size == 32) return launch_decode_gqa_mma<MmaTile<T, 128, 32>>(p, kmap, vmap, num_seqs, stream);
  } else if (head_dim == 64) {
    if (block_size == 16) return launch_decode_gqa_mma<MmaTile<T, 64, 16>>(p, kmap, vmap, num_seqs, stream);
    if (block_size == 8) return launch_decode_gqa_mma<MmaTile<T, 64, 8>>(p, kmap, vmap, num_seqs, stream);
    if (block_size == 32) return launch_decode_gqa_mma<MmaTile<T, 64, 32>>(p, kmap, vmap, num_seqs, stream);
  }
  return cudaErrorInvalidValue;
}

bool tile_one_copy() { return PKV_TILE_ONE_COPY != 0; }

}  // namespace pkv
