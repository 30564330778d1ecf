// Multi-query paged attention over an FP8 (E4M3) pool, 16 rows of a kv head per CTA in two 8-column
// groups that share each widened K/V fragment (pkv_mq_pairs.cuh); f16 and bf16 queries, head_dim 128.
#include "pkv_internal.h"
#include "pkv_mq_pairs.cuh"

namespace pkv {

namespace {

template <typename T>
cudaError_t dispatch(const DecodeParams& p, const MqParams& mq, const CUtensorMap& kmap, const CUtensorMap& vmap,
                     int head_dim, int block_size, int num_seqs, cudaStream_t stream) {
  if (head_dim != 128) return cudaErrorInvalidValue;
  if (block_size == 16) return launch_mq_pairs<T, 16>(p, mq, kmap, vmap, num_seqs, stream);
  if (block_size == 8) return launch_mq_pairs<T, 8>(p, mq, kmap, vmap, num_seqs, stream);
  if (block_size == 32) return launch_mq_pairs<T, 32>(p, mq, kmap, vmap, num_seqs, stream);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t decode_mq_pairs_fp8_f16(const DecodeParams& p, const MqParams& mq, const CUtensorMap& kmap,
                                    const CUtensorMap& vmap, int head_dim, int block_size, int num_seqs,
                                    cudaStream_t stream) {
  return dispatch<__half>(p, mq, kmap, vmap, head_dim, block_size, num_seqs, stream);
}

cudaError_t decode_mq_pairs_fp8_bf16(const DecodeParams& p, const MqParams& mq, const CUtensorMap& kmap,
                                     const CUtensorMap& vmap, int head_dim, int block_size, int num_seqs,
                                     cudaStream_t stream) {
  return dispatch<__nv_bfloat16>(p, mq, kmap, vmap, head_dim, block_size, num_seqs, stream);
}

}  // namespace pkv
