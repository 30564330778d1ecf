// CUDA-core decode kernels, f16 instantiations.
#include "pkv_decode_simt.cuh"
#include "pkv_internal.h"

namespace pkv {

cudaError_t decode_simt_f16(const DecodeParams& p, int head_dim, int block_size, int num_seqs,
                            cudaStream_t stream) {
  using T = __half;
  if (head_dim == 128) {
    if (block_size == 16) return launch_decode_simt<T, 128, 16>(p, num_seqs, stream);
    if (block_size == 8) return launch_decode_simt<T, 128, 8>(p, num_seqs, stream);
    if (block_size == 32) return launch_decode_simt<T, 128, 32>(p, num_seqs, stream);
  } else if (head_dim == 64) {
    if (block_size == 16) return launch_decode_simt<T, 64, 16>(p, num_seqs, stream);
    if (block_size == 8) return launch_decode_simt<T, 64, 8>(p, num_seqs, stream);
    if (block_size == 32) return launch_decode_simt<T, 64, 32>(p, num_seqs, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace pkv
