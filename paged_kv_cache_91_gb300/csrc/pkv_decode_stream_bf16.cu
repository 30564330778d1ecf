// Persistent equal-work decode kernels and their reduce, bf16 instantiations.
#include "pkv_decode_stream.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

template <int D, int BS>
cudaError_t dispatch(bool mma, const StreamParams* sp, const CUtensorMap* kmap, const CUtensorMap* vmap, int grid,
                     cudaStream_t stream, int num_seqs, int* ctas) {
  using T = __nv_bfloat16;
  if (mma) {
    using L = StreamLaunch<T, D, BS, true>;
    return sp ? L::launch(*sp, *kmap, *vmap, grid, stream) : L::occupancy(num_seqs, ctas);
  }
  using L = StreamLaunch<T, D, BS, false>;
  return sp ? L::launch(*sp, *kmap, *vmap, grid, stream) : L::occupancy(num_seqs, ctas);
}

cudaError_t dispatch_shape(int head_dim, int block_size, bool mma, const StreamParams* sp, const CUtensorMap* kmap,
                           const CUtensorMap* vmap, int grid, cudaStream_t stream, int num_seqs, int* ctas) {
  if (head_dim == 128) {
    if (block_size == 16) return dispatch<128, 16>(mma, sp, kmap, vmap, grid, stream, num_seqs, ctas);
    if (block_size == 8) return dispatch<128, 8>(mma, sp, kmap, vmap, grid, stream, num_seqs, ctas);
    if (block_size == 32) return dispatch<128, 32>(mma, sp, kmap, vmap, grid, stream, num_seqs, ctas);
  } else if (head_dim == 64) {
    if (block_size == 16) return dispatch<64, 16>(mma, sp, kmap, vmap, grid, stream, num_seqs, ctas);
    if (block_size == 8) return dispatch<64, 8>(mma, sp, kmap, vmap, grid, stream, num_seqs, ctas);
    if (block_size == 32) return dispatch<64, 32>(mma, sp, kmap, vmap, grid, stream, num_seqs, ctas);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t decode_stream_occupancy_bf16(int head_dim, int block_size, bool mma, int num_seqs, int* ctas) {
  return dispatch_shape(head_dim, block_size, mma, nullptr, nullptr, nullptr, 0, nullptr, num_seqs, ctas);
}

cudaError_t decode_stream_bf16(const StreamParams& sp, const CUtensorMap& kmap, const CUtensorMap& vmap,
                               int head_dim, int block_size, bool mma, int grid, cudaStream_t stream) {
  return dispatch_shape(head_dim, block_size, mma, &sp, &kmap, &vmap, grid, stream, sp.num_seqs, nullptr);
}

cudaError_t stream_reduce_bf16(const StreamParams& sp, int head_dim, int nwarps, cudaStream_t stream) {
  return launch_kernel(pkv_stream_reduce_kernel<__nv_bfloat16>, dim3(sp.ng, sp.num_seqs), dim3(128), 0, stream,
                       static_cast<__nv_bfloat16*>(sp.p.out), (const float*)sp.slot_o, (const float*)sp.slot_m,
                       (const float*)sp.slot_l, (const int*)sp.pre_out, sp.num_seqs, sp.p.num_heads, head_dim, sp.ng,
                       sp.gc, nwarps);
}

}  // namespace pkv
