// Host-side entry points shared between the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace pkv {

struct DecodeParams;

// CUDA-core decode (any group size; one CTA per query head).
cudaError_t decode_simt_f16(const DecodeParams& p, int head_dim, int block_size, int num_seqs,
                            cudaStream_t stream);
cudaError_t decode_simt_bf16(const DecodeParams& p, int head_dim, int block_size, int num_seqs,
                             cudaStream_t stream);

// CUDA-core decode over an FP8 (E4M3) cache; T is the query/output type.
cudaError_t decode_simt_fp8_f16(const DecodeParams& p, int head_dim, int block_size, int num_seqs,
                                cudaStream_t stream);
cudaError_t decode_simt_fp8_bf16(const DecodeParams& p, int head_dim, int block_size, int num_seqs,
                                 cudaStream_t stream);

// Tensor-core decode over an FP8 (E4M3) cache (head_dim 128, group <= 8, MHA included).
cudaError_t decode_mma_fp8_f16(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                               int head_dim, int block_size, int num_seqs, cudaStream_t stream);
cudaError_t decode_mma_fp8_bf16(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                int head_dim, int block_size, int num_seqs, cudaStream_t stream);

// Tensor-core grouped-query decode (2 <= group <= 8; one CTA per kv head).
cudaError_t decode_mma_f16(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                           int head_dim, int block_size, int num_seqs, cudaStream_t stream);
cudaError_t decode_mma_bf16(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                            int head_dim, int block_size, int num_seqs, cudaStream_t stream);

// Multi-query attention (several causal query tokens per sequence; pkv_decode_mq.cuh).
struct MqParams;
// wide: the 64-row tile (query rows in the MMA's M dimension) instead of the 8-column one.
// Whether the 16-bit tensor-core tiles take a head_dim-128 tile in one copy
// (the pool's tensor map is then make_pool_map_tc's).
bool tile_one_copy();

cudaError_t decode_mq_f16(const DecodeParams& p, const MqParams& mq, const CUtensorMap& kmap,
                          const CUtensorMap& vmap, int head_dim, int block_size, int num_seqs, int tile,
                          cudaStream_t stream);
cudaError_t decode_mq_bf16(const DecodeParams& p, const MqParams& mq, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, int head_dim, int block_size, int num_seqs, int tile,
                           cudaStream_t stream);
// Multi-query attention over an FP8 (E4M3) pool, head_dim 128: tile PKV_MQ_TILE_TENSOR (the pool
// through make_pool_map_fp8_rows) or the 8-column tile (make_pool_map).
cudaError_t decode_mq_fp8_f16(const DecodeParams& p, const MqParams& mq, const CUtensorMap& kmap,
                              const CUtensorMap& vmap, int head_dim, int block_size, int num_seqs, int tile,
                              cudaStream_t stream);
cudaError_t decode_mq_fp8_bf16(const DecodeParams& p, const MqParams& mq, const CUtensorMap& kmap,
                               const CUtensorMap& vmap, int head_dim, int block_size, int num_seqs, int tile,
                               cudaStream_t stream);
// The same over 16-row tiles of two 8-column groups (PKV_MQ_TILE_PAIRS; the pool through make_pool_map).
cudaError_t decode_mq_pairs_fp8_f16(const DecodeParams& p, const MqParams& mq, const CUtensorMap& kmap,
                                    const CUtensorMap& vmap, int head_dim, int block_size, int num_seqs,
                                    cudaStream_t stream);
cudaError_t decode_mq_pairs_fp8_bf16(const DecodeParams& p, const MqParams& mq, const CUtensorMap& kmap,
                                     const CUtensorMap& vmap, int head_dim, int block_size, int num_seqs,
                                     cudaStream_t stream);

// Set the calling thread's pkv_last_error_message() text.
void set_last_error_message(const char* msg);

// The device address of a device's error word (PKV_DEVERR_* bits), or null.
unsigned* device_error_word(int dev);

}  // namespace pkv
