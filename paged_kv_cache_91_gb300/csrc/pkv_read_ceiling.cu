// pkv_read_chunks: a measurement helper, not a step of the method. It reads
// chunks of a buffer in a given order, each chunk by one bulk copy into a
// per-warp shared-memory ring, and does nothing with the bytes. Timed over
// random whole chunks the size of one (block, kv head) tile, it gives the read
// ceiling of the decode's access pattern: every tile the decode reads is such a
// chunk at a random place in the pool. The bench reports each call against it.
#include <stdio.h>

#include "paged_kv.h"
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kReadWarps = 4;
constexpr int kReadPerWarp = 32;         // chunks per warp; the grid covers the rest
constexpr int kReadRingBytes = 48 * 1024;  // per CTA, as the FP8 decode ring

template <int CH>
constexpr int read_stages() {
  constexpr int s = kReadRingBytes / (kReadWarps * CH);
  return s < 2 ? 2 : (s > 12 ? 12 : s);
}

template <int CH>
__global__ void __launch_bounds__(kReadWarps * 32) pkv_read_chunks_kernel(const unsigned char* __restrict__ buf,
                                                                         long long num_chunks,
                                                                         const int32_t* __restrict__ order,
                                                                         long long num_reads, unsigned* err) {
  pdl_begin();
  constexpr int SPW = read_stages<CH>();
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned char* ring = smem + warp * SPW * CH;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kReadWarps * SPW * CH) + warp * SPW;
  const long long first = ((long long)blockIdx.x * kReadWarps + warp) * kReadPerWarp;
  const int n = (int)(num_reads - first < kReadPerWarp ? (num_reads - first > 0 ? num_reads - first : 0)
                                                       : kReadPerWarp);
  if (lane == 0) {
    for (int k = 0; k < SPW; ++k) mbar_init(bars + k, 1);
    fence_mbar_init();
  }
  __syncwarp();
  // lane i holds the chunk index of the warp's read i; an index outside the buffer is reported and skipped
  int idx = -1;
  if (lane < n) {
    const int c = order[first + lane];
    if (c >= 0 && c < num_chunks) {
      idx = c;
    } else {
      atomicOr(err, PKV_DEVERR_BLOCK_ID);
    }
  }
  auto issue = [&](int i) {
    const int c = __shfl_sync(kFull, idx, i);
    if (lane == 0) {
      uint64_t* bar = bars + (i % SPW);
      if (c >= 0) {
        mbar_arrive_expect_tx(bar, CH);
        bulk_g2s(ring + (i % SPW) * CH, buf + (size_t)c * CH, CH, bar);
      } else {
        mbar_arrive(bar);
      }
    }
  };
  const int nfirst = n < SPW ? n : SPW;
  for (int i = 0; i < nfirst; ++i) issue(i);
  int issued = nfirst;
  for (int i = 0; i < n; ++i) {
    if (!__all_sync(kFull, mbar_wait(bars + (i % SPW), (i / SPW) & 1))) {
      // a copy that never completes: report, then wait (bounded) for the copies still in flight
      if (lane == 0) {
        atomicOr(err, PKV_DEVERR_TIMEOUT);
        for (int j = i + 1; j < issued; ++j) mbar_wait(bars + (j % SPW), (j / SPW) & 1);
      }
      return;
    }
    __syncwarp();
    if (i + SPW < n) {
      issue(i + SPW);
      ++issued;
    }
  }
}

template <int CH>
cudaError_t launch_read(const unsigned char* buf, long long num_chunks, const int32_t* order, long long num_reads,
                        unsigned* err, cudaStream_t stream) {
  constexpr int SPW = read_stages<CH>();
  constexpr int smem = kReadWarps * SPW * CH + kReadWarps * SPW * 8;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(pkv_read_chunks_kernel<CH>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  const long long per_cta = (long long)kReadWarps * kReadPerWarp;
  const unsigned grid = (unsigned)((num_reads + per_cta - 1) / per_cta);
  return launch_kernel(pkv_read_chunks_kernel<CH>, dim3(grid), dim3(kReadWarps * 32), (size_t)smem, stream, buf,
                       num_chunks, order, num_reads, err);
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status_t pkv_read_chunks(const void* buffer, int64_t buffer_bytes, const int32_t* order,
                                        int64_t num_reads, int32_t chunk_bytes, cudaStream_t stream) {
  using namespace pkv;
  if (chunk_bytes != 1024 && chunk_bytes != 2048 && chunk_bytes != 4096 && chunk_bytes != 8192) {
    set_last_error_message("chunk_bytes must be 1024, 2048, 4096 or 8192");
    return PKV_ERR_UNSUPPORTED;
  }
  if (num_reads < 0 || buffer_bytes < 0) {
    set_last_error_message("num_reads and buffer_bytes must be >= 0");
    return PKV_ERR_INVALID_ARG;
  }
  if (num_reads == 0) return PKV_OK;
  if (!buffer || !order || (reinterpret_cast<uintptr_t>(buffer) & 15u)) {
    set_last_error_message("buffer (16-byte aligned) and order must be non-null");
    return PKV_ERR_INVALID_ARG;
  }
  if (num_reads > (1LL << 40)) {
    set_last_error_message("num_reads too large");
    return PKV_ERR_UNSUPPORTED;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_last_error_message(cudaGetErrorString(e));
    return PKV_ERR_CUDA;
  }
  unsigned* err = device_error_word(dev);
  if (!err) {
    set_last_error_message("device error word unavailable");
    return PKV_ERR_CUDA;
  }
  const long long chunks = buffer_bytes / chunk_bytes;
  const unsigned char* buf = static_cast<const unsigned char*>(buffer);
  switch (chunk_bytes) {
    case 1024: e = launch_read<1024>(buf, chunks, order, num_reads, err, stream); break;
    case 2048: e = launch_read<2048>(buf, chunks, order, num_reads, err, stream); break;
    case 4096: e = launch_read<4096>(buf, chunks, order, num_reads, err, stream); break;
    default: e = launch_read<8192>(buf, chunks, order, num_reads, err, stream); break;
  }
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof msg, "read kernel launch: %s", cudaGetErrorString(e));
    set_last_error_message(msg);
    return PKV_ERR_CUDA;
  }
  return PKV_OK;
}
