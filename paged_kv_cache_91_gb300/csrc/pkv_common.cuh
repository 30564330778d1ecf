// Shared device helpers for the paged KV cache kernels (sm_103a).
//
// Inline PTX for the Blackwell data movers used by the decode kernels:
// mbarrier transaction counting, the bulk (TMA) copy engine in its linear and
// tiled forms, plus the warp-level matrix helpers the grouped-query kernel uses.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "paged_kv.h"

namespace pkv {

constexpr unsigned kFull = 0xffffffffu;

#ifndef PKV_DECODE_WARPS
#define PKV_DECODE_WARPS 4  // warps per decode CTA (build-time tuning knob)
#endif
#ifndef PKV_DECODE_MIN_CTAS
#define PKV_DECODE_MIN_CTAS 1  // __launch_bounds__ minimum CTAs per SM (build-time tuning knob)
#endif
#ifndef PKV_GRID_HEAD_FASTEST
#define PKV_GRID_HEAD_FASTEST 0  // partitioned grid: 1 = blockIdx.x walks heads (build-time tuning knob)
#endif
#ifndef PKV_PROXY_FENCE
// 1: fence.proxy.async before every stage refill (build-time knob). With 0 the
// fence runs only where generic stores went into the stage (tail zeroing); reads
// of a stage have all returned their values before the refill is issued.
#define PKV_PROXY_FENCE 0
#endif
constexpr int kDecodeWarps = PKV_DECODE_WARPS;
// A warp keeps one physical block id per lane, so a partition spans at most
// kDecodeWarps * 32 blocks.
constexpr int kMaxPartitionBlocks = kDecodeWarps * 32;
// Upper bound on one wait for a bulk copy, in SM clock cycles (about 1 s at 2 GHz).
constexpr long long kWaitLimitCycles = 2000000000ll;

// Parameters of one decode launch (both decode kernels).
struct DecodeParams {
  void* out;
  const void* query;
  const unsigned char* key_cache;
  const unsigned char* value_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float* part_o;  // [S][H][max_partitions][D]   (split mode only)
  float* part_m;  // [S][H][max_partitions]
  float* part_l;  // [S][H][max_partitions]
  unsigned* err;  // per-device error word
  float scale_log2;  // scale * log2(e) (* k_scale for an FP8 cache): scores live in the base-2 domain
  float v_scale;     // FP8 cache: value of one V code unit (1 for 16-bit caches, unused there)
  int max_blocks_per_seq;
  int num_heads;
  int num_kv_heads;
  int group;  // num_heads / num_kv_heads
  int num_blocks;
  int partition_size;  // tokens, multiple of block_size
  int max_partitions;  // ceil(max_context_len / partition_size), >= 1
  int ctx_limit;       // min(max_context_len, max_blocks_per_seq * block_size)
};

#ifndef PKV_USE_PDL
#define PKV_USE_PDL 1  // launch with programmatic stream serialization (build-time knob)
#endif

// Programmatic dependent launch. Every kernel first waits until the kernels
// before it in the stream have completed and their writes are visible (a no-op
// without a programmatic dependency), then lets the next kernel start its launch
// while this one runs. Inputs are only read after the wait, so the stream
// order of reads and writes is that of ordinary launches.
__device__ __forceinline__ void pdl_begin() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch with programmatic stream serialization allowed (PKV_USE_PDL), else plainly.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = PKV_USE_PDL ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// ---------------------------------------------------------------------------
// mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete; false after `limit` SM cycles.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, long long limit = kWaitLimitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}

// ---------------------------------------------------------------------------
// bulk copies (TMA engine)

// Linear bulk copy global -> shared; completes `bytes` transactions on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Tiled 2D tensor copy global -> shared through a tensor map; x is the inner
// (contiguous) coordinate in elements and must be a multiple of 8 for 16-bit data.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// ---------------------------------------------------------------------------
// 16-bit element helpers

template <typename T>
struct Elem;

template <>
struct Elem<__half> {
  static __device__ __forceinline__ float2 to_float2(uint32_t packed) {
    __half2 h = *reinterpret_cast<__half2*>(&packed);
    return __half22float2(h);
  }
  static __device__ __forceinline__ __half from_float(float f) { return __float2half_rn(f); }
  static __device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
};

template <>
struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float2 to_float2(uint32_t packed) {
    return make_float2(__uint_as_float(packed << 16), __uint_as_float(packed & 0xffff0000u));
  }
  static __device__ __forceinline__ __nv_bfloat16 from_float(float f) { return __float2bfloat16_rn(f); }
  static __device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
};

// ---------------------------------------------------------------------------
// cache element formats of the CUDA-core tile: C is the type of the stored K/V
// elements. A 16-bit cache holds the inputs' bits; an E4M3 cache holds 8-bit
// codes whose values are code * scale (the scale is applied outside the tile).
// pair() widens the element pair in the low 2 * EB bytes of `w` (first element
// in the lower bytes) to fp32.

template <typename C>
struct CacheFmt {
  static constexpr int EB = 2;  // bytes per element
  static __device__ __forceinline__ float2 pair(uint32_t w) { return Elem<C>::to_float2(w); }
};

template <>
struct CacheFmt<__nv_fp8_e4m3> {
  static constexpr int EB = 1;
  // Every E4M3 value is exactly an fp16 value, so the widening is exact.
  static __device__ __forceinline__ float2 pair(uint32_t w) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xffffu), __NV_E4M3);
    return __half22float2(*reinterpret_cast<const __half2*>(&h));
  }
  // The four codes of w as two pairs: lo = (byte 0, byte 1), hi = (byte 2, byte 3).
  // One conversion instruction per 16-bit half of the register.
  static __device__ __forceinline__ void quad(uint32_t w, float2& lo, float2& hi) {
    uint32_t a, b;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(a), "=r"(b)
        : "r"(w));
    lo = __half22float2(*reinterpret_cast<const __half2*>(&a));
    hi = __half22float2(*reinterpret_cast<const __half2*>(&b));
  }
};

// ---------------------------------------------------------------------------
// warp-level matrix helpers (grouped-query kernel)

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p))
               : "memory");
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p))
               : "memory");
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

template <typename T>
struct Mma;

// D[16x8] += A[16x16] * B[16x8], fp32 accumulate
template <>
struct Mma<__half> {
  static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
};

template <>
struct Mma<__nv_bfloat16> {
  static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
};

// Partition bookkeeping common to both decode kernels. Returns false when the
// CTA has nothing to do (partition past the end of the context).
struct PartitionInfo {
  int ctx;   // clamped context length
  int tok0;  // first token of this partition
  int tok1;  // one past the last token of this partition
  int blk0;  // first logical block
  int nblk;  // logical blocks in this partition
  bool direct;  // the whole context is one partition: write the final output
};

__device__ __forceinline__ int clamp_context(const DecodeParams& p, int s, bool report) {
  int ctx = p.context_lens[s];
  if (ctx < 0 || ctx > p.ctx_limit) {
    if (report) atomicOr(p.err, PKV_DEVERR_CONTEXT);
    ctx = ctx < 0 ? 0 : p.ctx_limit;
  }
  return ctx;
}

}  // namespace pkv
