// C ABI of the paged KV cache library: argument validation, the cache-write
// kernel, the split-K log-sum-exp reduce kernel, dispatch of the decode kernels
// and the per-device error word. See include/paged_kv.h for the contract.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>

#include "paged_kv.h"
#include "pkv_common.cuh"
#include "pkv_decode_mq.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

// Decode partition when the call passes 0: 1024 tokens over both cache types, 2048 for batches whose
// contexts may exceed 8192 tokens (at most 128 blocks either way). Measured, decode call ms at 512 / 1024 /
// 2048 tokens (16-bit cache): workload 2 0.1995 / 0.1980 / 0.1988, workload 3 (contexts up to 8192) 0.1747
// / 0.1715 / 0.1718, workload 4 0.0662 / 0.0627 / 0.0619, workload 5 (32768) 1.485 / 1.464 / 1.454; FP8
// cache: workload 2 0.115 / 0.114 / 0.117, workload 3 0.114 / 0.104 / 0.107, workload 5 - / 0.771 / 0.760.
// A CTA's start and end cost more than the longer per-CTA tail.
constexpr int kDefaultPartition = 1024;
constexpr int kDefaultPartitionLong = 2048;
constexpr int kLongContext = 8192;
int default_partition(int max_context_len, int block_size) {
  const int P = max_context_len > kLongContext ? kDefaultPartitionLong : kDefaultPartition;
  const int cap = kMaxPartitionBlocks * block_size;
  return P < cap ? P : cap;
}
#ifndef PKV_MQ_WIDE_MIN_ROWS
// Multi-query rows per kv head from which the tensor-memory tile runs (build-time knob). Measured: at 16
// rows (two 8-column CTAs per kv head) the 8-column tile is 3-10% faster; from 20 rows on the tensor tile
// wins, by 1.5x at 32 rows.
#define PKV_MQ_WIDE_MIN_ROWS 17
#endif
#ifndef PKV_MQ_WIDE_MIN_ROWS_FP8
// The same over an FP8 pool, where the 8-column tile is relatively faster: 24 rows 0.266 against
// 0.362 ms, 32 rows even, 48 rows 0.509 against 0.371 ms (workload 3).
#define PKV_MQ_WIDE_MIN_ROWS_FP8 33
#endif
// Multi-query: every query row writes D + 2 partial floats per partition, so
// few long partitions measure fastest (capped at kMaxPartitionBlocks blocks).
constexpr int kDefaultPartitionMq = 2048;
int mq_default_partition(int block_size) {
  const int cap = kMaxPartitionBlocks * block_size;
  return kDefaultPartitionMq < cap ? kDefaultPartitionMq : cap;
}
constexpr int kMaxDevices = 64;

thread_local char g_msg[512] = "";

pkv_status_t fail(pkv_status_t st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof g_msg, fmt, ap);
  va_end(ap);
  return st;
}

pkv_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_head_dim(int d) { return d == 64 || d == 128; }
bool supported_block_size(int b) { return b == 8 || b == 16 || b == 32; }

}  // namespace

// Per-device error word; kernels get its address as an argument.
__device__ unsigned int g_pkv_error_word;

namespace {

unsigned* error_word(int dev) {
  static unsigned* ptrs[kMaxDevices] = {};
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  if (!ptrs[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_pkv_error_word) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<unsigned*>(ptr);
  }
  return ptrs[dev];
}

// ---------------------------------------------------------------------------
// cache write: one thread per 16-byte piece of a (token, kv head) row, K and V

__global__ void pkv_write_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                                 uint4* __restrict__ key_cache, uint4* __restrict__ value_cache,
                                 const int64_t* __restrict__ slot_mapping, int num_tokens, int num_kv_heads,
                                 int pieces_per_row, int block_size, long long num_slots, unsigned* err) {
  pdl_begin();
  const long long total = (long long)num_tokens * num_kv_heads * pieces_per_row;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
    const int c = (int)(idx % pieces_per_row);
    const long long r = idx / pieces_per_row;
    const int h = (int)(r % num_kv_heads);
    const int t = (int)(r / num_kv_heads);
    // the slot and the row pieces load together: the pieces do not depend on the slot
    const size_t src = ((size_t)t * num_kv_heads + h) * pieces_per_row + c;
    const long long slot = __ldg(slot_mapping + t);
    const uint4 kv = __ldg(key + src);
    const uint4 vv = __ldg(value + src);
    if (slot < 0) continue;  // padding token
    if (slot >= num_slots) {
      if (c == 0 && h == 0) atomicOr(err, PKV_DEVERR_SLOT);
      continue;
    }
    const long long blk = slot / block_size, off = slot - blk * block_size;
    const size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + off) * pieces_per_row + c;
    key_cache[dst] = kv;
    value_cache[dst] = vv;
  }
}

// ---------------------------------------------------------------------------
// quantizing cache write into an FP8 (E4M3) pool: one thread per 16 codes (16
// bytes) of a (token, kv head) row, K and V. code = E4M3(x / scale): the
// division correctly rounded in fp32, then round-to-nearest-even to E4M3 with
// saturation to +-448 (the satfinite conversion).

template <typename T>
__device__ __forceinline__ uint4 quantize16(const uint4 (&src)[2], float scale) {
  uint32_t out[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint4 r = src[k / 2];
    const uint32_t w0 = (k & 1) ? r.z : r.x, w1 = (k & 1) ? r.w : r.y;
    const float2 a = Elem<T>::to_float2(w0), b = Elem<T>::to_float2(w1);
    const __nv_fp8x2_storage_t lo =
        __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(a.x, scale), __fdiv_rn(a.y, scale)), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi =
        __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(b.x, scale), __fdiv_rn(b.y, scale)), __NV_SATFINITE, __NV_E4M3);
    out[k] = (uint32_t)lo | ((uint32_t)hi << 16);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

template <typename T>
__global__ void pkv_write_fp8_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                                     uint4* __restrict__ key_cache, uint4* __restrict__ value_cache,
                                     const int64_t* __restrict__ slot_mapping, int num_tokens, int num_kv_heads,
                                     int pieces_per_row, int block_size, long long num_slots, float k_scale,
                                     float v_scale, unsigned* err) {
  pdl_begin();
  const long long total = (long long)num_tokens * num_kv_heads * pieces_per_row;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
    const int c = (int)(idx % pieces_per_row);  // 16 output codes = 32 source bytes
    const long long r = idx / pieces_per_row;
    const int h = (int)(r % num_kv_heads);
    const int t = (int)(r / num_kv_heads);
    const size_t src = (((size_t)t * num_kv_heads + h) * pieces_per_row + c) * 2;
    const long long slot = __ldg(slot_mapping + t);
    if (slot < 0) continue;  // padding token: its rows are not read
    if (slot >= num_slots) {
      if (c == 0 && h == 0) atomicOr(err, PKV_DEVERR_SLOT);
      continue;
    }
    const uint4 kv[2] = {__ldg(key + src), __ldg(key + src + 1)};
    const uint4 vv[2] = {__ldg(value + src), __ldg(value + src + 1)};
    const long long blk = slot / block_size, off = slot - blk * block_size;
    const size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + off) * pieces_per_row + c;
    key_cache[dst] = quantize16<T>(kv, k_scale);
    value_cache[dst] = quantize16<T>(vv, v_scale);
  }
}

// ---------------------------------------------------------------------------
// split-K reduce: merge the partitions' (m_p, l_p, o_p) of one (seq, head) by
// log-sum-exp: out = sum_p w_p o_p / sum_p w_p with w_p = l_p 2^(m_p - max m).
// One warp per output row; lane p holds the weight of partition p (p < 32 per
// round) and each lane merges D/32 dims.

constexpr int kReduceRows = 4;
constexpr int kReduceEarly = 4;  // partitions whose partial outputs are fetched with the first loads

// The first round of loads for output row `row` (partials at base = row * max_partitions):
// this lane's partition (m, l) and the partial outputs of the first kReduceEarly partitions.
// All are in bounds whatever the row's partition count; entries past it are masked later.
template <int D>
__device__ __forceinline__ void reduce_load_row(const float* __restrict__ part_o, const float* __restrict__ part_m,
                                                const float* __restrict__ part_l, size_t base, int max_partitions,
                                                int lane, float& mp, float& lp, float (&o_early)[kReduceEarly][D / 32]) {
  constexpr int DPL = D / 32;
  mp = -INFINITY;
  lp = 0.f;
  if (lane < max_partitions) {
    mp = part_m[base + lane];
    lp = part_l[base + lane];
  }
#pragma unroll
  for (int k = 0; k < kReduceEarly; ++k) {
    if (k < max_partitions) {
      const float* o = part_o + (base + k) * D + lane * DPL;
      if constexpr (DPL == 4) {
        const float4 v = *reinterpret_cast<const float4*>(o);
        o_early[k][0] = v.x; o_early[k][1] = v.y; o_early[k][2] = v.z; o_early[k][3] = v.w;
      } else {
        const float2 v = *reinterpret_cast<const float2*>(o);
        o_early[k][0] = v.x; o_early[k][1] = v.y;
      }
    } else {
#pragma unroll
      for (int e = 0; e < DPL; ++e) o_early[k][e] = 0.f;
    }
  }
}

// Merge the np (> 1) partials of output row `row` into out[row][:], given the first round of loads.
template <typename T, int D>
__device__ __forceinline__ void reduce_combine_row(T* __restrict__ out, const float* __restrict__ part_o,
                                                   const float* __restrict__ part_m,
                                                   const float* __restrict__ part_l, size_t base, size_t row,
                                                   int np, float mp, float lp,
                                                   const float (&o_early)[kReduceEarly][D / 32], int lane) {
  constexpr int DPL = D / 32;
  if (lane >= np) mp = -INFINITY;
  // global max over all partitions (np may exceed 32)
  float M = mp;
  for (int p = 32 + lane; p < np; p += 32) M = fmaxf(M, part_m[base + p]);
  M = warp_max(M);
  float acc[DPL];
#pragma unroll
  for (int e = 0; e < DPL; ++e) acc[e] = 0.f;
  float W = 0.f;
  for (int p0 = 0; p0 < np; p0 += 32) {
    float wp = 0.f;
    if (p0 == 0) {
      wp = mp == -INFINITY ? 0.f : lp * fast_exp2(mp - M);
    } else if (p0 + lane < np) {
      const float m2 = part_m[base + p0 + lane];
      wp = m2 == -INFINITY ? 0.f : part_l[base + p0 + lane] * fast_exp2(m2 - M);
    }
    W += wp;
    const int cnt = np - p0 < 32 ? np - p0 : 32;
    int k = 0;
    if (p0 == 0) {
#pragma unroll
      for (int q = 0; q < kReduceEarly; ++q) {
        const float w = __shfl_sync(kFull, wp, q);
        if (q < cnt) {
#pragma unroll
          for (int e = 0; e < DPL; ++e) acc[e] = fmaf(w, o_early[q][e], acc[e]);
        }
      }
      k = kReduceEarly;
    }
    for (; k < cnt; ++k) {
      const float w = __shfl_sync(kFull, wp, k);
      const float* o = part_o + (base + p0 + k) * D + lane * DPL;
      if constexpr (DPL == 4) {
        const float4 v = *reinterpret_cast<const float4*>(o);
        acc[0] = fmaf(w, v.x, acc[0]);
        acc[1] = fmaf(w, v.y, acc[1]);
        acc[2] = fmaf(w, v.z, acc[2]);
        acc[3] = fmaf(w, v.w, acc[3]);
      } else {
        const float2 v = *reinterpret_cast<const float2*>(o);
        acc[0] = fmaf(w, v.x, acc[0]);
        acc[1] = fmaf(w, v.y, acc[1]);
      }
    }
  }
  W = warp_sum(W);
  const float inv = W > 0.f ? 1.f / W : 0.f;
  T* dst = out + row * D + lane * DPL;
  if constexpr (DPL == 4) {
    uint2 v;
    v.x = Elem<T>::pack2(acc[0] * inv, acc[1] * inv);
    v.y = Elem<T>::pack2(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(dst) = v;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = Elem<T>::pack2(acc[0] * inv, acc[1] * inv);
  }
}

// Decode: output row (seq, head), kReduceRows rows per CTA. One round of loads
// (the context length, and the row's first partials) precedes the partition
// count, which hides one memory round trip.
template <typename T, int D>
__global__ void __launch_bounds__(32 * kReduceRows)
    pkv_reduce_kernel(T* __restrict__ out, const float* __restrict__ part_o, const float* __restrict__ part_m,
                      const float* __restrict__ part_l, const int32_t* __restrict__ context_lens, int num_seqs,
                      int num_heads, int partition_size, int max_partitions, int ctx_limit) {
  pdl_begin();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t row = (size_t)blockIdx.x * kReduceRows + warp;  // seq * num_heads + h
  if (row >= (size_t)num_seqs * num_heads) return;
  const int s = (int)(row / num_heads);
  const size_t base = row * max_partitions;
  const int ctx_raw = context_lens[s];
  float mp, lp;
  float o_early[kReduceEarly][D / 32];
  reduce_load_row<D>(part_o, part_m, part_l, base, max_partitions, lane, mp, lp, o_early);
  const int ctx = ctx_raw < 0 ? 0 : (ctx_raw > ctx_limit ? ctx_limit : ctx_raw);
  const int np = (ctx + partition_size - 1) / partition_size;
  if (np <= 1) return;  // the decode kernel wrote this row directly
  reduce_combine_row<T, D>(out, part_o, part_m, part_l, base, row, np, mp, lp, o_early, lane);
}

// Multi-query: one CTA per (sequence, head). It reads the context length first and leaves at once
// when the context fits one partition (the attention kernel then wrote the rows directly); else
// its warps take the sequence's query rows (query token q0 + i, this head) in turn. No row has to
// search query_start_loc for its sequence.
template <typename T, int D>
__global__ void __launch_bounds__(32 * kReduceRows)
    pkv_reduce_mq_kernel(T* __restrict__ out, const float* __restrict__ part_o, const float* __restrict__ part_m,
                         const float* __restrict__ part_l, const int32_t* __restrict__ context_lens, int num_heads,
                         int partition_size, int max_partitions, int ctx_limit, const MqParams mq) {
  pdl_begin();
  const int s = blockIdx.x, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = context_lens[s];
  const int ctx = c < 0 ? 0 : (c > ctx_limit ? ctx_limit : c);
  const int np = (ctx + partition_size - 1) / partition_size;
  if (np <= 1) return;
  int q0 = 0;
  const int n = mq_query_len(mq, s, ctx, q0);
  if (n <= 0) return;  // n < 0: reported by the attention kernel, the rows are not written
  for (int i = warp; i < n; i += kReduceRows) {
    const size_t row = (size_t)(q0 + i) * num_heads + h;
    const size_t base = row * max_partitions;
    float mp, lp;
    float o_early[kReduceEarly][D / 32];
    reduce_load_row<D>(part_o, part_m, part_l, base, max_partitions, lane, mp, lp, o_early);
    reduce_combine_row<T, D>(out, part_o, part_m, part_l, base, row, np, mp, lp, o_early, lane);
  }
}

// Shared-prefix decode: the output row (s, h) merges the prefix stage's np1
// partials (every sequence attends the same prefix) with its own tail's
// partials, ceil(tail_len / P2) of them, by the same log-sum-exp rule as the
// split-K reduce: out = sum_p l_p 2^(m_p - M) o_p / sum_p l_p 2^(m_p - M),
// M = max_p m_p (each o_p already divided by its l_p). One warp per row, lane
// l holds dims l * D / 32 ...
template <typename T, int D>
__global__ void __launch_bounds__(32 * kReduceRows)
    pkv_merge_prefix_kernel(T* __restrict__ out, const float* __restrict__ o1, const float* __restrict__ m1,
                            const float* __restrict__ l1, int np1, const float* __restrict__ o2,
                            const float* __restrict__ m2, const float* __restrict__ l2, int np2, int p2,
                            const int32_t* __restrict__ tail_lens, int tail_limit, int num_seqs, int num_heads) {
  pdl_begin();
  constexpr int DPL = D / 32;
  constexpr int EARLY = 8;  // prefix partials whose outputs are requested in the first round of loads
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t row = (size_t)blockIdx.x * kReduceRows + warp;
  if (row >= (size_t)num_seqs * num_heads) return;
  const int s = (int)(row / num_heads);
  auto at = [&](int q) { return q < np1 ? row * np1 + q : row * np2 + (q - np1); };
  auto load_o = [&](int q, float (&v)[DPL]) {  // lane's dims of partial q's output
    const float* o = (q < np1 ? o1 : o2) + at(q) * D + lane * DPL;
    if constexpr (DPL == 4) {
      const float4 x = *reinterpret_cast<const float4*>(o);
      v[0] = x.x, v[1] = x.y, v[2] = x.z, v[3] = x.w;
    } else {
      const float2 x = *reinterpret_cast<const float2*>(o);
      v[0] = x.x, v[1] = x.y;
    }
  };
  // First round of loads, all independent: the tail length, the prefix partials' m and l (lane q holds
  // partial q) and the first EARLY prefix partials' outputs. The prefix count is known without the tail.
  const int t_raw = tail_lens[s];
  float mq = -INFINITY, lq = 0.f;
  if (lane < np1) {
    mq = m1[at(lane)];
    lq = l1[at(lane)];
  }
  const int ne = np1 < EARLY ? np1 : EARLY;
  float oe[EARLY][DPL];
#pragma unroll
  for (int q = 0; q < EARLY; ++q)
    if (q < ne) load_o(q, oe[q]);
  // Second round: the tail's partials (its length clamped as the tail stage clamped it), and the output of
  // the first partial past the early ones
  const int t = t_raw < 0 ? 0 : (t_raw > tail_limit ? tail_limit : t_raw);
  const int n = np1 + (t + p2 - 1) / p2;
  if (lane >= np1 && lane < n) {
    mq = m2[at(lane)];
    lq = l2[at(lane)];
  }
  float on[DPL];
  if (ne < n) load_o(ne, on);
  float M = mq;
  for (int q = 32 + lane; q < n; q += 32) M = fmaxf(M, q < np1 ? m1[at(q)] : m2[at(q)]);
  M = warp_max(M);
  // partial q < 32: its weight l_q 2^(m_q - M) sits in lane q
  const float wl = mq == -INFINITY ? 0.f : lq * fast_exp2(mq - M);
  float W = warp_sum(wl);
  float acc[DPL];
#pragma unroll
  for (int e = 0; e < DPL; ++e) acc[e] = 0.f;
#pragma unroll
  for (int q = 0; q < EARLY; ++q) {
    if (q < ne) {
      const float wk = __shfl_sync(kFull, wl, q);
#pragma unroll
      for (int e = 0; e < DPL; ++e) acc[e] = fmaf(wk, oe[q][e], acc[e]);
    }
  }
  const int n32 = n < 32 ? n : 32;
  if (ne < n32) {
    const float wk = __shfl_sync(kFull, wl, ne);
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[e] = fmaf(wk, on[e], acc[e]);
  }
#pragma unroll 4
  for (int q = ne + 1; q < n32; ++q) {  // independent loads of the remaining partial outputs
    const float wk = __shfl_sync(kFull, wl, q);
    float v[DPL];
    load_o(q, v);
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[e] = fmaf(wk, v[e], acc[e]);
  }
  for (int q0 = 32; q0 < n; q0 += 32) {  // more than 32 partials: weights 32 at a time
    float w = 0.f;
    if (q0 + lane < n) {
      const int q = q0 + lane;
      const float m = q < np1 ? m1[at(q)] : m2[at(q)];
      w = m == -INFINITY ? 0.f : (q < np1 ? l1[at(q)] : l2[at(q)]) * fast_exp2(m - M);
    }
    W += warp_sum(w);
    const int cnt = n - q0 < 32 ? n - q0 : 32;
#pragma unroll 4
    for (int k = 0; k < cnt; ++k) {
      const int q = q0 + k;
      const float wk = __shfl_sync(kFull, w, k);
      float v[DPL];
      load_o(q, v);
#pragma unroll
      for (int e = 0; e < DPL; ++e) acc[e] = fmaf(wk, v[e], acc[e]);
    }
  }
  const float inv = W > 0.f ? 1.f / W : 0.f;
  T* dst = out + row * D + lane * DPL;
  if constexpr (DPL == 4) {
    uint2 v;
    v.x = Elem<T>::pack2(acc[0] * inv, acc[1] * inv);
    v.y = Elem<T>::pack2(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(dst) = v;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = Elem<T>::pack2(acc[0] * inv, acc[1] * inv);
  }
}

// mq.query_start_loc == nullptr: decode rows (num_seqs * num_heads).
template <typename T>
cudaError_t launch_reduce(const DecodeParams& p, int num_seqs, int head_dim, cudaStream_t stream,
                          const MqParams& mq = MqParams{}) {
  T* out = static_cast<T*>(p.out);
  const float *po = p.part_o, *pm = p.part_m, *pl = p.part_l;
  if (mq.query_start_loc) {  // multi-query: a CTA per (sequence, head)
    const dim3 grid((unsigned)num_seqs, (unsigned)p.num_heads);
    if (head_dim == 128)
      return launch_kernel(pkv_reduce_mq_kernel<T, 128>, grid, dim3(32 * kReduceRows), 0, stream, out, po, pm, pl,
                           p.context_lens, p.num_heads, p.partition_size, p.max_partitions, p.ctx_limit, mq);
    return launch_kernel(pkv_reduce_mq_kernel<T, 64>, grid, dim3(32 * kReduceRows), 0, stream, out, po, pm, pl,
                         p.context_lens, p.num_heads, p.partition_size, p.max_partitions, p.ctx_limit, mq);
  }
  const size_t rows = (size_t)num_seqs * p.num_heads;
  const unsigned grid = (unsigned)((rows + kReduceRows - 1) / kReduceRows);
  if (head_dim == 128)
    return launch_kernel(pkv_reduce_kernel<T, 128>, dim3(grid), dim3(32 * kReduceRows), 0, stream, out, po, pm, pl,
                         p.context_lens, num_seqs, p.num_heads, p.partition_size, p.max_partitions, p.ctx_limit);
  return launch_kernel(pkv_reduce_kernel<T, 64>, dim3(grid), dim3(32 * kReduceRows), 0, stream, out, po, pm, pl,
                       p.context_lens, num_seqs, p.num_heads, p.partition_size, p.max_partitions, p.ctx_limit);
}

// ---------------------------------------------------------------------------
// copy-on-write block copy: every 16-byte piece of physical block src (all kv
// heads, K and V) goes to block dst. Grid: (pieces, pairs).

constexpr int kOrderBuckets = 1024;
// The sequences by context length, longest first: a counting sort into 1024 length classes of
// ceil(ctx_limit / 1024) tokens (the order within a class is arbitrary and does not change any result).
// One CTA. The 8-column and 128-row multi-query tiles dispatch their grids in this order.
__global__ void __launch_bounds__(1024)
    pkv_mq_order_kernel(const int32_t* __restrict__ context_lens, int num_seqs, int ctx_limit, int32_t* __restrict__ order) {
  pdl_begin();
  __shared__ int cnt[kOrderBuckets];
  __shared__ int wsum[32];
  const int t = threadIdx.x;
  cnt[t] = 0;
  __syncthreads();
  const int gran = max(1, (ctx_limit + kOrderBuckets - 1) / kOrderBuckets);
  auto key = [&](int s) {
    int c = context_lens[s];
    c = c < 0 ? 0 : (c > ctx_limit ? ctx_limit : c);
    return min(kOrderBuckets - 1, c / gran);
  };
  for (int s = t; s < num_seqs; s += kOrderBuckets) atomicAdd(&cnt[key(s)], 1);
  __syncthreads();
  // thread t takes class b = 1023 - t: its first position is the count of all longer classes
  const int b = kOrderBuckets - 1 - t;
  const int v = cnt[b];
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, x, o);
    if ((t & 31) >= o) x += y;
  }
  if ((t & 31) == 31) wsum[t >> 5] = x;
  __syncthreads();
  if (t < 32) {
    int w = wsum[t];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, w, o);
      if (t >= o) w += y;
    }
    wsum[t] = w;
  }
  __syncthreads();
  const int first = x - v + ((t >> 5) ? wsum[(t >> 5) - 1] : 0);
  cnt[b] = first;
  __syncthreads();
  for (int s = t; s < num_seqs; s += kOrderBuckets) order[atomicAdd(&cnt[key(s)], 1)] = s;
}


__global__ void pkv_copy_blocks_kernel(uint4* __restrict__ key_cache, uint4* __restrict__ value_cache,
                                       const int64_t* __restrict__ block_mapping, long long pieces_per_block,
                                       long long num_blocks, unsigned* err) {
  pdl_begin();
  const int pair = blockIdx.y;
  const long long src = block_mapping[2 * pair], dst = block_mapping[2 * pair + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(err, PKV_DEVERR_BLOCK_ID);
    return;
  }
  const uint4* ks = key_cache + src * pieces_per_block;
  const uint4* vs = value_cache + src * pieces_per_block;
  uint4* kd = key_cache + dst * pieces_per_block;
  uint4* vd = value_cache + dst * pieces_per_block;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < pieces_per_block; i += stride) {
    const uint4 k = __ldg(ks + i), v = __ldg(vs + i);
    kd[i] = k;
    vd[i] = v;
  }
}

// ---------------------------------------------------------------------------
// self-test of the bounded wait: an mbarrier expects 16 transaction bytes that
// no copy will ever deliver; the wait must give up after `limit` cycles and
// report PKV_DEVERR_TIMEOUT. Nothing is in flight when the kernel returns.

__global__ void pkv_wait_selftest_kernel(unsigned* err, long long limit) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&bar, 16);  // the phase now waits for 16 bytes that never come
  }
  __syncwarp();
  const bool done = __all_sync(kFull, mbar_wait(&bar, 0, limit));
  if (!done && threadIdx.x == 0) atomicOr(err, PKV_DEVERR_TIMEOUT);
}

// ---------------------------------------------------------------------------
// tensor maps for the grouped-query kernel

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
  }
  return fn;
}

// The pool viewed as a 2D array [num_blocks * num_kv_heads * block_size][head_dim],
// copied with the 128-byte swizzle in boxes of 128 bytes x block_size rows: 64
// dims of a 16-bit cache, or all 128 codes of an E4M3 cache.
bool make_pool_map(CUtensorMap* map, const void* base, long long rows, int head_dim, int block_size,
                   pkv_dtype_t dtype) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const bool fp8 = dtype == PKV_FP8_E4M3;
  const cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)head_dim * (fp8 ? 1 : 2)};
  const cuuint32_t box[2] = {fp8 ? 128u : 64u, (cuuint32_t)block_size};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUtensorMapDataType type = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                       : (dtype == PKV_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                           : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
  const CUresult r = enc(map, type,
                         2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// An FP8 pool as the tensor-memory multi-query tile reads it: each (block, kv head) tile lands as
// block_size rows of 128 codes, unswizzled (the tile widens them to f16 in shared memory).
bool make_pool_map_fp8_rows(CUtensorMap* map, const void* base, long long rows, int block_size) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {128, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {128u, (cuuint32_t)block_size};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The 16-bit pool as seen by the head_dim-128 tensor-core tiles: one copy per
// (block, kv head) tile of block_size rows, landing as 8-row atoms of
// 2 KB, each holding its rows' columns 0..63 (1 KB, 128-byte swizzled) then
// columns 64..127. Dimensions, innermost first: 64 columns, 8 rows of an atom
// (row stride), the two column halves (128 bytes apart), the atoms (8 rows
// apart).
bool make_pool_map_tc(CUtensorMap* map, const void* base, long long rows, int block_size, pkv_dtype_t dtype) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[4] = {64, 8, 2, (cuuint64_t)(rows / 8)};
  const cuuint64_t strides[3] = {256, 128, 2048};
  const cuuint32_t box[4] = {64, 8, 2, (cuuint32_t)(block_size / 8)};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  const CUtensorMapDataType type =
      dtype == PKV_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUresult r = enc(map, type, 4, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int max_partitions_for(int max_context_len, int partition_size) {
  const int n = (max_context_len + partition_size - 1) / partition_size;
  return n < 1 ? 1 : n;
}

std::atomic<int> g_mq_tile{PKV_MQ_TILE_AUTO};

// How one decode call runs and what workspace it needs.
struct Plan {
  bool mma;     // tensor-core grouped-query tile (else CUDA cores)
  int np;       // partitions per sequence
  size_t need;  // split-K workspace bytes
};

// One CTA per (partition of P tokens, head group, sequence). fp8: an FP8 (E4M3)
// cache, on the tensor-core tile for head_dim 128 and any group size up to 8 (MHA
// included), else the CUDA cores; a 16-bit cache takes the tensor-core tile for
// 2 <= G <= 8. Contexts longer than P leave one partial per partition.
Plan make_plan(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size, int max_context_len,
               int partition_size, bool fp8) {
  Plan pl{};
  const int G = num_heads / num_kv_heads;
  pl.mma = fp8 ? (G <= 8 && head_dim == 128) : (G >= 2 && G <= 8);
  const int P = partition_size ? partition_size : default_partition(max_context_len, block_size);
  pl.np = max_partitions_for(max_context_len, P);
  pl.need = pl.np > 1 ? (size_t)num_seqs * num_heads * pl.np * (head_dim + 2) * sizeof(float) : 0;
  return pl;
}

// A second stream (and its fork / join events) on which the shared-prefix call
// runs its prefix stage beside the tail stage. One per host thread and device,
// created on first use and kept until the process exits. null if creation failed
// (the call then runs its stages in order on the caller's stream).
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  bool tried = false;
};

SideStream* side_stream(int dev) {
  thread_local SideStream side[kMaxDevices];
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  SideStream& x = side[dev];
  if (!x.tried) {
    x.tried = true;
    if (cudaStreamCreateWithFlags(&x.s, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&x.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&x.join, cudaEventDisableTiming) != cudaSuccess)
      x.s = nullptr;
  }
  return x.s ? &x : nullptr;
}

size_t workspace_size(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                      int32_t block_size, int32_t max_context_len, int32_t partition_size, bool fp8) {
  if (num_seqs <= 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads || head_dim <= 0 ||
      block_size <= 0 || max_context_len < 0 || partition_size < 0)
    return 0;
  return make_plan(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_context_len, partition_size, fp8)
      .need;
}

// Both decode entry points. fp8: the caches hold E4M3 codes of value / k_scale
// and value / v_scale.
pkv_status_t decode_impl(void* out, const void* query, const void* key_cache, const void* value_cache,
                         const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens,
                         int32_t num_seqs, int32_t max_context_len, float scale, int32_t block_size,
                         int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                         pkv_dtype_t dtype, int32_t partition_size, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream, bool fp8, float k_scale, float v_scale) {
  g_msg[0] = '\0';
  if (num_seqs < 0) return fail(PKV_ERR_INVALID_ARG, "num_seqs < 0");
  if (dtype != PKV_F16 && dtype != PKV_BF16) return fail(PKV_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
  if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads)
    return fail(PKV_ERR_INVALID_ARG, "num_heads (%d) must be a positive multiple of num_kv_heads (%d)", num_heads,
                num_kv_heads);
  if (num_blocks <= 0 || max_blocks_per_seq <= 0)
    return fail(PKV_ERR_INVALID_ARG, "num_blocks and max_blocks_per_seq must be > 0");
  if (!supported_head_dim(head_dim)) return fail(PKV_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", head_dim);
  if (!supported_block_size(block_size))
    return fail(PKV_ERR_UNSUPPORTED, "block_size %d (supported: 8, 16, 32)", block_size);
  if (!isfinite(scale)) return fail(PKV_ERR_INVALID_ARG, "scale is not finite");
  if (fp8 && !(isfinite(k_scale) && isfinite(v_scale) && k_scale > 0.f && v_scale > 0.f))
    return fail(PKV_ERR_INVALID_ARG, "k_scale and v_scale must be finite and > 0");
  if (max_context_len < 0) return fail(PKV_ERR_INVALID_ARG, "max_context_len < 0");
  if ((long long)max_context_len > (long long)max_blocks_per_seq * block_size)
    return fail(PKV_ERR_INVALID_ARG, "max_context_len %d exceeds max_blocks_per_seq * block_size = %lld",
                max_context_len, (long long)max_blocks_per_seq * block_size);
  if (partition_size < 0) return fail(PKV_ERR_INVALID_ARG, "partition_size < 0");
  const int P = partition_size ? partition_size : default_partition(max_context_len, block_size);
  if (P % block_size || P < block_size || P > kMaxPartitionBlocks * block_size)
    return fail(PKV_ERR_UNSUPPORTED, "partition_size %d must be a multiple of block_size in [%d, %d]", P,
                block_size, kMaxPartitionBlocks * block_size);
  if (num_seqs > 65535 || num_heads > 65535)
    return fail(PKV_ERR_UNSUPPORTED, "num_seqs and num_heads must be <= 65535");
  if ((long long)num_blocks * num_kv_heads * block_size >= (1LL << 31))
    return fail(PKV_ERR_UNSUPPORTED, "pool rows num_blocks * num_kv_heads * block_size must be < 2^31");
  if (num_seqs == 0) return PKV_OK;
  if (!out || !query || !key_cache || !value_cache || !block_tables || !context_lens)
    return fail(PKV_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(out) || !aligned16(query) || !aligned16(key_cache) || !aligned16(value_cache))
    return fail(PKV_ERR_INVALID_ARG, "out, query and caches must be 16-byte aligned");

  const Plan pl = make_plan(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_context_len, P, fp8);
  if (pl.need) {
    if (!workspace) return fail(PKV_ERR_WORKSPACE, "workspace of %zu bytes required", pl.need);
    if (workspace_bytes < pl.need)
      return fail(PKV_ERR_WORKSPACE, "workspace of %zu bytes < %zu required", workspace_bytes, pl.need);
    if (!aligned16(workspace)) return fail(PKV_ERR_WORKSPACE, "workspace must be 16-byte aligned");
  }

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  unsigned* err = error_word(dev);
  if (!err) return fail(PKV_ERR_CUDA, "device error word unavailable on device %d", dev);

  DecodeParams p{};
  p.out = out;
  p.query = query;
  p.key_cache = static_cast<const unsigned char*>(key_cache);
  p.value_cache = static_cast<const unsigned char*>(value_cache);
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.err = err;
  p.scale_log2 = scale * 1.4426950408889634f * k_scale;
  p.v_scale = v_scale;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_heads = num_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = num_heads / num_kv_heads;
  p.num_blocks = num_blocks;
  p.partition_size = P;
  p.max_partitions = pl.np;
  p.ctx_limit = max_context_len;

  CUtensorMap kmap, vmap;
  memset(&kmap, 0, sizeof kmap);
  memset(&vmap, 0, sizeof vmap);
  if (pl.mma) {
    const long long rows = (long long)num_blocks * num_kv_heads * block_size;
    const pkv_dtype_t cache_dtype = fp8 ? PKV_FP8_E4M3 : dtype;
    const bool one_copy = !fp8 && head_dim == 128 && tile_one_copy();
    if (one_copy ? !make_pool_map_tc(&kmap, key_cache, rows, block_size, dtype) ||
                       !make_pool_map_tc(&vmap, value_cache, rows, block_size, dtype)
                 : !make_pool_map(&kmap, key_cache, rows, head_dim, block_size, cache_dtype) ||
                       !make_pool_map(&vmap, value_cache, rows, head_dim, block_size, cache_dtype))
      return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed for the KV pool");
  }

  if (pl.need) {
    float* ws = static_cast<float*>(workspace);
    const size_t rows = (size_t)num_seqs * num_heads * pl.np;
    p.part_o = ws;
    p.part_m = ws + rows * head_dim;
    p.part_l = p.part_m + rows;
  }
  if (fp8 && pl.mma) {
    e = dtype == PKV_F16 ? decode_mma_fp8_f16(p, kmap, vmap, head_dim, block_size, num_seqs, stream)
                         : decode_mma_fp8_bf16(p, kmap, vmap, head_dim, block_size, num_seqs, stream);
  } else if (fp8) {
    e = dtype == PKV_F16 ? decode_simt_fp8_f16(p, head_dim, block_size, num_seqs, stream)
                         : decode_simt_fp8_bf16(p, head_dim, block_size, num_seqs, stream);
  } else if (pl.mma) {
    e = dtype == PKV_F16 ? decode_mma_f16(p, kmap, vmap, head_dim, block_size, num_seqs, stream)
                         : decode_mma_bf16(p, kmap, vmap, head_dim, block_size, num_seqs, stream);
  } else {
    e = dtype == PKV_F16 ? decode_simt_f16(p, head_dim, block_size, num_seqs, stream)
                         : decode_simt_bf16(p, head_dim, block_size, num_seqs, stream);
  }
  if (e != cudaSuccess) return cuda_fail(e, "decode kernel launch");

  if (pl.np > 1) {
    e = dtype == PKV_F16 ? launch_reduce<__half>(p, num_seqs, head_dim, stream)
                         : launch_reduce<__nv_bfloat16>(p, num_seqs, head_dim, stream);
    if (e != cudaSuccess) return cuda_fail(e, "reduce kernel launch");
  }
  return PKV_OK;
}

// How a shared-prefix decode splits its work (paged_attention_decode_shared_prefix).
struct PrefixPlan {
  bool tensor;   // prefix stage on the tensor-memory tile (else the 8-column tile)
  int rt1;       // prefix row tiles per kv head (rows = num_seqs * group)
  int pp, np1;   // prefix partition size (tokens, whole 64-token tiles) and count
  int p2, np2;   // tail partition size and the most partitions a tail can have
  int rt2;       // tail row tiles per kv head (group rows)
};

PrefixPlan prefix_plan(int num_seqs, int group, int num_kv_heads, int block_size, int prefix_len,
                       int max_tail_len) {
  PrefixPlan pl{};
  const long long rows = (long long)num_seqs * group;
  // One threshold for 16-bit and FP8 pools: the partition count depends on the tile, and the workspace
  // size function does not know the pool's dtype.
  pl.tensor = rows >= PKV_MQ_WIDE_MIN_ROWS;
  const int rpt = pl.tensor ? 128 : 8;
  pl.rt1 = (int)((rows + rpt - 1) / rpt);
  // about 256 prefix CTAs, so that the whole GPU shares the prefix's tiles
  const long long per = (long long)num_kv_heads * (pl.rt1 > 0 ? pl.rt1 : 1);
  long long want = (256 + per - 1) / per;
  const int tiles = (prefix_len + 63) / 64;
  if (want > tiles) want = tiles;
  if (want < 1) want = 1;
  int pp = (int)(((prefix_len + want - 1) / want + 63) / 64 * 64);
  const int cap = kMaxPartitionBlocks * block_size;
  if (pp > cap) pp = cap;
  if (pp < 64) pp = 64;
  pl.pp = pp;
  pl.np1 = prefix_len > 0 ? (prefix_len + pp - 1) / pp : 0;
  pl.p2 = mq_default_partition(block_size);
  pl.np2 = max_partitions_for(max_tail_len, pl.p2);
  pl.rt2 = (group + 7) / 8;
  return pl;
}

}  // namespace

void set_last_error_message(const char* msg) { snprintf(g_msg, sizeof g_msg, "%s", msg); }

unsigned* device_error_word(int dev) { return error_word(dev); }

}  // namespace pkv

using namespace pkv;

extern "C" {

const char* pkv_status_string(pkv_status_t status) {
  switch (status) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
    case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
    case PKV_ERR_DEVICE_CHECK: return "PKV_ERR_DEVICE_CHECK";
  }
  return "PKV_UNKNOWN_STATUS";
}

const char* pkv_last_error_message(void) { return g_msg; }

pkv_status_t paged_kv_write(const void* key, const void* value, void* key_cache, void* value_cache,
                            const int64_t* slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                            int32_t head_dim, int32_t block_size, int32_t num_blocks, pkv_dtype_t dtype,
                            cudaStream_t stream) {
  g_msg[0] = '\0';
  if (num_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "num_tokens < 0");
  if (dtype != PKV_F16 && dtype != PKV_BF16) return fail(PKV_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
  if (num_kv_heads <= 0 || num_blocks <= 0) return fail(PKV_ERR_INVALID_ARG, "num_kv_heads and num_blocks must be > 0");
  if (!supported_head_dim(head_dim)) return fail(PKV_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", head_dim);
  if (!supported_block_size(block_size))
    return fail(PKV_ERR_UNSUPPORTED, "block_size %d (supported: 8, 16, 32)", block_size);
  if (num_tokens == 0) return PKV_OK;
  if (!key || !value || !key_cache || !value_cache || !slot_mapping)
    return fail(PKV_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(key) || !aligned16(value) || !aligned16(key_cache) || !aligned16(value_cache))
    return fail(PKV_ERR_INVALID_ARG, "key, value and caches must be 16-byte aligned");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  unsigned* err = error_word(dev);
  if (!err) return fail(PKV_ERR_CUDA, "device error word unavailable on device %d", dev);
  const int pieces = head_dim * 2 / 16;
  const long long total = (long long)num_tokens * num_kv_heads * pieces;
  const int threads = 256;
  long long blocks = (total + threads - 1) / threads;
  if (blocks > 65535LL * 16) blocks = 65535LL * 16;
  e = launch_kernel(pkv_write_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream,
                    static_cast<const uint4*>(key), static_cast<const uint4*>(value), static_cast<uint4*>(key_cache),
                    static_cast<uint4*>(value_cache), slot_mapping, num_tokens, num_kv_heads, pieces, block_size,
                    (long long)num_blocks * block_size, err);
  if (e != cudaSuccess) return cuda_fail(e, "paged_kv_write launch");
  return PKV_OK;
}

pkv_status_t paged_kv_write_fp8(const void* key, const void* value, void* key_cache, void* value_cache,
                                const int64_t* slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                                int32_t head_dim, int32_t block_size, int32_t num_blocks, pkv_dtype_t dtype,
                                float k_scale, float v_scale, cudaStream_t stream) {
  g_msg[0] = '\0';
  if (num_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "num_tokens < 0");
  if (dtype != PKV_F16 && dtype != PKV_BF16) return fail(PKV_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
  if (num_kv_heads <= 0 || num_blocks <= 0) return fail(PKV_ERR_INVALID_ARG, "num_kv_heads and num_blocks must be > 0");
  if (!supported_head_dim(head_dim)) return fail(PKV_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", head_dim);
  if (!supported_block_size(block_size))
    return fail(PKV_ERR_UNSUPPORTED, "block_size %d (supported: 8, 16, 32)", block_size);
  if (!(isfinite(k_scale) && isfinite(v_scale) && k_scale > 0.f && v_scale > 0.f))
    return fail(PKV_ERR_INVALID_ARG, "k_scale and v_scale must be finite and > 0");
  if (num_tokens == 0) return PKV_OK;
  if (!key || !value || !key_cache || !value_cache || !slot_mapping)
    return fail(PKV_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(key) || !aligned16(value) || !aligned16(key_cache) || !aligned16(value_cache))
    return fail(PKV_ERR_INVALID_ARG, "key, value and caches must be 16-byte aligned");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  unsigned* err = error_word(dev);
  if (!err) return fail(PKV_ERR_CUDA, "device error word unavailable on device %d", dev);
  const int pieces = head_dim / 16;  // 16 one-byte codes per 16-byte piece
  const long long total = (long long)num_tokens * num_kv_heads * pieces;
  const int threads = 256;
  long long blocks = (total + threads - 1) / threads;
  if (blocks > 65535LL * 16) blocks = 65535LL * 16;
  auto kern = dtype == PKV_F16 ? pkv_write_fp8_kernel<__half> : pkv_write_fp8_kernel<__nv_bfloat16>;
  e = launch_kernel(kern, dim3((unsigned)blocks), dim3(threads), 0, stream, static_cast<const uint4*>(key),
                    static_cast<const uint4*>(value), static_cast<uint4*>(key_cache),
                    static_cast<uint4*>(value_cache), slot_mapping, num_tokens, num_kv_heads, pieces, block_size,
                    (long long)num_blocks * block_size, k_scale, v_scale, err);
  if (e != cudaSuccess) return cuda_fail(e, "paged_kv_write_fp8 launch");
  return PKV_OK;
}

int32_t pkv_set_multi_query_tile(int32_t tile) {
  if (tile != PKV_MQ_TILE_AUTO && tile != PKV_MQ_TILE_COLUMNS && tile != PKV_MQ_TILE_ROWS &&
      tile != PKV_MQ_TILE_TENSOR && tile != PKV_MQ_TILE_PAIRS)
    return -1;
  return g_mq_tile.exchange(tile);
}

pkv_status_t paged_kv_copy_blocks(void* key_cache, void* value_cache, const int64_t* block_mapping,
                                  int32_t num_pairs, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                  int32_t num_blocks, pkv_dtype_t dtype, cudaStream_t stream) {
  g_msg[0] = '\0';
  if (num_pairs < 0) return fail(PKV_ERR_INVALID_ARG, "num_pairs < 0");
  if (dtype != PKV_F16 && dtype != PKV_BF16 && dtype != PKV_FP8_E4M3)
    return fail(PKV_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
  if (num_kv_heads <= 0 || num_blocks <= 0) return fail(PKV_ERR_INVALID_ARG, "num_kv_heads and num_blocks must be > 0");
  if (!supported_head_dim(head_dim)) return fail(PKV_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", head_dim);
  if (!supported_block_size(block_size))
    return fail(PKV_ERR_UNSUPPORTED, "block_size %d (supported: 8, 16, 32)", block_size);
  if (num_pairs > 65535) return fail(PKV_ERR_UNSUPPORTED, "num_pairs must be <= 65535 per call");
  if (num_pairs == 0) return PKV_OK;
  if (!key_cache || !value_cache || !block_mapping) return fail(PKV_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(key_cache) || !aligned16(value_cache))
    return fail(PKV_ERR_INVALID_ARG, "caches must be 16-byte aligned");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  unsigned* err = error_word(dev);
  if (!err) return fail(PKV_ERR_CUDA, "device error word unavailable on device %d", dev);
  const int elem_bytes = dtype == PKV_FP8_E4M3 ? 1 : 2;
  const long long pieces = (long long)num_kv_heads * block_size * head_dim * elem_bytes / 16;
  const int threads = 256;
  long long chunks = (pieces + threads * 4 - 1) / (threads * 4);  // about 4 pieces per thread
  if (chunks < 1) chunks = 1;
  e = launch_kernel(pkv_copy_blocks_kernel, dim3((unsigned)chunks, (unsigned)num_pairs), dim3(threads), 0, stream,
                    static_cast<uint4*>(key_cache), static_cast<uint4*>(value_cache), block_mapping, pieces,
                    (long long)num_blocks, err);
  if (e != cudaSuccess) return cuda_fail(e, "paged_kv_copy_blocks launch");
  return PKV_OK;
}

size_t paged_attention_workspace_size(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                      int32_t block_size, int32_t max_context_len, int32_t partition_size) {
  return workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_context_len, partition_size,
                        false);
}

size_t paged_attention_workspace_size_fp8(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                          int32_t head_dim, int32_t block_size, int32_t max_context_len,
                                          int32_t partition_size) {
  return workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_context_len, partition_size,
                        true);
}

pkv_status_t paged_attention_decode(void* out, const void* query, const void* key_cache, const void* value_cache,
                                    const int32_t* block_tables, int32_t max_blocks_per_seq,
                                    const int32_t* context_lens, int32_t num_seqs, int32_t max_context_len,
                                    float scale, int32_t block_size, int32_t num_heads, int32_t num_kv_heads,
                                    int32_t head_dim, int32_t num_blocks, pkv_dtype_t dtype,
                                    int32_t partition_size, void* workspace, size_t workspace_bytes,
                                    cudaStream_t stream) {
  return decode_impl(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                     max_context_len, scale, block_size, num_heads, num_kv_heads, head_dim, num_blocks, dtype,
                     partition_size, workspace, workspace_bytes, stream, false, 1.f, 1.f);
}

pkv_status_t paged_attention_decode_fp8(void* out, const void* query, const void* key_cache,
                                        const void* value_cache, const int32_t* block_tables,
                                        int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
                                        int32_t max_context_len, float scale, int32_t block_size,
                                        int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                        int32_t num_blocks, pkv_dtype_t dtype, float k_scale, float v_scale,
                                        int32_t partition_size, void* workspace, size_t workspace_bytes,
                                        cudaStream_t stream) {
  return decode_impl(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                     max_context_len, scale, block_size, num_heads, num_kv_heads, head_dim, num_blocks, dtype,
                     partition_size, workspace, workspace_bytes, stream, true, k_scale, v_scale);
}

namespace {
// Split-K partials of a multi-query call, at the start of its workspace.
size_t mq_partials_bytes(int num_query_tokens, int num_heads, int head_dim, int block_size, int max_context_len,
                         int partition_size) {
  const int P = partition_size ? partition_size : mq_default_partition(block_size);
  const int np = max_partitions_for(max_context_len, P);
  return np > 1 ? (size_t)num_query_tokens * num_heads * np * (head_dim + 2) * sizeof(float) : 0;
}
// The sequence order of the 128-row tile, after the partials: one int32 per sequence, and a sequence
// with query tokens has at least one, so num_query_tokens entries bound it.
size_t mq_order_bytes(int n) { return ((size_t)n * sizeof(int32_t) + 255) / 256 * 256; }
}  // namespace

size_t paged_attention_multi_query_workspace_size(int32_t num_query_tokens, int32_t num_heads, int32_t num_kv_heads,
                                                  int32_t head_dim, int32_t block_size, int32_t max_context_len,
                                                  int32_t partition_size) {
  if (num_query_tokens < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads || head_dim <= 0 ||
      block_size <= 0 || max_context_len < 0 || partition_size < 0)
    return 0;
  return mq_partials_bytes(num_query_tokens, num_heads, head_dim, block_size, max_context_len, partition_size) +
         mq_order_bytes(num_query_tokens);
}

namespace {
// Both multi-query entry points. fp8: the caches hold E4M3 codes of value / k_scale and
// value / v_scale; only the 8-column tile (head_dim 128) reads them.
pkv_status_t mq_impl(void* out, const void* query, const void* key_cache, const void* value_cache,
                     const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens,
                     const int32_t* query_start_loc, int32_t num_seqs, int32_t num_query_tokens,
                     int32_t max_query_len, int32_t max_context_len, float scale, int32_t block_size,
                     int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                     pkv_dtype_t dtype, int32_t partition_size, void* workspace, size_t workspace_bytes,
                     cudaStream_t stream, bool fp8, float k_scale, float v_scale) {
  g_msg[0] = '\0';
  if (num_seqs < 0 || num_query_tokens < 0 || max_query_len < 0)
    return fail(PKV_ERR_INVALID_ARG, "num_seqs, num_query_tokens and max_query_len must be >= 0");
  if (dtype != PKV_F16 && dtype != PKV_BF16) return fail(PKV_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
  if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads)
    return fail(PKV_ERR_INVALID_ARG, "num_heads (%d) must be a positive multiple of num_kv_heads (%d)", num_heads,
                num_kv_heads);
  if (num_blocks <= 0 || max_blocks_per_seq <= 0)
    return fail(PKV_ERR_INVALID_ARG, "num_blocks and max_blocks_per_seq must be > 0");
  if (!supported_head_dim(head_dim)) return fail(PKV_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", head_dim);
  if (!supported_block_size(block_size))
    return fail(PKV_ERR_UNSUPPORTED, "block_size %d (supported: 8, 16, 32)", block_size);
  if (!isfinite(scale)) return fail(PKV_ERR_INVALID_ARG, "scale is not finite");
  if (fp8 && !(isfinite(k_scale) && isfinite(v_scale) && k_scale > 0.f && v_scale > 0.f))
    return fail(PKV_ERR_INVALID_ARG, "k_scale and v_scale must be finite and > 0");
  if (fp8 && head_dim != 128)
    return fail(PKV_ERR_UNSUPPORTED, "multi-query over an FP8 pool needs head_dim 128 (got %d)", head_dim);
  if (max_context_len < 0) return fail(PKV_ERR_INVALID_ARG, "max_context_len < 0");
  if ((long long)max_context_len > (long long)max_blocks_per_seq * block_size)
    return fail(PKV_ERR_INVALID_ARG, "max_context_len %d exceeds max_blocks_per_seq * block_size = %lld",
                max_context_len, (long long)max_blocks_per_seq * block_size);
  if (max_query_len > max_context_len)
    return fail(PKV_ERR_INVALID_ARG, "max_query_len %d exceeds max_context_len %d", max_query_len, max_context_len);
  if (partition_size < 0) return fail(PKV_ERR_INVALID_ARG, "partition_size < 0");
  const int P = partition_size ? partition_size : mq_default_partition(block_size);
  if (P % block_size || P < block_size || P > kMaxPartitionBlocks * block_size)
    return fail(PKV_ERR_UNSUPPORTED, "partition_size %d must be a multiple of block_size in [%d, %d]", P,
                block_size, kMaxPartitionBlocks * block_size);
  const int G = num_heads / num_kv_heads;
  // Many rows per kv head go to a tile with query rows in the MMA's M, a few
  // to the 8-column tile, which reads no padding rows.
  // Over an FP8 pool, 9 to 32 rows run as 16-row pairs of 8-column groups, which widen each code once.
  const long long kv_rows = (long long)max_query_len * G;
  int tile = g_mq_tile.load(std::memory_order_relaxed);
  if (tile == PKV_MQ_TILE_AUTO)
    tile = kv_rows >= (fp8 ? PKV_MQ_WIDE_MIN_ROWS_FP8 : PKV_MQ_WIDE_MIN_ROWS) ? PKV_MQ_TILE_TENSOR
           : fp8 && kv_rows > 8                                             ? PKV_MQ_TILE_PAIRS
                                                                            : PKV_MQ_TILE_COLUMNS;
  if (fp8 && tile == PKV_MQ_TILE_ROWS) tile = PKV_MQ_TILE_COLUMNS;  // no FP8 form of the 64-row tile
  if (!fp8 && tile == PKV_MQ_TILE_PAIRS) tile = PKV_MQ_TILE_COLUMNS;  // the pairs exist for FP8 only
  const int rows_per_tile = tile == PKV_MQ_TILE_TENSOR ? 128
                            : tile == PKV_MQ_TILE_ROWS ? 64
                            : tile == PKV_MQ_TILE_PAIRS ? 16
                                                        : 8;
  const long long row_tiles = ((long long)max_query_len * G + rows_per_tile - 1) / rows_per_tile;
  if (num_seqs > 65535 || num_heads > 65535 || (long long)num_kv_heads * row_tiles > 65535)
    return fail(PKV_ERR_UNSUPPORTED,
                "num_seqs, num_heads and num_kv_heads * ceil(max_query_len * group / %d) must be <= 65535",
                rows_per_tile);
  if ((long long)num_blocks * num_kv_heads * block_size >= (1LL << 31))
    return fail(PKV_ERR_UNSUPPORTED, "pool rows num_blocks * num_kv_heads * block_size must be < 2^31");
  if ((long long)num_query_tokens * num_heads >= (1LL << 31))
    return fail(PKV_ERR_UNSUPPORTED, "num_query_tokens * num_heads must be < 2^31");
  if (num_seqs == 0 || num_query_tokens == 0 || max_query_len == 0) return PKV_OK;
  if (!out || !query || !key_cache || !value_cache || !block_tables || !context_lens || !query_start_loc)
    return fail(PKV_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(out) || !aligned16(query) || !aligned16(key_cache) || !aligned16(value_cache))
    return fail(PKV_ERR_INVALID_ARG, "out, query and caches must be 16-byte aligned");
  const int np = max_partitions_for(max_context_len, P);
  // the partials are required; room for the sequence order after them is optional (without it the
  // tiles run the sequences in index order)
  const size_t need = mq_partials_bytes(num_query_tokens, num_heads, head_dim, block_size, max_context_len,
                                        partition_size);
  if (need) {
    if (!workspace) return fail(PKV_ERR_WORKSPACE, "workspace of %zu bytes required", need);
    if (workspace_bytes < need)
      return fail(PKV_ERR_WORKSPACE, "workspace of %zu bytes < %zu required", workspace_bytes, need);
    if (!aligned16(workspace)) return fail(PKV_ERR_WORKSPACE, "workspace must be 16-byte aligned");
  }

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  unsigned* err = error_word(dev);
  if (!err) return fail(PKV_ERR_CUDA, "device error word unavailable on device %d", dev);

  DecodeParams p{};
  p.out = out;
  p.query = query;
  p.key_cache = static_cast<const unsigned char*>(key_cache);
  p.value_cache = static_cast<const unsigned char*>(value_cache);
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.err = err;
  p.scale_log2 = scale * 1.4426950408889634f * (fp8 ? k_scale : 1.f);  // scores in the base-2 domain
  p.v_scale = fp8 ? v_scale : 1.f;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_heads = num_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = G;
  p.num_blocks = num_blocks;
  p.partition_size = P;
  p.max_partitions = np;
  p.ctx_limit = max_context_len;
  if (need) {
    float* ws = static_cast<float*>(workspace);
    const size_t rows = (size_t)num_query_tokens * num_heads * np;
    p.part_o = ws;
    p.part_m = ws + rows * head_dim;
    p.part_l = p.part_m + rows;
  }
  MqParams mq{};
  mq.query_start_loc = query_start_loc;
  mq.num_query_tokens = num_query_tokens;
  mq.max_query_len = max_query_len;
  mq.row_tiles = (int)row_tiles;
  const size_t order_at = (need + 255) / 256 * 256;
  if (tile != PKV_MQ_TILE_ROWS && num_seqs > 1 && workspace && aligned16(workspace) &&
      workspace_bytes >= order_at + (size_t)num_seqs * sizeof(int32_t)) {
    int32_t* order = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(workspace) + order_at);
    e = launch_kernel(pkv_mq_order_kernel, dim3(1), dim3(kOrderBuckets), 0, stream, context_lens, num_seqs,
                      max_context_len, order);
    if (e != cudaSuccess) return cuda_fail(e, "sequence order kernel launch");
    mq.order = order;
  }

  CUtensorMap kmap, vmap;
  memset(&kmap, 0, sizeof kmap);
  memset(&vmap, 0, sizeof vmap);
  const long long rows = (long long)num_blocks * num_kv_heads * block_size;
  const bool tc_map = !fp8 && head_dim == 128 && (tile == PKV_MQ_TILE_TENSOR || tile_one_copy());
  const bool fp8_rows = fp8 && tile == PKV_MQ_TILE_TENSOR;
  const pkv_dtype_t cache_dtype = fp8 ? PKV_FP8_E4M3 : dtype;
  if (fp8_rows ? !make_pool_map_fp8_rows(&kmap, key_cache, rows, block_size) ||
                     !make_pool_map_fp8_rows(&vmap, value_cache, rows, block_size)
      : tc_map ? !make_pool_map_tc(&kmap, key_cache, rows, block_size, dtype) ||
                     !make_pool_map_tc(&vmap, value_cache, rows, block_size, dtype)
               : !make_pool_map(&kmap, key_cache, rows, head_dim, block_size, cache_dtype) ||
                     !make_pool_map(&vmap, value_cache, rows, head_dim, block_size, cache_dtype))
    return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed for the KV pool");
  if (fp8 && tile == PKV_MQ_TILE_PAIRS)
    e = dtype == PKV_F16 ? decode_mq_pairs_fp8_f16(p, mq, kmap, vmap, head_dim, block_size, num_seqs, stream)
                         : decode_mq_pairs_fp8_bf16(p, mq, kmap, vmap, head_dim, block_size, num_seqs, stream);
  else if (fp8)
    e = dtype == PKV_F16 ? decode_mq_fp8_f16(p, mq, kmap, vmap, head_dim, block_size, num_seqs, tile, stream)
                         : decode_mq_fp8_bf16(p, mq, kmap, vmap, head_dim, block_size, num_seqs, tile, stream);
  else
    e = dtype == PKV_F16 ? decode_mq_f16(p, mq, kmap, vmap, head_dim, block_size, num_seqs, tile, stream)
                         : decode_mq_bf16(p, mq, kmap, vmap, head_dim, block_size, num_seqs, tile, stream);
  if (e != cudaSuccess) return cuda_fail(e, "multi-query kernel launch");
  if (np > 1) {
    e = dtype == PKV_F16 ? launch_reduce<__half>(p, num_seqs, head_dim, stream, mq)
                         : launch_reduce<__nv_bfloat16>(p, num_seqs, head_dim, stream, mq);
    if (e != cudaSuccess) return cuda_fail(e, "reduce kernel launch");
  }
  return PKV_OK;
}
}  // namespace

pkv_status_t paged_attention_multi_query(void* out, const void* query, const void* key_cache,
                                         const void* value_cache, const int32_t* block_tables,
                                         int32_t max_blocks_per_seq, const int32_t* context_lens,
                                         const int32_t* query_start_loc, int32_t num_seqs, int32_t num_query_tokens,
                                         int32_t max_query_len, int32_t max_context_len, float scale,
                                         int32_t block_size, int32_t num_heads, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t num_blocks, pkv_dtype_t dtype,
                                         int32_t partition_size, void* workspace, size_t workspace_bytes,
                                         cudaStream_t stream) {
  return mq_impl(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq, context_lens,
                 query_start_loc, num_seqs, num_query_tokens, max_query_len, max_context_len, scale, block_size,
                 num_heads, num_kv_heads, head_dim, num_blocks, dtype, partition_size, workspace, workspace_bytes,
                 stream, false, 1.f, 1.f);
}

pkv_status_t paged_attention_multi_query_fp8(void* out, const void* query, const void* key_cache,
                                             const void* value_cache, const int32_t* block_tables,
                                             int32_t max_blocks_per_seq, const int32_t* context_lens,
                                             const int32_t* query_start_loc, int32_t num_seqs,
                                             int32_t num_query_tokens, int32_t max_query_len,
                                             int32_t max_context_len, float scale, int32_t block_size,
                                             int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                             int32_t num_blocks, pkv_dtype_t dtype, float k_scale, float v_scale,
                                             int32_t partition_size, void* workspace, size_t workspace_bytes,
                                             cudaStream_t stream) {
  return mq_impl(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq, context_lens,
                 query_start_loc, num_seqs, num_query_tokens, max_query_len, max_context_len, scale, block_size,
                 num_heads, num_kv_heads, head_dim, num_blocks, dtype, partition_size, workspace, workspace_bytes,
                 stream, true, k_scale, v_scale);
}

size_t paged_attention_shared_prefix_workspace_size(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                                    int32_t head_dim, int32_t block_size, int32_t prefix_len,
                                                    int32_t max_tail_len) {
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads || head_dim <= 0 ||
      block_size <= 0 || prefix_len < 0 || max_tail_len < 0)
    return 0;
  const PrefixPlan pl = prefix_plan(num_seqs, num_heads / num_kv_heads, num_kv_heads, block_size, prefix_len,
                                    max_tail_len);
  return (size_t)num_seqs * num_heads * (pl.np1 + pl.np2) * (head_dim + 2) * sizeof(float);
}

namespace {
// Both shared-prefix entry points. fp8: the caches hold E4M3 codes of value / k_scale and
// value / v_scale (head_dim 128); the stages run the multi-query kernels' FP8 forms.
pkv_status_t shared_prefix_impl(void* out, const void* query, const void* key_cache, const void* value_cache,
                                const int32_t* prefix_blocks, int32_t prefix_len, const int32_t* block_tables,
                                int32_t max_blocks_per_seq, const int32_t* tail_lens, int32_t num_seqs,
                                int32_t max_tail_len, float scale, int32_t block_size, int32_t num_heads,
                                int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks, pkv_dtype_t dtype,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream, bool fp8,
                                float k_scale, float v_scale) {
  g_msg[0] = '\0';
  if (num_seqs < 0 || prefix_len < 0 || max_tail_len < 0)
    return fail(PKV_ERR_INVALID_ARG, "num_seqs, prefix_len and max_tail_len must be >= 0");
  if (dtype != PKV_F16 && dtype != PKV_BF16) return fail(PKV_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
  if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads)
    return fail(PKV_ERR_INVALID_ARG, "num_heads (%d) must be a positive multiple of num_kv_heads (%d)", num_heads,
                num_kv_heads);
  if (num_blocks <= 0) return fail(PKV_ERR_INVALID_ARG, "num_blocks must be > 0");
  if (!supported_head_dim(head_dim)) return fail(PKV_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", head_dim);
  if (!supported_block_size(block_size))
    return fail(PKV_ERR_UNSUPPORTED, "block_size %d (supported: 8, 16, 32)", block_size);
  if (!isfinite(scale)) return fail(PKV_ERR_INVALID_ARG, "scale is not finite");
  if (fp8 && !(isfinite(k_scale) && isfinite(v_scale) && k_scale > 0.f && v_scale > 0.f))
    return fail(PKV_ERR_INVALID_ARG, "k_scale and v_scale must be finite and > 0");
  if (fp8 && head_dim != 128)
    return fail(PKV_ERR_UNSUPPORTED, "the shared-prefix call over an FP8 pool needs head_dim 128 (got %d)", head_dim);
  if (prefix_len % block_size)
    return fail(PKV_ERR_INVALID_ARG, "prefix_len %d must be a whole number of blocks of %d", prefix_len, block_size);
  if (max_tail_len > 0 && (max_blocks_per_seq <= 0 || (long long)max_tail_len > (long long)max_blocks_per_seq * block_size))
    return fail(PKV_ERR_INVALID_ARG, "max_tail_len %d exceeds max_blocks_per_seq * block_size", max_tail_len);
  const int G = num_heads / num_kv_heads;
  const PrefixPlan pl = prefix_plan(num_seqs, G, num_kv_heads, block_size, prefix_len, max_tail_len);
  if (num_seqs > 65535 || (long long)num_kv_heads * pl.rt1 > 65535 || (long long)num_kv_heads * pl.rt2 > 65535)
    return fail(PKV_ERR_UNSUPPORTED, "num_seqs and the kv heads' row tiles must be <= 65535");
  if ((long long)num_blocks * num_kv_heads * block_size >= (1LL << 31))
    return fail(PKV_ERR_UNSUPPORTED, "pool rows num_blocks * num_kv_heads * block_size must be < 2^31");
  if ((long long)num_seqs * num_heads >= (1LL << 31)) return fail(PKV_ERR_UNSUPPORTED, "num_seqs * num_heads >= 2^31");
  if (num_seqs == 0) return PKV_OK;
  if (!out || !query || !key_cache || !value_cache || !tail_lens || (prefix_len > 0 && !prefix_blocks) ||
      (max_tail_len > 0 && !block_tables))
    return fail(PKV_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(out) || !aligned16(query) || !aligned16(key_cache) || !aligned16(value_cache))
    return fail(PKV_ERR_INVALID_ARG, "out, query and caches must be 16-byte aligned");
  const size_t need = paged_attention_shared_prefix_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim,
                                                                   block_size, prefix_len, max_tail_len);
  if (!workspace) return fail(PKV_ERR_WORKSPACE, "workspace of %zu bytes required", need);
  if (workspace_bytes < need) return fail(PKV_ERR_WORKSPACE, "workspace of %zu bytes < %zu required", workspace_bytes, need);
  if (!aligned16(workspace)) return fail(PKV_ERR_WORKSPACE, "workspace must be 16-byte aligned");

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  unsigned* err = error_word(dev);
  if (!err) return fail(PKV_ERR_CUDA, "device error word unavailable on device %d", dev);

  const size_t rows = (size_t)num_seqs * num_heads;
  float* ws = static_cast<float*>(workspace);
  float *o1 = ws, *m1 = o1 + rows * pl.np1 * head_dim, *l1 = m1 + rows * pl.np1;
  float *o2 = l1 + rows * pl.np1, *m2 = o2 + rows * pl.np2 * head_dim, *l2 = m2 + rows * pl.np2;

  DecodeParams base{};
  base.out = out;
  base.query = query;
  base.key_cache = static_cast<const unsigned char*>(key_cache);
  base.value_cache = static_cast<const unsigned char*>(value_cache);
  base.err = err;
  base.scale_log2 = scale * 1.4426950408889634f * (fp8 ? k_scale : 1.f);  // scores in the base-2 domain
  base.v_scale = fp8 ? v_scale : 1.f;
  base.num_heads = num_heads;
  base.num_kv_heads = num_kv_heads;
  base.group = G;
  base.num_blocks = num_blocks;

  const long long pool_rows = (long long)num_blocks * num_kv_heads * block_size;
  auto maps = [&](int tile, CUtensorMap* km, CUtensorMap* vm) {
    memset(km, 0, sizeof *km);
    memset(vm, 0, sizeof *vm);
    if (fp8 && tile == PKV_MQ_TILE_TENSOR)
      return make_pool_map_fp8_rows(km, key_cache, pool_rows, block_size) &&
             make_pool_map_fp8_rows(vm, value_cache, pool_rows, block_size);
    if (fp8)
      return make_pool_map(km, key_cache, pool_rows, head_dim, block_size, PKV_FP8_E4M3) &&
             make_pool_map(vm, value_cache, pool_rows, head_dim, block_size, PKV_FP8_E4M3);
    if (head_dim == 128 && (tile == PKV_MQ_TILE_TENSOR || tile_one_copy()))
      return make_pool_map_tc(km, key_cache, pool_rows, block_size, dtype) &&
             make_pool_map_tc(vm, value_cache, pool_rows, block_size, dtype);
    return make_pool_map(km, key_cache, pool_rows, head_dim, block_size, dtype) &&
           make_pool_map(vm, value_cache, pool_rows, head_dim, block_size, dtype);
  };
  auto run = [&](const DecodeParams& p, const MqParams& mq, const CUtensorMap& km, const CUtensorMap& vm, int seqs,
                 int tile, cudaStream_t st) {
    if (fp8)
      return dtype == PKV_F16 ? decode_mq_fp8_f16(p, mq, km, vm, head_dim, block_size, seqs, tile, st)
                              : decode_mq_fp8_bf16(p, mq, km, vm, head_dim, block_size, seqs, tile, st);
    return dtype == PKV_F16 ? decode_mq_f16(p, mq, km, vm, head_dim, block_size, seqs, tile, st)
                            : decode_mq_bf16(p, mq, km, vm, head_dim, block_size, seqs, tile, st);
  };
  CUtensorMap kmap, vmap;
  // The prefix stage runs on a side stream beside the tail stage when both exist:
  // the fork event orders it after everything queued on `stream`, the join event
  // orders the merge after it.
  SideStream* side = pl.np1 > 0 && max_tail_len > 0 ? side_stream(dev) : nullptr;
  cudaStream_t prefix_stream = stream;
  if (side) {
    e = cudaEventRecord(side->fork, stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side->s, side->fork, 0);
    if (e != cudaSuccess) return cuda_fail(e, "side stream fork");
    prefix_stream = side->s;
  }
  // 1. the prefix, once: all num_seqs * group rows of a kv head as the query rows of one context
  if (pl.np1 > 0) {
    const int tile = pl.tensor ? PKV_MQ_TILE_TENSOR : PKV_MQ_TILE_COLUMNS;
    if (!maps(tile, &kmap, &vmap)) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed for the KV pool");
    DecodeParams p = base;
    p.block_tables = prefix_blocks;
    p.max_blocks_per_seq = prefix_len / block_size;
    p.partition_size = pl.pp;
    p.max_partitions = pl.np1;
    p.ctx_limit = prefix_len;
    p.part_o = o1;
    p.part_m = m1;
    p.part_l = l1;
    MqParams mq{};
    mq.mode = MQ_ONE_SEQ;
    mq.num_query_tokens = num_seqs;
    mq.max_query_len = num_seqs;
    mq.row_tiles = pl.rt1;
    mq.ctx_const = prefix_len;
    mq.causal = 0;
    mq.partials = 1;
    e = run(p, mq, kmap, vmap, 1, tile, prefix_stream);
    if (e != cudaSuccess) return cuda_fail(e, "shared-prefix kernel launch");
  }
  // 2. each sequence's tail: one query token per sequence over its own blocks
  if (max_tail_len > 0) {
    if (!maps(PKV_MQ_TILE_COLUMNS, &kmap, &vmap))
      return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed for the KV pool");
    DecodeParams p = base;
    p.block_tables = block_tables;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.context_lens = tail_lens;
    p.partition_size = pl.p2;
    p.max_partitions = pl.np2;
    p.ctx_limit = max_tail_len;
    p.part_o = o2;
    p.part_m = m2;
    p.part_l = l2;
    MqParams mq{};
    mq.mode = MQ_ONE_PER_SEQ;
    mq.num_query_tokens = num_seqs;
    mq.max_query_len = 1;
    mq.row_tiles = pl.rt2;
    mq.partials = 1;
    e = run(p, mq, kmap, vmap, num_seqs, PKV_MQ_TILE_COLUMNS, stream);
    if (e != cudaSuccess) return cuda_fail(e, "shared-prefix tail kernel launch");
  }
  if (side) {
    e = cudaEventRecord(side->join, side->s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, side->join, 0);
    if (e != cudaSuccess) return cuda_fail(e, "side stream join");
  }
  // 3. merge
  const unsigned grid = (unsigned)((rows + kReduceRows - 1) / kReduceRows);
  const dim3 blk(32 * kReduceRows);
  if (dtype == PKV_F16)
    e = head_dim == 128
            ? launch_kernel(pkv_merge_prefix_kernel<__half, 128>, dim3(grid), blk, 0, stream, static_cast<__half*>(out),
                            (const float*)o1, (const float*)m1, (const float*)l1, pl.np1, (const float*)o2,
                            (const float*)m2, (const float*)l2, pl.np2, pl.p2, tail_lens, max_tail_len, num_seqs,
                            num_heads)
            : launch_kernel(pkv_merge_prefix_kernel<__half, 64>, dim3(grid), blk, 0, stream, static_cast<__half*>(out),
                            (const float*)o1, (const float*)m1, (const float*)l1, pl.np1, (const float*)o2,
                            (const float*)m2, (const float*)l2, pl.np2, pl.p2, tail_lens, max_tail_len, num_seqs,
                            num_heads);
  else
    e = head_dim == 128
            ? launch_kernel(pkv_merge_prefix_kernel<__nv_bfloat16, 128>, dim3(grid), blk, 0, stream,
                            static_cast<__nv_bfloat16*>(out), (const float*)o1, (const float*)m1, (const float*)l1,
                            pl.np1, (const float*)o2, (const float*)m2, (const float*)l2, pl.np2, pl.p2, tail_lens,
                            max_tail_len, num_seqs, num_heads)
            : launch_kernel(pkv_merge_prefix_kernel<__nv_bfloat16, 64>, dim3(grid), blk, 0, stream,
                            static_cast<__nv_bfloat16*>(out), (const float*)o1, (const float*)m1, (const float*)l1,
                            pl.np1, (const float*)o2, (const float*)m2, (const float*)l2, pl.np2, pl.p2, tail_lens,
                            max_tail_len, num_seqs, num_heads);
  if (e != cudaSuccess) return cuda_fail(e, "shared-prefix merge launch");
  return PKV_OK;
}
}  // namespace

pkv_status_t paged_attention_decode_shared_prefix(void* out, const void* query, const void* key_cache,
                                                  const void* value_cache, const int32_t* prefix_blocks,
                                                  int32_t prefix_len, const int32_t* block_tables,
                                                  int32_t max_blocks_per_seq, const int32_t* tail_lens,
                                                  int32_t num_seqs, int32_t max_tail_len, float scale,
                                                  int32_t block_size, int32_t num_heads, int32_t num_kv_heads,
                                                  int32_t head_dim, int32_t num_blocks, pkv_dtype_t dtype,
                                                  void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return shared_prefix_impl(out, query, key_cache, value_cache, prefix_blocks, prefix_len, block_tables,
                            max_blocks_per_seq, tail_lens, num_seqs, max_tail_len, scale, block_size, num_heads,
                            num_kv_heads, head_dim, num_blocks, dtype, workspace, workspace_bytes, stream, false,
                            1.f, 1.f);
}

pkv_status_t paged_attention_decode_shared_prefix_fp8(void* out, const void* query, const void* key_cache,
                                                      const void* value_cache, const int32_t* prefix_blocks,
                                                      int32_t prefix_len, const int32_t* block_tables,
                                                      int32_t max_blocks_per_seq, const int32_t* tail_lens,
                                                      int32_t num_seqs, int32_t max_tail_len, float scale,
                                                      int32_t block_size, int32_t num_heads, int32_t num_kv_heads,
                                                      int32_t head_dim, int32_t num_blocks, pkv_dtype_t dtype,
                                                      float k_scale, float v_scale, void* workspace,
                                                      size_t workspace_bytes, cudaStream_t stream) {
  return shared_prefix_impl(out, query, key_cache, value_cache, prefix_blocks, prefix_len, block_tables,
                            max_blocks_per_seq, tail_lens, num_seqs, max_tail_len, scale, block_size, num_heads,
                            num_kv_heads, head_dim, num_blocks, dtype, workspace, workspace_bytes, stream, true,
                            k_scale, v_scale);
}

pkv_status_t pkv_selftest_wait_timeout(int64_t limit_cycles, cudaStream_t stream) {
  g_msg[0] = '\0';
  if (limit_cycles <= 0 || limit_cycles > kWaitLimitCycles)
    return fail(PKV_ERR_INVALID_ARG, "limit_cycles must be in (0, %lld]", kWaitLimitCycles);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  unsigned* err = error_word(dev);
  if (!err) return fail(PKV_ERR_CUDA, "device error word unavailable on device %d", dev);
  pkv_wait_selftest_kernel<<<1, 32, 0, stream>>>(err, (long long)limit_cycles);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return PKV_OK;
}

pkv_status_t paged_kv_device_errors(uint32_t* flags, int32_t clear) {
  g_msg[0] = '\0';
  if (!flags) return fail(PKV_ERR_INVALID_ARG, "flags is null");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  unsigned v = 0;
  e = cudaMemcpyFromSymbol(&v, g_pkv_error_word, sizeof v);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  if (clear) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_pkv_error_word, &zero, sizeof zero);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
  }
  *flags = v;
  return PKV_OK;
}

}  // extern "C"
