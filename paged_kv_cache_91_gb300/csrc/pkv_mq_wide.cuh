// Multi-query paged attention for many query rows per kv head (long
// chunked-prefill chunks): query rows in the MMA's M dimension.
//
// Same computation as pkv_mq_mma_kernel (pkv_decode_mq.cuh): the R = q_len * G
// (query token, head) rows of a (sequence, kv head), row r being query token
// r / G at position ctx - q_len + r / G, each attending the positions up to
// its own. Here a CTA takes 16 * NW rows and every warp owns 16 of them, the M
// of m16n8k16:
//   S[16 rows x 16 tokens] = Q[16 x D] . K^T   (Q fragments stay in registers;
//                                               K^T fragments come from ldmatrix)
//   O[16 rows x D] += P[16 x 16] . V           (P's score fragments are already
//                                               the A fragments; V^T from
//                                               ldmatrix.trans)
// so every K/V tile in shared memory serves 16 * NW rows at once, where the
// 8-column tile (pkv_decode_mq.cuh) serves 8. The warps share one ring of
// stages: a stage is refilled by the copy engine once all NW warps have
// released it (an "empty" mbarrier with NW arrivals), and its tail rows past
// the context are zeroed in the V fragments rather than in shared memory,
// since other warps may be reading the stage.
#pragma once

#include "pkv_decode_mq.cuh"

namespace pkv {

template <typename T, int D, int BS, int NW, int ST>
struct MqWideShape {
  static constexpr int TILE = BS * D * 2;  // one (block, kv head) tile, 16-bit elements
  static constexpr int STAGE = 2 * TILE;   // K tile + V tile
  static constexpr int RING = ST * STAGE;
  static constexpr int BARS = RING;  // full[ST] then empty[ST]
  static constexpr int SMEM = BARS + 2 * ST * 8 + 1024;  // + slack to align the ring to 1024 bytes
  static constexpr int ROWS = 16 * NW;                   // query rows per CTA
  static constexpr int KT = D / 16;                      // k-steps of S, 16-dim groups of O
  static constexpr int IDS = (kMaxPartitionBlocks + 31) / 32;  // block ids per lane
  static_assert(TILE % 1024 == 0 || BS * 128 % 1024 == 0, "swizzle atoms need 1024-byte aligned boxes");
};

#ifndef PKV_MQ_WIDE_MIN_CTAS
#define PKV_MQ_WIDE_MIN_CTAS 3  // __launch_bounds__ minimum CTAs per SM (build-time tuning knob)
#endif

template <typename T, int D, int BS, int NW, int ST>
__global__ void __launch_bounds__(NW * 32, PKV_MQ_WIDE_MIN_CTAS)
    pkv_mq_wide_kernel(const DecodeParams p, const MqParams mq, const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap) {
  pdl_begin();
  using Sh = MqWideShape<T, D, BS, NW, ST>;
  constexpr int KT = Sh::KT;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Sh::BARS);
  uint64_t* empty = full + ST;
  __shared__ int failed;

  const int part = blockIdx.x;
  const int kvh = blockIdx.y / mq.row_tiles, rt = blockIdx.y % mq.row_tiles;
  const int s = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, qd = lane & 3;
  const int G = p.group;
  const bool reporter = part == 0 && blockIdx.y == 0 && threadIdx.x == 0;
  const int ctx = mq_context(p, mq, s, reporter);
  int q0 = 0;
  const int q_len = mq_query_len(mq, s, ctx, q0);
  if (q_len < 0) {
    if (reporter) atomicOr(p.err, PKV_DEVERR_QUERY);
    return;
  }
  const int R = q_len * G;
  const int row0 = rt * Sh::ROWS;
  if (row0 >= R) return;
  const int P = p.partition_size;
  const int tok0 = part * P;
  if (tok0 >= ctx) return;
  const int lim_cta = mq_limit(mq, ctx, q_len, min(row0 + Sh::ROWS, R) - 1, G);  // the CTA's last row's limit
  const int tok1 = min(min(tok0 + P, ctx), lim_cta);
  const bool direct = !mq.partials && ctx <= P;
  const int blk0 = tok0 / BS;
  const int nblk = tok1 > tok0 ? (tok1 - tok0 + BS - 1) / BS : 0;

  // this warp's rows, this lane's two rows (g and g + 8) and their limits
  const int wrow0 = row0 + 16 * warp;
  const bool wactive = wrow0 < R;
  const int rA = wrow0 + g, rB = wrow0 + g + 8;
  const int limA = rA < R ? mq_limit(mq, ctx, q_len, rA, G) : 0;
  const int limB = rB < R ? mq_limit(mq, ctx, q_len, rB, G) : 0;
  const int lim_w = wactive ? mq_limit(mq, ctx, q_len, min(wrow0 + 16, R) - 1, G) : 0;

  if (threadIdx.x == 0) {
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
#pragma unroll
    for (int k = 0; k < ST; ++k) {
      mbar_init(full + k, 1);
      mbar_init(empty + k, NW);
    }
    fence_mbar_init();
    failed = 0;
  }
  __syncthreads();

  // physical block ids of the partition, lane l holding blocks l, l + 32, ...; bad ids become -1
  int ids[Sh::IDS];
#pragma unroll
  for (int u = 0; u < Sh::IDS; ++u) {
    const int b = lane + 32 * u;
    ids[u] = -1;
    if (b < nblk) {
      const int v = p.block_tables[(size_t)s * p.max_blocks_per_seq + blk0 + b];
      if ((unsigned)v < (unsigned)p.num_blocks) {
        ids[u] = v;
      } else if (warp == 0) {
        atomicOr(p.err, PKV_DEVERR_BLOCK_ID);
      }
    }
  }
  auto block_id = [&](int i) {  // all lanes of the warp call this
    int v = -1;
#pragma unroll
    for (int u = 0; u < Sh::IDS; ++u) {
      const int x = __shfl_sync(kFull, ids[u], i & 31);
      if ((i >> 5) == u) v = x;
    }
    return v;
  };
  // Warp 0 brings block i into stage i % ST (lane 0 issues).
  auto issue = [&](int i) {
    const int phys = block_id(i);
    if (lane == 0) {
      uint64_t* bar = full + (i % ST);
      unsigned char* st = smem + (i % ST) * Sh::STAGE;
      if (phys >= 0) {
        mbar_arrive_expect_tx(bar, Sh::STAGE);
        const int y = (phys * p.num_kv_heads + kvh) * BS;
        copy_tile16<D, BS>(st, &kmap, y, bar);
        copy_tile16<D, BS>(st + Sh::TILE, &vmap, y, bar);
      } else {
        mbar_arrive(bar);  // complete the phase without data; the block is skipped
      }
    }
  };
  int issued = 0;
  if (warp == 0) {
    const int n = nblk < ST ? nblk : ST;
    for (int i = 0; i < n; ++i) issue(i);
    issued = n;
  }

  // Q fragments (A operand, rows g and g + 8 of this warp), in registers for the whole loop
  uint32_t qa[KT][4];
  {
    const T* qA = rA < R ? reinterpret_cast<const T*>(p.query) +
                               ((size_t)(q0 + rA / G) * p.num_heads + kvh * G + rA % G) * D
                         : nullptr;
    const T* qB = rB < R ? reinterpret_cast<const T*>(p.query) +
                               ((size_t)(q0 + rB / G) * p.num_heads + kvh * G + rB % G) * D
                         : nullptr;
#pragma unroll
    for (int kk = 0; kk < KT; ++kk) {
      const int d0 = kk * 16 + 2 * qd;
      qa[kk][0] = qA ? *reinterpret_cast<const uint32_t*>(qA + d0) : 0u;
      qa[kk][1] = qB ? *reinterpret_cast<const uint32_t*>(qB + d0) : 0u;
      qa[kk][2] = qA ? *reinterpret_cast<const uint32_t*>(qA + d0 + 8) : 0u;
      qa[kk][3] = qB ? *reinterpret_cast<const uint32_t*>(qB + d0 + 8) : 0u;
    }
  }
  const float sl2 = p.scale_log2;

  float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
  float acc[2 * KT][4];  // O[rows g, g+8][dims 8j + 2qd, + 1]
#pragma unroll
  for (int j = 0; j < 2 * KT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

  constexpr int CH = BS >= 16 ? BS / 16 : 1;
  const int mi = lane >> 3, r8 = lane & 7;
  bool ok = true;
  for (int i = 0; i < nblk; ++i) {
    const int k = i % ST;
    if (!__all_sync(kFull, mbar_wait(full + k, (i / ST) & 1))) {
      ok = false;
      if (lane == 0) failed = 1;
    }
    const int base = (blk0 + i) * BS;  // position of the block's first token
    const int phys = block_id(i);
    if (ok && phys >= 0 && wactive && base < lim_w) {
      const unsigned char* Ks = smem + k * Sh::STAGE;
      const unsigned char* Vs = Ks + Sh::TILE;
      const int nvalid = min(BS, tok1 - base);
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        if (c * 16 < nvalid) {
          const int nv = min(16, nvalid - c * 16);  // valid tokens of this 16-token chunk
          // S = Q . K^T for 16 tokens (n-tile 0: tokens 0-7, n-tile 1: 8-15)
          // (four accumulation chains: even and odd k-steps of each n-tile)
          float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
          {
            float s2[4] = {0.f, 0.f, 0.f, 0.f}, s3[4] = {0.f, 0.f, 0.f, 0.f};
            const int tk = (mi >> 1) * 8 + r8;
            const int t = BS >= 16 ? c * 16 + tk : (tk & (BS - 1));
#pragma unroll
            for (int kk = 0; kk < KT; ++kk) {
              uint32_t b[4];
              ldmatrix_x4(b, Ks + swz_offset<BS, D / 64>(t, 2 * kk + (mi & 1)));
              if (kk & 1) {
                Mma<T>::run(s2, qa[kk], b[0], b[1]);
                Mma<T>::run(s3, qa[kk], b[2], b[3]);
              } else {
                Mma<T>::run(s0, qa[kk], b[0], b[1]);
                Mma<T>::run(s1, qa[kk], b[2], b[3]);
              }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              s0[e] += s2[e];
              s1[e] += s3[e];
            }
          }
          // masks: chunk token u at position base + c*16 + u sees row A iff u < nv and position < limA
          const int pos = base + c * 16;
          const int u0 = 2 * qd, u1 = 2 * qd + 1, u8 = 8 + 2 * qd, u9 = 9 + 2 * qd;
          float xA[4], xB[4];
          xA[0] = u0 < nv && pos + u0 < limA ? s0[0] * sl2 : -INFINITY;
          xA[1] = u1 < nv && pos + u1 < limA ? s0[1] * sl2 : -INFINITY;
          xA[2] = u8 < nv && pos + u8 < limA ? s1[0] * sl2 : -INFINITY;
          xA[3] = u9 < nv && pos + u9 < limA ? s1[1] * sl2 : -INFINITY;
          xB[0] = u0 < nv && pos + u0 < limB ? s0[2] * sl2 : -INFINITY;
          xB[1] = u1 < nv && pos + u1 < limB ? s0[3] * sl2 : -INFINITY;
          xB[2] = u8 < nv && pos + u8 < limB ? s1[2] * sl2 : -INFINITY;
          xB[3] = u9 < nv && pos + u9 < limB ? s1[3] * sl2 : -INFINITY;
          float mxA = fmaxf(fmaxf(xA[0], xA[1]), fmaxf(xA[2], xA[3]));
          float mxB = fmaxf(fmaxf(xB[0], xB[1]), fmaxf(xB[2], xB[3]));
          mxA = fmaxf(mxA, __shfl_xor_sync(kFull, mxA, 1));
          mxB = fmaxf(mxB, __shfl_xor_sync(kFull, mxB, 1));
          mxA = fmaxf(mxA, __shfl_xor_sync(kFull, mxA, 2));
          mxB = fmaxf(mxB, __shfl_xor_sync(kFull, mxB, 2));
          // lazy rescaling: a row's reference m moves only when a score exceeds it by more than 8
          const bool upA = mxA > mA + 8.f, upB = mxB > mB + 8.f;
          if (__any_sync(kFull, upA || upB)) {
            const float nA = upA ? mxA : mA, nB = upB ? mxB : mB;
            const float aA = fast_exp2(mA - (nA == -INFINITY ? 0.f : nA));
            const float aB = fast_exp2(mB - (nB == -INFINITY ? 0.f : nB));
            lA *= aA;
            lB *= aB;
#pragma unroll
            for (int j = 0; j < 2 * KT; ++j) {
              acc[j][0] *= aA;
              acc[j][1] *= aA;
              acc[j][2] *= aB;
              acc[j][3] *= aB;
            }
            mA = nA;
            mB = nB;
          }
          const float msA = mA == -INFINITY ? 0.f : mA, msB = mB == -INFINITY ? 0.f : mB;
          // P as the A operand of PV: rows g (a0, a2) and g + 8 (a1, a3), tokens 2qd.. (a0, a1) and 8+2qd.. (a2, a3)
          uint32_t pa[4];
          pa[0] = Elem<T>::pack2(fast_exp2(xA[0] - msA), fast_exp2(xA[1] - msA));
          pa[1] = Elem<T>::pack2(fast_exp2(xB[0] - msB), fast_exp2(xB[1] - msB));
          pa[2] = Elem<T>::pack2(fast_exp2(xA[2] - msA), fast_exp2(xA[3] - msA));
          pa[3] = Elem<T>::pack2(fast_exp2(xB[2] - msB), fast_exp2(xB[3] - msB));
          {
            const float2 f0 = Elem<T>::to_float2(pa[0]), f2 = Elem<T>::to_float2(pa[2]);
            const float2 f1 = Elem<T>::to_float2(pa[1]), f3 = Elem<T>::to_float2(pa[3]);
            lA += (f0.x + f0.y) + (f2.x + f2.y);  // this lane's part of row g's sum
            lB += (f1.x + f1.y) + (f3.x + f3.y);
          }
          // value rows past the context may hold NaN: their halves of the V fragments are zeroed
          uint32_t vm01 = 0xffffffffu, vm89 = 0xffffffffu;
          if (nv < 16) {
            vm01 = (u0 < nv ? 0x0000ffffu : 0u) | (u1 < nv ? 0xffff0000u : 0u);
            vm89 = (u8 < nv ? 0x0000ffffu : 0u) | (u9 < nv ? 0xffff0000u : 0u);
          }
          {
            const int tk = (mi & 1) * 8 + r8;
            const int t = BS >= 16 ? c * 16 + tk : (tk & (BS - 1));
#pragma unroll
            for (int j = 0; j < KT; ++j) {
              uint32_t v[4];
              ldmatrix_x4_trans(v, Vs + swz_offset<BS, D / 64>(t, 2 * j + (mi >> 1)));
              Mma<T>::run(acc[2 * j], pa, v[0] & vm01, v[1] & vm89);
              Mma<T>::run(acc[2 * j + 1], pa, v[2] & vm01, v[3] & vm89);
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + k);  // this warp is done with the stage
    if (warp == 0 && i + ST < nblk) {
      // refill the stage once every warp has released it
      if (!__all_sync(kFull, mbar_wait(empty + k, (i / ST) & 1))) {
        if (lane == 0) failed = 1;
        ok = false;
      }
      if (ok) {
        issue(i + ST);
        ++issued;
      }
    }
    if (!ok) break;
  }

  // row sums: add the four lanes of each row
  lA += __shfl_xor_sync(kFull, lA, 1);
  lB += __shfl_xor_sync(kFull, lB, 1);
  lA += __shfl_xor_sync(kFull, lA, 2);
  lB += __shfl_xor_sync(kFull, lB, 2);

  __syncthreads();
  if (warp == 0) {
    // every issued copy has landed before the CTA's shared memory goes away
    const int first = issued > ST ? issued - ST : 0;
    for (int j = first; j < issued; ++j) mbar_wait(full + (j % ST), (j / ST) & 1);
  }
  const bool bad = failed != 0;
  if (bad && threadIdx.x == 0) atomicOr(p.err, PKV_DEVERR_TIMEOUT);

  // each warp writes its own rows
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const int r = h2 ? rB : rA;
    if (r >= R) continue;
    const float m = h2 ? mB : mA;
    const float l = h2 ? lB : lA;
    const float inv = !bad && l > 0.f ? 1.f / l : 0.f;
    const size_t row = (size_t)(q0 + r / G) * p.num_heads + kvh * G + r % G;
#pragma unroll
    for (int j = 0; j < 2 * KT; ++j) {
      const int d = 8 * j + 2 * qd;
      const float o0 = acc[j][2 * h2] * inv, o1 = acc[j][2 * h2 + 1] * inv;
      if (direct) {
        *reinterpret_cast<uint32_t*>(reinterpret_cast<T*>(p.out) + row * D + d) = Elem<T>::pack2(o0, o1);
      } else {
        *reinterpret_cast<float2*>(p.part_o + (row * p.max_partitions + part) * D + d) = make_float2(o0, o1);
      }
    }
    if (!direct && qd == 0) {
      p.part_m[row * p.max_partitions + part] = bad ? -INFINITY : m;
      p.part_l[row * p.max_partitions + part] = bad ? 0.f : l;
    }
  }
}

#ifndef PKV_MQ_WIDE_STAGES
#define PKV_MQ_WIDE_STAGES 4  // ring stages per CTA of the wide multi-query kernel (build-time knob)
#endif

template <typename T, int D, int BS>
cudaError_t launch_mq_wide(const DecodeParams& p, const MqParams& mq, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, int num_seqs, cudaStream_t stream) {
  constexpr int NW = 4, ST = PKV_MQ_WIDE_STAGES;
  using Sh = MqWideShape<T, D, BS, NW, ST>;
  auto kern = pkv_mq_wide_kernel<T, D, BS, NW, ST>;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  const dim3 grid(p.max_partitions, p.num_kv_heads * mq.row_tiles, num_seqs);
  return launch_kernel(kern, grid, dim3(NW * 32), Sh::SMEM, stream, p, mq, kmap, vmap);
}

}  // namespace pkv
