// Multi-query paged attention over an FP8 (E4M3) pool with 16 (query token,
// head) rows of one kv head per CTA: two 8-column groups in the n dimension of
// the MMA, over one K/V ring.
//
// The 8-column tile (pkv_decode_mq.cuh with MmaTileE4M3) gives a kv head with
// 9 to 32 rows two to four CTAs, each of which streams the context and widens
// every K and V code to f16 for its own 8 rows. Widening costs more issue slots
// than the MMAs it feeds (pkv_decode_mma_fp8.cuh). Here each 16-byte K or V
// chunk is loaded and widened once per CTA and feeds the MMAs of both groups,
// so a 16-row kv head costs one pass over its context instead of two.
//
// Everything else is the 8-column tile's: the warps split the partition's
// blocks, each with its own ring of (K, V) block tiles filled by tensor-map
// copies, each column has its own causal limit and online-softmax state, the
// warps merge through shared memory, and a context longer than one partition
// leaves (m, l, o) partials for the log-sum-exp reduce.
#pragma once

#include "pkv_decode_mma_fp8.cuh"
#include "pkv_decode_mq.cuh"

#ifndef PKV_MQ_PAIRS_MIN_CTAS
#define PKV_MQ_PAIRS_MIN_CTAS 3  // __launch_bounds__ minimum CTAs per SM (build-time tuning knob)
#endif

namespace pkv {

// One lane's running state for its two columns (2 (lane % 4), + 1) of a group.
struct PairCols {
  float m0, m1, l0, l1;  // running maxima (base 2) and sums
  float sla, slb;        // score multipliers (per-column 2^-k of a bf16 query)
  int lim0, lim1;        // causal limits: positions below them are seen
};

template <typename T_, int BS_>
struct E4M3Pairs {
  using Base = MmaTileE4M3<T_, 128, BS_>;
  using T = T_;
  static constexpr int D = 128;
  static constexpr int BS = BS_;
  static constexpr int KT = Base::KT;
  static constexpr int CH = Base::CH;
  static constexpr int TILE = Base::TILE;
  using QB = typename Base::QB;

  // The exponentials of one group's four scores against its references, with the
  // lazy rescale of MmaTileE4M3::run (a reference moves only when a score exceeds
  // it by more than 8), and P^T as the PV MMA's B operand (b0, b1).
  template <bool CAUSAL>
  static __device__ __forceinline__ void softmax(const float (&sacc)[4], bool va, bool vb, int ta, int tok_base,
                                                 PairCols& cs, float (&acc)[KT][4], uint32_t& b0, uint32_t& b1) {
    bool va0 = va, va1 = va, vb0 = vb, vb1 = vb;
    if constexpr (CAUSAL) {
      va0 = va && tok_base + ta < cs.lim0;
      va1 = va && tok_base + ta < cs.lim1;
      vb0 = vb && tok_base + ta + 8 < cs.lim0;
      vb1 = vb && tok_base + ta + 8 < cs.lim1;
    }
    const float x00 = va0 ? sacc[0] * cs.sla : -INFINITY;
    const float x01 = va1 ? sacc[1] * cs.slb : -INFINITY;
    const float x10 = vb0 ? sacc[2] * cs.sla : -INFINITY;
    const float x11 = vb1 ? sacc[3] * cs.slb : -INFINITY;
    // each lane tests its own scores and the warp votes; the max is reduced across the lanes only when
    // some score exceeds its column's reference by more than 8
    float mx0 = fmaxf(x00, x10), mx1 = fmaxf(x01, x11);
    if (__any_sync(kFull, mx0 > cs.m0 + 8.f || mx1 > cs.m1 + 8.f)) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, o));
      }
      const bool up0 = mx0 > cs.m0 + 8.f, up1 = mx1 > cs.m1 + 8.f;
      const float mn0 = up0 ? mx0 : cs.m0, mn1 = up1 ? mx1 : cs.m1;
      float al0 = fast_exp2(cs.m0 - mn0), al1 = fast_exp2(cs.m1 - mn1);
      if constexpr (CAUSAL) {  // a column that keeps its m may still hold -inf there
        if (!up0) al0 = 1.f;
        if (!up1) al1 = 1.f;
      }
      cs.l0 *= al0;
      cs.l1 *= al1;
#pragma unroll
      for (int mt = 0; mt < KT; ++mt) {
        acc[mt][0] *= al0;
        acc[mt][1] *= al1;
        acc[mt][2] *= al0;
        acc[mt][3] *= al1;
      }
      cs.m0 = mn0;
      cs.m1 = mn1;
    }
    float r0 = cs.m0, r1 = cs.m1;
    if constexpr (CAUSAL) {  // a column that has seen nothing yet: against 0 (its x are all -inf)
      if (r0 == -INFINITY) r0 = 0.f;
      if (r1 == -INFINITY) r1 = 0.f;
    }
    const uint32_t pa = Elem<__half>::pack2(fast_exp2(x00 - r0), fast_exp2(x01 - r1));
    const uint32_t pb = Elem<__half>::pack2(fast_exp2(x10 - r0), fast_exp2(x11 - r1));
    const float2 fa = Elem<__half>::to_float2(pa), fb = Elem<__half>::to_float2(pb);
    cs.l0 += fa.x + fb.x;  // this lane's rows only; Base::finish adds the lanes of a column
    cs.l1 += fa.y + fb.y;
    b0 = movmatrix_trans(pa);
    b1 = movmatrix_trans(pb);
  }

  // Fold one (block, kv head) tile into both groups: tokens 0 .. nvalid-1 take
  // part, column limits as in cs. The operand layouts are MmaTileE4M3's; the
  // widened K and V fragments are shared by the groups. Zeroes the value rows
  // past nvalid in shared memory (the stage then needs a proxy fence before the
  // copy engine refills it).
  template <bool CAUSAL>
  static __device__ __forceinline__ void run(unsigned char* Ks, unsigned char* Vs, int nvalid,
                                             const QB (&qb)[2], int lane, PairCols (&cs)[2],
                                             float (&acc)[2][KT][4], int tok_base) {
    const int g = lane >> 2, qd = lane & 3;
    if (nvalid < BS) {
      const int nz = (BS - nvalid) * 8;
      for (int idx = lane; idx < nz; idx += 32)
        *reinterpret_cast<uint4*>(Vs + (nvalid + idx / 8) * 128 + (idx % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
      __syncwarp();
    }
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      if (c * 16 < nvalid) {
        const int ta = c * 16 + g, tb = BS >= 16 ? ta + 8 : ta;
        const uint4 ka0 = *reinterpret_cast<const uint4*>(Ks + Base::off(ta, 2 * qd));
        const uint4 ka1 = *reinterpret_cast<const uint4*>(Ks + Base::off(ta, 2 * qd + 1));
        const uint4 kb0 = *reinterpret_cast<const uint4*>(Ks + Base::off(tb, 2 * qd));
        const uint4 kb1 = *reinterpret_cast<const uint4*>(Ks + Base::off(tb, 2 * qd + 1));
        const uint32_t wa[8] = {ka0.x, ka0.y, ka0.z, ka0.w, ka1.x, ka1.y, ka1.z, ka1.w};
        const uint32_t wb[8] = {kb0.x, kb0.y, kb0.z, kb0.w, kb1.x, kb1.y, kb1.z, kb1.w};
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < KT; ++j) {
          uint32_t a[4];
          e4m3x4_to_f16x2(wa[j], a[0], a[2]);
          e4m3x4_to_f16x2(wb[j], a[1], a[3]);
          Mma<__half>::run(s0, a, qb[0][j][0], qb[0][j][1]);
          Mma<__half>::run(s1, a, qb[1][j][0], qb[1][j][1]);
        }
        const bool va = ta < nvalid;
        const bool vb = BS >= 16 && ta + 8 < nvalid;
        uint32_t b[2][2];
        softmax<CAUSAL>(s0, va, vb, ta, tok_base, cs[0], acc[0], b[0][0], b[0][1]);
        softmax<CAUSAL>(s1, va, vb, ta, tok_base, cs[1], acc[1], b[1][0], b[1][1]);
        const int v0 = c * 16 + 2 * qd, v8 = BS >= 16 ? v0 + 8 : v0;
        const uint4 X0 = *reinterpret_cast<const uint4*>(Vs + Base::off(v0, g));
        const uint4 X1 = *reinterpret_cast<const uint4*>(Vs + Base::off(v0 + 1, g));
        const uint4 X8 = *reinterpret_cast<const uint4*>(Vs + Base::off(v8, g));
        const uint4 X9 = *reinterpret_cast<const uint4*>(Vs + Base::off(v8 + 1, g));
        const uint32_t x0[4] = {X0.x, X0.y, X0.z, X0.w}, x1[4] = {X1.x, X1.y, X1.z, X1.w};
        const uint32_t x8[4] = {X8.x, X8.y, X8.z, X8.w}, x9[4] = {X9.x, X9.y, X9.z, X9.w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint32_t lo01 = prmt(x0[w], x1[w], 0x5140), hi01 = prmt(x0[w], x1[w], 0x7362);
          const uint32_t lo89 = prmt(x8[w], x9[w], 0x5140), hi89 = prmt(x8[w], x9[w], 0x7362);
          uint32_t ae[4], ao[4];
          e4m3x4_to_f16x2(lo01, ae[0], ae[1]);
          e4m3x4_to_f16x2(lo89, ae[2], ae[3]);
          e4m3x4_to_f16x2(hi01, ao[0], ao[1]);
          e4m3x4_to_f16x2(hi89, ao[2], ao[3]);
#pragma unroll
          for (int gi = 0; gi < 2; ++gi) {
            Mma<__half>::run(acc[gi][2 * w], ae, b[gi][0], b[gi][1]);
            Mma<__half>::run(acc[gi][2 * w + 1], ao, b[gi][0], b[gi][1]);
          }
        }
      }
    }
  }
};

// Shared memory of the pair kernel: the 8-column tile's per-warp rings, at
// least large enough to hold the merge scratch of 16 columns.
template <int BS, int NW, int RING_BYTES>
struct PairShape {
  static constexpr int TILE = BS * 128;
  static constexpr int STAGE = 2 * TILE;
  static constexpr int RED_PER_WARP = (16 * 128 + 32) * 4;  // o[16][D], m[16], l[16]
  static constexpr int SPW_RING = mma_stages<STAGE, RING_BYTES>();
  static constexpr int SPW_RED = (RED_PER_WARP + STAGE - 1) / STAGE;
  static constexpr int SPW = SPW_RING > SPW_RED ? SPW_RING : SPW_RED;
  using Sh = MmaShape<128, BS, NW, SPW, TILE>;
  static_assert(RED_PER_WARP <= SPW * STAGE, "merge scratch reuses the warp's ring");
};

template <typename T, int BS, int NW, int SPW>
__global__ void __launch_bounds__(NW * 32, PKV_MQ_PAIRS_MIN_CTAS)
    pkv_mq_pairs_kernel(const DecodeParams p, const MqParams mq, const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap) {
  pdl_begin();
  using Tile = E4M3Pairs<T, BS>;
  using Base = typename Tile::Base;
  constexpr int D = 128;
  using Sh = MmaShape<D, BS, NW, SPW, Tile::TILE>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  const int part = blockIdx.x;
  const int kvh = blockIdx.y / mq.row_tiles, rt = blockIdx.y % mq.row_tiles;
  const int s = mq.order ? mq.order[blockIdx.z] : (int)blockIdx.z;  // long contexts first
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
  const int row0 = rt * 16;
  if (row0 >= R) return;  // no rows in this tile
  const int ncol = min(16, R - row0);
  const int P = p.partition_size;
  const int tok0 = part * P;
  if (tok0 >= ctx) return;
  const int lim_max = mq_limit(mq, ctx, q_len, row0 + ncol - 1, G);
  const int tok1 = min(min(tok0 + P, ctx), lim_max);
  const bool direct = !mq.partials && ctx <= P;
  const int blk0 = tok0 / BS;
  const int nblk = tok1 > tok0 ? (tok1 - tok0 + BS - 1) / BS : 0;
  const int nmine = warp < nblk ? (nblk - warp + NW - 1) / NW : 0;

  if (threadIdx.x == 0) {
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
  }

  int my_phys = -1;
  if (lane < nmine) {
    const int v = p.block_tables[(size_t)s * p.max_blocks_per_seq + blk0 + warp + NW * lane];
    if ((unsigned)v < (unsigned)p.num_blocks) {
      my_phys = v;
    } else {
      atomicOr(p.err, PKV_DEVERR_BLOCK_ID);
    }
  }

  unsigned char* ring = smem + warp * SPW * Sh::STAGE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sh::BARS) + warp * SPW;
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < SPW; ++k) mbar_init(bars + k, 1);
    fence_mbar_init();
  }
  __syncwarp();

  unsigned zeroed = 0;  // stages whose tail rows were zeroed since their last refill
  auto issue = [&](int i) {
    const int phys = __shfl_sync(kFull, my_phys, i);
    if (lane == 0) {
      uint64_t* bar = bars + (i % SPW);
      unsigned char* st = ring + (i % SPW) * Sh::STAGE;
      if (phys >= 0) {
        if (PKV_PROXY_FENCE || ((zeroed >> (i % SPW)) & 1u)) fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, Sh::STAGE);
        Base::issue_tiles(st, &kmap, &vmap, (phys * p.num_kv_heads + kvh) * BS, bar);
      } else {
        mbar_arrive(bar);
      }
    }
  };
  const int nfirst = nmine < SPW ? nmine : SPW;
  for (int i = 0; i < nfirst; ++i) issue(i);
  int issued = nfirst;

  // this lane's query column n = lane / 4 in each group (rows row0 + n and row0 + 8 + n), and the
  // limits of its two accumulator columns in each group
  typename Tile::QB qb[2];
  PairCols cs[2];
  const int j0 = (lane & 3) * 2;
#pragma unroll
  for (int gi = 0; gi < 2; ++gi) {
    const int n = 8 * gi + (lane >> 2);
    const T* qrow = nullptr;
    if (n < ncol) {
      const int r = row0 + n;
      qrow = reinterpret_cast<const T*>(p.query) + ((size_t)(q0 + r / G) * p.num_heads + kvh * G + r % G) * D;
    }
    Base::load_qb_row(qb[gi], qrow, lane, p.scale_log2, cs[gi].sla, cs[gi].slb);
    const int c0 = 8 * gi + j0;
    cs[gi].lim0 = c0 < ncol ? mq_limit(mq, ctx, q_len, row0 + c0, G) : 0;
    cs[gi].lim1 = c0 + 1 < ncol ? mq_limit(mq, ctx, q_len, row0 + c0 + 1, G) : 0;
    cs[gi].m0 = cs[gi].m1 = -INFINITY;
    cs[gi].l0 = cs[gi].l1 = 0.f;
  }
  float acc[2][Tile::KT][4];
#pragma unroll
  for (int gi = 0; gi < 2; ++gi)
#pragma unroll
    for (int mt = 0; mt < Tile::KT; ++mt) acc[gi][mt][0] = acc[gi][mt][1] = acc[gi][mt][2] = acc[gi][mt][3] = 0.f;

  int failed_at = -1;
  for (int i = 0; i < nmine; ++i) {
    const int phys = __shfl_sync(kFull, my_phys, i);
    const int k = i % SPW;
    const bool ready = __all_sync(kFull, mbar_wait(bars + k, (i / SPW) & 1));
    if (!ready) {
      failed_at = i;
      break;
    }
    if (phys >= 0) {
      unsigned char* Ks = ring + k * Sh::STAGE;
      const int lb = warp + NW * i;
      const int base = (blk0 + lb) * BS;
      const int nvalid = min(BS, tok1 - base);
      Tile::template run<true>(Ks, Ks + Sh::TILE, nvalid, qb, lane, cs, acc, base);
      if (nvalid < BS) zeroed |= 1u << k;
    }
    __syncwarp();
    if (i + SPW < nmine) {
      issue(i + SPW);
      zeroed &= ~(1u << k);
      ++issued;
    }
  }

  if (failed_at >= 0) {
    if (lane == 0) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
    for (int j = failed_at; j < issued; ++j) mbar_wait(bars + (j % SPW), (j / SPW) & 1);
#pragma unroll
    for (int gi = 0; gi < 2; ++gi) {
      cs[gi].m0 = cs[gi].m1 = -INFINITY;
      cs[gi].l0 = cs[gi].l1 = 0.f;
#pragma unroll
      for (int mt = 0; mt < Tile::KT; ++mt)
        acc[gi][mt][0] = acc[gi][mt][1] = acc[gi][mt][2] = acc[gi][mt][3] = 0.f;
    }
  }

  // merge the warps: each warp writes o[16][D], m[16], l[16] into its own ring slice
  float* red = reinterpret_cast<float*>(ring);
  float* red_m = red + 16 * D;
  float* red_l = red_m + 16;
#pragma unroll
  for (int gi = 0; gi < 2; ++gi) {
    Base::finish(cs[gi].l0, cs[gi].l1);
    Base::store_acc(red + 8 * gi * D, acc[gi], lane);
    if (lane < 4) {
      red_m[8 * gi + j0] = cs[gi].m0;
      red_m[8 * gi + j0 + 1] = cs[gi].m1;
      red_l[8 * gi + j0] = cs[gi].l0;
      red_l[8 * gi + j0 + 1] = cs[gi].l1;
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < ncol * D; idx += NW * 32) {
    const int n = idx / D, d = idx - n * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, reinterpret_cast<float*>(smem + w * SPW * Sh::STAGE)[16 * D + n]);
    float L = 0.f, o = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float* rw = reinterpret_cast<float*>(smem + w * SPW * Sh::STAGE);
      const float mw = rw[16 * D + n];
      const float f = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
      L += rw[16 * D + 16 + n] * f;
      o += rw[n * D + d] * f;
    }
    o = L > 0.f ? o / L : 0.f;
    o *= p.v_scale * Base::UNIT;  // V codes -> values
    const int r = row0 + n;
    const size_t row = (size_t)(q0 + r / G) * p.num_heads + kvh * G + r % G;  // output row (query token, head)
    if (direct) {
      reinterpret_cast<T*>(p.out)[row * D + d] = Elem<T>::from_float(o);
    } else {
      p.part_o[(row * p.max_partitions + part) * D + d] = o;
      if (d == 0) {
        p.part_m[row * p.max_partitions + part] = M;
        p.part_l[row * p.max_partitions + part] = L;
      }
    }
  }
}

template <typename T, int BS, int RING_BYTES = PKV_MMA_FP8_RING_BYTES>
cudaError_t launch_mq_pairs(const DecodeParams& p, const MqParams& mq, const CUtensorMap& kmap,
                            const CUtensorMap& vmap, int num_seqs, cudaStream_t stream) {
  constexpr int NW = kDecodeWarps;
  using PS = PairShape<BS, NW, RING_BYTES>;
  using Sh = typename PS::Sh;
  auto kern = pkv_mq_pairs_kernel<T, BS, NW, PS::SPW>;
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
