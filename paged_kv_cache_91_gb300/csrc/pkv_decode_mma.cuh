// Grouped-query decode attention over the paged KV pool on the tensor cores,
// serving all G = H / Hkv query heads of one kv head together, so each KV tile
// is read from HBM once per group ("Sparse Computation and Memory Management
// ...": GQA, 32 Q heads / 8 KV heads).
//
// With G >= 2 the per-block work is a dense contraction: for a 16-token slice
// of a block, S^T[16 x G] = K[16 x D] . Q^T[D x G] and O^T[D x G] += V^T[D x 16] .
// P^T[16 x G]. Both run as m16n8k16 warp MMAs with fp32 accumulation; the G
// query heads sit in the n = 8 dimension (G <= 8). The score fragment is turned
// into the PV operand in registers with movmatrix, so P never touches shared
// memory. P is rounded to the cache dtype for the PV product, and the running
// sum l adds the same rounded values, so weights and normaliser agree.
//
// Tiles come in through a 2D tensor map in boxes of 64 head dims x block_size
// tokens with the 128-byte swizzle, which makes every ldmatrix phase
// conflict-free. MmaTile holds the per-tile arithmetic of the grid kernel
// below (one CTA per (partition, kv head, sequence), per-warp rings).
#pragma once

#include "pkv_common.cuh"

namespace pkv {

#ifndef PKV_TILE_ONE_COPY
#define PKV_TILE_ONE_COPY 1  // head_dim 128: one 4-D copy per (block, kv head) tile (build-time knob)
#endif

// Byte offset of 16-byte piece `piece` (of D/8) of token row `t` inside a
// 16-bit (block, kv head) tile of NBOX = D/64 column halves in 128-byte
// swizzled rows. With one copy per tile the tile is a run of 8-row atoms of
// NBOX x 1024 bytes (each atom: its rows' columns 0..63, then 64..127, the
// layout a 4-D tensor map of the pool delivers); otherwise NBOX boxes of BS
// rows x 128 bytes, one per column half. For NBOX = 1 the two coincide.
template <int BS, int NBOX = 2>
__device__ __forceinline__ int swz_offset(int t, int piece) {
  const int box = piece >> 3, chunk = piece & 7;
  if (PKV_TILE_ONE_COPY)
    return (t >> 3) * (NBOX * 1024) + box * 1024 + (t & 7) * 128 + ((chunk ^ (t & 7)) << 4);
  return box * (BS * 128) + t * 128 + ((chunk ^ (t & 7)) << 4);
}

// Tiled 4D tensor copy global -> shared through a tensor map (x innermost).
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int x, int y, int z, int w,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
      "%5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
      : "memory");
}

// One (block, kv head) tile of a 16-bit pool into `dst` in the swz_offset
// layout; y is the tile's first row in the pool.
template <int D, int BS>
__device__ __forceinline__ void copy_tile16(unsigned char* dst, const CUtensorMap* map, int y, uint64_t* bar) {
  if constexpr (D == 128 && PKV_TILE_ONE_COPY) {
    tma_load_4d(dst, map, 0, 0, 0, y / 8, bar);
  } else {
#pragma unroll
    for (int b = 0; b < D / 64; ++b) tma_load_2d(dst + b * (BS * 128), map, 64 * b, y, bar);
  }
}

template <typename T_, int D_, int BS_>
struct MmaTile {
  using T = T_;  // query / output type, also the cache type
  static constexpr int D = D_;
  static constexpr int BS = BS_;
  static constexpr bool FP8 = false;
  static constexpr int MIN_CTAS = PKV_DECODE_MIN_CTAS;
  static constexpr int NBOX = D / 64;       // swizzled boxes per tile (64 dims x BS rows each)
  static constexpr int BOXB = BS * 128;     // bytes of one box
  static constexpr int TILE = NBOX * BOXB;  // = BS * D * 2
  static constexpr int CH = BS >= 16 ? BS / 16 : 1;  // 16-token slices per block
  static constexpr int KT = D / 16;                  // k-steps of the score MMA / m-tiles of PV
  using QB = uint32_t[KT][2];                        // Q^T operand registers
  static_assert(TILE == BS * D * 2, "tile bytes");
  static_assert(BOXB % 1024 == 0, "swizzle atoms need 1024-byte aligned boxes");

  // Q^T as the B operand of the score MMA: lane holds head n = lane / 4,
  // dims 2 (lane % 4) + {0, 1} (+ 8) of each 16-dim k-step. Heads >= G are zero.
  // `q` points at the group's first query row (G rows of D), global or shared.
  // sa, sb: the score multipliers of the lane's two columns (here both sl2).
  static __device__ __forceinline__ void load_qb(uint32_t (&qb)[KT][2], const T* q, int G, int lane, float sl2,
                                                 float& sa, float& sb) {
    sa = sl2;
    sb = sl2;
    load_qb_row(qb, (lane >> 2) < G ? q + (lane >> 2) * D : nullptr, lane);
  }

  // The same operand with column n = lane / 4 taken from the query row `qr`
  // (nullptr: a zero column).
  static __device__ __forceinline__ void load_qb_row(uint32_t (&qb)[KT][2], const T* qr, int lane) {
    const int kq = (lane & 3) * 2;
#pragma unroll
    for (int kk = 0; kk < KT; ++kk) {
      if (qr) {
        qb[kk][0] = *reinterpret_cast<const uint32_t*>(qr + kk * 16 + kq);
        qb[kk][1] = *reinterpret_cast<const uint32_t*>(qr + kk * 16 + 8 + kq);
      } else {
        qb[kk][0] = 0u;
        qb[kk][1] = 0u;
      }
    }
  }

  // Fold one (block, kv head) tile into the lane's running state for its two
  // heads (columns j0 = 2 (lane % 4), j0 + 1): tokens 0 .. nvalid-1 take part.
  // CAUSAL: besides, column j0 sees only tokens whose position tok_base + t is
  // below lim0 (lim1 for j0 + 1); a column may then see no token of a tile.
  // Zeroes the value rows past nvalid in shared memory (the stage then needs a
  // proxy fence before the copy engine refills it).
  template <bool CAUSAL = false>
  static __device__ __forceinline__ void run(unsigned char* Ks, unsigned char* Vs, int nvalid,
                                             const uint32_t (&qb)[KT][2], int lane, float sla, float slb,
                                             float& m0, float& m1, float& l0, float& l1, float (&acc)[KT][4],
                                             int tok_base = 0, int lim0 = 0, int lim1 = 0) {
    const int mi = lane >> 3;  // which 8x8 matrix this lane addresses in ldmatrix
    const int r8 = lane & 7;   // row inside that matrix
    const int r0 = lane >> 2;  // accumulator rows r0 and r0 + 8
    if (nvalid < BS) {
      // value rows past the context may hold anything (even NaN): zero them so
      // that their zero weights contribute exactly zero
      const int nz = (BS - nvalid) * (D / 8);
      for (int idx = lane; idx < nz; idx += 32) {
        const int t = nvalid + idx / (D / 8), piece = idx % (D / 8);
        *reinterpret_cast<uint4*>(Vs + swz_offset<BS, NBOX>(t, piece)) = make_uint4(0u, 0u, 0u, 0u);
      }
      __syncwarp();
    }
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      if (c * 16 < nvalid) {
        // scores S^T[token][head] for 16 tokens, in two accumulation chains
        float sacc[4] = {0.f, 0.f, 0.f, 0.f};
        {
          float sacc2[4] = {0.f, 0.f, 0.f, 0.f};
          const int rr = r8 + ((mi & 1) << 3);  // A rows 0..15
          const int t = BS >= 16 ? c * 16 + rr : (rr & (BS - 1));
#pragma unroll
          for (int kk = 0; kk < KT; ++kk) {
            uint32_t a[4];
            ldmatrix_x4(a, Ks + swz_offset<BS, NBOX>(t, kk * 2 + (mi >> 1)));
            if (kk & 1) {
              Mma<T>::run(sacc2, a, qb[kk][0], qb[kk][1]);
            } else {
              Mma<T>::run(sacc, a, qb[kk][0], qb[kk][1]);
            }
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) sacc[e] += sacc2[e];
        }
        const int ta = c * 16 + r0, tb = ta + 8;
        const bool va = (BS >= 16 || r0 < BS) && ta < nvalid;
        const bool vb = BS >= 16 && tb < nvalid;
        bool va0 = va, va1 = va, vb0 = vb, vb1 = vb;
        if constexpr (CAUSAL) {
          va0 = va && tok_base + ta < lim0;
          va1 = va && tok_base + ta < lim1;
          vb0 = vb && tok_base + tb < lim0;
          vb1 = vb && tok_base + tb < lim1;
        }
        const float x00 = va0 ? sacc[0] * sla : -INFINITY;
        const float x01 = va1 ? sacc[1] * slb : -INFINITY;
        const float x10 = vb0 ? sacc[2] * sla : -INFINITY;
        const float x11 = vb1 ? sacc[3] * slb : -INFINITY;
        // Lazy rescaling: a column's reference m moves (and its state is rescaled) only when one of its
        // scores exceeds m by more than 8, so p = 2^(x - m) <= 2^8. Each lane tests its own scores and the
        // warp votes; the max is reduced across the lanes only when some score does exceed.
        float mx0 = fmaxf(x00, x10), mx1 = fmaxf(x01, x11);
        if (__any_sync(kFull, mx0 > m0 + 8.f || mx1 > m1 + 8.f)) {
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, o));
            mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, o));
          }
          const bool up0 = mx0 > m0 + 8.f, up1 = mx1 > m1 + 8.f;
          const float mn0 = up0 ? mx0 : m0, mn1 = up1 ? mx1 : m1;
          // a column that keeps its m may still hold -inf there (it has seen nothing yet): factor 1
          const float al0 = up0 ? fast_exp2(m0 - mn0) : 1.f, al1 = up1 ? fast_exp2(m1 - mn1) : 1.f;
          l0 *= al0;
          l1 *= al1;
#pragma unroll
          for (int mt = 0; mt < KT; ++mt) {
            acc[mt][0] *= al0;
            acc[mt][1] *= al1;
            acc[mt][2] *= al0;
            acc[mt][3] *= al1;
          }
          m0 = mn0;
          m1 = mn1;
        }
        // a column that has seen no token yet keeps m = -inf (all its x are -inf): exponentiate against 0
        const float ms0 = m0 == -INFINITY ? 0.f : m0, ms1 = m1 == -INFINITY ? 0.f : m1;
        const uint32_t pa = Elem<T>::pack2(fast_exp2(x00 - ms0), fast_exp2(x01 - ms1));
        const uint32_t pb = Elem<T>::pack2(fast_exp2(x10 - ms0), fast_exp2(x11 - ms1));
        const float2 fa = Elem<T>::to_float2(pa), fb = Elem<T>::to_float2(pb);
        // l: this lane's rows only (the weights PV multiplies); finish() adds the lanes of a column
        l0 += fa.x + fb.x;
        l1 += fa.y + fb.y;
        // P^T as the B operand of the PV MMA: transpose the 8x8 score fragments
        const uint32_t b0 = movmatrix_trans(pa), b1 = movmatrix_trans(pb);
        {
          const int tr = r8 + ((mi >> 1) << 3);  // stored V rows 0..15
          const int t = BS >= 16 ? c * 16 + tr : (tr & (BS - 1));
#pragma unroll
          for (int mt = 0; mt < KT; ++mt) {
            uint32_t a[4];
            ldmatrix_x4_trans(a, Vs + swz_offset<BS, NBOX>(t, mt * 2 + (mi & 1)));
            Mma<T>::run(acc[mt], a, b0, b1);
          }
        }
      }
    }
  }

  // The running sums are complete after every tile here.
  // Complete the running sums: add the per-lane partial sums of each column.
  static __device__ __forceinline__ void finish(float& l0, float& l1) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0 += __shfl_xor_sync(kFull, l0, o);
      l1 += __shfl_xor_sync(kFull, l1, o);
    }
  }

  // The accumulators as red[head][dim] (head = column, dims in natural order).
  static __device__ __forceinline__ void store_acc(float* red, const float (&acc)[KT][4], int lane) {
    const int j0 = (lane & 3) * 2, r0 = lane >> 2;
#pragma unroll
    for (int mt = 0; mt < KT; ++mt) {
      const int d0 = mt * 16 + r0;
      red[j0 * D + d0] = acc[mt][0];
      red[(j0 + 1) * D + d0] = acc[mt][1];
      red[j0 * D + d0 + 8] = acc[mt][2];
      red[(j0 + 1) * D + d0 + 8] = acc[mt][3];
    }
  }

  // Issue the tensor-map copies of one (block, kv head) tile pair into a stage.
  static __device__ __forceinline__ void issue_tiles(unsigned char* st, const CUtensorMap* kmap,
                                                     const CUtensorMap* vmap, int y, uint64_t* bar) {
    copy_tile16<D, BS>(st, kmap, y, bar);
    copy_tile16<D, BS>(st + TILE, vmap, y, bar);
  }
};

template <int D, int BS, int NW, int SPW, int TILE_BYTES = BS * D * 2>
struct MmaShape {
  static constexpr int TILE = TILE_BYTES;
  static constexpr int STAGE = 2 * TILE;  // K tile + V tile
  static constexpr int RING = NW * SPW * STAGE;
  static constexpr int BARS = RING;
  static constexpr int SMEM_USED = BARS + ((NW * SPW * 8 + 15) / 16) * 16;
  static constexpr int SMEM = SMEM_USED + 1024;  // slack to align the ring to 1024 bytes
  static constexpr int RED_PER_WARP = (8 * D + 16) * 4;
  static_assert(RED_PER_WARP <= SPW * STAGE, "reduction scratch reuses the warp's ring");
};

// Tile: MmaTile (16-bit cache) or MmaTileE4M3 (FP8 cache, pkv_decode_mma_fp8.cuh).
template <typename Tile, int NW, int SPW>
__global__ void __launch_bounds__(NW * 32, Tile::MIN_CTAS)
    pkv_decode_gqa_mma_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap kmap,
                              const __grid_constant__ CUtensorMap vmap) {
  pdl_begin();
  using T = typename Tile::T;
  constexpr int D = Tile::D, BS = Tile::BS;
  using Sh = MmaShape<D, BS, NW, SPW, Tile::TILE>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  const int part = PKV_GRID_HEAD_FASTEST ? blockIdx.y : blockIdx.x;
  const int kvh = PKV_GRID_HEAD_FASTEST ? blockIdx.x : blockIdx.y;
  const int s = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;
  const int ctx = clamp_context(p, s, part == 0 && kvh == 0 && threadIdx.x == 0);
  const int P = p.partition_size;
  const int tok0 = part * P;
  const size_t row0 = (size_t)s * p.num_heads + (size_t)kvh * G;  // first query head row

  if (ctx == 0) {
    if (part == 0) {
      T* out = reinterpret_cast<T*>(p.out) + row0 * D;
      for (int i = threadIdx.x; i < G * D; i += NW * 32) out[i] = Elem<T>::from_float(0.f);
    }
    return;
  }
  if (tok0 >= ctx) return;
  const int tok1 = min(tok0 + P, ctx);
  const bool direct = ctx <= P;
  const int blk0 = tok0 / BS;
  const int nblk = (tok1 - tok0 + BS - 1) / BS;
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
        // generic stores (tail zeroing) into this stage must be ordered before the copy's writes
        if (PKV_PROXY_FENCE || ((zeroed >> (i % SPW)) & 1u)) fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, Sh::STAGE);
        Tile::issue_tiles(st, &kmap, &vmap, (phys * p.num_kv_heads + kvh) * BS, bar);
      } else {
        mbar_arrive(bar);
      }
    }
  };
  const int nfirst = nmine < SPW ? nmine : SPW;
  for (int i = 0; i < nfirst; ++i) issue(i);
  int issued = nfirst;

  typename Tile::QB qb;
  float sla, slb;  // score multipliers of this lane's two columns
  Tile::load_qb(qb, reinterpret_cast<const T*>(p.query) + row0 * D, G, lane, p.scale_log2, sla, slb);

  // running state of this lane's two heads (columns j0 = 2 (lane % 4), j0 + 1)
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float acc[Tile::KT][4];
#pragma unroll
  for (int mt = 0; mt < Tile::KT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;

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
      const int nvalid = min(BS, tok1 - (blk0 + lb) * BS);
      Tile::run(Ks, Ks + Sh::TILE, nvalid, qb, lane, sla, slb, m0, m1, l0, l1, acc);
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
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
#pragma unroll
    for (int mt = 0; mt < Tile::KT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
  }

  Tile::finish(l0, l1);

  // merge the warps: each warp writes [head][D] accumulators, m, l into its own ring slice
  float* red = reinterpret_cast<float*>(ring);
  float* red_m = red + 8 * D;
  float* red_l = red_m + 8;
  const int j0 = (lane & 3) * 2;
  Tile::store_acc(red, acc, lane);
  if (lane < 4) {
    red_m[j0] = m0;
    red_m[j0 + 1] = m1;
    red_l[j0] = l0;
    red_l[j0 + 1] = l1;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * D; idx += NW * 32) {
    const int g = idx / D, d = idx - g * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, reinterpret_cast<float*>(smem + w * SPW * Sh::STAGE)[8 * D + g]);
    float L = 0.f, o = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float* rw = reinterpret_cast<float*>(smem + w * SPW * Sh::STAGE);
      const float mw = rw[8 * D + g];
      const float f = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
      L += rw[8 * D + 8 + g] * f;
      o += rw[g * D + d] * f;
    }
    o = L > 0.f ? o / L : 0.f;
    if constexpr (Tile::FP8) o *= p.v_scale * Tile::UNIT;  // V codes in MMA units -> values
    const size_t row = row0 + g;
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

#ifndef PKV_MMA_RING_BYTES
#define PKV_MMA_RING_BYTES (64 * 1024)  // ring bytes per CTA (build-time tuning knob)
#endif

template <int STAGE_BYTES, int RING_BYTES = PKV_MMA_RING_BYTES>
constexpr int mma_stages() {
  constexpr int spw = RING_BYTES / (kDecodeWarps * STAGE_BYTES);
  return spw < 1 ? 1 : (spw > 6 ? 6 : spw);
}

// Tile: MmaTile<T, D, BS> or MmaTileE4M3<T, D, BS>; RING_BYTES: ring bytes per CTA.
template <typename Tile, int RING_BYTES = PKV_MMA_RING_BYTES>
cudaError_t launch_decode_gqa_mma(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                  int num_seqs, cudaStream_t stream) {
  constexpr int NW = kDecodeWarps;
  constexpr int SPW = mma_stages<2 * Tile::TILE, RING_BYTES>();
  using Sh = MmaShape<Tile::D, Tile::BS, NW, SPW, Tile::TILE>;
  auto kern = pkv_decode_gqa_mma_kernel<Tile, NW, SPW>;
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
  const dim3 grid(PKV_GRID_HEAD_FASTEST ? p.num_kv_heads : p.max_partitions,
                  PKV_GRID_HEAD_FASTEST ? p.max_partitions : p.num_kv_heads, num_seqs);
  return launch_kernel(kern, grid, dim3(NW * 32), Sh::SMEM, stream, p, kmap, vmap);
}

}  // namespace pkv
