// Decode attention over the paged KV pool on the CUDA cores: used for MHA (one
// query head per kv head, where the per-block work is a matrix-vector product)
// and as the general path for group sizes the tensor-core kernel does not take.
//
// Method: "KV Cache와 PagedAttention 완전 해부", 부록 -- walk the sequence's
// blocks through the block table, score each block's keys, update a running
// softmax, accumulate the weighted values; "vLLM: LLM 서빙 메모리 최적화의
// 교과서", eq. (4).
//
// SimtTile holds the per-tile arithmetic of the grid kernel below, which runs
// one CTA per (context partition, query head, sequence): each warp owns a
// private ring of SPW stages, each stage the K tile and V tile of one (physical
// block, kv head) pair brought in by two linear bulk copies (TMA engine)
// completing on the stage's mbarrier; warp w takes the partition's blocks w,
// w+NW, ... and refills the stage it just consumed. A single-partition context writes its output
// directly; longer ones write (m, l, o) partials that pkv_reduce_kernel merges.
#pragma once

#include "pkv_common.cuh"

namespace pkv {

template <int D, int BS, int EB = 2>
struct SimtTileShape {
  static constexpr int TPC = BS < 16 ? BS : 16;  // tokens per score chunk
  static constexpr int CPB = BS / TPC;           // chunks per block
  static constexpr int LPT = 32 / TPC;           // lanes per token in the score pass
  static constexpr int DPL = D / LPT;            // head dims per lane in the score pass
  static constexpr int EPP = 16 / EB;            // elements per 16-byte piece
  static constexpr int NCH = DPL / EPP;          // 16-byte pieces per lane in the score pass
  static constexpr int DPV = D / 32;             // head dims per lane in the value pass
  static constexpr int ROWB = D * EB;            // bytes of one cached row
  static constexpr int TILE = BS * ROWB;         // bytes of one (block, kv head) tile
  static_assert(NCH == 1 || NCH == 2 || NCH == 4 || NCH == 8, "score-pass piece count");
  static_assert(DPV == 2 || DPV == 4, "value-pass width");
};

// Start piece of each lane in the score pass. Lane (t, pt) reads row t at byte
// pt * NCH * 16 + piece * 16. A warp's 16-byte loads are served 8 lanes at a
// time, and the 8 lanes must hit 8 different 16-byte bank groups; rows are 64,
// 128 or 256 bytes apart, so without a rotation several lanes of one group land
// in the same bank group. rotation_conflict_free() checks every case below.
template <int ROWB, int LPT, int NCH>
__host__ __device__ constexpr int qk_rotation(int lane) {
  const int t = lane / LPT, pt = lane % LPT;
  if (NCH == 1) return 0;
  if (NCH >= 8) return lane & 7;
  if (NCH == 4 && LPT == 2) return t & 3;
  if (NCH == 4) return ((pt >> 1) + 2 * t) & 3;
  if (ROWB == 64) return (t >> 1) & 1;  // NCH == 2, two lanes per 64-byte row
  return t & 1;                          // NCH == 2, four lanes per 128-byte row
}

template <int ROWB, int LPT, int NCH>
constexpr bool rotation_conflict_free() {
  for (int phase = 0; phase < 4; ++phase) {
    for (int i = 0; i < NCH; ++i) {
      unsigned used = 0;
      for (int k = 0; k < 8; ++k) {
        const int lane = phase * 8 + k;
        const int piece = (i + qk_rotation<ROWB, LPT, NCH>(lane)) & (NCH - 1);
        const int addr = (lane / LPT) * ROWB + (lane % LPT) * NCH * 16 + piece * 16;
        const unsigned bit = 1u << ((addr / 16) % 8);
        if (used & bit) return false;
        used |= bit;
      }
    }
  }
  return true;
}

// T: query/output type; C: cache element type (T itself, or __nv_fp8_e4m3).
template <typename T, typename C, int D, int BS>
struct SimtTile {
  using Fmt = CacheFmt<C>;
  static constexpr int EB = Fmt::EB;
  using Sh = SimtTileShape<D, BS, EB>;
  static_assert(rotation_conflict_free<Sh::ROWB, Sh::LPT, Sh::NCH>(), "score-pass bank conflicts");
  static constexpr int PAIR = 2 * EB;  // bytes of one element pair

  static __device__ __forceinline__ int rotation(int lane) { return qk_rotation<Sh::ROWB, Sh::LPT, Sh::NCH>(lane); }

  // This lane's slice of one query row for the score pass, scaled into the
  // base-2 domain and stored in rotated piece order. `q` is the row's first
  // element, in global or shared memory, 16-byte aligned.
  static __device__ __forceinline__ void load_q(float (&qreg)[Sh::DPL], const T* q, int lane, float scale_log2) {
    const int pt = lane % Sh::LPT;
    const int rot = rotation(lane);
#pragma unroll
    for (int i = 0; i < Sh::NCH; ++i) {
      const int piece = (i + rot) & (Sh::NCH - 1);
#pragma unroll
      for (int k = 0; k < Sh::EPP / 8; ++k) {
        const uint4 raw = *reinterpret_cast<const uint4*>(q + pt * Sh::DPL + piece * Sh::EPP + k * 8);
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = Elem<T>::to_float2(w[e]);
          qreg[i * Sh::EPP + k * 8 + 2 * e] = f.x * scale_log2;
          qreg[i * Sh::EPP + k * 8 + 2 * e + 1] = f.y * scale_log2;
        }
      }
    }
  }

  // Fold one (block, kv head) tile into the warp's running state (m, l, acc):
  // tokens 0 .. nvalid-1 of the tile take part, the rest are never read.
  static __device__ __forceinline__ void run(const unsigned char* Ks, const unsigned char* Vs, int nvalid,
                                             const float (&qreg)[Sh::DPL], int lane, float& m, float& l,
                                             float (&acc)[Sh::DPV]) {
    const int tl = lane / Sh::LPT, pt = lane % Sh::LPT;
    const int rot = rotation(lane);
#pragma unroll
    for (int c = 0; c < Sh::CPB; ++c) {
      if (c * Sh::TPC < nvalid) {
        // scores of this chunk's tokens: LPT lanes per token, fp32 accumulation
        const unsigned char* krow = Ks + (c * Sh::TPC + tl) * Sh::ROWB + pt * (Sh::NCH * 16);
        float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i2 = 0; i2 < Sh::NCH; ++i2) {
          const int piece = (i2 + rot) & (Sh::NCH - 1);
          const uint4 raw = *reinterpret_cast<const uint4*>(krow + piece * 16);
          const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
          for (int j = 0; j < Sh::EPP / 2; ++j) {  // element pairs of the piece
            float2 f;
            if constexpr (EB == 1) {
              if (j & 1) continue;  // pairs j, j + 1 come from one word
              float2 f2;
              Fmt::quad(w[j / 2], f, f2);
              a[(2 * j + 2) & 3] = fmaf(qreg[i2 * Sh::EPP + 2 * j + 2], f2.x, a[(2 * j + 2) & 3]);
              a[(2 * j + 3) & 3] = fmaf(qreg[i2 * Sh::EPP + 2 * j + 3], f2.y, a[(2 * j + 3) & 3]);
            } else {
              f = Fmt::pair(w[j]);
            }
            a[(2 * j) & 3] = fmaf(qreg[i2 * Sh::EPP + 2 * j], f.x, a[(2 * j) & 3]);
            a[(2 * j + 1) & 3] = fmaf(qreg[i2 * Sh::EPP + 2 * j + 1], f.y, a[(2 * j + 1) & 3]);
          }
        }
        float sc = (a[0] + a[1]) + (a[2] + a[3]);
#pragma unroll
        for (int o = Sh::LPT / 2; o > 0; o >>= 1) sc += __shfl_xor_sync(kFull, sc, o);
        const int nv = min(Sh::TPC, nvalid - c * Sh::TPC);
        sc = tl < nv ? sc : -INFINITY;  // tokens past the context do not take part

        // Running softmax with a lazily moved reference: m moves (and l and acc are
        // rescaled) only when a score exceeds it by more than 8, so every weight is
        // at most 2^8. Each lane tests its token and the warp votes; the max is
        // reduced (over the TPC distinct tokens: the LPT lanes of a token hold the
        // same score) only then.
        if (__any_sync(kFull, sc > m + 8.f)) {
          float mx = sc;
#pragma unroll
          for (int o = Sh::LPT; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
          const float alpha = fast_exp2(m - mx);  // 0 while m is still -inf (l and acc are 0 then)
          l *= alpha;
#pragma unroll
          for (int e = 0; e < Sh::DPV; ++e) acc[e] *= alpha;
          m = mx;
        }
        const float pr = fast_exp2(sc - m);
        if (pt == 0) l += pr;  // one lane per token; the lanes' sums are added after the last tile

        // weighted values: lane owns DPV consecutive head dims. A full chunk runs
        // without per-token branches so its loads can all be in flight at once;
        // a partial chunk never reads rows past the context.
        const unsigned char* vrow = Vs + (c * Sh::TPC) * Sh::ROWB + lane * (Sh::DPV * EB);
        if (nv == Sh::TPC) {
#pragma unroll
          for (int tt = 0; tt < Sh::TPC; ++tt) pv_row(acc, __shfl_sync(kFull, pr, tt * Sh::LPT), vrow + tt * Sh::ROWB);
        } else {
#pragma unroll
          for (int tt = 0; tt < Sh::TPC; ++tt) {
            const float w = __shfl_sync(kFull, pr, tt * Sh::LPT);
            if (tt < nv) pv_row(acc, w, vrow + tt * Sh::ROWB);
          }
        }
      }
    }
  }

  // acc[e] += w * V[row][lane dims e]
  static __device__ __forceinline__ void pv_row(float (&acc)[Sh::DPV], float w, const unsigned char* v) {
    constexpr int BYTES = Sh::DPV * EB;  // 8, 4 or 2
    uint32_t raw[2];
    if constexpr (BYTES == 8) {
      const uint2 r = *reinterpret_cast<const uint2*>(v);
      raw[0] = r.x;
      raw[1] = r.y;
    } else if constexpr (BYTES == 4) {
      raw[0] = *reinterpret_cast<const uint32_t*>(v);
    } else {
      raw[0] = *reinterpret_cast<const uint16_t*>(v);
    }
    if constexpr (EB == 1 && Sh::DPV == 4) {
      float2 f0, f1;
      Fmt::quad(raw[0], f0, f1);
      acc[0] = fmaf(w, f0.x, acc[0]);
      acc[1] = fmaf(w, f0.y, acc[1]);
      acc[2] = fmaf(w, f1.x, acc[2]);
      acc[3] = fmaf(w, f1.y, acc[3]);
    } else {
#pragma unroll
      for (int j = 0; j < Sh::DPV / 2; ++j) {
        const float2 f = Fmt::pair(raw[j * PAIR / 4] >> (8 * ((j * PAIR) % 4)));
        acc[2 * j] = fmaf(w, f.x, acc[2 * j]);
        acc[2 * j + 1] = fmaf(w, f.y, acc[2 * j + 1]);
      }
    }
  }
};

template <int D, int BS, int NW, int SPW, int EB = 2>
struct SimtShape : SimtTileShape<D, BS, EB> {
  static constexpr int STAGE = 2 * SimtTileShape<D, BS, EB>::TILE;  // K tile + V tile
  static constexpr int RING = NW * SPW * STAGE;
  static constexpr int BARS = RING;  // mbarriers follow the ring
  static constexpr int RED = BARS + ((NW * SPW * 8 + 15) / 16) * 16;
  static constexpr int SMEM = RED + NW * (D + 2) * 4;
};

template <typename T, typename C, int D, int BS, int NW, int SPW>
__global__ void __launch_bounds__(NW * 32, PKV_DECODE_MIN_CTAS) pkv_decode_simt_kernel(const DecodeParams p) {
  pdl_begin();
  using Tile = SimtTile<T, C, D, BS>;
  using Sh = SimtShape<D, BS, NW, SPW, Tile::EB>;
  extern __shared__ __align__(128) unsigned char smem[];

  const int part = PKV_GRID_HEAD_FASTEST ? blockIdx.y : blockIdx.x;
  const int h = PKV_GRID_HEAD_FASTEST ? blockIdx.x : blockIdx.y;
  const int s = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kvh = h / p.group;
  const int ctx = clamp_context(p, s, part == 0 && h == 0 && threadIdx.x == 0);
  const int P = p.partition_size;
  const int tok0 = part * P;
  const size_t out_row = (size_t)s * p.num_heads + h;

  if (ctx == 0) {  // empty context: zero output
    if (part == 0) {
      T* out = reinterpret_cast<T*>(p.out) + out_row * D;
      for (int d = threadIdx.x; d < D; d += NW * 32) out[d] = Elem<T>::from_float(0.f);
    }
    return;
  }
  if (tok0 >= ctx) return;  // partition past the end of this context
  const int tok1 = min(tok0 + P, ctx);
  const bool direct = ctx <= P;
  const int blk0 = tok0 / BS;
  const int nblk = (tok1 - tok0 + BS - 1) / BS;
  const int nmine = warp < nblk ? (nblk - warp + NW - 1) / NW : 0;  // <= 32 (host-checked)

  // physical block ids of this warp's blocks, one per lane; bad entries become -1
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

  const size_t head_off = (size_t)kvh * Sh::TILE;
  const size_t block_stride = (size_t)p.num_kv_heads * Sh::TILE;
  // Bring block i of this warp into stage i % SPW (all lanes call; lane 0 issues).
  auto issue = [&](int i) {
    const int phys = __shfl_sync(kFull, my_phys, i);
    if (lane == 0) {
      uint64_t* bar = bars + (i % SPW);
      unsigned char* st = ring + (i % SPW) * Sh::STAGE;
      if (phys >= 0) {
        if (PKV_PROXY_FENCE) fence_proxy_async_smem();  // earlier reads of this stage before the copy's writes
        mbar_arrive_expect_tx(bar, Sh::STAGE);
        const size_t off = (size_t)phys * block_stride + head_off;
        bulk_g2s(st, p.key_cache + off, Sh::TILE, bar);
        bulk_g2s(st + Sh::TILE, p.value_cache + off, Sh::TILE, bar);
      } else {
        mbar_arrive(bar);  // complete the phase without data; the block is skipped
      }
    }
  };
  const int nfirst = nmine < SPW ? nmine : SPW;
  for (int i = 0; i < nfirst; ++i) issue(i);
  int issued = nfirst;

  float qreg[Sh::DPL];
  Tile::load_q(qreg, reinterpret_cast<const T*>(p.query) + out_row * D, lane, p.scale_log2);

  float m = -INFINITY, l = 0.f;
  float acc[Sh::DPV];
#pragma unroll
  for (int e = 0; e < Sh::DPV; ++e) acc[e] = 0.f;

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
      const unsigned char* Ks = ring + k * Sh::STAGE;
      const int lb = warp + NW * i;
      const int nvalid = min(BS, tok1 - (blk0 + lb) * BS);
      Tile::run(Ks, Ks + Sh::TILE, nvalid, qreg, lane, m, l, acc);
    }
    __syncwarp();
    if (i + SPW < nmine) {
      issue(i + SPW);
      ++issued;
    }
  }

  if (failed_at >= 0) {
    // a copy did not arrive in time: report, let the other copies land, give a defined result
    if (lane == 0) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
    for (int j = failed_at; j < issued; ++j) mbar_wait(bars + (j % SPW), (j / SPW) & 1);
    m = -INFINITY;
    l = 0.f;
#pragma unroll
    for (int e = 0; e < Sh::DPV; ++e) acc[e] = 0.f;
  }
  l = warp_sum(l);  // the tiles' sums were kept per lane

  // merge the warps' running states
  float* red = reinterpret_cast<float*>(smem + Sh::RED);
  float* red_m = red + NW * D;
  float* red_l = red_m + NW;
#pragma unroll
  for (int e = 0; e < Sh::DPV; ++e) red[warp * D + lane * Sh::DPV + e] = acc[e];
  if (lane == 0) {
    red_m[warp] = m;
    red_l[warp] = l;
  }
  __syncthreads();
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < NW; ++w) M = fmaxf(M, red_m[w]);
  float f[NW];
  float L = 0.f;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    f[w] = red_m[w] == -INFINITY ? 0.f : fast_exp2(red_m[w] - M);
    L += red_l[w] * f[w];
  }
  float inv = L > 0.f ? 1.f / L : 0.f;
  if constexpr (Tile::EB == 1) inv *= p.v_scale;  // V codes -> values
  for (int d = threadIdx.x; d < D; d += NW * 32) {
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) o += red[w * D + d] * f[w];
    o *= inv;
    if (direct) {
      reinterpret_cast<T*>(p.out)[out_row * D + d] = Elem<T>::from_float(o);
    } else {
      p.part_o[(out_row * p.max_partitions + part) * D + d] = o;
    }
  }
  if (!direct && threadIdx.x == 0) {
    p.part_m[out_row * p.max_partitions + part] = M;
    p.part_l[out_row * p.max_partitions + part] = L;
  }
}

#ifndef PKV_SIMT_RING_BYTES
#define PKV_SIMT_RING_BYTES (64 * 1024)  // ring bytes per CTA (build-time tuning knob)
#endif

// Stages per warp: about PKV_SIMT_RING_BYTES of ring per CTA, 1 to 6 stages.
template <int D, int BS, int EB = 2>
constexpr int simt_stages() {
  constexpr int stage = 2 * BS * D * EB;
  constexpr int spw = (PKV_SIMT_RING_BYTES) / (kDecodeWarps * stage);
  return spw < 1 ? 1 : (spw > 6 ? 6 : spw);
}

// C: cache element type (T for a 16-bit cache, __nv_fp8_e4m3 for an FP8 cache).
template <typename T, int D, int BS, typename C = T>
cudaError_t launch_decode_simt(const DecodeParams& p, int num_seqs, cudaStream_t stream) {
  constexpr int NW = kDecodeWarps;
  constexpr int EB = CacheFmt<C>::EB;
  constexpr int SPW = simt_stages<D, BS, EB>();
  using Sh = SimtShape<D, BS, NW, SPW, EB>;
  auto kern = pkv_decode_simt_kernel<T, C, D, BS, NW, SPW>;
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
  const dim3 grid(PKV_GRID_HEAD_FASTEST ? p.num_heads : p.max_partitions,
                  PKV_GRID_HEAD_FASTEST ? p.max_partitions : p.num_heads, num_seqs);
  return launch_kernel(kern, grid, dim3(NW * 32), Sh::SMEM, stream, p);
}

}  // namespace pkv
