// Decode attention over the paged KV pool on the CUDA cores: used for MHA (one
// query head per kv head, where the per-block work is a matrix-vector product)
// and as the general path for group sizes the tensor-core kernel does not take.
//
// Method: "KV Cache와 PagedAttention 완전 해부", 부록 -- walk the sequence's
// blocks through the block table, score each block's keys, update a running
// softmax, accumulate the weighted values; "vLLM: LLM 서빙 메모리 최적화의
// 교과서", eq. (4).
//
// SimtTile holds the per-tile arithmetic shared by the grid kernel below and the
// persistent kernel (pkv_decode_stream.cuh). The grid kernel runs one CTA per
// (context partition, query head, sequence): each warp owns a private ring of
// SPW stages, each stage the K tile and V tile of one (physical block, kv head)
// pair brought in by two linear bulk copies (TMA engine) completing on the
// stage's mbarrier; warp w takes the partition's blocks w, w+NW, ... and refills
// the stage it just consumed. A single-partition context writes its output
// directly; longer ones write (m, l, o) partials that pkv_reduce_kernel merges.
#pragma once

#include "pkv_common.cuh"

namespace pkv {

template <int D, int BS>
struct SimtTileShape {
  static constexpr int TPC = BS < 16 ? BS : 16;  // tokens per score chunk
  static constexpr int CPB = BS / TPC;           // chunks per block
  static constexpr int LPT = 32 / TPC;           // lanes per token in the score pass
  static constexpr int DPL = D / LPT;            // head dims per lane in the score pass
  static constexpr int NCH = DPL / 8;            // 16-byte pieces per lane in the score pass
  static constexpr int DPV = D / 32;             // head dims per lane in the value pass
  static constexpr int TILE = BS * D * 2;        // bytes of one (block, kv head) tile
  static_assert(NCH == 2 || NCH == 4 || NCH == 8, "score-pass piece count");
  static_assert(DPV == 2 || DPV == 4, "value-pass width");
};

// Start piece of each lane in the score pass. Rows of a tile are 128 or 256
// bytes apart, so without a rotation the lanes of one shared-memory phase hit
// the same 16-byte bank group; these rotations make every phase conflict-free.
template <int LPT, int NCH>
__device__ __forceinline__ int qk_rotation(int lane) {
  const int t = lane / LPT, pt = lane % LPT;
  if constexpr (NCH >= 8) {
    return lane & 7;
  } else if constexpr (NCH == 4 && LPT == 2) {
    return t & 3;
  } else if constexpr (NCH == 4) {
    return ((pt >> 1) + 2 * t) & 3;
  } else {
    return t & 1;
  }
}

template <typename T, int D, int BS>
struct SimtTile {
  using Sh = SimtTileShape<D, BS>;

  // This lane's slice of one query row for the score pass, scaled into the
  // base-2 domain and stored in rotated piece order. `q` is the row's first
  // element, in global or shared memory, 16-byte aligned.
  static __device__ __forceinline__ void load_q(float (&qreg)[Sh::DPL], const T* q, int lane, float scale_log2) {
    const int pt = lane % Sh::LPT;
    const int rot = qk_rotation<Sh::LPT, Sh::NCH>(lane);
#pragma unroll
    for (int i = 0; i < Sh::NCH; ++i) {
      const int piece = (i + rot) & (Sh::NCH - 1);
      const uint4 raw = *reinterpret_cast<const uint4*>(q + pt * Sh::DPL + piece * 8);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = Elem<T>::to_float2(w[e]);
        qreg[i * 8 + 2 * e] = f.x * scale_log2;
        qreg[i * 8 + 2 * e + 1] = f.y * scale_log2;
      }
    }
  }

  // Fold one (block, kv head) tile into the warp's running state (m, l, acc):
  // tokens 0 .. nvalid-1 of the tile take part, the rest are never read.
  static __device__ __forceinline__ void run(const unsigned char* Ks, const unsigned char* Vs, int nvalid,
                                             const float (&qreg)[Sh::DPL], int lane, float& m, float& l,
                                             float (&acc)[Sh::DPV]) {
    const int tl = lane / Sh::LPT, pt = lane % Sh::LPT;
    const int rot = qk_rotation<Sh::LPT, Sh::NCH>(lane);
#pragma unroll
    for (int c = 0; c < Sh::CPB; ++c) {
      if (c * Sh::TPC < nvalid) {
        // scores of this chunk's tokens: LPT lanes per token, fp32 accumulation
        const unsigned char* krow = Ks + (c * Sh::TPC + tl) * (D * 2) + pt * (Sh::DPL * 2);
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int i2 = 0; i2 < Sh::NCH; ++i2) {
          const int piece = (i2 + rot) & (Sh::NCH - 1);
          const uint4 raw = *reinterpret_cast<const uint4*>(krow + piece * 16);
          const float2 f0 = Elem<T>::to_float2(raw.x), f1 = Elem<T>::to_float2(raw.y);
          const float2 f2 = Elem<T>::to_float2(raw.z), f3 = Elem<T>::to_float2(raw.w);
          a0 = fmaf(qreg[i2 * 8 + 0], f0.x, a0);
          a1 = fmaf(qreg[i2 * 8 + 1], f0.y, a1);
          a2 = fmaf(qreg[i2 * 8 + 2], f1.x, a2);
          a3 = fmaf(qreg[i2 * 8 + 3], f1.y, a3);
          a0 = fmaf(qreg[i2 * 8 + 4], f2.x, a0);
          a1 = fmaf(qreg[i2 * 8 + 5], f2.y, a1);
          a2 = fmaf(qreg[i2 * 8 + 6], f3.x, a2);
          a3 = fmaf(qreg[i2 * 8 + 7], f3.y, a3);
        }
        float sc = (a0 + a1) + (a2 + a3);
#pragma unroll
        for (int o = Sh::LPT / 2; o > 0; o >>= 1) sc += __shfl_xor_sync(kFull, sc, o);
        const int nv = min(Sh::TPC, nvalid - c * Sh::TPC);
        sc = tl < nv ? sc : -INFINITY;  // tokens past the context do not take part

        // running softmax update; the LPT lanes of a token hold the same score,
        // so the reductions run over the TPC distinct tokens only
        float mx = sc;
#pragma unroll
        for (int o = Sh::LPT; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
        const float mnew = fmaxf(m, mx);
        const float alpha = fast_exp2(m - mnew);
        const float pr = fast_exp2(sc - mnew);
        float ps = pr;
#pragma unroll
        for (int o = Sh::LPT; o < 32; o <<= 1) ps += __shfl_xor_sync(kFull, ps, o);
        l = l * alpha + ps;
        m = mnew;
#pragma unroll
        for (int e = 0; e < Sh::DPV; ++e) acc[e] *= alpha;

        // weighted values: lane owns DPV consecutive head dims. A full chunk runs
        // without per-token branches so its loads can all be in flight at once;
        // a partial chunk never reads rows past the context.
        const unsigned char* vrow = Vs + (c * Sh::TPC) * (D * 2) + lane * (Sh::DPV * 2);
        if (nv == Sh::TPC) {
#pragma unroll
          for (int tt = 0; tt < Sh::TPC; ++tt) pv_row(acc, __shfl_sync(kFull, pr, tt * Sh::LPT), vrow + tt * (D * 2));
        } else {
#pragma unroll
          for (int tt = 0; tt < Sh::TPC; ++tt) {
            const float w = __shfl_sync(kFull, pr, tt * Sh::LPT);
            if (tt < nv) pv_row(acc, w, vrow + tt * (D * 2));
          }
        }
      }
    }
  }

  // acc[e] += w * V[row][lane dims e]
  static __device__ __forceinline__ void pv_row(float (&acc)[Sh::DPV], float w, const unsigned char* v) {
    if constexpr (Sh::DPV == 4) {
      const uint2 raw = *reinterpret_cast<const uint2*>(v);
      const float2 f0 = Elem<T>::to_float2(raw.x), f1 = Elem<T>::to_float2(raw.y);
      acc[0] = fmaf(w, f0.x, acc[0]);
      acc[1] = fmaf(w, f0.y, acc[1]);
      acc[2] = fmaf(w, f1.x, acc[2]);
      acc[3] = fmaf(w, f1.y, acc[3]);
    } else {
      const uint32_t raw = *reinterpret_cast<const uint32_t*>(v);
      const float2 f0 = Elem<T>::to_float2(raw);
      acc[0] = fmaf(w, f0.x, acc[0]);
      acc[1] = fmaf(w, f0.y, acc[1]);
    }
  }
};

template <int D, int BS, int NW, int SPW>
struct SimtShape : SimtTileShape<D, BS> {
  static constexpr int STAGE = 2 * SimtTileShape<D, BS>::TILE;  // K tile + V tile
  static constexpr int RING = NW * SPW * STAGE;
  static constexpr int BARS = RING;  // mbarriers follow the ring
  static constexpr int RED = BARS + ((NW * SPW * 8 + 15) / 16) * 16;
  static constexpr int SMEM = RED + NW * (D + 2) * 4;
};

template <typename T, int D, int BS, int NW, int SPW>
__global__ void __launch_bounds__(NW * 32, PKV_DECODE_MIN_CTAS) pkv_decode_simt_kernel(const DecodeParams p) {
  pdl_begin();
  using Sh = SimtShape<D, BS, NW, SPW>;
  using Tile = SimtTile<T, D, BS>;
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
  const float inv = L > 0.f ? 1.f / L : 0.f;
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
template <int D, int BS>
constexpr int simt_stages() {
  constexpr int stage = 2 * BS * D * 2;
  constexpr int spw = (PKV_SIMT_RING_BYTES) / (kDecodeWarps * stage);
  return spw < 1 ? 1 : (spw > 6 ? 6 : spw);
}

template <typename T, int D, int BS>
cudaError_t launch_decode_simt(const DecodeParams& p, int num_seqs, cudaStream_t stream) {
  constexpr int NW = kDecodeWarps;
  constexpr int SPW = simt_stages<D, BS>();
  using Sh = SimtShape<D, BS, NW, SPW>;
  auto kern = pkv_decode_simt_kernel<T, D, BS, NW, SPW>;
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
