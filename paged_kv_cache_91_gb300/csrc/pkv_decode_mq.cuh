// Multi-query paged attention: several query tokens per sequence over the
// paged pool, each attending the positions up to its own. This is the
// attention of a chunked-prefill chunk batched with decode tokens, or of the
// tokens a speculative step verifies ("Sparse Computation and Memory
// Management for Efficient LLM Inference", the chunked prefill paragraph and
// Speculative Decoding; causal a_ij over j <= i: "vLLM: LLM 서빙 메모리 최적화의
// 교과서", 01 Problem Definition).
//
// Sequence s has q_len = query_start_loc[s+1] - query_start_loc[s] query rows
// (packed, [T][H][D]); they are its last q_len context positions, so query
// token i (position ctx - q_len + i) sees the first ctx - q_len + i + 1 tokens.
//
// The tensor-core tile (MmaTile) already puts 8 "columns" in the MMA's n
// dimension; here a column is one (query token, query head) row of a kv head
// rather than one head. The R = q_len * G rows of (sequence, kv head) -- row
// r is query token r / G, head kvh * G + r % G -- are cut into tiles of 8, and
// each CTA runs one (partition, kv head x row tile, sequence): its warps walk
// the partition's blocks as in the decode kernel, each column with its own
// causal limit, and merge. Blocks past the tile's largest limit are not read.
// Contexts longer than one partition leave per-(row, head) partials for the
// log-sum-exp reduce, exactly as in decode.
#pragma once

#include "pkv_decode_mma.cuh"

namespace pkv {

// Extra parameters of a multi-query launch. The defaults give the call's own
// meaning: query_start_loc packs each sequence's query tokens, which are its
// last q_len positions and attend causally.
struct MqParams {
  const int32_t* query_start_loc = nullptr;  // [num_seqs + 1] (mode MQ_PACKED)
  int num_query_tokens = 0;                  // host bound on query_start_loc entries
  int max_query_len = 0;                     // host bound on every q_len
  int row_tiles = 1;                         // ceil(max_query_len * G / rows per CTA)
  int mode = 0;        // MQ_PACKED, MQ_ONE_PER_SEQ (query token s of sequence s) or MQ_ONE_SEQ
                       // (sequence 0 holds all num_query_tokens tokens)
  int ctx_const = -1;  // >= 0: every sequence's context length (context_lens is not read)
  int causal = 1;      // 0: every query row sees the whole context
  int partials = 0;    // 1: write (m, l, o) partials even for a single-partition context
  const int32_t* order = nullptr;  // if set, the sequence of grid index z (longest context first)
};
constexpr int MQ_PACKED = 0, MQ_ONE_PER_SEQ = 1, MQ_ONE_SEQ = 2;

// Context length of sequence s, clamped like clamp_context.
__device__ __forceinline__ int mq_context(const DecodeParams& p, const MqParams& mq, int s, bool report) {
  if (mq.ctx_const >= 0) return mq.ctx_const < p.ctx_limit ? mq.ctx_const : p.ctx_limit;
  return clamp_context(p, s, report);
}

// q_len of sequence s and its first query row q0, or -1 (and PKV_DEVERR_QUERY)
// if query_start_loc is inconsistent with the bounds or the (clamped) context.
// One query token per sequence over an empty context gives 0 (no rows).
__device__ __forceinline__ int mq_query_len(const MqParams& mq, int s, int ctx, int& q0) {
  if (mq.mode == MQ_ONE_PER_SEQ) {
    q0 = s;
    return ctx > 0 ? 1 : 0;
  }
  if (mq.mode == MQ_ONE_SEQ) {
    q0 = 0;
    return s == 0 ? mq.num_query_tokens : 0;
  }
  q0 = mq.query_start_loc[s];
  const int q1 = mq.query_start_loc[s + 1];
  const int n = q1 - q0;
  if (q0 < 0 || n < 0 || q1 > mq.num_query_tokens || n > mq.max_query_len || (mq.causal && n > ctx)) return -1;
  return n;
}

// Positions [0, limit) that query row r (token r / G of the sequence's q_len) sees.
__device__ __forceinline__ int mq_limit(const MqParams& mq, int ctx, int q_len, int r, int G) {
  return mq.causal ? ctx - q_len + r / G + 1 : ctx;
}

template <typename Tile, int NW, int SPW>
__global__ void __launch_bounds__(NW * 32, Tile::MIN_CTAS)
    pkv_mq_mma_kernel(const DecodeParams p, const MqParams mq, const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap) {
  pdl_begin();
  using T = typename Tile::T;
  constexpr int D = Tile::D, BS = Tile::BS;
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
  const int row0 = rt * 8;
  if (row0 >= R) return;  // no rows in this tile
  const int ncol = min(8, R - row0);
  const int P = p.partition_size;
  const int tok0 = part * P;
  if (tok0 >= ctx) return;
  // the tile's last row sees the most tokens; nothing past its limit is read
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
        Tile::issue_tiles(st, &kmap, &vmap, (phys * p.num_kv_heads + kvh) * BS, bar);
      } else {
        mbar_arrive(bar);
      }
    }
  };
  const int nfirst = nmine < SPW ? nmine : SPW;
  for (int i = 0; i < nfirst; ++i) issue(i);
  int issued = nfirst;

  // this lane's query column (n = lane / 4) and its two accumulator columns' limits
  const T* qrow = nullptr;
  {
    const int n = lane >> 2, r = row0 + n;
    if (n < ncol) qrow = reinterpret_cast<const T*>(p.query) + ((size_t)(q0 + r / G) * p.num_heads + kvh * G + r % G) * D;
  }
  const int j0 = (lane & 3) * 2;
  const int lim0 = j0 < ncol ? mq_limit(mq, ctx, q_len, row0 + j0, G) : 0;
  const int lim1 = j0 + 1 < ncol ? mq_limit(mq, ctx, q_len, row0 + j0 + 1, G) : 0;
  typename Tile::QB qb;
  float sla = p.scale_log2, slb = p.scale_log2;  // score multipliers of this lane's two columns
  if constexpr (Tile::FP8)
    Tile::load_qb_row(qb, qrow, lane, p.scale_log2, sla, slb);  // per-column f16 scaling of a bf16 query
  else
    Tile::load_qb_row(qb, qrow, lane);

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
      const int base = (blk0 + lb) * BS;
      const int nvalid = min(BS, tok1 - base);
      Tile::template run<true>(Ks, Ks + Sh::TILE, nvalid, qb, lane, sla, slb, m0, m1, l0, l1, acc, base, lim0,
                               lim1);
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

  // merge the warps: each warp writes [column][D] accumulators, m, l into its own ring slice
  float* red = reinterpret_cast<float*>(ring);
  float* red_m = red + 8 * D;
  float* red_l = red_m + 8;
  Tile::store_acc(red, acc, lane);
  if (lane < 4) {
    red_m[j0] = m0;
    red_m[j0 + 1] = m1;
    red_l[j0] = l0;
    red_l[j0 + 1] = l1;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < ncol * D; idx += NW * 32) {
    const int n = idx / D, d = idx - n * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, reinterpret_cast<float*>(smem + w * SPW * Sh::STAGE)[8 * D + n]);
    float L = 0.f, o = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float* rw = reinterpret_cast<float*>(smem + w * SPW * Sh::STAGE);
      const float mw = rw[8 * D + n];
      const float f = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
      L += rw[8 * D + 8 + n] * f;
      o += rw[n * D + d] * f;
    }
    o = L > 0.f ? o / L : 0.f;
    if constexpr (Tile::FP8) o *= p.v_scale * Tile::UNIT;  // V codes -> values
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

template <typename Tile, int RING_BYTES = PKV_MMA_RING_BYTES>
cudaError_t launch_mq_mma(const DecodeParams& p, const MqParams& mq, const CUtensorMap& kmap,
                          const CUtensorMap& vmap, int num_seqs, cudaStream_t stream) {
  constexpr int NW = kDecodeWarps;
  constexpr int SPW = mma_stages<2 * Tile::TILE, RING_BYTES>();
  using Sh = MmaShape<Tile::D, Tile::BS, NW, SPW, Tile::TILE>;
  auto kern = pkv_mq_mma_kernel<Tile, NW, SPW>;
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
