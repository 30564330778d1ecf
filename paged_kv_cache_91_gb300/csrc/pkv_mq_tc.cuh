// Multi-query paged attention on the fifth-generation tensor cores (tcgen05):
// 128 query rows per CTA in the MMA's M dimension, scores and outputs
// accumulated in tensor memory.
//
// Same computation as the other multi-query tiles (pkv_decode_mq.cuh): the
// R = q_len * G (query token, head) rows of a (sequence, kv head), row r being
// query token r / G at position ctx - q_len + r / G and attending the positions
// up to its own ("vLLM: LLM 서빙 메모리 최적화의 교과서", 01 Problem Definition:
// a_ij over j <= i; the blocked form o_i = sum_j V_j A_ij^T of "Efficient
// Memory Management for LLM Serving with PagedAttention", §4.1 Eq. (4)). A
// CTA takes 128 rows of one (partition, kv head, sequence) and walks the
// partition in tiles of 64 tokens (64 / block_size pool blocks):
//   S_j = Q . K_j^T      M 128, N 64,  K = head_dim   -> tensor memory (fp32)
//   P_j = exp2(S_j * scale * log2 e - m_ref)          one thread per row,
//                                                      16-bit, over S_j's columns
//   O  += P_j . V_j      M 128, N = head_dim, K 64    A from tensor memory
//
// Roles (7 or 8 warps): warp 0 copies K tiles into a three-slot ring and warp
// 2 V tiles into a two-slot ring, one copy per pool block (a copy takes about
// 100 cycles to issue, so one warp for both fell behind); one thread of warp 1
// issues the MMAs (over a 16-bit pool the S MMAs only, and one thread of warp
// 7 the PV MMAs); warps 3..6 each own 32 rows (their tensor-memory lane
// quarter) for the softmax, write P_j back into tensor memory where S_j was,
// and finally normalise and store O. A
// K slot is refilled as soon as its S MMA has completed, a V slot (and the S/P
// buffer) once its PV has. S/P is double-buffered in tensor memory, so S_{j+1}
// is usually ready when the softmax of tile j ends, and the softmax never
// waits for the previous PV except to rescale O. The running max is a lazily
// moved reference: O's row is rescaled only when a score exceeds the reference
// by more than 2^8, which keeps P within the 16-bit range. Two CTAs share an
// SM, so one CTA's start and end overlap the other's streaming.
//
// FP8 (E4M3) pool (F8): each K/V tile's codes land, one copy per pool block,
// in the upper half of the tile's f16 slot; the copy warp that issued them
// widens them in place into the f16 operand layout (the codes convert to f16
// exactly) and only then signals the MMA thread. A bf16 query is scaled per row
// by a power of two into f16, so both MMAs multiply f16; the output takes
// v_scale.
//
// Every wait is bounded: a copy or MMA that does not complete makes the CTA
// stop, set PKV_DEVERR_TIMEOUT and write an empty result.
#pragma once

#include <type_traits>

#include "pkv_decode_mma_fp8.cuh"
#include "pkv_decode_mq.cuh"
#include "pkv_tcgen05.cuh"

namespace pkv {

#ifndef PKV_MQ_TC_PREFETCH
// 16-bit pool: the blocks of the tile this many tiles ahead of the one being copied are prefetched into
// L2 (0: none; build-time knob). Measured: 2 tiles ahead took workload 2's 128-token chunks from 0.298 to
// 0.290 ms and workload 3's 32-token chunks from 0.270 to 0.266 ms; 4 ahead was slower. Over an FP8 pool
// the copy warps also widen the codes, and the extra work there cost 3%, so FP8 pools are not prefetched.
#define PKV_MQ_TC_PREFETCH 2
#endif

#ifndef PKV_MQ_TC_COPY_WARPS
#define PKV_MQ_TC_COPY_WARPS 2  // 1: one warp copies K and V; 2: one warp each (build-time knob)
#endif

template <typename T, int D, int BS, bool F8 = false>
struct MqTcShape {
  static constexpr int ROWS = 128;                // query rows per CTA (M)
  static constexpr int NT = 64;                   // tokens per K/V tile
  static constexpr int NBT = NT / BS;             // pool blocks per tile
  static constexpr int DH = D / 64;               // 128-byte halves of a 16-bit row
  // A K or V tile in shared memory: 8-token atoms of DH x 1024 bytes (atom
  // stride ATOM), each holding the 128-byte rows of its 8 tokens for columns
  // 0..63, then (head_dim 128) for columns 64..127 -- the layout one copy of a
  // whole pool block lands in (see make_pool_map_tc on the host).
  static constexpr int ATOM = DH * 1024;
  static constexpr int TILE = NT / 8 * ATOM;
  static constexpr int KST = 3, VST = 2;          // K and V ring slots
  static constexpr int OFF_K = DH * ROWS * 128;   // after Q
  static constexpr int OFF_V = OFF_K + KST * TILE;
  static constexpr int OFF_BARS = OFF_V + VST * TILE;
  // k_full[3], k_empty[3], v_full[2], pv_done[2] (PV_j done: V slot and S/P buffer j % 2 free),
  // s_full[2], p_full[2] (per S/P buffer: no row can reach tile j + 2 before PV_j), fin, q_full,
  // and for an FP8 pool k_raw[3], v_raw[2] (the codes have landed; k_full / v_full then mean widened)
  static constexpr int NBARS = 22;  // (+ fin_pv, the PV warp's completion barrier, last)
  static constexpr int HALF = TILE / 2;           // FP8 pool: the codes of a tile land in its slot's upper half
  static constexpr int OFF_MISC = OFF_BARS + NBARS * 8;  // tensor-memory base, abort flag
  static constexpr int SMEM_USED = OFF_MISC + 8;
  // The operands need 1024-byte aligned atoms; the dynamic shared memory of a
  // CTA without static shared variables starts 1024-aligned (checked at run
  // time), so no slack is reserved. At most two CTAs per SM: their tensor
  // memory (2 x 256 columns) is then always free.
  static constexpr int SMEM_MIN = 233472 / 3 + 1024;
  static constexpr int SMEM = SMEM_USED > SMEM_MIN ? SMEM_USED : SMEM_MIN;
  static constexpr int TMEM_COLS = 256;           // O at columns [0, D), S/P buffers at 128 and 192
  static constexpr int S_COL = 128;
  static constexpr int IDS = (kMaxPartitionBlocks + 31) / 32;
  static constexpr int CW = PKV_MQ_TC_COPY_WARPS;  // copy warps: warp 0 (and warp 2 for V)
  static constexpr int SW = CW + 1;                // first of the four row warps
  // 16-bit pool: a warp of its own issues the PV MMAs (measured: workload 2 with 128- and 64-token
  // chunks 0.2861 / 0.2579 ms against 0.2893 / 0.2687 with one issuing thread, workload 3 with
  // 32-token chunks 0.2589 against 0.2656). Over an FP8 pool it measured mixed (workload 3 0.3543
  // against 0.3460), so one thread issues both there.
  static constexpr bool SPLIT = !F8 && CW == 2;
  static constexpr int PVW = SW + 4;               // the PV warp (when SPLIT)
  static constexpr int THREADS = (SW + 4 + (SPLIT ? 1 : 0)) * 32;
  static_assert(BS * 128 % 1024 == 0, "a block's rows must fill whole 1024-byte swizzle atoms");
  static_assert(NT % BS == 0 && NBT <= 32, "tile of whole blocks");
  static_assert(2 * (SMEM + 1024) <= 233472, "two CTAs per SM");
};

// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for `parity` on `bar`; false if another role gave up (`abort` set) or
// the wait passed the cycle limit (then `abort` is set here).
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > kWaitLimitCycles) {
      *abort = 1;
      return false;
    }
  }
}

// 16 bytes from global to shared memory without a register round trip;
// `bytes` = 0 writes zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Bring `bytes` (a multiple of 16) at the 16-byte aligned global address into L2, without waiting.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Thread `row` of the rows' warps brings its query row (rows r = rt * ROWS + row, query token
// r / G, head kvh * G + r % G; zeros past q_len * G) into Q's A-operand layout: 128-byte swizzled
// rows, columns 64.. in the next ROWS x 128 bytes. Out of line, which keeps the softmax loop's
// registers free.
template <typename T, int D, int ROWS>
__device__ __noinline__ void mq_tc_fetch_q(unsigned char* Qs, int row, const T* query, int q0, int kvh, int rt,
                                           int q_len, int G, int num_heads) {
  const int r = rt * ROWS + row;
  const bool act = r < q_len * G;
  const T* src = query;
  if (act) src += ((size_t)(q0 + r / G) * num_heads + kvh * G + r % G) * D;
  const uint32_t dst = smem_u32(Qs) + row * 128, rx = row & 7;
  if (act) {
#pragma unroll
    for (int c = 0; c < D / 8; ++c) cp_async16(dst + (c / 8) * (ROWS * 128) + (((c % 8) ^ rx) << 4), src + c * 8, 16u);
  } else {
#pragma unroll
    for (int c = 0; c < D / 8; ++c)
      *reinterpret_cast<uint4*>(Qs + row * 128 + (c / 8) * (ROWS * 128) + (((c % 8) ^ rx) << 4)) = make_uint4(0, 0, 0, 0);
  }
}

// FP8 pool: widen the E4M3 codes of one 64-token tile, landed as 64 rows of 128 codes at src (the
// upper half of the slot), into the slot's f16 operand layout at dst (8-token atoms of two
// 128-byte-swizzled 1 KB halves, columns 0..63 then 64..127), in place. Lane (t = lane / 4, quarter
// q = lane % 4) takes codes 32q .. 32q + 31 of token 8a + t of every atom a. The whole tile is read
// into registers before anything is written (the output overwrites the codes).
__device__ __forceinline__ void mq_tc_widen_tile(unsigned char* dst, const unsigned char* src, int lane) {
  const int t8 = lane >> 2, q = lane & 3;
  // An 8-lane phase of a 16-byte load covers two token rows 128 bytes apart; odd rows fetch their
  // second 16 bytes first, so that the two rows fall on different banks.
  const int h0 = (t8 & 1) * 16, h1 = 16 - h0;
  uint4 c[8][2];
#pragma unroll
  for (int a = 0; a < 8; ++a) {
    const int t = 8 * a + t8;
    const uint4 x = *reinterpret_cast<const uint4*>(src + t * 128 + 32 * q + h0);
    const uint4 y = *reinterpret_cast<const uint4*>(src + t * 128 + 32 * q + h1);
    c[a][0] = h0 ? y : x;
    c[a][1] = h0 ? x : y;
  }
  __syncwarp();
#pragma unroll
  for (int a = 0; a < 8; ++a) {
    const uint32_t w[8] = {c[a][0].x, c[a][0].y, c[a][0].z, c[a][0].w, c[a][1].x, c[a][1].y, c[a][1].z, c[a][1].w};
    unsigned char* row = dst + a * 2048 + (q >> 1) * 1024 + t8 * 128;
    // Lanes q = 2, 3 store their chunks in the order 2, 3, 0, 1: an 8-lane phase of the 16-byte stores then
    // covers 8 distinct 16-byte bank groups (in order, lanes q and q + 2 would hit the same one).
    const bool rot = (q >> 1) != 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int kk = rot ? (k ^ 2) : k;
      const uint32_t wa = rot ? w[2 * (k ^ 2)] : w[2 * k];
      const uint32_t wb = rot ? w[2 * (k ^ 2) + 1] : w[2 * k + 1];
      uint32_t h[4];
      e4m3x4_to_f16x2(wa, h[0], h[1]);
      e4m3x4_to_f16x2(wb, h[2], h[3]);
      const int cc = (q & 1) * 4 + kk;
      *reinterpret_cast<uint4*>(row + ((cc ^ t8) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
    }
  }
}

// FP8 pool with a bf16 query: thread `row` stores its query row (as in mq_tc_fetch_q) in f16,
// multiplied by 2^k so that its largest magnitude lies in [2^14, 2^15) (every bf16 value keeps its
// 8 significant bits unless it lies below 2^-14 of that range, where its contribution is far below
// the fp32 accumulation error); returns 2^-k, which the row's score multiplier takes back. Zeros
// and 1 past q_len * G.
template <int D, int ROWS>
__device__ __noinline__ float mq_tc_fetch_q_bf16_as_f16(unsigned char* Qs, int row, const __nv_bfloat16* query,
                                                         int q0, int kvh, int rt, int q_len, int G, int num_heads) {
  const int r = rt * ROWS + row;
  const uint32_t rx = row & 7;
  if (r >= q_len * G) {
#pragma unroll
    for (int c = 0; c < D / 8; ++c)
      *reinterpret_cast<uint4*>(Qs + row * 128 + (c / 8) * (ROWS * 128) + (((c % 8) ^ rx) << 4)) = make_uint4(0, 0, 0, 0);
    return 1.f;
  }
  const uint4* src = reinterpret_cast<const uint4*>(query + ((size_t)(q0 + r / G) * num_heads + kvh * G + r % G) * D);
  // two passes over the row (the second reads it from cache): its largest magnitude, then the stores
  float amax = 0.f;
#pragma unroll 4
  for (int c = 0; c < D / 8; ++c) {
    const uint4 v = src[c];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = Elem<__nv_bfloat16>::to_float2(w[e]);
      amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
  const int ex = static_cast<int>((__float_as_uint(amax) >> 23) & 0xff) - 127;  // floor(log2(amax))
  int k = amax > 0.f ? 14 - ex : 0;
  k = k < -60 ? -60 : (k > 60 ? 60 : k);
  const float pw = __uint_as_float(static_cast<uint32_t>(127 + k) << 23);
#pragma unroll 4
  for (int c = 0; c < D / 8; ++c) {
    const uint4 v = src[c];
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = Elem<__nv_bfloat16>::to_float2(w[e]);
      w[e] = Elem<__half>::pack2(f.x * pw, f.y * pw);
    }
    *reinterpret_cast<uint4*>(Qs + row * 128 + (c / 8) * (ROWS * 128) + (((c % 8) ^ rx) << 4)) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
  return __uint_as_float(static_cast<uint32_t>(127 - k) << 23);
}

template <typename T, int D, int BS, bool F8 = false>
// Two CTAs per SM: 6 warps x 168 registers (3 warps per SM quarter), or 7 x 128 (4 per quarter).
__global__ void __maxnreg__(PKV_MQ_TC_COPY_WARPS == 2 ? 128 : 168)
    pkv_mq_tc_kernel(const DecodeParams p, const MqParams mq, const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap) {
  pdl_begin();
  using Sh = MqTcShape<T, D, BS, F8>;
  // FP8 pool: both MMAs multiply f16 (the codes widen exactly; a bf16 query is scaled into f16)
  using TP = typename std::conditional<F8, __half, T>::type;  // the type of P (and, with F8, of Q, K and V)
  static_assert(!F8 || (D == 128 && Sh::CW == 2), "an FP8 pool: head_dim 128, one copy warp each for K and V");
  constexpr int NT = Sh::NT, NBT = Sh::NBT, DH = Sh::DH;
  extern __shared__ __align__(1024) unsigned char smem[];
  constexpr int KST = Sh::KST;
  uint64_t* k_full = reinterpret_cast<uint64_t*>(smem + Sh::OFF_BARS);
  uint64_t* k_empty = k_full + 3;
  uint64_t* v_full = k_full + 6;
  uint64_t* pv_done = k_full + 8;
  uint64_t* s_full = k_full + 10;
  uint64_t* p_full = k_full + 12;
  uint64_t* fin = k_full + 14;
  uint64_t* q_full = k_full + 15;
  uint64_t* k_raw = k_full + 16;  // FP8 pool only
  uint64_t* v_raw = k_full + 19;
  uint64_t* fin_pv = k_full + 21;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Sh::OFF_MISC);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  unsigned char* Qs = smem;
  auto k_slot = [&](int j) { return smem + Sh::OFF_K + (j % KST) * Sh::TILE; };
  auto v_slot = [&](int j) { return smem + Sh::OFF_V + (j & 1) * Sh::TILE; };

  const int part = blockIdx.x;
  const int kvh = blockIdx.y / mq.row_tiles, rt = blockIdx.y % mq.row_tiles;
  // with an order, grid index z runs over the sequences longest context first, so that the long
  // items start early and the grid's end is made of short ones
  const int s = mq.order ? mq.order[blockIdx.z] : (int)blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;
  const bool reporter = part == 0 && blockIdx.y == 0 && threadIdx.x == 0;
  if (smem_u32(smem) & 1023u) {  // not expected on any supported GPU; nothing is written
    if (threadIdx.x == 0) atomicOr(p.err, PKV_DEVERR_LAYOUT);
    return;
  }
  // The first copies need the partition's block ids. In the first partition, which has tokens
  // whenever the context does, the copy warps load them together with the context length (as far
  // as the table row goes; masked below), so that the first copy waits for one memory round trip
  // rather than two. Later partitions are often past the context and load them once it is known.
  // (Requesting the query rows early as well measured slower.)
  const bool srole = warp >= Sh::SW && warp < Sh::SW + 4;
  const int row = 32 * (warp & 3) + lane;
  const bool early = part == 0;
  int raw[Sh::IDS];
  auto load_raw = [&] {
    const int bb = part * p.partition_size / BS;
#pragma unroll
    for (int u = 0; u < Sh::IDS; ++u) {
      const int b = lane + 32 * u;
      raw[u] = b < p.partition_size / BS && bb + b < p.max_blocks_per_seq
                   ? p.block_tables[(size_t)s * p.max_blocks_per_seq + bb + b]
                   : -1;
    }
  };
  if (early && (warp == 0 || (Sh::CW == 2 && warp == 2))) load_raw();
  const int ctx = mq_context(p, mq, s, reporter);
  int q0 = 0;
  const int q_len = mq_query_len(mq, s, ctx, q0);
  if (q_len < 0) {
    if (reporter) atomicOr(p.err, PKV_DEVERR_QUERY);
    return;
  }
  const int R = q_len * G;
  const int row0 = rt * Sh::ROWS;
  const int P = p.partition_size;
  const int tok0 = part * P;
  if (row0 >= R || tok0 >= ctx) return;
  const int lim_cta = mq_limit(mq, ctx, q_len, min(row0 + Sh::ROWS, R) - 1, G);  // the CTA's last row's limit
  const int tok1 = min(min(tok0 + P, ctx), lim_cta);
  const bool direct = !mq.partials && ctx <= P;
  const int ntile = tok1 > tok0 ? (tok1 - tok0 + NT - 1) / NT : 0;
  const int blk0 = tok0 / BS;

  // softmax rows: warps SW.., thread row = 32 (warp % 4) + lane (its tensor-memory lane)
  const int r = row0 + row;
  const bool active = srole && r < R;
  const size_t orow = active ? (size_t)(q0 + r / G) * p.num_heads + kvh * G + r % G : 0;  // output row

  if (ntile == 0) {  // no visible token in this partition: an empty partial (ctx > P here)
    if (active) {
      for (int d = 0; d < D; d += 4)
        *reinterpret_cast<float4*>(p.part_o + (orow * p.max_partitions + part) * D + d) = make_float4(0, 0, 0, 0);
      p.part_m[orow * p.max_partitions + part] = -INFINITY;
      p.part_l[orow * p.max_partitions + part] = 0.f;
    }
    return;
  }

  if (threadIdx.x == 0) {
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
    for (int k = 0; k < 12; ++k) mbar_init(k_full + k, 1);
    for (int k = 16; k < 21; ++k) mbar_init(k_full + k, 1);
    mbar_init(p_full, 128);
    mbar_init(p_full + 1, 128);
    mbar_init(fin, 1);
    mbar_init(fin_pv, 1);
    mbar_init(q_full, 128);
    fence_mbar_init();
    *abort = 0;
  }
  if (warp == 1) tc::alloc(tmem_slot, Sh::TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *tmem_slot;

  if (warp == 0 || (Sh::CW == 2 && warp == 2)) {
    // ---- copies: K tile j into slot j % 3 of the K ring, V tile j into slot j % 2 of the V ring
    // (one warp for both, or warp 0 for K and warp 2 for V)
    const bool do_k = Sh::CW == 1 || warp == 0, do_v = Sh::CW == 1 || warp == 2;
    if (!early) load_raw();
    int ids[Sh::IDS];  // lane l: block ids l, l + 32, ... of the partition; -1 for a bad id
    const int nblk = (tok1 - tok0 + BS - 1) / BS;
#pragma unroll
    for (int u = 0; u < Sh::IDS; ++u) {
      const int b = lane + 32 * u;
      ids[u] = -1;
      if (b < nblk) {
        if ((unsigned)raw[u] < (unsigned)p.num_blocks) {
          ids[u] = raw[u];
        } else if (do_k) {
          atomicOr(p.err, PKV_DEVERR_BLOCK_ID);
        }
      }
    }
    if constexpr (F8) {
      // FP8 pool: this warp's tiles (K: 3 slots, freed by S; V: 2 slots, freed by PV). Either widen
      // the oldest tile whose codes have landed, or copy the next tile's codes into its slot's upper
      // half once the slot is free, whichever is ready first.
      const int NS = do_k ? KST : 2;
      uint64_t* landed = do_k ? k_raw : v_raw;
      uint64_t* widened = do_k ? k_full : v_full;
      uint64_t* freed = do_k ? k_empty : pv_done;
      auto slot = [&](int j) { return do_k ? k_slot(j) : v_slot(j); };
      int ni = 0, nc = 0;  // tiles issued, tiles widened
      long long t_last = clock64();
      while (nc < ntile) {
        int act = -1;  // 0: widen tile nc, 1: copy tile ni
        if (lane == 0) {
          if (nc < ni && mbar_test_wait(landed + nc % NS, (nc / NS) & 1))
            act = 0;
          else if (ni < ntile && (ni < NS || mbar_test_wait(freed + ni % NS, ((ni / NS) - 1) & 1)))
            act = 1;
          else if (*abort || clock64() - t_last > kWaitLimitCycles)
            act = 2;
        }
        act = __shfl_sync(kFull, act, 0);
        if (act == 2) {
          if (lane == 0) *abort = 1;
          break;
        }
        if (act < 0) {
          __nanosleep(64);
          continue;
        }
        if (act == 0) {
          mq_tc_widen_tile(slot(nc), slot(nc) + Sh::HALF, lane);
          fence_proxy_async_smem();  // generic stores, read by the MMAs
          __syncwarp();
          if (lane == 0) mbar_arrive(widened + nc % NS);
          ++nc;
        } else {
          const int j = ni;
          int phys = -1;  // lane i < NBT: block j * NBT + i of the partition
#pragma unroll
          for (int u = 0; u < Sh::IDS; ++u) {
            const int b = j * NBT + (lane & (NBT - 1));
            const int x = __shfl_sync(kFull, ids[u], b & 31);
            if ((b >> 5) == u) phys = x;
          }
          if (lane >= NBT || j * NBT + lane >= nblk) phys = -1;
          const unsigned mask = __ballot_sync(kFull, phys >= 0);
          uint64_t* bar = landed + j % NS;
          if (lane == 0) {
            fence_proxy_async_smem();  // the widening (and the rows' zeros) wrote this slot: before the copies
            mbar_arrive_expect_tx(bar, __popc(mask) * BS * 128);
          }
          __syncwarp();
          if (phys >= 0)  // block i of the tile: BS rows of 128 codes at row i * BS of the upper half
            tma_load_2d(slot(j) + Sh::HALF + lane * BS * 128, do_k ? &kmap : &vmap, 0,
                        (phys * p.num_kv_heads + kvh) * BS, bar);
          ++ni;
        }
        t_last = clock64();
      }
      // no copy may still be landing when the CTA leaves
      if (lane == 0)
        for (int j = nc; j < ni; ++j) mbar_wait(landed + j % NS, (j / NS) & 1);
    } else {
    // Copy whichever slot frees first: K tile nk once S_{nk-3} is done, V tile
    // nv (never ahead of K) once PV_{nv-2} is done.
    int nk = 0, nv = 0;
    unsigned zeroed = 0;  // V slots whose tail rows the rows zeroed (generic stores)
    long long t_last = clock64();
    while (do_v ? nv < ntile : nk < ntile) {
      int which = -1;  // 0: K tile nk, 1: V tile nv
      if (lane == 0) {
        if (do_k && nk < ntile && (nk < KST || mbar_test_wait(k_empty + nk % KST, ((nk / KST) - 1) & 1)))
          which = 0;
        else if (do_v && nv < (do_k ? nk : ntile) &&
                 (nv < 2 || mbar_test_wait(pv_done + (nv & 1), ((nv >> 1) - 1) & 1)))
          which = 1;
        else if (*abort || clock64() - t_last > kWaitLimitCycles)
          which = 2;
      }
      which = __shfl_sync(kFull, which, 0);
      if (which == 2) {
        if (lane == 0) *abort = 1;
        break;
      }
      if (which < 0) {
        __nanosleep(64);  // leave the issue slots to the rows' warp on this SM quarter
        continue;
      }
      const int j = which ? nv : nk;
      int phys = -1;  // lane i < NBT: block j * NBT + i of the partition
#pragma unroll
      for (int u = 0; u < Sh::IDS; ++u) {
        const int b = j * NBT + (lane & (NBT - 1));
        const int x = __shfl_sync(kFull, ids[u], b & 31);
        if ((b >> 5) == u) phys = x;
      }
      if (lane >= NBT || j * NBT + lane >= nblk) phys = -1;
      const unsigned mask = __ballot_sync(kFull, phys >= 0);
      uint64_t* bar = which ? v_full + (j & 1) : k_full + j % KST;
      if (lane == 0) {
        if (which && ((zeroed >> (j & 1)) & 1u)) fence_proxy_async_smem();  // the rows' zeros precede the copies
        mbar_arrive_expect_tx(bar, __popc(mask) * DH * BS * 128);
        t_last = clock64();
      }
      if (which) {  // the rows zero this tile's V tail (the same test as theirs)
        const bool z = mask != (1u << NBT) - 1u || tok0 + j * NT + NT > ctx;
        zeroed = (zeroed & ~(1u << (j & 1))) | ((z ? 1u : 0u) << (j & 1));
      }
      __syncwarp();
      if (phys >= 0) {
        const int y = (phys * p.num_kv_heads + kvh) * BS;
        unsigned char* dst = (which ? v_slot(j) : k_slot(j)) + lane * (BS / 8) * Sh::ATOM;
        if constexpr (DH == 2)
          tma_load_4d(dst, which ? &vmap : &kmap, 0, 0, 0, y / 8, bar);  // the block's BS rows, both halves
        else
          tma_load_2d(dst, which ? &vmap : &kmap, 0, y, bar);
      }
      if (PKV_MQ_TC_PREFETCH > 0 && j + PKV_MQ_TC_PREFETCH < ntile) {  // a later tile's blocks into L2
        const int jp = j + PKV_MQ_TC_PREFETCH;
        int pp = -1;
#pragma unroll
        for (int u = 0; u < Sh::IDS; ++u) {
          const int b = jp * NBT + (lane & (NBT - 1));
          const int x = __shfl_sync(kFull, ids[u], b & 31);
          if ((b >> 5) == u) pp = x;
        }
        if (lane < NBT && jp * NBT + lane < nblk && pp >= 0)
          prefetch_l2((which ? p.value_cache : p.key_cache) + ((size_t)pp * p.num_kv_heads + kvh) * BS * D * 2,
                      BS * D * 2);
      }
      if (which) ++nv; else ++nk;
    }
    // no copy may still be landing when the CTA leaves
    if (lane == 0) {
      for (int j = nk > KST ? nk - KST : 0; j < nk; ++j) mbar_wait(k_full + j % KST, (j / KST) & 1);
      for (int j = nv > 2 ? nv - 2 : 0; j < nv; ++j) mbar_wait(v_full + (j & 1), (j >> 1) & 1);
    }
    }
  } else if (Sh::SPLIT && (warp == 1 || warp == Sh::PVW)) {
    // ---- MMA issue, 16-bit pool: one thread of warp 1 the S MMAs, one of the PV warp the PV MMAs, each
    // in tile order with blocking waits (a tcgen05.mma holds its issuing thread while the tensor core
    // takes it in, so with one thread S and PV queued behind each other)
    if (lane == 0) {
      constexpr bool BF = std::is_same<TP, __nv_bfloat16>::value;
      constexpr uint32_t IDESC_S = tc::idesc_f16(BF, Sh::ROWS, NT, false, false);
      constexpr uint32_t IDESC_O = tc::idesc_f16(BF, Sh::ROWS, D, false, true);
      if (warp == 1) {
        // S_j once K_j has landed and PV_{j-2}, the last reader of its S/P buffer, is done
        const uint32_t q_addr = smem_u32(Qs);
        bool ok = tc_wait(q_full, 0, abort);  // the rows have written Q
        for (int j = 0; ok && j < ntile; ++j) {
          ok = tc_wait(k_full + j % KST, (j / KST) & 1, abort) &&
               (j < 2 || tc_wait(pv_done + (j & 1), ((j >> 1) - 1) & 1, abort));
          if (!ok) break;
          tc::fence_after_sync();
          const uint32_t k_addr = smem_u32(k_slot(j));
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint64_t a = tc::desc_sw128(q_addr + (k / 4) * (Sh::ROWS * 128) + (k % 4) * 32, 16, 1024);
            const uint64_t b = tc::desc_sw128(k_addr + (k / 4) * 1024 + (k % 4) * 32, 16, Sh::ATOM);
            tc::mma_f16(tbase + Sh::S_COL + (j & 1) * NT, a, b, IDESC_S, k > 0);
          }
          tc::commit(s_full + (j & 1));
          tc::commit(k_empty + j % KST);
        }
        tc::commit(fin);  // every S MMA issued above has completed once this arrives
        mbar_wait(fin, 0);
      } else {
        // O += P_j . V_j once P_j is written and V_j has landed; then V slot j % 2 and S/P buffer j % 2
        // are free
        for (int j = 0; j < ntile; ++j) {
          const bool ok = tc_wait(p_full + (j & 1), (j >> 1) & 1, abort) &&
                          tc_wait(v_full + (j & 1), (j >> 1) & 1, abort);
          if (!ok) break;
          tc::fence_after_sync();
          const uint32_t v_addr = smem_u32(v_slot(j));
#pragma unroll
          for (int k = 0; k < NT / 16; ++k) {
            const uint64_t b = tc::desc_sw128(v_addr + k * 2 * Sh::ATOM, 1024, Sh::ATOM);
            tc::mma_f16_ta(tbase, tbase + Sh::S_COL + (j & 1) * NT + k * 8, b, IDESC_O, j > 0 || k > 0);
          }
          tc::commit(pv_done + (j & 1));
        }
        tc::commit(fin_pv);  // every PV MMA issued above has completed once this arrives
        mbar_wait(fin_pv, 0);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- MMA issue (one thread)
    if (lane == 0) {
      constexpr bool BF = std::is_same<TP, __nv_bfloat16>::value;
      constexpr uint32_t IDESC_S = tc::idesc_f16(BF, Sh::ROWS, NT, false, false);
      constexpr uint32_t IDESC_O = tc::idesc_f16(BF, Sh::ROWS, D, false, true);
      const uint32_t q_addr = smem_u32(Qs);
      auto issue_s = [&](int j) {  // S_j = Q . K_j^T into S/P buffer j % 2, then K slot j % 3 is free
        const uint32_t k_addr = smem_u32(k_slot(j));
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint64_t a = tc::desc_sw128(q_addr + (k / 4) * (Sh::ROWS * 128) + (k % 4) * 32, 16, 1024);
          const uint64_t b = tc::desc_sw128(k_addr + (k / 4) * 1024 + (k % 4) * 32, 16, Sh::ATOM);
          tc::mma_f16(tbase + Sh::S_COL + (j & 1) * NT, a, b, IDESC_S, k > 0);
        }
        tc::commit(s_full + (j & 1));
        tc::commit(k_empty + j % KST);
      };
      auto issue_pv = [&](int j) {  // O += P_j . V_j, then V slot j % 2 and S/P buffer j % 2 are free
        const uint32_t v_addr = smem_u32(v_slot(j));
#pragma unroll
        for (int k = 0; k < NT / 16; ++k) {
          const uint64_t b = tc::desc_sw128(v_addr + k * 2 * Sh::ATOM, 1024, Sh::ATOM);
          tc::mma_f16_ta(tbase, tbase + Sh::S_COL + (j & 1) * NT + k * 8, b, IDESC_O, j > 0 || k > 0);
        }
        tc::commit(pv_done + (j & 1));
      };
      // Issue whichever is ready: S_ns once K_ns has landed and PV_{ns-2} (the
      // last reader of its buffer) is done; PV_npv once P_npv is written and
      // V_npv has landed.
      int ns = 0, npv = 0;
      bool q_in = false;  // the rows have written Q
      long long t_last = clock64();
      while (npv < ntile) {
        bool progressed = false;
        if (!q_in) q_in = mbar_test_wait(q_full, 0);
        if (q_in && ns < ntile && mbar_test_wait(k_full + ns % KST, (ns / KST) & 1) &&
            (ns < 2 || mbar_test_wait(pv_done + (ns & 1), ((ns >> 1) - 1) & 1))) {
          tc::fence_after_sync();
          issue_s(ns++);
          progressed = true;
        } else if (npv < ns && mbar_test_wait(p_full + (npv & 1), (npv >> 1) & 1) &&
                   mbar_test_wait(v_full + (npv & 1), (npv >> 1) & 1)) {
          tc::fence_after_sync();
          issue_pv(npv++);
          progressed = true;
        }
        if (progressed) {
          t_last = clock64();
        } else if (__nanosleep(32), *abort) {
          break;
        } else if (clock64() - t_last > kWaitLimitCycles) {
          *abort = 1;
          break;
        }
      }
      tc::commit(fin);  // every MMA issued above has completed once this arrives
      mbar_wait(fin, 0);
    }
    __syncwarp();
  } else if (srole) {
    // ---- softmax rows
    // the query rows (zeros past R), copied while the copy warps start: tell the MMA thread once landed
    float qscale = 1.f;  // FP8 pool, bf16 query: the 2^-k the row was scaled by
    if constexpr (F8 && std::is_same<T, __nv_bfloat16>::value) {
      qscale = mq_tc_fetch_q_bf16_as_f16<D, Sh::ROWS>(Qs, row, reinterpret_cast<const __nv_bfloat16*>(p.query), q0,
                                                      kvh, rt, q_len, G, p.num_heads);
    } else {
      mq_tc_fetch_q<T, D, Sh::ROWS>(Qs, row, reinterpret_cast<const T*>(p.query), q0, kvh, rt, q_len, G, p.num_heads);
      cp_async_wait_all();
    }
    fence_proxy_async_smem();  // generic-proxy writes, read by the S MMAs
    mbar_arrive(q_full);
    const int lim = active ? mq_limit(mq, ctx, q_len, r, G) : 0;  // this row sees positions < lim
    const int vis = min(lim, tok1);
    const float sl2 = p.scale_log2 * qscale;
    const bool neg = sl2 < 0.f;  // a negative scale: the largest score comes from the smallest product
    const uint32_t all = (1u << NBT) - 1u;
    // which blocks of each tile were fetched: the same test as the producer's
    int ids[Sh::IDS];
    const int nblk = (tok1 - tok0 + BS - 1) / BS;
#pragma unroll
    for (int u = 0; u < Sh::IDS; ++u) {
      const int b = lane + 32 * u;
      ids[u] = 0;
      if (b < nblk) ids[u] = (unsigned)p.block_tables[(size_t)s * p.max_blocks_per_seq + blk0 + b] < (unsigned)p.num_blocks;
    }
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < ntile; ++j) {
      const int tb = tok0 + j * NT;
      // (tensor-memory accesses are warp-wide: a warp leaves the loop as a whole)
      ok = tc_wait(s_full + (j & 1), (j >> 1) & 1, abort);
      if (!__all_sync(kFull, ok)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      uint32_t sr[2][32];
      tc::ld32(tc::taddr(tbase, 32 * (warp & 3), Sh::S_COL + (j & 1) * NT), sr[0]);
      tc::ld32(tc::taddr(tbase, 32 * (warp & 3), Sh::S_COL + (j & 1) * NT + 32), sr[1]);
      tc::wait_ld();
      int fetched = 0;
#pragma unroll
      for (int u = 0; u < Sh::IDS; ++u) {
        const int b = j * NBT + (lane & (NBT - 1));
        const int x = __shfl_sync(kFull, ids[u], b & 31);
        if ((b >> 5) == u) fetched = x;
      }
      const uint32_t mask = __ballot_sync(kFull, lane < NBT && fetched) & all;
      const int nv = vis - tb;  // leading tokens of the tile this row may see
      // x[t] * mul is the score in the base-2 domain. A tile the row sees whole keeps the raw products
      // (mul = sl2): the max of the raw scores, times sl2, is the max of the scaled ones (the min, for a
      // negative scale), and each weight is then one fused multiply-add into exp2. A partial tile scales
      // first and masks with -inf (mul = 1).
      float x[NT];
      float mq[4];  // four independent max (or min) chains
      float mx, mul;
      if (nv >= NT && mask == all) {
        mul = sl2;
        if (neg) {
          mq[0] = mq[1] = mq[2] = mq[3] = INFINITY;
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            x[t] = __uint_as_float(sr[t >> 5][t & 31]);
            mq[t & 3] = fminf(mq[t & 3], x[t]);
          }
          mx = fminf(fminf(mq[0], mq[1]), fminf(mq[2], mq[3])) * sl2;
        } else {
          mq[0] = mq[1] = mq[2] = mq[3] = -INFINITY;
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            x[t] = __uint_as_float(sr[t >> 5][t & 31]);
            mq[t & 3] = fmaxf(mq[t & 3], x[t]);
          }
          mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * sl2;
        }
      } else {
        mul = 1.f;
        mq[0] = mq[1] = mq[2] = mq[3] = -INFINITY;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const bool see = t < nv && ((mask >> (t / BS)) & 1u);
          x[t] = see ? __uint_as_float(sr[t >> 5][t & 31]) * sl2 : -INFINITY;
          mq[t & 3] = fmaxf(mq[t & 3], x[t]);
        }
        mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
      }
      const bool move = mx > m_ref + 8.f;
      const bool resc = j > 0 && move && m_ref != -INFINITY;  // O's row holds terms to rescale
      const float f = resc ? fast_exp2(m_ref - mx) : 1.f;
      if (move) m_ref = mx;
      // P row as 16-bit pairs (exp2(-inf) = 0 for masked tokens; a row that has seen nothing yet keeps
      // m_ref = -inf and gets zeros). l sums the fp32 weights before their rounding to 16 bits, which
      // moves the result by at most the rounding unit times the row's largest |v| (2^-9 for bf16 P).
      uint32_t pw[NT / 2];
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
      if (m_ref != -INFINITY) {
        const float nm = -m_ref;
#pragma unroll
        for (int u = 0; u < NT / 2; ++u) {
          const float p0 = fast_exp2(fmaf(x[2 * u], mul, nm)), p1 = fast_exp2(fmaf(x[2 * u + 1], mul, nm));
          pw[u] = Elem<TP>::pack2(p0, p1);
          ls[u & 3] += p0 + p1;
        }
      } else {
#pragma unroll
        for (int u = 0; u < NT / 2; ++u) pw[u] = 0u;
      }
      if (__any_sync(kFull, resc)) {  // the whole warp moves its rows' O (factor 1 for rows that keep theirs)
        ok = tc_wait(pv_done + ((j - 1) & 1), ((j - 1) >> 1) & 1, abort);  // once PV_{j-1} is done
        if (!__all_sync(kFull, ok)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tc::ld32(tc::taddr(tbase, 32 * (warp & 3), c * 32), o);
          tc::wait_ld();
#pragma unroll
          for (int u = 0; u < 32; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * f);
          tc::st32(tc::taddr(tbase, 32 * (warp & 3), c * 32), o);
        }
        tc::wait_st();
      }
      l = l * f + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
      tc::st32(tc::taddr(tbase, 32 * (warp & 3), Sh::S_COL + (j & 1) * NT), pw);  // P_j over S_j
      tc::wait_st();
      // V rows past the context, or of blocks not fetched, may hold anything (NaN):
      // zero them once V_j has landed, since P = 0 times NaN is NaN in the MMA
      if (mask != all || tb + NT > ctx) {
        ok = tc_wait(v_full + (j & 1), (j >> 1) & 1, abort);
        if (!__all_sync(kFull, ok)) {
          ok = false;
          break;
        }
        unsigned char* vs = v_slot(j);
        for (int i = threadIdx.x - 32 * Sh::SW; i < NT * 8 * DH; i += 128) {
          const int t = i / (8 * DH), c = i % (8 * DH);
          if (!((mask >> (t / BS)) & 1u) || tb + t >= ctx)
            *reinterpret_cast<uint4*>(vs + (t / 8) * Sh::ATOM + (c / 8) * 1024 + tc::sw128(t % 8, c % 8)) =
                make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();  // the zeros precede the PV's reads
      }
      tc::fence_before_sync();
      mbar_arrive(p_full + (j & 1));
    }
    // epilogue: O / l
    if (ok) ok = tc_wait(pv_done + ((ntile - 1) & 1), ((ntile - 1) >> 1) & 1, abort);
    tc::fence_after_sync();
    ok = ok && !*abort;
    // 1 / l (FP8 pool: times the value of one V code)
    const float inv = ok && l > 0.f ? (F8 ? p.v_scale : 1.f) / l : 0.f;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      tc::ld32(tc::taddr(tbase, 32 * (warp & 3), c * 32), o);
      tc::wait_ld();
      if (!active) continue;
      if (direct) {
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<T*>(p.out) + orow * D + c * 32);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = Elem<T>::pack2(__uint_as_float(o[8 * u + 2 * e]) * inv, __uint_as_float(o[8 * u + 2 * e + 1]) * inv);
          dst[u] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      } else {
        float4* dst = reinterpret_cast<float4*>(p.part_o + (orow * p.max_partitions + part) * D + c * 32);
#pragma unroll
        for (int u = 0; u < 8; ++u)  // partials are normalised by their own l (inv = 0 after a failure)
          dst[u] = make_float4(__uint_as_float(o[4 * u]) * inv, __uint_as_float(o[4 * u + 1]) * inv,
                               __uint_as_float(o[4 * u + 2]) * inv, __uint_as_float(o[4 * u + 3]) * inv);
      }
    }
    if (active && !direct) {
      p.part_m[orow * p.max_partitions + part] = ok ? m_ref : -INFINITY;
      p.part_l[orow * p.max_partitions + part] = ok ? l : 0.f;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (*abort && threadIdx.x == 0) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
  if (warp == 1) {
    tc::fence_after_sync();
    tc::dealloc(tbase, Sh::TMEM_COLS);
  }
}

template <typename T, int D, int BS, bool F8 = false>
cudaError_t launch_mq_tc(const DecodeParams& p, const MqParams& mq, const CUtensorMap& kmap,
                         const CUtensorMap& vmap, int num_seqs, cudaStream_t stream) {
  using Sh = MqTcShape<T, D, BS, F8>;
  auto kern = pkv_mq_tc_kernel<T, D, BS, F8>;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM);
    if (e != cudaSuccess) return e;
    // two CTAs need nearly all of the SM's shared memory: ask for the largest carveout
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  const dim3 grid(p.max_partitions, p.num_kv_heads * mq.row_tiles, num_seqs);
  return launch_kernel(kern, grid, dim3(Sh::THREADS), Sh::SMEM, stream, p, mq, kmap, vmap);
}

}  // namespace pkv
