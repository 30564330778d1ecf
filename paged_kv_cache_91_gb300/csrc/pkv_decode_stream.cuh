// Persistent decode attention with equal work per warp.
//
// The decode step's work is the set of (sequence s, head group g, block j)
// tiles: for every sequence, every head group (a query head on the CUDA-core
// path, a kv head with its G query heads on the tensor-core path) reads the
// sequence's ceil(ctx / B) blocks. Flattened with j innermost, that is a list
// of T tiles in which each (s, g) pair -- a "segment" -- is one contiguous run.
// A persistent grid of W warps (one wave) splits the list into W equal ranges;
// each warp streams its range through a private ring of bulk-copied stages
// without ever draining it, so every warp moves the same number of bytes and no
// CTA waits on an empty partition.
//
// A warp keeps one running softmax per segment ("KV Cache와 PagedAttention 완전
// 해부", 부록; "vLLM: LLM 서빙 메모리 최적화의 교과서", eq. (4)). A segment that
// lies wholly inside one warp's range is normalised and written to `out` by that
// warp. A segment cut by range boundaries leaves one (m, l, o) partial per warp
// that touches it -- at most two per warp, its first and its last segment -- and
// pkv_stream_reduce_kernel merges them by log-sum-exp.
//
// Each warp finds the segment of its tiles by binary search over a prefix of
// blocks per sequence that every CTA builds in shared memory, 32 tiles at a
// time and well ahead of use. The query rows of a segment ride into shared
// memory in the same stage as the segment's first tile, so a new segment costs
// no extra round trip to HBM.
#pragma once

#include "pkv_decode_mma.cuh"
#include "pkv_decode_simt.cuh"

namespace pkv {

constexpr int kStreamMaxSeqs = 2048;   // prefix arrays live in shared memory
constexpr int kStreamMaxWarps = 2048;  // bounds the partial slots in the workspace

#ifndef PKV_STREAM_WARPS
#define PKV_STREAM_WARPS 4  // warps per persistent CTA (build-time tuning knob)
#endif
#ifndef PKV_STREAM_RING_BYTES
#define PKV_STREAM_RING_BYTES (64 * 1024)  // K/V ring bytes per persistent CTA (build-time tuning knob)
#endif
constexpr int kStreamWarps = PKV_STREAM_WARPS;

template <bool MMA, int D>
struct StreamQ {
  // bytes reserved per stage for a segment's query rows (16-byte multiple;
  // 1024-byte multiple on the tensor-core path so tiles stay swizzle-aligned)
  static constexpr int BYTES = MMA ? 8 * D * 2 : D * 2;
};

// Stages per warp of the persistent kernel: PKV_STREAM_RING_BYTES of K/V tiles,
// 1 to 8 stages, and never more than fits in 227 KB of shared memory next to
// the largest prefix arrays.
template <int D, int BS, bool MMA>
constexpr int stream_stages() {
  constexpr int kv = 2 * BS * D * 2;
  constexpr int full = kv + StreamQ<MMA, D>::BYTES;
  constexpr int room = 232448 - (2 * kStreamMaxSeqs + 1) * 4 - 1024 - 1024;
  constexpr int by_ring = (PKV_STREAM_RING_BYTES) / (kStreamWarps * kv);
  constexpr int by_smem = room / (kStreamWarps * full);
  constexpr int spw = by_ring < by_smem ? by_ring : by_smem;
  return spw < 1 ? 1 : (spw > 8 ? 8 : spw);
}

struct StreamParams {
  DecodeParams p;
  int num_seqs;
  int ng;  // head groups per sequence
  int gc;  // query heads per group (1, or G on the tensor-core path)
  int* pre_out;  // workspace: blocks-per-sequence prefix [S + 1], written by CTA 0
  float* slot_o;  // workspace: [W][2][gc][D] normalised partial outputs
  float* slot_m;  // workspace: [W][2][gc]
  float* slot_l;  // workspace: [W][2][gc]
};

template <int D, int BS, int NW, int SPW, bool MMA>
struct StreamShape {
  static constexpr int TILE = BS * D * 2;
  static constexpr int STAGE = 2 * TILE + StreamQ<MMA, D>::BYTES;
  static constexpr int RING = NW * SPW * STAGE;
  static constexpr int BARS = RING;
  static constexpr int PRE = BARS + ((NW * SPW * 8 + 127) / 128) * 128;  // ints follow the barriers
  static constexpr int ALIGN = MMA ? 1024 : 128;
  static_assert(STAGE % 16 == 0, "stage alignment");
  static_assert(!MMA || STAGE % 1024 == 0, "swizzled tiles need 1024-byte aligned stages");
  static constexpr int smem_bytes(int num_seqs) { return PRE + (2 * num_seqs + 1) * 4 + ALIGN; }
};

// metadata flag bits of one tile
constexpr int kFlagFirst = 1 << 8;      // first tile of its segment within this warp
constexpr int kFlagLast = 1 << 9;       // last tile of its segment within this warp
constexpr int kFlagComplete = 1 << 10;  // the whole segment lies in this warp's range
constexpr int kFlagSlot1 = 1 << 11;     // a split segment that starts inside the range (partial slot 1)

template <typename T, int D, int BS, int NW, int SPW, bool MMA>
__global__ void __launch_bounds__(NW * 32, 1)
    pkv_decode_stream_kernel(const StreamParams sp, const __grid_constant__ CUtensorMap kmap,
                             const __grid_constant__ CUtensorMap vmap) {
  pdl_begin();
  using Sh = StreamShape<D, BS, NW, SPW, MMA>;
  using ST = SimtTile<T, T, D, BS>;
  using MT = MmaTile<T, D, BS>;
  const DecodeParams& p = sp.p;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + Sh::ALIGN - 1) & ~static_cast<uintptr_t>(Sh::ALIGN - 1));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = sp.num_seqs, ng = sp.ng, gc = sp.gc;
  int* pre = reinterpret_cast<int*>(smem + Sh::PRE);  // [S + 1]
  int* ctxs = pre + S + 1;                            // [S], clamped

  // ---- blocks-per-sequence prefix (every CTA builds its own copy)
  {
    constexpr int NT = NW * 32;
    const int per = (S + NT - 1) / NT;
    const int i0 = threadIdx.x * per;
    int sum = 0;
    for (int i = i0; i < i0 + per && i < S; ++i) {
      const int c = clamp_context(p, i, blockIdx.x == 0);
      ctxs[i] = c;
      sum += (c + BS - 1) / BS;
    }
    int incl = sum;  // inclusive scan of the per-thread sums across the CTA
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += v;
    }
    __shared__ int warp_tot[NW];
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w) before += warp_tot[w];
    int run = before + incl - sum;  // exclusive prefix of this thread's first element
    if (threadIdx.x == 0) pre[0] = 0;
    for (int i = i0; i < i0 + per && i < S; ++i) {
      run += (ctxs[i] + BS - 1) / BS;
      pre[i + 1] = run;
    }
    __syncthreads();
    if (blockIdx.x == 0)
      for (int i = threadIdx.x; i <= S; i += NT) sp.pre_out[i] = pre[i];
  }

  // ---- this warp's range of the flattened tile list
  const int total = ng * pre[S];
  const int nwarps = gridDim.x * NW;
  const int R = (total + nwarps - 1) / nwarps;
  const int w = blockIdx.x * NW + warp;
  const int r0 = min(w * R, total), r1 = min(r0 + R, total);
  const int n = r1 - r0;

  unsigned char* ring = smem + warp * SPW * Sh::STAGE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sh::BARS) + warp * SPW;
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < SPW; ++k) mbar_init(bars + k, 1);
    fence_mbar_init();
  }
  if (MMA && threadIdx.x == 0) {
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
  }
  __syncwarp();
  if (n <= 0) return;

  // Metadata of tile r0 + b for this lane's b (32 tiles per batch): physical
  // block, first query row of the segment, and valid tokens | flags.
  auto meta = [&](int b, int& phys, int& qrow, int& flags) {
    phys = -1;
    qrow = 0;
    flags = 0;
    const int f = r0 + b;
    if (b >= n) return;
    int lo = 0, hi = S - 1;  // the last sequence whose tiles start at or before f
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (ng * pre[mid] <= f) lo = mid; else hi = mid - 1;
    }
    const int s = lo;
    const int nb = pre[s + 1] - pre[s];
    const int local = f - ng * pre[s];
    const int g = local / nb;
    const int j = local - g * nb;
    const int a = ng * pre[s] + g * nb;  // first tile of the segment
    const int v = p.block_tables[(size_t)s * p.max_blocks_per_seq + j];
    if ((unsigned)v < (unsigned)p.num_blocks) {
      phys = v;
    } else {
      atomicOr(p.err, PKV_DEVERR_BLOCK_ID);
    }
    qrow = s * p.num_heads + g * gc;
    flags = min(BS, ctxs[s] - j * BS);
    if (j == 0 || f == r0) flags |= kFlagFirst;
    if (j == nb - 1 || f == r1 - 1) flags |= kFlagLast;
    if (a >= r0 && a + nb <= r1) flags |= kFlagComplete;
    if (a > r0) flags |= kFlagSlot1;
  };
  int ph[2], qr[2], fl[2];  // two batches: tiles [32k, 32k + 32) live in set k & 1
  meta(lane, ph[0], qr[0], fl[0]);
  meta(32 + lane, ph[1], qr[1], fl[1]);
  auto get = [&](int i, int& phys, int& qrow, int& flags) {
    const int set = (i >> 5) & 1, src = i & 31;
    phys = __shfl_sync(kFull, set ? ph[1] : ph[0], src);
    qrow = __shfl_sync(kFull, set ? qr[1] : qr[0], src);
    flags = __shfl_sync(kFull, set ? fl[1] : fl[0], src);
  };

  const int qbytes = gc * D * 2;
  unsigned zeroed = 0;  // stages whose tail rows were zeroed since their last refill
  auto issue = [&](int i) {
    int phys, qrow, flags;
    get(i, phys, qrow, flags);
    if (lane == 0) {
      uint64_t* bar = bars + (i % SPW);
      unsigned char* st = ring + (i % SPW) * Sh::STAGE;
      const bool first = flags & kFlagFirst;
      const uint32_t bytes = (phys >= 0 ? 2 * Sh::TILE : 0) + (first ? qbytes : 0);
      if (bytes) {
        // generic stores (tail zeroing) into this stage must be ordered before the copy's writes
        if (PKV_PROXY_FENCE || ((zeroed >> (i % SPW)) & 1u)) fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, bytes);
        if (phys >= 0) {
          const int kvh = (qrow % p.num_heads) / p.group;  // kv head of the segment's query rows
          if constexpr (MMA) {
            MT::issue_tiles(st, &kmap, &vmap, (phys * p.num_kv_heads + kvh) * BS, bar);
          } else {
            const size_t off = ((size_t)phys * p.num_kv_heads + kvh) * Sh::TILE;
            bulk_g2s(st, p.key_cache + off, Sh::TILE, bar);
            bulk_g2s(st + Sh::TILE, p.value_cache + off, Sh::TILE, bar);
          }
        }
        if (first)
          bulk_g2s(st + 2 * Sh::TILE, static_cast<const unsigned char*>(p.query) + (size_t)qrow * D * 2, qbytes,
                   bar);
      } else {
        mbar_arrive(bar);
      }
    }
  };
  const int nfirst = n < SPW ? n : SPW;
  for (int i = 0; i < nfirst; ++i) issue(i);
  int issued = nfirst;

  // running state of the current segment
  float m = -INFINITY, l = 0.f, m1 = -INFINITY, l1 = 0.f;
  float qreg[MMA ? 1 : ST::Sh::DPL];
  float acc_s[MMA ? 1 : ST::Sh::DPV];
  uint32_t qb[MMA ? MT::KT : 1][2];
  float acc_m[MMA ? MT::KT : 1][4];

  int failed_at = -1;
  for (int i = 0; i < n; ++i) {
    int phys, qrow, flags;
    get(i, phys, qrow, flags);
    const int k = i % SPW;
    const bool ready = __all_sync(kFull, mbar_wait(bars + k, (i / SPW) & 1));
    if (!ready) {
      failed_at = i;
      break;
    }
    unsigned char* st = ring + k * Sh::STAGE;
    if (flags & kFlagFirst) {
      m = m1 = -INFINITY;
      l = l1 = 0.f;
      const T* qs = reinterpret_cast<const T*>(st + 2 * Sh::TILE);
      if constexpr (MMA) {
#pragma unroll
        for (int mt = 0; mt < MT::KT; ++mt) acc_m[mt][0] = acc_m[mt][1] = acc_m[mt][2] = acc_m[mt][3] = 0.f;
        float sl_unused0, sl_unused1;
        MT::load_qb(qb, qs, gc, lane, p.scale_log2, sl_unused0, sl_unused1);
      } else {
#pragma unroll
        for (int e = 0; e < ST::Sh::DPV; ++e) acc_s[e] = 0.f;
        ST::load_q(qreg, qs, lane, p.scale_log2);
      }
    }
    if (phys >= 0) {
      const int nvalid = flags & 0xff;
      if constexpr (MMA) {
        MT::run(st, st + Sh::TILE, nvalid, qb, lane, p.scale_log2, p.scale_log2, m, m1, l, l1, acc_m);
        if (nvalid < BS) zeroed |= 1u << k;
      } else {
        ST::run(st, st + Sh::TILE, nvalid, qreg, lane, m, l, acc_s);
      }
    }
    if (flags & kFlagLast) {
      // finish the segment: the final output, or this warp's partial of it
      const bool complete = flags & kFlagComplete;
      const size_t slot = (size_t)w * 2 + ((flags & kFlagSlot1) ? 1 : 0);
      if constexpr (MMA) {
        const int j0 = (lane & 3) * 2, r0l = lane >> 2;
        const float inv0 = l > 0.f ? 1.f / l : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
        for (int mt = 0; mt < MT::KT; ++mt) {
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int j = j0 + h2;
            if (j < gc) {
              const float inv = h2 ? inv1 : inv0;
              const int d0 = mt * 16 + r0l;
              const float o0 = acc_m[mt][h2] * inv, o1 = acc_m[mt][2 + h2] * inv;
              if (complete) {
                T* orow = reinterpret_cast<T*>(p.out) + (size_t)(qrow + j) * D;
                orow[d0] = Elem<T>::from_float(o0);
                orow[d0 + 8] = Elem<T>::from_float(o1);
              } else {
                float* prow = sp.slot_o + (slot * gc + j) * D;
                prow[d0] = o0;
                prow[d0 + 8] = o1;
              }
            }
          }
        }
        if (!complete && lane < 4) {
          if (j0 < gc) {
            sp.slot_m[slot * gc + j0] = m;
            sp.slot_l[slot * gc + j0] = l;
          }
          if (j0 + 1 < gc) {
            sp.slot_m[slot * gc + j0 + 1] = m1;
            sp.slot_l[slot * gc + j0 + 1] = l1;
          }
        }
      } else {
        constexpr int DPV = ST::Sh::DPV;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        if (complete) {
          T* orow = reinterpret_cast<T*>(p.out) + (size_t)qrow * D + lane * DPV;
          if constexpr (DPV == 4) {
            uint2 v;
            v.x = Elem<T>::pack2(acc_s[0] * inv, acc_s[1] * inv);
            v.y = Elem<T>::pack2(acc_s[2] * inv, acc_s[3] * inv);
            *reinterpret_cast<uint2*>(orow) = v;
          } else {
            *reinterpret_cast<uint32_t*>(orow) = Elem<T>::pack2(acc_s[0] * inv, acc_s[1] * inv);
          }
        } else {
          float* prow = sp.slot_o + slot * D + lane * DPV;
#pragma unroll
          for (int e = 0; e < DPV; ++e) prow[e] = acc_s[e] * inv;
          if (lane == 0) {
            sp.slot_m[slot] = m;
            sp.slot_l[slot] = l;
          }
        }
      }
    }
    __syncwarp();
    if (i + SPW < n) {
      issue(i + SPW);
      zeroed &= ~(1u << k);
      ++issued;
    }
    if ((i & 31) == 31) {
      // tiles up to i are consumed and issued: refill their set with the batch after
      // the next one (its block-table loads overlap the copies now in flight)
      const int b = i + 33;
      int a0, a1, a2;
      meta(b + lane, a0, a1, a2);
      if (((b >> 5) & 1) == 0) {
        ph[0] = a0; qr[0] = a1; fl[0] = a2;
      } else {
        ph[1] = a0; qr[1] = a1; fl[1] = a2;
      }
    }
  }

  if (failed_at >= 0) {
    // a copy did not arrive in time: report and let the other copies land
    if (lane == 0) atomicOr(p.err, PKV_DEVERR_TIMEOUT);
    for (int j = failed_at; j < issued; ++j) mbar_wait(bars + (j % SPW), (j / SPW) & 1);
  }
}

// Merge the partials of every split segment, and zero the rows of empty contexts.
// One CTA per (head group, sequence).
template <typename T>
__global__ void pkv_stream_reduce_kernel(T* __restrict__ out, const float* __restrict__ slot_o,
                                         const float* __restrict__ slot_m, const float* __restrict__ slot_l,
                                         const int* __restrict__ pre, int num_seqs, int num_heads, int head_dim,
                                         int ng, int gc, int nwarps) {
  pdl_begin();
  __shared__ float s_max[8], s_inv[8];
  const int g = blockIdx.x, s = blockIdx.y;
  const int nb = pre[s + 1] - pre[s];
  const size_t qrow = (size_t)s * num_heads + (size_t)g * gc;
  if (nb == 0) {
    for (int i = threadIdx.x; i < gc * head_dim; i += blockDim.x) out[qrow * head_dim + i] = Elem<T>::from_float(0.f);
    return;
  }
  const int total = ng * pre[num_seqs];
  const int R = (total + nwarps - 1) / nwarps;
  const int a = ng * pre[s] + g * nb;
  const int w_lo = a / R, w_hi = (a + nb - 1) / R;
  if (w_lo == w_hi) return;  // written whole by one warp
  const int nc = w_hi - w_lo + 1;
  const bool lo_slot1 = a != w_lo * R;  // the first contributor holds it in its slot 1
  auto slot_of = [&](int k) -> size_t { return (size_t)(w_lo + k) * 2 + ((k == 0 && lo_slot1) ? 1 : 0); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int j = warp; j < gc; j += blockDim.x >> 5) {
    float M = -INFINITY;
    for (int k = lane; k < nc; k += 32) M = fmaxf(M, slot_m[slot_of(k) * gc + j]);
    M = warp_max(M);
    float W = 0.f;
    for (int k = lane; k < nc; k += 32) {
      const float mk = slot_m[slot_of(k) * gc + j];
      if (mk != -INFINITY) W += slot_l[slot_of(k) * gc + j] * fast_exp2(mk - M);
    }
    W = warp_sum(W);
    if (lane == 0) {
      s_max[j] = M;
      s_inv[j] = W > 0.f ? 1.f / W : 0.f;
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < gc * head_dim; i += blockDim.x) {
    const int j = i / head_dim, d = i - j * head_dim;
    const float M = s_max[j];
    float o = 0.f;
    for (int k = 0; k < nc; ++k) {
      const size_t sl = slot_of(k) * gc + j;
      const float mk = slot_m[sl];
      if (mk != -INFINITY) o += slot_l[sl] * fast_exp2(mk - M) * slot_o[sl * head_dim + d];
    }
    out[(qrow + j) * head_dim + d] = Elem<T>::from_float(o * s_inv[j]);
  }
}

template <typename T, int D, int BS, bool MMA>
struct StreamLaunch {
  static constexpr int NW = kStreamWarps;
  static constexpr int SPW = stream_stages<D, BS, MMA>();
  using Sh = StreamShape<D, BS, NW, SPW, MMA>;
  static constexpr auto kernel() { return pkv_decode_stream_kernel<T, D, BS, NW, SPW, MMA>; }

  // CTAs of this kernel one SM holds with the prefix arrays of num_seqs sequences
  static cudaError_t occupancy(int num_seqs, int* ctas) {
    static bool configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
      e = cudaFuncSetAttribute(kernel(), cudaFuncAttributeMaxDynamicSharedMemorySize,
                               Sh::smem_bytes(kStreamMaxSeqs));
      if (e != cudaSuccess) return e;
      configured[dev] = true;
    }
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, kernel(), NW * 32, Sh::smem_bytes(num_seqs));
  }

  static cudaError_t launch(const StreamParams& sp, const CUtensorMap& kmap, const CUtensorMap& vmap, int grid,
                            cudaStream_t stream) {
    return launch_kernel(kernel(), dim3(grid), dim3(NW * 32), Sh::smem_bytes(sp.num_seqs), stream, sp, kmap, vmap);
  }
};

}  // namespace pkv
