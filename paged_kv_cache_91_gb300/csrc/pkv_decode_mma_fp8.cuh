// Decode attention over an FP8 (E4M3) KV pool on the tensor cores.
//
// The contraction of MmaTile (pkv_decode_mma.cuh) for an 8-bit cache: for a
// 16-token slice of a block, S^T[16 x G] = K[16 x D] . Q^T[D x G] and
// O^T[D x G] += V^T[D x 16] . P^T[16 x G] as m16n8k16 f16 MMAs with fp32
// accumulation, the G <= 8 query heads of one kv head in the n = 8 dimension.
// Used for every group size up to 8, MHA included: the MMA does a whole
// 16 x 16 x 8 multiply-add step per instruction, where the CUDA cores would
// spend one instruction per element and head.
//
// Widening. Every E4M3 value is exactly an f16 value. One conversion
// instruction widens the two codes of a 16-bit half of a register into an f16
// pair; applied to the two halves of a loaded word it costs about one
// integer-pipe instruction per pair, half of what an integer bit rearrangement
// or the conversion intrinsic's repacking costs (measured on this GPU).
//
// Layout. The tile arrives through a 2D tensor map as BS rows of 128 bytes
// (D = 128 codes) with the 128-byte swizzle: 16-byte chunk c of row t sits at
// chunk position c ^ (t % 8). Lane (g = lane / 4, qd = lane % 4) uses only whole
// 16-byte chunks, each one conflict-free load, by choosing which head dim sits
// at which MMA position:
//   score MMA, k-step j: positions 2qd, 2qd+1 are dims 32qd + 4j + 0, + 1 and
//     positions 2qd+8, 2qd+9 are dims 32qd + 4j + 2, + 3 (the two halves of one
//     word), so the lane reads bytes 32qd .. 32qd+31 of token rows g and g + 8;
//     Q^T uses the same dim order.
//   PV MMA, m-tile i: row g is dim 16g + 2i, row g + 8 is dim 16g + 2i + 1, so
//     the lane needs chunk g of token rows 2qd, 2qd+1, 2qd+8, 2qd+9; a byte
//     permute pairs the two token rows of each dim in a 16-bit half.
// Every dim still meets every other factor once, so S and O are unchanged.
//
// The MMA multiplies f16 by f16. An f16 query is used as it is. A bf16 query is
// multiplied by 2^k (k per head, so that its largest magnitude lies in
// [2^14, 2^15)) and rounded to f16, which keeps all of its 8 significant bits
// except in components below 2^-14 of that scaled range, whose contribution is
// far below the fp32 accumulation error; the score multiplier undoes 2^k. P is
// rounded to f16 for the PV product and l sums the same rounded values.
#pragma once

#include <type_traits>

#include "pkv_decode_mma.cuh"

#ifndef PKV_MMA_FP8_MIN_CTAS
#define PKV_MMA_FP8_MIN_CTAS 4  // __launch_bounds__ minimum CTAs per SM (build-time tuning knob)
#endif
#ifndef PKV_MMA_FP8_RING_BYTES
#define PKV_MMA_FP8_RING_BYTES (48 * 1024)  // ring bytes per CTA (build-time tuning knob)
#endif

namespace pkv {

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) { return __byte_perm(a, b, sel); }

// The E4M3 codes of w as two f16 pairs: lo = (byte 0, byte 1), hi = (byte 2,
// byte 3), the first code of each pair in the low half. Exact.
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

template <typename T_, int D_, int BS_>
struct MmaTileE4M3 {
  using T = T_;  // query / output type (f16 or bf16); the cache holds E4M3 codes
  static constexpr int D = D_;
  static constexpr int BS = BS_;
  static constexpr bool FP8 = true;
  static constexpr float UNIT = 1.f;  // K and V enter the MMAs at their code values
  static constexpr int MIN_CTAS = PKV_MMA_FP8_MIN_CTAS;  // resident CTAs per SM the registers must allow
  static_assert(D == 128, "one 128-byte swizzle span per cached row");
  static constexpr int TILE = BS * D;                // bytes of one (block, kv head) tile
  static constexpr int CH = BS >= 16 ? BS / 16 : 1;  // 16-token slices per block
  static constexpr int KT = D / 16;                  // k-steps of the score MMA / m-tiles of PV
  using QB = uint32_t[KT][2];                        // Q^T operand registers
  static_assert(TILE % 1024 == 0, "swizzle atoms need 1024-byte aligned tiles");

  // Byte offset of 16-byte chunk c of row t.
  static __device__ __forceinline__ int off(int t, int c) { return t * 128 + ((c ^ (t & 7)) << 4); }

  // Q^T as the B operand: lane (head g = lane / 4, quad qd) holds, for k-step j,
  // dims 32qd + 4j + {0, 1} (qb[j][0]) and + {2, 3} (qb[j][1]) of head g in
  // f16. sa, sb: sl2 * 2^-k of the lane's columns (heads 2qd, 2qd + 1). Heads
  // >= G are zero.
  static __device__ __forceinline__ void load_qb(QB& qb, const T* q, int G, int lane, float sl2, float& sa,
                                                 float& sb) {
    load_qb_row(qb, (lane >> 2) < G ? q + (lane >> 2) * D : nullptr, lane, sl2, sa, sb);
  }

  // The same operand with column n = lane / 4 taken from the query row `qr`
  // (nullptr: a zero column), each column with its own 2^-k.
  static __device__ __forceinline__ void load_qb_row(QB& qb, const T* qr, int lane, float sl2, float& sa,
                                                     float& sb) {
    const int qd = lane & 3;
    uint32_t w[16];  // qr[32qd .. 32qd + 31] as 16-bit pairs
    if (qr) {
      const uint4* src = reinterpret_cast<const uint4*>(qr + 32 * qd);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint4 v = src[u];
        w[4 * u] = v.x;
        w[4 * u + 1] = v.y;
        w[4 * u + 2] = v.z;
        w[4 * u + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 16; ++e) w[e] = 0u;
    }
    float inv = 1.f;  // 2^-k of column lane / 4
    if constexpr (!std::is_same<T, __half>::value) {
      float amax = 0.f;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float2 v = Elem<T>::to_float2(w[e]);
        amax = fmaxf(amax, fmaxf(fabsf(v.x), fabsf(v.y)));
      }
      amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
      // floor(log2(amax)) from the exponent field; k keeps the scaled maximum in [2^14, 2^15)
      const int ex = static_cast<int>((__float_as_uint(amax) >> 23) & 0xff) - 127;
      int k = amax > 0.f ? 14 - ex : 0;
      k = k < -60 ? -60 : (k > 60 ? 60 : k);
      const float pw = __uint_as_float(static_cast<uint32_t>(127 + k) << 23);
      inv = __uint_as_float(static_cast<uint32_t>(127 - k) << 23);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float2 v = Elem<T>::to_float2(w[e]);
        w[e] = Elem<__half>::pack2(v.x * pw, v.y * pw);
      }
    }
    // w[2j] holds dims 4j, 4j+1 and w[2j+1] dims 4j+2, 4j+3 (relative to 32qd)
#pragma unroll
    for (int j = 0; j < KT; ++j) {
      qb[j][0] = w[2 * j];
      qb[j][1] = w[2 * j + 1];
    }
    sa = sl2 * UNIT * __shfl_sync(kFull, inv, (2 * qd) * 4);
    sb = sl2 * UNIT * __shfl_sync(kFull, inv, (2 * qd + 1) * 4);
  }

  // Fold one (block, kv head) tile into the lane's running state for its two
  // heads (columns 2 (lane % 4) and + 1): tokens 0 .. nvalid-1 take part. acc is
  // in V's code units. CAUSAL: besides, the first column sees only tokens whose
  // position tok_base + t is below lim0 (the second: lim1), so a column may see
  // no token of a tile, or of all tiles so far (its m then stays -inf). Zeroes
  // the value rows past nvalid in shared memory (the stage then needs a proxy
  // fence before the copy engine refills it).
  template <bool CAUSAL = false>
  static __device__ __forceinline__ void run(unsigned char* Ks, unsigned char* Vs, int nvalid, const QB& qb,
                                             int lane, float sla, float slb, float& m0, float& m1, float& l0,
                                             float& l1, float (&acc)[KT][4], int tok_base = 0, int lim0 = 0,
                                             int lim1 = 0) {
    const int g = lane >> 2, qd = lane & 3;
    if (nvalid < BS) {
      // value rows past the context may hold anything (NaN codes too): zero them
      // so that their zero weights contribute exactly zero
      const int nz = (BS - nvalid) * 8;
      for (int idx = lane; idx < nz; idx += 32)
        *reinterpret_cast<uint4*>(Vs + (nvalid + idx / 8) * 128 + (idx % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
      __syncwarp();
    }
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      if (c * 16 < nvalid) {
        // K rows of this lane: c*16 + g and + 8 (with BS = 8 the second aliases the first; masked)
        const int ta = c * 16 + g, tb = BS >= 16 ? ta + 8 : ta;
        const uint4 ka0 = *reinterpret_cast<const uint4*>(Ks + off(ta, 2 * qd));
        const uint4 ka1 = *reinterpret_cast<const uint4*>(Ks + off(ta, 2 * qd + 1));
        const uint4 kb0 = *reinterpret_cast<const uint4*>(Ks + off(tb, 2 * qd));
        const uint4 kb1 = *reinterpret_cast<const uint4*>(Ks + off(tb, 2 * qd + 1));
        const uint32_t wa[8] = {ka0.x, ka0.y, ka0.z, ka0.w, ka1.x, ka1.y, ka1.z, ka1.w};
        const uint32_t wb[8] = {kb0.x, kb0.y, kb0.z, kb0.w, kb1.x, kb1.y, kb1.z, kb1.w};
        float sacc[4] = {0.f, 0.f, 0.f, 0.f}, sacc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < KT; ++j) {
          uint32_t a[4];  // rows g, g + 8 at positions 2qd.. (dims +0, +1) and 2qd+8.. (dims +2, +3)
          e4m3x4_to_f16x2(wa[j], a[0], a[2]);
          e4m3x4_to_f16x2(wb[j], a[1], a[3]);
          if (j & 1) {
            Mma<__half>::run(sacc2, a, qb[j][0], qb[j][1]);
          } else {
            Mma<__half>::run(sacc, a, qb[j][0], qb[j][1]);
          }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[e] += sacc2[e];
        const bool va = ta < nvalid;
        const bool vb = BS >= 16 && ta + 8 < nvalid;
        bool va0 = va, va1 = va, vb0 = vb, vb1 = vb;
        if constexpr (CAUSAL) {
          va0 = va && tok_base + ta < lim0;
          va1 = va && tok_base + ta < lim1;
          vb0 = vb && tok_base + ta + 8 < lim0;
          vb1 = vb && tok_base + ta + 8 < lim1;
        }
        const float x00 = va0 ? sacc[0] * sla : -INFINITY;
        const float x01 = va1 ? sacc[1] * slb : -INFINITY;
        const float x10 = vb0 ? sacc[2] * sla : -INFINITY;
        const float x11 = vb1 ? sacc[3] * slb : -INFINITY;
        // Lazy rescaling: a column's reference m moves (and its state is rescaled)
        // only when a score exceeds it by more than 8, so p = 2^(x - m) <= 2^8. Each
        // lane tests its own scores and the warp votes; the max is reduced across
        // the lanes only when some score does exceed.
        float mx0 = fmaxf(x00, x10), mx1 = fmaxf(x01, x11);
        if (__any_sync(kFull, mx0 > m0 + 8.f || mx1 > m1 + 8.f)) {
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, o));
            mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, o));
          }
          const bool up0 = mx0 > m0 + 8.f, up1 = mx1 > m1 + 8.f;
          const float mn0 = up0 ? mx0 : m0, mn1 = up1 ? mx1 : m1;
          float al0 = fast_exp2(m0 - mn0), al1 = fast_exp2(m1 - mn1);
          if constexpr (CAUSAL) {  // a column that keeps its m may still hold -inf there
            if (!up0) al0 = 1.f;
            if (!up1) al1 = 1.f;
          }
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
        float r0 = m0, r1 = m1;  // exponentials against the reference
        if constexpr (CAUSAL) {  // a column that has seen nothing yet: against 0 (its x are all -inf)
          if (r0 == -INFINITY) r0 = 0.f;
          if (r1 == -INFINITY) r1 = 0.f;
        }
        const uint32_t pa = Elem<__half>::pack2(fast_exp2(x00 - r0), fast_exp2(x01 - r1));
        const uint32_t pb = Elem<__half>::pack2(fast_exp2(x10 - r0), fast_exp2(x11 - r1));
        const float2 fa = Elem<__half>::to_float2(pa), fb = Elem<__half>::to_float2(pb);
        // l: this lane's rows only; finish() adds the lanes of a column
        l0 += fa.x + fb.x;
        l1 += fa.y + fb.y;
        // P^T as the B operand of the PV MMA: transpose the 8x8 score fragments
        const uint32_t b0 = movmatrix_trans(pa), b1 = movmatrix_trans(pb);
        // V: chunk g (dims 16g .. 16g+15) of token rows 2qd, 2qd+1, 2qd+8, 2qd+9
        // (with BS = 8 the last two alias the first two; their weights are zero)
        const int v0 = c * 16 + 2 * qd, v8 = BS >= 16 ? v0 + 8 : v0;
        const uint4 X0 = *reinterpret_cast<const uint4*>(Vs + off(v0, g));
        const uint4 X1 = *reinterpret_cast<const uint4*>(Vs + off(v0 + 1, g));
        const uint4 X8 = *reinterpret_cast<const uint4*>(Vs + off(v8, g));
        const uint4 X9 = *reinterpret_cast<const uint4*>(Vs + off(v8 + 1, g));
        const uint32_t x0[4] = {X0.x, X0.y, X0.z, X0.w}, x1[4] = {X1.x, X1.y, X1.z, X1.w};
        const uint32_t x8[4] = {X8.x, X8.y, X8.z, X8.w}, x9[4] = {X9.x, X9.y, X9.z, X9.w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          // byte b of word w is dim 16g + 4w + b. For the token rows (r, r'):
          // lo = [r.b0, r'.b0, r.b1, r'.b1] and hi = [r.b2, r'.b2, r.b3, r'.b3], so
          // each 16-bit half pairs the two rows at one dim
          const uint32_t lo01 = prmt(x0[w], x1[w], 0x5140), hi01 = prmt(x0[w], x1[w], 0x7362);
          const uint32_t lo89 = prmt(x8[w], x9[w], 0x5140), hi89 = prmt(x8[w], x9[w], 0x7362);
          // m-tile 2w: dims 16g + 4w (row g) and + 1 (row g + 8); m-tile 2w + 1: + 2 and + 3
          uint32_t ae[4], ao[4];
          e4m3x4_to_f16x2(lo01, ae[0], ae[1]);
          e4m3x4_to_f16x2(lo89, ae[2], ae[3]);
          e4m3x4_to_f16x2(hi01, ao[0], ao[1]);
          e4m3x4_to_f16x2(hi89, ao[2], ao[3]);
          Mma<__half>::run(acc[2 * w], ae, b0, b1);
          Mma<__half>::run(acc[2 * w + 1], ao, b0, b1);
        }
      }
    }
  }

  // Complete the running sums: add the per-lane partial sums of each column.
  static __device__ __forceinline__ void finish(float& l0, float& l1) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0 += __shfl_xor_sync(kFull, l0, o);
      l1 += __shfl_xor_sync(kFull, l1, o);
    }
  }

  // The accumulators as red[head][dim]: acc[i] rows g and g + 8 are dims
  // 16g + 2i and 16g + 2i + 1.
  static __device__ __forceinline__ void store_acc(float* red, const float (&acc)[KT][4], int lane) {
    const int g = lane >> 2, j0 = (lane & 3) * 2;
#pragma unroll
    for (int i = 0; i < KT; ++i) {
      const int d = 16 * g + 2 * i;
      *reinterpret_cast<float2*>(red + j0 * D + d) = make_float2(acc[i][0], acc[i][2]);
      *reinterpret_cast<float2*>(red + (j0 + 1) * D + d) = make_float2(acc[i][1], acc[i][3]);
    }
  }

  // Issue the tensor-map copies of one (block, kv head) tile pair into a stage.
  static __device__ __forceinline__ void issue_tiles(unsigned char* st, const CUtensorMap* kmap,
                                                     const CUtensorMap* vmap, int y, uint64_t* bar) {
    tma_load_2d(st, kmap, 0, y, bar);
    tma_load_2d(st + TILE, vmap, 0, y, bar);
  }
};

}  // namespace pkv
