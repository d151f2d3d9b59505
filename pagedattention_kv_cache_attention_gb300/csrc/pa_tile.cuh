// pa_tile.cuh -- the per-sub-tile arithmetic of the paged decode kernel over
// a 16-bit KV cache, and the sub-tile geometry and softmax step it shares with
// the FP8 path.
//
// A sub-tile is 16 consecutive rows of one physical block, K or V, staged in
// shared memory by 2-D TMA copies in 128-byte boxes of 16 rows with the
// 128-byte swizzle: 16-byte unit u of row r sits at unit u ^ (r & 7) of its
// 128-byte line.  Against it a warp computes, for the 8 query columns of its
// MMA tile ("LLM Serving Engine Shootout", 3.1 PagedAttention Mechanics: the
// logits of one query against the gathered keys, then the softmax-weighted
// values):
//   S^T[16 tokens, 8 columns] = K[16, d] Q^T[d, 8]        (qk_subtile)
//   O^T[d, 8] += V^T[d, 16] P^T[16, 8]                     (pv_subtile)
// on mma.sync m16n8k16 with fp32 accumulation.  Fragment ownership: lane
// (g = lane / 4, c = lane % 4) holds S^T rows (tokens) g and g + 8 of columns
// 2c and 2c + 1, and the B operand Q^T of column g.
#pragma once

#include <stdint.h>

#include "pa_device.cuh"

namespace pa {

constexpr int kTile = 16;  // tokens per sub-tile (one MMA row block)
constexpr unsigned kFull = 0xffffffffu;

// Geometry of one sub-tile in shared memory.  Rows of 128 bytes or more are
// staged in 128-byte box rows with the 128-byte swizzle; the 64-byte rows of
// an FP8 cache at head_dim 64 in 64-byte box rows with the 64-byte swizzle
// (16-byte unit u of row r at unit u ^ ((r >> 1) & 3)).
template <int D, bool F8> struct Shape {
  static constexpr int kElem = F8 ? 1 : 2;               // bytes per cached element
  static constexpr int kRowBytes = D * kElem;
  static constexpr int kBoxRow = kRowBytes < 128 ? kRowBytes : 128;  // bytes per box row
  static constexpr int kBoxElems = kBoxRow / kElem;      // elements per box row
  static constexpr int kBoxes = kRowBytes / kBoxRow;     // boxes per row
  static constexpr int kBoxBytes = kTile * kBoxRow;      // one box of 16 rows
  static constexpr int kTileBytes = kTile * kRowBytes;   // K (or V) of one sub-tile
  static constexpr int kQChunks = D / 32;                // 16-byte q chunks per lane
  static constexpr int kMTiles = D / 16;                 // m16 tiles of the P.V product
};

// Address of 16-byte unit u of row r of an FP8 sub-tile (one box per row).
template <int D>
__device__ __forceinline__ const uint8_t *f8_unit(const uint8_t *tile, int r, int u) {
  return D == 128 ? tile + r * 128 + ((u ^ (r & 7)) << 4)
                  : tile + r * 64 + ((u ^ ((r >> 1) & 3)) << 4);
}

// 16-bit caches: the 16-byte chunk (8 elements) of a head_dim row that lane
// column c reads in QK^T step i.  Every chunk is read by exactly one (i, c);
// chunks read by one quarter-warp in one step are all even or all odd, which
// with the swizzle puts them in distinct banks.
__device__ __forceinline__ int q_chunk(int i, int c) { return 2 * c + (i & 1) + 8 * (i >> 1); }

// Output dimensions of P.V m-tile mt held by lane row g: row g of the MMA is
// dimension dA, row g + 8 is dB.
template <int D, bool F8> __device__ __forceinline__ int pv_dim_a(int g, int mt) {
  return F8 && D == 128 ? 16 * g + mt : 8 * g + mt;
}
template <int D, bool F8> __device__ __forceinline__ int pv_dim_b(int g, int mt) {
  return F8 && D == 128 ? 16 * g + 8 + mt : (D == 128 ? 64 + 8 * g + mt : 8 * g + 4 + mt);
}

// S^T = K Q^T for one 16-bit sub-tile: sc[0..1] = tokens g (columns 2c, 2c+1),
// sc[2..3] = tokens g + 8.
template <typename MT, int D>
__device__ __forceinline__ void qk_subtile_16(const uint8_t *Ks, const uint4 (&qf)[D / 32], int g,
                                              int c, float (&sc)[4]) {
  using Sh = Shape<D, false>;
  sc[0] = sc[1] = sc[2] = sc[3] = 0.f;
#pragma unroll
  for (int i = 0; i < Sh::kQChunks; ++i) {
    const int ch = q_chunk(i, c);
    const uint8_t *box = Ks + (ch >> 3) * Sh::kBoxBytes;
    const int sw = ((ch & 7) ^ g) << 4;  // rows g and g+8 share (row & 7) = g
    const uint4 ka = *reinterpret_cast<const uint4 *>(box + g * 128 + sw);
    const uint4 kb = *reinterpret_cast<const uint4 *>(box + (g + 8) * 128 + sw);
    Elem<MT>::mma(sc, ka.x, kb.x, ka.y, kb.y, qf[i].x, qf[i].y);
    Elem<MT>::mma(sc, ka.z, kb.z, ka.w, kb.w, qf[i].z, qf[i].w);
  }
}

// 2^x for the softmax probabilities and rescale factors: the PTX approximate
// base-2 exponential (relative error near 2^-22; results below 2^-126 flush
// to zero, i.e. probabilities that small relative to the running maximum are
// dropped, far below what the fp32 accumulation resolves).  2^-inf = 0.
__device__ __forceinline__ float softmax_exp2(float x) { return ex2_approx(x); }

// One online-softmax step in base 2 (log2(e) is folded into scale_log2) over
// the NSUB sub-tiles of a pipeline step, for the lane's columns 2c (m0, l0)
// and 2c + 1 (m1, l1): tokens at or past nvalid[h] of sub-tile h get logit
// -inf; the running maxima take one butterfly reduction over the step's token
// rows; the accumulator is rescaled only when some maximum grew.  The running
// sums stay per lane (summed over the token rows at the end).  p receives the
// step's probabilities 2^(x - m) in the S^T fragment layout.
template <int NSUB, int MTILES>
__device__ __forceinline__ void softmax_step(const float (&sc)[NSUB][4], const int (&nvalid)[NSUB],
                                             int g, float scale_log2, float &m0, float &m1,
                                             float &l0, float &l1, float (&acc)[MTILES][4],
                                             float (&p)[NSUB][4]) {
  const float NEG_INF = -INFINITY;
  float x[NSUB][4];
  float mx0 = NEG_INF, mx1 = NEG_INF;
#pragma unroll
  for (int h = 0; h < NSUB; ++h) {
    const bool v_lo = g < nvalid[h], v_hi = g + 8 < nvalid[h];
    x[h][0] = v_lo ? sc[h][0] * scale_log2 : NEG_INF;
    x[h][1] = v_lo ? sc[h][1] * scale_log2 : NEG_INF;
    x[h][2] = v_hi ? sc[h][2] * scale_log2 : NEG_INF;
    x[h][3] = v_hi ? sc[h][3] * scale_log2 : NEG_INF;
    mx0 = fmaxf(mx0, fmaxf(x[h][0], x[h][2]));
    mx1 = fmaxf(mx1, fmaxf(x[h][1], x[h][3]));
  }
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, off));
    mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, off));
  }
  const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
  const float r0 = mn0 == NEG_INF ? 0.f : mn0;  // no valid token yet: any finite reference
  const float r1 = mn1 == NEG_INF ? 0.f : mn1;
  const float al0 = softmax_exp2(m0 - r0), al1 = softmax_exp2(m1 - r1);
  float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
  for (int h = 0; h < NSUB; ++h) {
    p[h][0] = softmax_exp2(x[h][0] - r0);
    p[h][1] = softmax_exp2(x[h][1] - r1);
    p[h][2] = softmax_exp2(x[h][2] - r0);
    p[h][3] = softmax_exp2(x[h][3] - r1);
    ps0 += p[h][0] + p[h][2];
    ps1 += p[h][1] + p[h][3];
  }
  l0 = l0 * al0 + ps0;
  l1 = l1 * al1 + ps1;
  m0 = mn0;
  m1 = mn1;
  if (__any_sync(kFull, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
    for (int mt = 0; mt < MTILES; ++mt) {
      acc[mt][0] *= al0;
      acc[mt][1] *= al1;
      acc[mt][2] *= al0;
      acc[mt][3] *= al1;
    }
  }
}

// P^T as the B operand of the P.V product, carried as hi + lo in the MMA type
// (hi = P rounded, lo = the exact fp32 remainder rounded), so the product
// keeps ~16 (bf16) or ~22 (fp16) bits of P instead of 8 or 11.  p[0..3] are
// the probabilities of the lane's S^T fragment; each part is moved from the
// accumulator layout to the B-operand layout by an 8x8 transpose.
template <typename MT>
__device__ __forceinline__ void p_operands(const float (&p)[4], uint32_t &pb0, uint32_t &pb1,
                                           uint32_t &pr0, uint32_t &pr1) {
  const uint32_t h01 = Elem<MT>::pack(p[0], p[1]);
  const uint32_t h23 = Elem<MT>::pack(p[2], p[3]);
  const float2 f01 = Elem<MT>::unpack(h01), f23 = Elem<MT>::unpack(h23);
  pb0 = movmatrix_trans(h01);
  pb1 = movmatrix_trans(h23);
  pr0 = movmatrix_trans(Elem<MT>::pack(p[0] - f01.x, p[1] - f01.y));
  pr1 = movmatrix_trans(Elem<MT>::pack(p[2] - f23.x, p[3] - f23.y));
}

// O^T += V^T P^T for one 16-bit sub-tile.  The lane reads V rows 2c, 2c+1,
// 2c+8, 2c+9 (unit g of every box); rows at or past nvalid are zeroed, so
// whatever those slots hold (even NaN) cannot reach the accumulator.
template <typename MT, int D>
__device__ __forceinline__ void pv_subtile_16(const uint8_t *Vs, int nvalid, int g, int c,
                                              uint32_t pb0, uint32_t pb1, uint32_t pr0,
                                              uint32_t pr1, float (&acc)[D / 16][4]) {
  using Sh = Shape<D, false>;
  uint4 v[4][Sh::kBoxes];
#pragma unroll
  for (int ri = 0; ri < 4; ++ri) {
    const int r = 2 * c + (ri & 1) + 8 * (ri >> 1);
    const bool keep = r < nvalid;
#pragma unroll
    for (int b = 0; b < Sh::kBoxes; ++b) {
      const uint4 xv =
          *reinterpret_cast<const uint4 *>(Vs + b * Sh::kBoxBytes + r * 128 + ((g ^ (r & 7)) << 4));
      v[ri][b] = keep ? xv : make_uint4(0, 0, 0, 0);
    }
  }
#pragma unroll
  for (int mt = 0; mt < Sh::kMTiles; ++mt) {
    // output dim of MMA row g is (box A, element eA) of chunk g; row g+8 is (box B, eB)
    constexpr int bA = 0;
    constexpr int bB = Sh::kBoxes - 1;
    const int eA = mt;
    const int eB = D == 128 ? mt : 4 + mt;
    const uint32_t a0 = pair_of(v[0][bA], v[1][bA], eA);
    const uint32_t a1 = pair_of(v[0][bB], v[1][bB], eB);
    const uint32_t a2 = pair_of(v[2][bA], v[3][bA], eA);
    const uint32_t a3 = pair_of(v[2][bB], v[3][bB], eB);
    Elem<MT>::mma(acc[mt], a0, a1, a2, a3, pb0, pb1);
    Elem<MT>::mma(acc[mt], a0, a1, a2, a3, pr0, pr1);
  }
}

// Writes the lane's share of a finished partial, columns 2c (o0, ok0) and
// 2c + 1 (o1, ok1): o[d] = acc * inv from the P.V fragments.
template <int D, bool F8>
__device__ __forceinline__ void store_partial_o(float *o0, float *o1, bool ok0, bool ok1,
                                                const float (&acc)[D / 16][4], float inv0,
                                                float inv1, int g) {
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) {
    const int dA = pv_dim_a<D, F8>(g, mt);
    const int dB = pv_dim_b<D, F8>(g, mt);
    if (ok0) {
      o0[dA] = acc[mt][0] * inv0;
      o0[dB] = acc[mt][2] * inv0;
    }
    if (ok1) {
      o1[dA] = acc[mt][1] * inv1;
      o1[dB] = acc[mt][3] * inv1;
    }
  }
}

}  // namespace pa
