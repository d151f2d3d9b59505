// pa_prefix.cu -- decode attention over the shared prefix of groups of
// sequences whose block tables point at the same physical blocks.
//
// Copy-on-write block sharing ("LLM Serving Engine Shootout", 3.2 Copy-on-Write
// and 4 RadixAttention; "Serving engines", How vLLM works) lets many sequences
// reference one copy of a prefix's K/V.  The plain decode kernel still reads
// those blocks once per sequence (the L2 serves the repeats when it can hold
// them).  Here each K/V sub-tile of a group's prefix leaves memory once per
// group: one CTA serves 16 query columns -- (member sequence, query head)
// pairs of one KV head -- so every staged tile feeds 16 query rows at once
// (a group with more columns takes several CTAs, which read the same tiles
// through the L2 at about the same time).
//
// Work split with the decode kernel.  The prefix is cut at the decode's own
// partition boundaries (partition p = tokens [p P, (p+1) P), P the partition
// size).  For member m with context ctx_m (np_m partitions) and shared prefix
// length L_m, the partitions p < first_m = min(floor(L_m / P), np_m - 1) are
// computed here and written as split partials (m, l, o) into the decode
// workspace; the decode kernel then computes partitions first_m .. np_m - 1 of
// the sequence and joins them all by log-sum-exp exactly as for a plain split.
// Every partition computed here lies wholly inside the contexts of the
// members it is written for, so no per-column token mask is needed.
//
// CTA (partition p x chunk of a group, KV head, group): four warps
// over 16 query columns (column = member * G + query head).  The arithmetic is
// the plain orientation S[columns, tokens] = Q K^T, O += P V on mma.sync
// m16n8k16 (fp32 accumulate): every warp holds the 16 rows and takes every
// fourth 16-token sub-tile of the partition.  K and V^T fragments come straight from the
// swizzled tiles by ldmatrix (V transposed in the load), and the softmax's P
// feeds the P.V product from the S accumulators without a transpose (the
// accumulator layout of two 8-token n-tiles is the A layout of one k16 step),
// split into hi + lo parts as in the decode kernel.  The four token quarters
// are merged by log-sum-exp at the end.  Each warp streams its own sub-tiles
// (warp w: w, w + 4, ...) through a private ring of two shared-memory stages
// loaded by 2-D TMA copies, so no warp waits for another.  The partition's
// block ids come from the table of the first member that takes the partition
// from here, once, into shared memory; the other members' entries must be the
// same blocks (checked, PA_DEVERR_PREFIX otherwise).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tile.cuh"

namespace pa {

namespace {

constexpr int kPxWarps = 4;                                // token quarters of one row tile
constexpr int kPxRows = 16;                                // query rows (columns) per CTA
#ifndef PA_PREFIX_STAGES
#define PA_PREFIX_STAGES 2
#endif
constexpr int kPxStages = PA_PREFIX_STAGES;                // ring stages per warp
constexpr int kPxMaxSub = kMaxSharedPrefixPartition / kTile;  // sub-tiles per partition

// L2 policy for prefix tiles that another CTA of the launch reads again (a
// group split over several chunks).
__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

template <typename T, int D>
__global__ void __launch_bounds__(kPxWarps * 32)
    pa_shared_prefix_kernel(const __grid_constant__ CUtensorMap kmap,
                            const __grid_constant__ CUtensorMap vmap, const DecodeArgs a) {
  using Sh = Shape<D, false>;
  constexpr int NW = kPxWarps, S = kPxStages;
  constexpr int kStepBytes = 2 * Sh::kTileBytes;  // K and V of one sub-tile
  extern __shared__ uint8_t smem_raw[];
  // 128-byte swizzled TMA destinations need 1024-byte alignment.
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + NW * S * kStepBytes);  // [NW][S]
  int *row_of = reinterpret_cast<int *>(bars + NW * S);  // [kPxMaxSub] pool row, -1 = skip
  int *first_of = row_of + kPxMaxSub;  // [32] first_m of each member of this CTA
  int *ctl = first_of + 32;  // source member, member count, first member, timeout, bad id

  // the chunks of one (partition, KV head, group) run back to back, so the
  // tiles they share are still in the L2 for the second
  const int p = blockIdx.x / a.chunks, chunk = blockIdx.x % a.chunks;
  const int kvh = blockIdx.y, grp = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int G = a.group, P = a.part_tokens;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < NW * S; ++s) mbar_init(&bars[s], 1);
    ctl[3] = 0;
    ctl[4] = 0;
    fence_barrier_init();
  }

  // tables, lengths and the pool may come from the kernel launched just before
  grid_dependency_wait();
  // the decode grid that follows may start now: it streams the sequences'
  // own partitions while this grid runs, and waits for this grid's partials
  // only before it joins them
  grid_launch_dependents();

  // ---- this CTA's members and the partitions they take from here (warp 0,
  // one member per lane)
  if (warp == 0) {
    const int g0 = a.group_start[grp], g1 = a.group_start[grp + 1];
    const bool group_ok = g0 >= 0 && g1 >= g0 && g1 <= a.num_seqs &&
                          g1 - g0 <= a.max_group_size && (grp > 0 || g0 == 0) &&
                          (grp < a.num_groups - 1 || g1 == a.num_seqs);
    const bool reporter = p == 0 && kvh == 0;  // one CTA per chunk reports bad input
    if (!group_ok && reporter && chunk == 0 && lane == 0) atomicOr(a.err, kErrPrefix);
    const int m0 = g0 + chunk * a.members_per_cta;
    const int nm = group_ok ? max(0, min(a.members_per_cta, g1 - m0)) : 0;
    int first = 0;
    if (lane < nm) {
      const int seq = m0 + lane;
      int ctx = a.context_lens[seq];
      // the decode kernel flags a bad length; here it only means "nothing shared"
      if (ctx < 0 || ctx > (a.max_blocks_per_seq << a.bs_log2) || ctx > a.max_context_len)
        ctx = 0;
      const int np = ctx > 0 ? (ctx + P - 1) / P : 1;
      const int pl = a.prefix_lens[seq];
      if (pl != a.prefix_lens[g0] && reporter) atomicOr(a.err, kErrPrefix);
      first = min(max(pl, 0) / P, np - 1);
    }
    first_of[lane] = first;
    const unsigned takers = __ballot_sync(kFull, lane < nm && p < first);
    if (lane == 0) {
      ctl[0] = takers ? __ffs(takers) - 1 : -1;
      ctl[1] = nm;
      ctl[2] = m0;
    }
  }
  // the partition's sub-tiles as pool rows, read (speculatively, by warp 1,
  // while warp 0 finds the members) from the table of the chunk's first
  // member, which is the source whenever that member takes the partition
  const int n_sub = P / kTile;
  const int t0 = p * P;
  const int bs_mask = (1 << a.bs_log2) - 1;
  auto load_rows = [&](const int32_t *row, int u0, int du) -> bool {
    bool bad = false;
    for (int u = u0; u < n_sub; u += du) {
      const int t = t0 + u * kTile;
      const int lb = t >> a.bs_log2;
      const int phys = lb < a.max_blocks_per_seq ? row[lb] : -1;
      int r = -1;
      if (phys >= 0 && static_cast<int64_t>(phys) < a.num_blocks)
        r = ((phys * a.num_kv_heads + kvh) << a.bs_log2) + (t & bs_mask);
      else
        bad = true;
      row_of[u] = r;
    }
    return bad;
  };
  if (warp == 1) {
    const int m0s = a.group_start[grp] + chunk * a.members_per_cta;
    if (m0s >= 0 && m0s < a.num_seqs &&
        load_rows(a.block_tables + static_cast<int64_t>(m0s) * a.max_blocks_per_seq, lane, 32))
      atomicOr(&ctl[4], 1);
  }
  __syncthreads();
  const int src = ctl[0];
  if (src < 0) return;  // no member takes this partition from here (uniform)
  const int nm = ctl[1], m0 = ctl[2];
  // p < first_src <= np_src - 1: the partition ends inside the source's
  // context, so every table entry it needs is inside the source's row
  const int32_t *src_row =
      a.block_tables + static_cast<int64_t>(m0 + src) * a.max_blocks_per_seq;
  if (src != 0) {
    const bool bad = load_rows(src_row, threadIdx.x, NW * 32);
    __syncthreads();
    if (bad) atomicOr(a.err, kErrBadBlock);
  } else if (ctl[4] && threadIdx.x == 0) {
    atomicOr(a.err, kErrBadBlock);
  }

  const uint64_t policy = a.chunks > 1 ? l2_policy_evict_normal() : l2_policy_evict_first();
  // each warp streams its own sub-tiles (th, th + NW, ...) through a private
  // ring of S stages: lane 0 loads local sub-tile k into stage k % S
  const int th = warp;
  uint8_t *my_stages = smem + warp * S * kStepBytes;
  uint64_t *my_bars = bars + warp * S;
  const int my_n = n_sub > th ? (n_sub - th + NW - 1) / NW : 0;
  auto issue = [&](int k) {
    const int s = k % S;
    const int r = row_of[th + k * NW];
    if (r < 0) {
      mbar_arrive(&my_bars[s]);  // nothing to load: complete the phase at once
      return;
    }
    mbar_arrive_expect_tx(&my_bars[s], 2 * Sh::kTileBytes);
    uint8_t *st = my_stages + s * kStepBytes;
#pragma unroll
    for (int b = 0; b < Sh::kBoxes; ++b) {
      tma_load_2d(st + b * Sh::kBoxBytes, &kmap, b * Sh::kBoxElems, r, &my_bars[s], policy);
      tma_load_2d(st + Sh::kTileBytes + b * Sh::kBoxBytes, &vmap, b * Sh::kBoxElems, r,
                  &my_bars[s], policy);
    }
  };
  if (lane == 0) {
    for (int k = 0; k < S && k < my_n; ++k) issue(k);
  }
  // every other taker must reference the same blocks (checked once per
  // partition, while the first stages load; it only sets a flag)
  if (kvh == 0) {
    const int lb0 = t0 >> a.bs_log2;
    const int nlb = ((t0 + P - 1) >> a.bs_log2) - lb0 + 1;
    for (int it = threadIdx.x; it < nm * nlb; it += NW * 32) {
      const int i = it / nlb, lb = lb0 + it % nlb;
      if (i != src && p < first_of[i] &&
          a.block_tables[static_cast<int64_t>(m0 + i) * a.max_blocks_per_seq + lb] != src_row[lb])
        atomicOr(a.err, kErrPrefix);
    }
  }

  // ---- every warp holds the CTA's 16 query rows (MMA rows g and g + 8 are
  // columns g and g + 8)
  const int colA = g, colB = g + 8;
  const int iA = colA / G, iB = colB / G;         // their members
  // Q as the A operand: qa[ks] holds rows g, g+8 and dims 16 ks + 2c (+1),
  // 16 ks + 8 + 2c (+1); zero for padding columns
  uint32_t qa[D / 16][4];
  {
    const T *qA = iA < nm ? static_cast<const T *>(a.query) +
                                (static_cast<int64_t>(m0 + iA) * a.num_q_heads + kvh * G +
                                 colA % G) * D
                          : nullptr;
    const T *qB = iB < nm ? static_cast<const T *>(a.query) +
                                (static_cast<int64_t>(m0 + iB) * a.num_q_heads + kvh * G +
                                 colB % G) * D
                          : nullptr;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const int d0 = 16 * ks + 2 * c;
      qa[ks][0] = qA ? *reinterpret_cast<const uint32_t *>(qA + d0) : 0u;
      qa[ks][1] = qB ? *reinterpret_cast<const uint32_t *>(qB + d0) : 0u;
      qa[ks][2] = qA ? *reinterpret_cast<const uint32_t *>(qA + d0 + 8) : 0u;
      qa[ks][3] = qB ? *reinterpret_cast<const uint32_t *>(qB + d0 + 8) : 0u;
    }
  }
  // ldmatrix row of this lane: matrix mi = lane / 8, row r8 = lane % 8
  const int mi = lane >> 3, r8 = lane & 7;
  // K (B operand of S = Q K^T, non-transposed): matrices (tokens 0-7 | 8-15) x
  // (16-byte chunk 2 ks | 2 ks + 1) give b0, b1 of token n-tiles 0 and 1
  const int k_tok = r8 + 8 * (mi >> 1), k_chunk = mi & 1;
  // V (B operand of O += P V, transposed): matrices (tokens 0-7 | 8-15) x
  // (dims 16 j .. +7 | 16 j + 8 .. +15) give b0, b1 of dim n-tiles 2j, 2j+1
  const int v_tok = r8 + 8 * (mi & 1), v_chunk = mi >> 1;
  auto row_addr = [&](const uint8_t *tile, int tok, int chunk) {
    return tile + (chunk >> 3) * Sh::kBoxBytes + tok * 128 + (((chunk & 7) ^ (tok & 7)) << 4);
  };

  float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
  float acc[D / 8][4];  // O rows g, g+8; dims 8 nt + 2c (+1)
#pragma unroll
  for (int nt = 0; nt < D / 8; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;

  bool timed_out = false;
  int k_stop = my_n;
#pragma unroll 1
  for (int k = 0; k < my_n; ++k) {
    const int s = k % S;
    if (!__all_sync(kFull, mbar_wait_bounded(&my_bars[s], (k / S) & 1))) {
      if (lane == 0) atomicOr(a.err, kErrTimeout);
      timed_out = true;
      k_stop = k;
      break;
    }
    // partitions here hold only whole sub-tiles inside every taker's
    // context; a sub-tile whose block id was refused was not loaded at all
    if (row_of[th + k * NW] >= 0) {
      const uint8_t *Ks = my_stages + s * kStepBytes;
      const uint8_t *Vs = Ks + Sh::kTileBytes;
      // ---- S[16 rows, 16 tokens] = Q K^T (token n-tiles 0 and 1)
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t b[4];
        ldmatrix_x4(b, row_addr(Ks, k_tok, 2 * ks + k_chunk));
        Elem<T>::mma(sc[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b[0], b[1]);
        Elem<T>::mma(sc[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b[2], b[3]);
      }
      // ---- online softmax in base 2 over the 16 tokens of rows g and g+8
      float x[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) x[j][e] = sc[j][e] * a.scale_log2;
      float mxA = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
      float mxB = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
#pragma unroll
      for (int off = 1; off < 4; off <<= 1) {
        mxA = fmaxf(mxA, __shfl_xor_sync(kFull, mxA, off));
        mxB = fmaxf(mxB, __shfl_xor_sync(kFull, mxB, off));
      }
      const float nA = fmaxf(mA, mxA), nB = fmaxf(mB, mxB);
      const float rA = nA == -INFINITY ? 0.f : nA;  // any finite reference
      const float rB = nB == -INFINITY ? 0.f : nB;
      const float alA = softmax_exp2(mA - rA), alB = softmax_exp2(mB - rB);
      float pr[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        pr[j][0] = softmax_exp2(x[j][0] - rA);
        pr[j][1] = softmax_exp2(x[j][1] - rA);
        pr[j][2] = softmax_exp2(x[j][2] - rB);
        pr[j][3] = softmax_exp2(x[j][3] - rB);
      }
      lA = lA * alA + (pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1]);
      lB = lB * alB + (pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3]);
      mA = nA;
      mB = nB;
      if (__any_sync(kFull, alA != 1.f || alB != 1.f)) {
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt) {
          acc[nt][0] *= alA;
          acc[nt][1] *= alA;
          acc[nt][2] *= alB;
          acc[nt][3] *= alB;
        }
      }
      // ---- P as the A operand straight from the S fragments, hi + lo
      uint32_t ph[4], pl[4];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const float p0 = pr[j][2 * r], p1 = pr[j][2 * r + 1];
          const uint32_t h = Elem<T>::pack(p0, p1);
          const float2 f = Elem<T>::unpack(h);
          ph[2 * j + r] = h;
          pl[2 * j + r] = Elem<T>::pack(p0 - f.x, p1 - f.y);
        }
      }
      // ---- O[16 rows, d] += P V (dim n-tiles 2j, 2j+1 per transposed load)
#pragma unroll
      for (int j = 0; j < D / 16; ++j) {
        uint32_t b[4];
        ldmatrix_x4_trans(b, row_addr(Vs, v_tok, 2 * j + v_chunk));
        Elem<T>::mma(acc[2 * j], ph[0], ph[1], ph[2], ph[3], b[0], b[1]);
        Elem<T>::mma(acc[2 * j], pl[0], pl[1], pl[2], pl[3], b[0], b[1]);
        Elem<T>::mma(acc[2 * j + 1], ph[0], ph[1], ph[2], ph[3], b[2], b[3]);
        Elem<T>::mma(acc[2 * j + 1], pl[0], pl[1], pl[2], pl[3], b[2], b[3]);
      }
    }

    // refill this stage with the warp's sub-tile k + S
    __syncwarp();
    if (lane == 0 && k + S < my_n) {
      fence_proxy_async_smem();
      issue(k + S);
    }
  }

  // ---- row sums over the quad, then the four token quarters are merged by
  // log-sum-exp (warps 1-3 hand their state to warp 0 through the idle stage
  // area, lane for lane: all four hold the same rows and dims)
#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    lA += __shfl_xor_sync(kFull, lA, off);
    lB += __shfl_xor_sync(kFull, lB, off);
  }
  if (timed_out) {
    // a wait ran out: let this warp's copies already in flight land before
    // the CTA leaves (bounded again); the partition's partials are not written
    for (int kk = k_stop; kk < min(k_stop + S, my_n); ++kk)
      (void)mbar_wait_bounded(&my_bars[kk % S], (kk / S) & 1);
    if (lane == 0) atomicOr(&ctl[3], 1);
  }
  __syncthreads();
  if (ctl[3]) return;
  constexpr int kMerge = D / 2 + 4;  // floats per lane: acc, then mA, mB, lA, lB
  float *xchg = reinterpret_cast<float *>(smem) + lane;  // [warp - 1][i][lane]
  if (warp > 0) {
    float *x = xchg + (warp - 1) * kMerge * 32;
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) x[(4 * nt + e) * 32] = acc[nt][e];
    x[(D / 2 + 0) * 32] = mA;
    x[(D / 2 + 1) * 32] = mB;
    x[(D / 2 + 2) * 32] = lA;
    x[(D / 2 + 3) * 32] = lB;
  }
  __syncthreads();
  if (warp == 0) {
    float MA = mA, MB = mB;
#pragma unroll
    for (int w = 0; w < NW - 1; ++w) {
      MA = fmaxf(MA, xchg[(w * kMerge + D / 2 + 0) * 32]);
      MB = fmaxf(MB, xchg[(w * kMerge + D / 2 + 1) * 32]);
    }
    const float refA = MA == -INFINITY ? 0.f : MA, refB = MB == -INFINITY ? 0.f : MB;
    float fA[NW], fB[NW];
    fA[0] = exp2f(mA - refA);
    fB[0] = exp2f(mB - refB);
    float LA = lA * fA[0], LB = lB * fB[0];
#pragma unroll
    for (int w = 1; w < NW; ++w) {
      const float *x = xchg + (w - 1) * kMerge * 32;
      fA[w] = exp2f(x[(D / 2 + 0) * 32] - refA);
      fB[w] = exp2f(x[(D / 2 + 1) * 32] - refB);
      LA += x[(D / 2 + 2) * 32] * fA[w];
      LB += x[(D / 2 + 3) * 32] * fB[w];
    }
    const float invA = LA > 0.f ? 1.f / LA : 0.f, invB = LB > 0.f ? 1.f / LB : 0.f;
    const bool okA = iA < nm && p < first_of[iA];
    const bool okB = iB < nm && p < first_of[iB];
    const int64_t prA =
        (static_cast<int64_t>(m0 + iA) * a.num_q_heads + kvh * G + colA % G) * a.num_parts + p;
    const int64_t prB =
        (static_cast<int64_t>(m0 + iB) * a.num_q_heads + kvh * G + colB % G) * a.num_parts + p;
    if (c == 0) {
      if (okA) {
        a.ws_m[prA] = MA;
        a.ws_l[prA] = LA;
      }
      if (okB) {
        a.ws_m[prB] = MB;
        a.ws_l[prB] = LB;
      }
    }
    float *oA = okA ? a.ws_o + prA * D : nullptr;
    float *oB = okB ? a.ws_o + prB * D : nullptr;
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      float o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        o[e] = acc[nt][e] * (e < 2 ? fA[0] : fB[0]);
#pragma unroll
        for (int w = 1; w < NW; ++w)
          o[e] += xchg[((w - 1) * kMerge + 4 * nt + e) * 32] * (e < 2 ? fA[w] : fB[w]);
      }
      const int dd = 8 * nt + 2 * c;
      if (okA) *reinterpret_cast<float2 *>(oA + dd) = make_float2(o[0] * invA, o[1] * invA);
      if (okB) *reinterpret_cast<float2 *>(oB + dd) = make_float2(o[2] * invB, o[3] * invB);
    }
  }
}

template <typename T, int D>
cudaError_t launch_prefix_t(const DecodeArgs &a, const CUtensorMap &km, const CUtensorMap &vm,
                            cudaStream_t stream) {
  constexpr size_t step = 2 * Shape<D, false>::kTileBytes;
  constexpr size_t smem =
      1024 + kPxWarps * kPxStages * (step + 8) + (kPxMaxSub + 32 + 8) * 4;
  auto kern = pa_shared_prefix_kernel<T, D>;
  static SmemLimitOnce smem_limit;
  const cudaError_t e = smem_limit.ensure(kern, smem);
  if (e != cudaSuccess) return e;
  return launch_dependent(
      kern,
      dim3(static_cast<unsigned>(a.num_parts * a.chunks), static_cast<unsigned>(a.num_kv_heads),
           static_cast<unsigned>(a.num_groups)),
      dim3(kPxWarps * 32), smem, stream, km, vm, a);
}

}  // namespace

int shared_prefix_members_per_cta(int group) { return kPxRows / group; }

cudaError_t launch_shared_prefix(const DecodeArgs &a, const void *k_cache, const void *v_cache,
                                 int64_t pool_rows, int head_dim, int dtype, cudaStream_t stream,
                                 bool *map_failed) {
  CUtensorMap km, vm;
  *map_failed = false;
  if (!encode_pool_map(&km, k_cache, pool_rows, head_dim, dtype, false) ||
      !encode_pool_map(&vm, v_cache, pool_rows, head_dim, dtype, false)) {
    *map_failed = true;
    return cudaErrorInvalidValue;
  }
  if (dtype == 0)
    return head_dim == 128 ? launch_prefix_t<__half, 128>(a, km, vm, stream)
                           : launch_prefix_t<__half, 64>(a, km, vm, stream);
  return head_dim == 128 ? launch_prefix_t<__nv_bfloat16, 128>(a, km, vm, stream)
                         : launch_prefix_t<__nv_bfloat16, 64>(a, km, vm, stream);
}

}  // namespace pa
