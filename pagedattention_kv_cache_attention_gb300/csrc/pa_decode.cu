// pa_decode.cu -- paged decode attention and the log-sum-exp partition join.
//
// What is computed ("LLM Serving Engine Shootout", 3.1 PagedAttention
// Mechanics): for each sequence i and query head h, the logits
// scale * q . k_j over the sequence's tokens j, with k_j (and v_j) read from
// physical block BlockTable[i][j / block_size], row j % block_size (zhichai.net
// section 1 diagram), a softmax over those logits, and the softmax-weighted
// sum of the v_j.
//
// How (sm_103a):
//  * One CTA per (KV head, sequence, partition).  It serves all G query heads
//    of the KV head, so every K/V tile leaves HBM once per group.
//  * The unit of work is a 16-token sub-tile: 16 consecutive rows of one
//    physical block ([16, head_dim] contiguous in the pool layout
//    [num_blocks, num_kv_heads, block_size, head_dim]).  Warp w of a CTA takes
//    sub-tiles w, w + NW, ... of the partition and owns a private ring of S
//    shared-memory stages
//    (4 warps x 2 stages: 64 KB per CTA, three CTAs per SM).
//    Lane 0 of the warp loads each sub-tile's K and V with 2-D TMA copies
//    (128-byte rows, 128-byte swizzle) through the block table, completion
//    counted on one mbarrier per stage.  The warp's lanes keep the block ids
//    of its next 32 sub-tiles in registers (one per lane), so the table lookup
//    never sits on the issue path.
//  * QK^T is a tensor-core contraction S^T[16 tokens, 8 heads] =
//    K[16, d] Q^T[d, 8] (mma.sync m16n8k16, fp32 accumulate; the query group
//    is padded to 8 heads).  The 16-byte K chunks a lane reads are chosen so
//    that, with the 128-byte swizzle, every quarter-warp hits 32 distinct
//    banks; Q is loaded once into registers in the matching order.
//  * fp32 online softmax on the accumulator fragments (max over tokens by
//    three butterfly shuffles; the running sum stays per thread until the end).
//  * P.V is the second contraction O^T[d, 8] += V^T[d, 16] P^T[16, 8]: P is
//    split into hi + lo parts in the KV dtype (two MMAs, so P keeps ~16 or
//    ~22 bits), each moved into the B-operand layout by an 8x8 transpose
//    (movmatrix); V^T fragments are assembled from 16-byte shared-memory
//    reads with byte permutes.
//  * Warps merge their (m, l, acc) through shared memory at the end.  Without
//    a split the CTA writes the output; with a split it writes the
//    partition's (m, l, normalised o) to the workspace and
//    pa_decode_reduce_kernel joins partitions by log-sum-exp.
//  * Tokens past the context length inside a sub-tile get logit -inf and a
//    zeroed V row, so whatever those slots hold (even NaN) cannot reach the
//    output.
//  * Both kernels are launched as programmatic dependents of the previous
//    kernel in the stream: the decode kernel sets up its barriers while the
//    scatter finishes and waits (griddepcontrol.wait) before its first global
//    read; the join waits for the decode grid, which lets it launch as its
//    last CTAs finish.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>
#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tile.cuh"

namespace pa {

namespace {

// Atomic add with acquire-release semantics at GPU scope; returns the old value.
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned *p, unsigned v) {
  unsigned old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}

// Each partition CTA adds kJoinArrive to its (sequence, KV head) counter: after
// k arrivals both 16-bit halves hold k, so a counter that did not start at zero
// (a workspace whose counter words were not cleared) is recognised.
constexpr unsigned kJoinArrive = 0x00010001u;

// Log-sum-exp join of the np partitions of one (sequence, KV head), run by the
// CTA that finished last: out = sum_p w_p o_p / sum_p w_p, w_p = l_p 2^(m_p - M),
// M = max_p m_p, for the G query heads of the KV head.  Thread items are
// 4-element chunks of one head's output; partitions are taken 8 at a time with
// a running maximum, so every group costs one round trip to L2.  The partials
// were written by other CTAs of this grid: they are read through L2 (ld.cg).
template <typename T, int D, int NW>
__device__ __forceinline__ void join_partitions(const DecodeArgs &a, int seq, int kvh, int np) {
  constexpr int kQuads = D / 4;
  constexpr int kGroup = 8;
  const int G = a.group;
  for (int item = threadIdx.x; item < G * kQuads; item += NW * 32) {
    const int h = item / kQuads, c4 = item % kQuads;
    const int64_t row = static_cast<int64_t>(seq) * a.num_q_heads + kvh * G + h;
    const float *mrow = a.ws_m + row * a.num_parts;
    const float *lrow = a.ws_l + row * a.num_parts;
    const float *orow = a.ws_o + row * a.num_parts * D + c4 * 4;
    float M = -INFINITY, L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p0 = 0; p0 < np; p0 += kGroup) {
      float mp[kGroup], lp[kGroup];
      float4 op[kGroup];
#pragma unroll
      for (int u = 0; u < kGroup; ++u) {
        if (p0 + u < np) {
          mp[u] = __ldcg(mrow + p0 + u);
          lp[u] = __ldcg(lrow + p0 + u);
          op[u] = __ldcg(reinterpret_cast<const float4 *>(orow + static_cast<int64_t>(p0 + u) * D));
        } else {
          mp[u] = -INFINITY;
          lp[u] = 0.f;
          op[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      float Mn = M;
#pragma unroll
      for (int u = 0; u < kGroup; ++u) Mn = fmaxf(Mn, mp[u]);
      const float ref = Mn == -INFINITY ? 0.f : Mn;  // no token yet: any finite reference
      const float al = exp2f(M - ref);
      L *= al;
      acc.x *= al;
      acc.y *= al;
      acc.z *= al;
      acc.w *= al;
#pragma unroll
      for (int u = 0; u < kGroup; ++u) {
        const float wgt = lp[u] * exp2f(mp[u] - ref);
        L += wgt;
        acc.x += wgt * op[u].x;
        acc.y += wgt * op[u].y;
        acc.z += wgt * op[u].z;
        acc.w += wgt * op[u].w;
      }
      M = Mn;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const uint2 pk = make_uint2(Elem<T>::pack(acc.x * inv, acc.y * inv),
                                Elem<T>::pack(acc.z * inv, acc.w * inv));
    *reinterpret_cast<uint2 *>(static_cast<T *>(a.out) + row * D + c4 * 4) = pk;
  }
}

// The same join, by a CTA that holds one partition of the row itself: its
// unnormalised (M, L, o) of output elements 8 ch .. 8 ch + 7 are folded with
// the partials of partitions [0, np) (written by another grid, complete by
// now), and o leaves normalised.
template <int D>
__device__ __forceinline__ void join_into(const DecodeArgs &a, int64_t row, int ch, int np,
                                          float M, float L, float (&o)[8]) {
  constexpr int kGroup = 4;
  const float *mrow = a.ws_m + row * a.num_parts;
  const float *lrow = a.ws_l + row * a.num_parts;
  const float *orow = a.ws_o + row * a.num_parts * D + ch * 8;
  float W = L;  // the own partition's weight; L o_norm = o out_scale
#pragma unroll
  for (int e = 0; e < 8; ++e) o[e] *= a.out_scale;
  for (int p0 = 0; p0 < np; p0 += kGroup) {
    float mp[kGroup], lp[kGroup];
    float4 oa[kGroup], ob[kGroup];
#pragma unroll
    for (int u = 0; u < kGroup; ++u) {
      if (p0 + u < np) {
        mp[u] = __ldcg(mrow + p0 + u);
        lp[u] = __ldcg(lrow + p0 + u);
        const float4 *src =
            reinterpret_cast<const float4 *>(orow + static_cast<int64_t>(p0 + u) * D);
        oa[u] = __ldcg(src);
        ob[u] = __ldcg(src + 1);
      } else {
        mp[u] = -INFINITY;
        lp[u] = 0.f;
        oa[u] = ob[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    float Mn = M;
#pragma unroll
    for (int u = 0; u < kGroup; ++u) Mn = fmaxf(Mn, mp[u]);
    const float ref = Mn == -INFINITY ? 0.f : Mn;  // no token yet: any finite reference
    const float al = exp2f(M - ref);
    W *= al;
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] *= al;
#pragma unroll
    for (int u = 0; u < kGroup; ++u) {
      const float wgt = lp[u] * exp2f(mp[u] - ref);
      W += wgt;
      o[0] += wgt * oa[u].x;
      o[1] += wgt * oa[u].y;
      o[2] += wgt * oa[u].z;
      o[3] += wgt * oa[u].w;
      o[4] += wgt * ob[u].x;
      o[5] += wgt * ob[u].y;
      o[6] += wgt * ob[u].z;
      o[7] += wgt * ob[u].w;
    }
    M = Mn;
  }
  const float inv = W > 0.f ? 1.f / W : 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) o[e] *= inv;
}

// T: query/output type (and the MMA type); F8: the caches hold FP8 E4M3 codes
// (T is then fp16), converted exactly to fp16 in registers.  NSUB: 16-token
// sub-tiles per pipeline step (their MMA chains are independent and share one
// softmax reduction).
// WP ("warp partitions"): each warp takes a whole partition (CTA x serves
// partitions x NW .. x NW + NW - 1 of its sequence and KV head) and writes that
// partition's partial from its own registers, with no merge across warps; used
// when the partitions are joined by the reduce kernel (more of them than the
// in-kernel join takes), so a CTA pays one pipeline ramp and one epilogue for
// NW partitions -- short partitions gain the most.  Otherwise the NW warps
// share one partition.
template <typename T, int D, int NW, int S, bool F8, int NSUB, bool WP>
__global__ void __launch_bounds__(NW * 32)
    pa_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap, const DecodeArgs a) {
  using Sh = Shape<D, F8>;
  static_assert(!F8 || sizeof(T) == 2, "FP8 caches: 16-bit queries");
  // MMA operand type: the query type, except over FP8 caches, whose codes are
  // exact in fp16 (and not all in bf16's exponent range with fp16's
  // precision): there the queries are carried in fp16 (see the q load)
  using MT = typename std::conditional<F8, __half, T>::type;
  // (a step's sub-tiles never straddle a 32-entry block-id window)
  static_assert(NSUB == 1 || NSUB == 2 || NSUB == 4, "1, 2 or 4 sub-tiles per step");
  static_assert(S * NSUB <= 16, "stage bits");
  constexpr int kStepBytes = 2 * NSUB * Sh::kTileBytes;  // K and V of one step
  extern __shared__ uint8_t smem_raw[];
  // 128-byte swizzled TMA destinations need 1024-byte alignment.
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + NW * S * kStepBytes);

  const int kvh = blockIdx.y, seq = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int part = WP ? blockIdx.x * NW + warp : blockIdx.x;
  const int g = lane >> 2, c = lane & 3;

  uint8_t *my_stages = smem + warp * S * kStepBytes;
  uint64_t *my_bars = bars + warp * S;
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < S; ++s) mbar_init(&my_bars[s], 1);
    fence_barrier_init();
  }
  __syncwarp();

  // inputs (the pool above all) may come from the kernel launched just before.
  // After the shared-prefix kernel (launched between the scatter and this
  // grid) the wait moves to the epilogue: that kernel lets this grid start
  // once each of its CTAs has itself waited for the scatter, so the pool is
  // complete here, and only the join needs its partials.
  const bool after_shared_pass = a.prefix_lens != nullptr;
  if (!after_shared_pass) grid_dependency_wait();

  // Step k of warp w covers sub-tiles (w + k NW) NSUB + h, h < NSUB, of the
  // partition (WP: sub-tiles k NSUB + h of the warp's own partition).  A
  // "local" sub-tile index l = k NSUB + h numbers the warp's sub-tiles in
  // order; lane l of a window holds the block id of local sub-tile (window
  // base + l).  The first window is read before the context
  // length arrives (entries past the sequence are read from the table row but
  // never used).
  const int t_begin = part * a.part_tokens;
  const int full_sub = (a.part_tokens + kTile - 1) / kTile;
  const int32_t *bt_row = a.block_tables + static_cast<int64_t>(seq) * a.max_blocks_per_seq;
  const int bs_mask = (1 << a.bs_log2) - 1;
  auto sub_of = [&](int l) {
    return WP ? l : (warp + (l / NSUB) * NW) * NSUB + (l % NSUB);
  };
  auto table_entry = [&](int l) -> int {
    const int u = sub_of(l);
    if (u >= full_sub) return -1;
    const int lb = (t_begin + u * kTile) >> a.bs_log2;
    return lb < a.max_blocks_per_seq ? bt_row[lb] : -1;
  };
  int win = table_entry(lane);

  int ctx = a.context_lens[seq];
  const int prefix_len = a.prefix_lens != nullptr ? a.prefix_lens[seq] : 0;
  if (ctx < 0 || ctx > (a.max_blocks_per_seq << a.bs_log2) || ctx > a.max_context_len) {
    if (threadIdx.x == 0 && part == 0 && kvh == 0) atomicOr(a.err, kErrBadLen);
    ctx = 0;
  }
  if (part > 0 && t_begin >= ctx) return;  // partition past the end: nothing to write
  // partitions of this sequence that have tokens (partition 0 also stands for
  // an empty context)
  const int np_seq = ctx > 0 ? (ctx + a.part_tokens - 1) / a.part_tokens : 1;
  // partitions [0, first) lie inside a prefix the sequence shares with its
  // group, and the shared-prefix kernel has written their partials; the last
  // partition always stays here, so some CTA of this grid joins
  const int first = min(max(prefix_len, 0) / a.part_tokens, np_seq - 1);
  if (part < first) return;
  const int t_end = min(ctx, t_begin + a.part_tokens);
  const int n_sub = t_end > t_begin ? (t_end - t_begin + kTile - 1) / kTile : 0;
  const int n_grp = (n_sub + NSUB - 1) / NSUB;
  // this warp's steps
  const int my_n = WP ? n_grp : (n_grp > warp ? (n_grp - warp + NW - 1) / NW : 0);

  // physical block of local sub-tile l, -1 if past the partition or invalid
  // (an invalid entry is flagged and its tokens are masked)
  auto checked = [&](int l, int phys) -> int {
    if (l >= my_n * NSUB || sub_of(l) >= n_sub) return -1;
    if (phys < 0 || static_cast<int64_t>(phys) >= a.num_blocks) {
      atomicOr(a.err, kErrBadBlock);
      return -1;
    }
    return phys;
  };
  auto sub_token = [&](int l) { return t_begin + sub_of(l) * kTile; };

  const uint64_t policy = l2_policy_evict_first();
  // lane 0: start loading the sub-tiles of step k into stage s
  auto issue = [&](int k, const int (&phys)[NSUB], int s) {
    uint64_t *bar = &my_bars[s];
    uint32_t bytes = 0;
#pragma unroll
    for (int h = 0; h < NSUB; ++h) bytes += phys[h] >= 0 ? 2 * Sh::kTileBytes : 0;
    if (bytes == 0) {
      mbar_arrive(bar);  // nothing to load: complete the phase at once
      return;
    }
    mbar_arrive_expect_tx(bar, bytes);
    uint8_t *st = my_stages + s * kStepBytes;
#pragma unroll
    for (int h = 0; h < NSUB; ++h) {
      if (phys[h] < 0) continue;
      const int tok = sub_token(k * NSUB + h);
      const int y = ((phys[h] * a.num_kv_heads + kvh) << a.bs_log2) + (tok & bs_mask);
#pragma unroll
      for (int b = 0; b < Sh::kBoxes; ++b) {
        tma_load_2d(st + h * Sh::kTileBytes + b * Sh::kBoxBytes, &kmap, b * Sh::kBoxElems, y,
                    bar, policy);
        tma_load_2d(st + (NSUB + h) * Sh::kTileBytes + b * Sh::kBoxBytes, &vmap,
                    b * Sh::kBoxElems, y, bar, policy);
      }
    }
  };

  // block ids of the warp's local sub-tiles [win_base, win_base + 32) and the next 32
  int win_base = 0;
  win = checked(lane, win);
  int win_next = my_n * NSUB > 32 ? checked(32 + lane, table_entry(32 + lane)) : -1;
  uint32_t stage_ok = 0;  // bit s NSUB + h: sub-tile h of the step in stage s is valid
#pragma unroll
  for (int s = 0; s < S; ++s) {
    if (s < my_n) {
      int phys[NSUB];
#pragma unroll
      for (int h = 0; h < NSUB; ++h) {
        phys[h] = __shfl_sync(kFull, win, s * NSUB + h);
        stage_ok |= (phys[h] >= 0 ? 1u : 0u) << (s * NSUB + h);
      }
      if (lane == 0) issue(s, phys, s);
    }
  }

  // query fragments (B operand of S^T = K Q^T) of head g: 16-bit caches use
  // chunks q_chunk(i, c); FP8 caches use 16-dim units 2c + j (two chunks each)
  const int G = a.group;
  uint4 qf[Sh::kQChunks];
  float scale_log2 = a.scale_log2;
  {
    const T *qrow = static_cast<const T *>(a.query) +
                    (static_cast<int64_t>(seq) * a.num_q_heads + kvh * G + g) * D;
#pragma unroll
    for (int i = 0; i < Sh::kQChunks; ++i) {
      // FP8: lane c reads 16-dim units c D/64 + j of each K row (j < D/64)
      const int ch = F8 ? 2 * (c * (D / 64) + (i >> 1)) + (i & 1) : q_chunk(i, c);
      qf[i] = g < G ? *reinterpret_cast<const uint4 *>(qrow + ch * 8) : make_uint4(0, 0, 0, 0);
    }
    if constexpr (F8 && !std::is_same<T, __half>::value) {
      // bf16 queries over FP8 caches: the warp holds all G x D query values;
      // scale them by 2^e so the largest magnitude lands in [2^14, 2^15),
      // then round to fp16 (exact for every value down to 2^-31 of the
      // largest: bf16 carries 8 significant bits, and fp16 holds 8 bits at
      // every magnitude from 2^-17 up), and fold 2^-e into the softmax scale
      float mx = 0.f;
#pragma unroll
      for (int i = 0; i < Sh::kQChunks; ++i)
#pragma unroll
        for (int w2 = 0; w2 < 4; ++w2) {
          const float2 v = Elem<T>::unpack(word_of(qf[i], w2));
          mx = fmaxf(mx, fmaxf(fabsf(v.x), fabsf(v.y)));
        }
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
      const int ex = static_cast<int>((__float_as_uint(mx) >> 23) & 0xffu) - 127;
      const int e = min(120, 14 - ex);
      const float f = ldexpf(1.f, e);
#pragma unroll
      for (int i = 0; i < Sh::kQChunks; ++i) {
        uint32_t w4[4];
#pragma unroll
        for (int w2 = 0; w2 < 4; ++w2) {
          const float2 v = Elem<T>::unpack(word_of(qf[i], w2));
          w4[w2] = Elem<__half>::pack(v.x * f, v.y * f);
        }
        qf[i] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
      scale_log2 = ldexpf(scale_log2, -e);
    }
  }

  const float NEG_INF = -INFINITY;
  float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;  // heads 2c, 2c+1
  float acc[Sh::kMTiles][4];
#pragma unroll
  for (int mt = 0; mt < Sh::kMTiles; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;

  bool timed_out = false;
  int k_stop = my_n;
#pragma unroll 1
  for (int k = 0; k < my_n; ++k) {
    const int s = k % S;
    const uint32_t parity = (k / S) & 1;
    const bool arrived = __all_sync(kFull, mbar_wait_bounded(&my_bars[s], parity));
    if (!arrived) {
      if (lane == 0) atomicOr(a.err, kErrTimeout);
      timed_out = true;
      k_stop = k;
      break;
    }
    const uint8_t *stage = my_stages + s * kStepBytes;
    int nvalid[NSUB];
#pragma unroll
    for (int h = 0; h < NSUB; ++h) {
      const bool ok = (stage_ok >> (s * NSUB + h)) & 1u;
      nvalid[h] = ok ? max(0, min(kTile, t_end - sub_token(k * NSUB + h))) : 0;
    }

    // ---- S^T = K Q^T per sub-tile: rows g and g+8 (tokens), columns 2c, 2c+1 (heads)
    float sc[NSUB][4];
#pragma unroll
    for (int h = 0; h < NSUB; ++h) {
      const uint8_t *Ks = stage + h * Sh::kTileBytes;
      if constexpr (!F8) {
        qk_subtile_16<MT, D>(Ks, qf, g, c, sc[h]);
      } else {
        sc[h][0] = sc[h][1] = sc[h][2] = sc[h][3] = 0.f;
        // unit c D/64 + j of rows g and g+8 holds 16 dims: four k16 steps
        // (rows g and g+8 share their swizzle, so each quarter-warp hits 8
        // distinct 16-byte units of one 128-byte span)
#pragma unroll
        for (int j = 0; j < D / 64; ++j) {
          const int u = c * (D / 64) + j;
          uint32_t ka[8], kb[8];
          e4m3x16_to_half(*reinterpret_cast<const uint4 *>(f8_unit<D>(Ks, g, u)), ka);
          e4m3x16_to_half(*reinterpret_cast<const uint4 *>(f8_unit<D>(Ks, g + 8, u)), kb);
          const uint32_t q[8] = {qf[2 * j].x, qf[2 * j].y, qf[2 * j].z, qf[2 * j].w,
                                 qf[2 * j + 1].x, qf[2 * j + 1].y, qf[2 * j + 1].z,
                                 qf[2 * j + 1].w};
#pragma unroll
          for (int t = 0; t < 4; ++t)
            Elem<MT>::mma(sc[h], ka[2 * t], kb[2 * t], ka[2 * t + 1], kb[2 * t + 1], q[2 * t],
                         q[2 * t + 1]);
        }
      }
    }

    // ---- online softmax in base 2 (log2(e) folded into the scale), one
    // reduction over all NSUB x 16 tokens of the step
    float p[NSUB][4];
    softmax_step<NSUB, Sh::kMTiles>(sc, nvalid, g, scale_log2, m0, m1, l0, l1, acc, p);

#pragma unroll
    for (int h = 0; h < NSUB; ++h) {
      // P^T as the B operand (tokens 2c,2c+1 | 2c+8,2c+9 ; head g), hi + lo
      uint32_t pb0, pb1, pr0, pr1;
      p_operands<MT>(p[h], pb0, pb1, pr0, pr1);
      const uint8_t *Vs = stage + (NSUB + h) * Sh::kTileBytes;

      // ---- O^T += V^T P^T : V rows 2c, 2c+1, 2c+8, 2c+9; unit g of every box
      if constexpr (!F8) {
        pv_subtile_16<MT, D>(Vs, nvalid[h], g, c, pb0, pb1, pr0, pr1, acc);
      } else {
        // MMA row g of m-tile mt is dim dA = pv_dim_a(g, mt), row g+8 is dB:
        // at head_dim 128 the 16 dims 16g .. 16g+15 (unit g of each row), at
        // 64 the 8 dims 8g .. 8g+7 (half g % 2 of unit g / 2); each byte
        // interleave of two rows yields the (token 2c, token 2c+1) pairs of
        // two m-tiles, still E4M3
        constexpr int kHi = D == 128 ? 8 : 4;  // byte of dB within the lane's dims
        uint4 v8[4];
#pragma unroll
        for (int ri = 0; ri < 4; ++ri) {
          const int r = 2 * c + (ri & 1) + 8 * (ri >> 1);
          uint4 xv;
          if constexpr (D == 128) {
            xv = *reinterpret_cast<const uint4 *>(f8_unit<D>(Vs, r, g));
          } else {
            const uint2 half_unit =
                *reinterpret_cast<const uint2 *>(f8_unit<D>(Vs, r, g >> 1) + (g & 1) * 8);
            xv = make_uint4(half_unit.x, half_unit.y, 0u, 0u);
          }
          v8[ri] = r < nvalid[h] ? xv : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int mt = 0; mt < Sh::kMTiles; mt += 2) {
          const uint32_t w0 = interleave_bytes(v8[0], v8[1], mt);
          const uint32_t w1 = interleave_bytes(v8[0], v8[1], kHi + mt);
          const uint32_t w2 = interleave_bytes(v8[2], v8[3], mt);
          const uint32_t w3 = interleave_bytes(v8[2], v8[3], kHi + mt);
          {
            const uint32_t a0 = e4m3x2_lo_to_f16x2(w0), a1 = e4m3x2_lo_to_f16x2(w1);
            const uint32_t a2 = e4m3x2_lo_to_f16x2(w2), a3 = e4m3x2_lo_to_f16x2(w3);
            Elem<MT>::mma(acc[mt], a0, a1, a2, a3, pb0, pb1);
            Elem<MT>::mma(acc[mt], a0, a1, a2, a3, pr0, pr1);
          }
          {
            const uint32_t a0 = e4m3x2_hi_to_f16x2(w0), a1 = e4m3x2_hi_to_f16x2(w1);
            const uint32_t a2 = e4m3x2_hi_to_f16x2(w2), a3 = e4m3x2_hi_to_f16x2(w3);
            Elem<MT>::mma(acc[mt + 1], a0, a1, a2, a3, pb0, pb1);
            Elem<MT>::mma(acc[mt + 1], a0, a1, a2, a3, pr0, pr1);
          }
        }
      }
    }

    // ---- refill this stage with step k + S
    __syncwarp();
    const int nk = k + S;
    if (nk < my_n) {
      if (nk * NSUB >= win_base + 32) {
        win_base += 32;
        win = win_next;
        win_next = checked(win_base + 32 + lane, table_entry(win_base + 32 + lane));
      }
      int phys[NSUB];
#pragma unroll
      for (int h = 0; h < NSUB; ++h) {
        phys[h] = __shfl_sync(kFull, win, nk * NSUB + h - win_base);
        stage_ok = (stage_ok & ~(1u << (s * NSUB + h))) |
                   ((phys[h] >= 0 ? 1u : 0u) << (s * NSUB + h));
      }
      if (lane == 0) {
        fence_proxy_async_smem();
        issue(nk, phys, s);
      }
    }
  }

  if (timed_out) {
    // let copies already in flight land before the CTA leaves (bounded again)
    for (int kk = k_stop; kk < min(k_stop + S, my_n); ++kk)
      (void)mbar_wait_bounded(&my_bars[kk % S], (kk / S) & 1);
  }
  // the shared-prefix grid's partials are complete from here on (and this
  // grid's completion implies that grid's, for the reduce launched after it)
  if (after_shared_pass) grid_dependency_wait();

  // per-warp row sums over the 8 token rows (lanes differing in g)
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(kFull, l0, off);
    l1 += __shfl_xor_sync(kFull, l1, off);
  }

  if constexpr (WP) {
    // the warp's partition is complete: write its (m, l, o) for heads 2c and
    // 2c + 1 straight from the fragments (o normalised, times the V scale)
    const int64_t row0 = static_cast<int64_t>(seq) * a.num_q_heads + kvh * G;
    const int h0 = 2 * c, h1 = 2 * c + 1;
    const float inv0 = l0 > 0.f ? a.out_scale / l0 : 0.f;
    const float inv1 = l1 > 0.f ? a.out_scale / l1 : 0.f;
    const int64_t pr0 = (row0 + h0) * a.num_parts + part, pr1 = (row0 + h1) * a.num_parts + part;
    if (g == 0) {
      if (h0 < G) {
        a.ws_m[pr0] = m0;
        a.ws_l[pr0] = l0;
      }
      if (h1 < G) {
        a.ws_m[pr1] = m1;
        a.ws_l[pr1] = l1;
      }
    }
    store_partial_o<D, F8>(a.ws_o + pr0 * D, a.ws_o + pr1 * D, h0 < G, h1 < G, acc, inv0, inv1,
                           g);
    grid_launch_dependents();
    return;
  }

  // ---- merge warps through shared memory (stages are idle now)
  __syncthreads();
  float *wacc = reinterpret_cast<float *>(smem);  // [NW][8][D]
  float *wml = wacc + NW * 8 * D;                 // [NW][8][2]
  if (g == 0) {
    wml[(warp * 8 + 2 * c) * 2 + 0] = m0;
    wml[(warp * 8 + 2 * c) * 2 + 1] = l0;
    wml[(warp * 8 + 2 * c + 1) * 2 + 0] = m1;
    wml[(warp * 8 + 2 * c + 1) * 2 + 1] = l1;
  }
#pragma unroll
  for (int mt = 0; mt < Sh::kMTiles; ++mt) {
    const int dA = pv_dim_a<D, F8>(g, mt);
    const int dB = pv_dim_b<D, F8>(g, mt);
    float *h0 = wacc + (warp * 8 + 2 * c) * D;
    float *h1 = h0 + D;
    h0[dA] = acc[mt][0];
    h1[dA] = acc[mt][1];
    h0[dB] = acc[mt][2];
    h1[dB] = acc[mt][3];
  }
  __syncthreads();

  // A shared-prefix sequence whose partitions but this one all come from the
  // shared-prefix grid (complete since the wait above): this CTA joins them
  // at once, from its own merge, with no counter and no partial of its own.
  const bool join_here = a.fuse_join && first > 0 && np_seq - first == 1;
  constexpr int kChunks = D / 8;
  for (int item = threadIdx.x; item < G * kChunks; item += NW * 32) {
    const int h = item / kChunks, ch = item % kChunks;
    float M = NEG_INF;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, wml[(w * 8 + h) * 2]);
    float L = 0.f, o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float mw = wml[(w * 8 + h) * 2];
      const float f = mw == NEG_INF ? 0.f : exp2f(mw - M);
      L += wml[(w * 8 + h) * 2 + 1] * f;
      const float *src = wacc + (w * 8 + h) * D + ch * 8;
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] += src[e] * f;
    }
    const int64_t row = static_cast<int64_t>(seq) * a.num_q_heads + kvh * G + h;
    if (join_here) {
      join_into<D>(a, row, ch, first, M, L, o);
    } else {
      const float inv = L > 0.f ? a.out_scale / L : 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] *= inv;
    }
    if (a.num_parts == 1 || (a.fuse_join && np_seq == 1) || join_here) {
      uint4 pk;
      pk.x = Elem<T>::pack(o[0], o[1]);
      pk.y = Elem<T>::pack(o[2], o[3]);
      pk.z = Elem<T>::pack(o[4], o[5]);
      pk.w = Elem<T>::pack(o[6], o[7]);
      *reinterpret_cast<uint4 *>(static_cast<T *>(a.out) + row * D + ch * 8) = pk;
    } else {
      const int64_t pr = row * a.num_parts + part;
      float4 *dst = reinterpret_cast<float4 *>(a.ws_o + pr * D + ch * 8);
      dst[0] = make_float4(o[0], o[1], o[2], o[3]);
      dst[1] = make_float4(o[4], o[5], o[6], o[7]);
      if (ch == 0) {
        a.ws_m[pr] = M;
        a.ws_l[pr] = L;
      }
    }
  }
  if (a.fuse_join && np_seq > 1 && !join_here) {
    // count this partition in; the CTA that completes the count joins them
    // all (with a shared prefix, the partials of partitions below `first`
    // come from the shared-prefix grid, which finished before this one began).  The barrier orders every thread's partial stores before thread 0's
    // acquire-release add, which publishes them (release, cumulative) and, for
    // the last CTA, makes every other CTA's partials visible (acquire).
    __syncthreads();
    uint32_t *last_flag = reinterpret_cast<uint32_t *>(wml + NW * 8 * 2);
    if (threadIdx.x == 0) {
      unsigned *cnt = a.ws_cnt + static_cast<int64_t>(seq) * a.num_kv_heads + kvh;
      const unsigned prev = atom_add_acq_rel_gpu(cnt, kJoinArrive);
      const unsigned k = prev & 0xffffu;
      const unsigned arrivals = static_cast<unsigned>(np_seq - first);  // CTAs that count in
      uint32_t last = 0;
      if ((prev >> 16) != k || k >= arrivals) {
        atomicOr(a.err, kErrWorkspace);  // the counter did not start at zero
      } else if (k == arrivals - 1) {
        last = 1;
        atomicExch(cnt, 0u);  // every partition has arrived: ready for the next call
      }
      *last_flag = last;
    }
    __syncthreads();
    if (*last_flag) join_partitions<T, D, NW>(a, seq, kvh, np_seq);
  }
  grid_launch_dependents();
}

// Log-sum-exp join of partitions when a call has more of them than the decode
// kernel joins itself (and behind the exported pa_decode_reduce).  A CTA of
// four warps serves 4 / WPR output rows (sequence, query head), WPR warps per
// row: warp j of a row takes partitions j, j + WPR, ... with a running
// maximum, sixteen partitions per round trip to memory (each lane holds
// head_dim / 32 output elements of every partition it reads), and the row's
// warps combine their (M, L, acc) through shared memory.  The host picks WPR
// from the partition count: one warp per row when rows hold few partitions
// (fewer, fuller CTAs), four when they hold many (a row of 256 partitions then
// costs four round trips per warp).
constexpr int kReduceWarps = 4;

template <typename T, int D>
__global__ void __launch_bounds__(kReduceWarps * 32) pa_decode_reduce_kernel(const ReduceArgs a) {
  constexpr int kPer = D / 32;  // output elements per lane
  constexpr int kGroup = 16;    // partitions in flight per warp
  __shared__ float s_m[kReduceWarps], s_l[kReduceWarps];
  __shared__ __align__(16) float s_acc[kReduceWarps][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wpr = a.warps_per_row;               // 1, 2 or 4
  const int j = warp % wpr;                      // this warp's place in its row
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (kReduceWarps / wpr) + warp / wpr;
  grid_dependency_wait();  // the partials come from the decode grid
  const bool row_ok = row < static_cast<int64_t>(a.num_seqs) * a.num_q_heads;
  int np = 0;
  if (row_ok) {
    const int seq = static_cast<int>(row / a.num_q_heads);
    int ctx = a.context_lens[seq];
    // the same validity test as the decode kernel, so a length it refused
    // joins no partitions (none of them were written by this call)
    if (ctx < 0 || ctx > a.max_context_len || ctx > a.table_tokens) {
      if (lane == 0 && j == 0 && row % a.num_q_heads == 0) atomicOr(a.err, kErrBadLen);
      ctx = 0;
    }
    np = ctx > 0 ? (ctx + a.partition_size - 1) / a.partition_size : 0;
  }
  const int64_t rr = row_ok ? row : 0;
  const float *m = a.ws_m + rr * a.num_parts;
  const float *l = a.ws_l + rr * a.num_parts;
  const float *o = a.ws_o + rr * a.num_parts * D + lane * kPer;

  float M = -INFINITY, L = 0.f, acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
  for (int p0 = j; p0 < np; p0 += wpr * kGroup) {
    float mp[kGroup], lp[kGroup], op[kGroup][kPer];
#pragma unroll
    for (int u = 0; u < kGroup; ++u) {
      const int p = p0 + u * wpr;
      if (p < np) {
        mp[u] = m[p];
        lp[u] = l[p];
        const float *src = o + static_cast<int64_t>(p) * D;
        if constexpr (kPer == 4) {
          const float4 v = *reinterpret_cast<const float4 *>(src);
          op[u][0] = v.x;
          op[u][1] = v.y;
          op[u][2] = v.z;
          op[u][3] = v.w;
        } else {
          const float2 v = *reinterpret_cast<const float2 *>(src);
          op[u][0] = v.x;
          op[u][1] = v.y;
        }
      } else {
        mp[u] = -INFINITY;
        lp[u] = 0.f;
#pragma unroll
        for (int e = 0; e < kPer; ++e) op[u][e] = 0.f;
      }
    }
    float Mn = M;
#pragma unroll
    for (int u = 0; u < kGroup; ++u) Mn = fmaxf(Mn, mp[u]);
    const float ref = Mn == -INFINITY ? 0.f : Mn;  // no token yet: any finite reference
    const float al = exp2f(M - ref);
    L *= al;
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] *= al;
#pragma unroll
    for (int u = 0; u < kGroup; ++u) {
      const float wgt = lp[u] * exp2f(mp[u] - ref);
      L += wgt;
#pragma unroll
      for (int e = 0; e < kPer; ++e) acc[e] += wgt * op[u][e];
    }
    M = Mn;
  }

  if (lane == 0) {
    s_m[warp] = M;
    s_l[warp] = L;
  }
#pragma unroll
  for (int e = 0; e < kPer; ++e) s_acc[warp][lane * kPer + e] = acc[e];
  __syncthreads();
  if (j == 0 && row_ok) {
    // the row's warps are warp .. warp + wpr - 1
    float Mt = -INFINITY;
    for (int w = warp; w < warp + wpr; ++w) Mt = fmaxf(Mt, s_m[w]);
    const float ref = Mt == -INFINITY ? 0.f : Mt;
    float Lt = 0.f, out[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) out[e] = 0.f;
    for (int w = warp; w < warp + wpr; ++w) {
      const float f = exp2f(s_m[w] - ref);
      Lt += s_l[w] * f;
#pragma unroll
      for (int e = 0; e < kPer; ++e) out[e] += s_acc[w][lane * kPer + e] * f;
    }
    const float inv = Lt > 0.f ? 1.f / Lt : 0.f;
    uint32_t packed[kPer / 2];
#pragma unroll
    for (int e = 0; e < kPer / 2; ++e)
      packed[e] = Elem<T>::pack(out[2 * e] * inv, out[2 * e + 1] * inv);
    T *dst = static_cast<T *>(a.out) + row * D + lane * kPer;
    if constexpr (kPer == 4) {
      *reinterpret_cast<uint2 *>(dst) = make_uint2(packed[0], packed[1]);
    } else {
      *reinterpret_cast<uint32_t *>(dst) = packed[0];
    }
  }
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

// The pool viewed as a 2-D tensor [num_blocks * num_kv_heads * block_size rows,
// head_dim] loaded in boxes of 16 rows x 128 bytes with the 128-byte swizzle
// (rows of 64 bytes -- an FP8 cache at head_dim 64 -- in 64-byte boxes with
// the 64-byte swizzle).
bool encode_pool_map(CUtensorMap *map, const void *pool, int64_t rows, int head_dim, int dtype,
                     bool fp8) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const int elem = fp8 ? 1 : 2;
  const int box_row = head_dim * elem < 128 ? head_dim * elem : 128;  // bytes
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(head_dim) * elem};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_row / elem), static_cast<cuuint32_t>(kTile)};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType ty = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                     : (dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
  CUresult r = enc(map, ty, 2, const_cast<void *>(pool), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE,
                   box_row == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

template <typename T, int D, int NW, int S, bool F8, int NSUB, bool WP>
cudaError_t launch_decode_w(const DecodeArgs &a, const CUtensorMap &km, const CUtensorMap &vm,
                            cudaStream_t stream) {
  using Sh = Shape<D, F8>;
  constexpr size_t step = 2 * NSUB * Sh::kTileBytes;
  constexpr size_t smem = 1024 + static_cast<size_t>(NW) * S * step + NW * S * 8;
  static_assert(static_cast<size_t>(NW) * 8 * D * 4 + NW * 8 * 2 * 4 + 16 <=
                    static_cast<size_t>(NW) * S * step,
                "merge buffers and the join flag must fit in the stage area");
  auto kern = pa_decode_kernel<T, D, NW, S, F8, NSUB, WP>;
  static SmemLimitOnce smem_limit;
  const cudaError_t e = smem_limit.ensure(kern, smem);
  if (e != cudaSuccess) return e;
  const unsigned gx = WP ? static_cast<unsigned>((a.num_parts + NW - 1) / NW)
                         : static_cast<unsigned>(a.num_parts);
  return launch_dependent(kern, dim3(gx, a.num_kv_heads, a.num_seqs), dim3(NW * 32), smem, stream,
                          km, vm, a);
}

// Warp partitions when the partitions are joined by the reduce kernel; one
// partition per CTA otherwise (including the in-kernel join).
template <typename T, int D, int NW, int S, bool F8, int NSUB>
cudaError_t launch_decode_t(const DecodeArgs &a, const CUtensorMap &km, const CUtensorMap &vm,
                            cudaStream_t stream) {
  return a.num_parts > 1 && !a.fuse_join
             ? launch_decode_w<T, D, NW, S, F8, NSUB, true>(a, km, vm, stream)
             : launch_decode_w<T, D, NW, S, F8, NSUB, false>(a, km, vm, stream);
}

template <typename T, int D>
cudaError_t launch_reduce_t(const ReduceArgs &a, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(a.num_seqs) * a.num_q_heads;
  const int rows_per_cta = kReduceWarps / a.warps_per_row;
  return launch_dependent(pa_decode_reduce_kernel<T, D>,
                          dim3(static_cast<unsigned>((rows + rows_per_cta - 1) / rows_per_cta)),
                          dim3(kReduceWarps * 32), 0, stream, a);
}

}  // namespace

// Warps per CTA and TMA stages per warp of the decode kernel.
#ifndef PA_DECODE_WARPS
#define PA_DECODE_WARPS 4
#endif
#ifndef PA_DECODE_STAGES
#define PA_DECODE_STAGES 2
#endif
constexpr int kWarps = PA_DECODE_WARPS;
constexpr int kStages = PA_DECODE_STAGES;

// Sub-tiles per pipeline step.  FP8 tiles carry half the bytes, so two of
// them per step keep the bytes per step, and the per-step latency chain is
// shared by twice the tokens.
#ifndef PA_DECODE_NSUB
#define PA_DECODE_NSUB 1
#endif
#ifndef PA_DECODE_NSUB_F8
#define PA_DECODE_NSUB_F8 2
#endif
#ifndef PA_DECODE_STAGES_F8
#define PA_DECODE_STAGES_F8 2
#endif
// head_dim 64: half the bytes per sub-tile, so more sub-tiles share a step
#ifndef PA_DECODE_NSUB_D64
#define PA_DECODE_NSUB_D64 2
#endif
#ifndef PA_DECODE_NSUB_F8_D64
#define PA_DECODE_NSUB_F8_D64 2
#endif
constexpr int kNsub = PA_DECODE_NSUB;
constexpr int kNsubF8 = PA_DECODE_NSUB_F8;
constexpr int kStagesF8 = PA_DECODE_STAGES_F8;
constexpr int kNsubD64 = PA_DECODE_NSUB_D64;
constexpr int kNsubF8D64 = PA_DECODE_NSUB_F8_D64;

cudaError_t launch_decode(const DecodeArgs &a, const void *k_cache, const void *v_cache,
                          int64_t pool_rows, int head_dim, int dtype, bool kv_fp8,
                          cudaStream_t stream, bool *map_failed) {
  CUtensorMap km, vm;
  *map_failed = false;
  if (!encode_pool_map(&km, k_cache, pool_rows, head_dim, dtype, kv_fp8) ||
      !encode_pool_map(&vm, v_cache, pool_rows, head_dim, dtype, kv_fp8)) {
    *map_failed = true;
    return cudaErrorInvalidValue;
  }
  if (kv_fp8) {
    if (head_dim == 128)
      return dtype == 0
                 ? launch_decode_t<__half, 128, kWarps, kStagesF8, true, kNsubF8>(a, km, vm, stream)
                 : launch_decode_t<__nv_bfloat16, 128, kWarps, kStagesF8, true, kNsubF8>(a, km, vm,
                                                                                         stream);
    return dtype == 0
               ? launch_decode_t<__half, 64, kWarps, kStagesF8, true, kNsubF8D64>(a, km, vm, stream)
               : launch_decode_t<__nv_bfloat16, 64, kWarps, kStagesF8, true, kNsubF8D64>(a, km, vm,
                                                                                         stream);
  }
  if (dtype == 0) {
    return head_dim == 128
               ? launch_decode_t<__half, 128, kWarps, kStages, false, kNsub>(a, km, vm, stream)
               : launch_decode_t<__half, 64, kWarps, kStages, false, kNsubD64>(a, km, vm, stream);
  }
  return head_dim == 128
             ? launch_decode_t<__nv_bfloat16, 128, kWarps, kStages, false, kNsub>(a, km, vm,
                                                                                   stream)
             : launch_decode_t<__nv_bfloat16, 64, kWarps, kStages, false, kNsubD64>(a, km, vm,
                                                                                    stream);
}

cudaError_t launch_reduce(const ReduceArgs &a, int head_dim, int dtype, cudaStream_t stream) {
  if (dtype == 0)
    return head_dim == 128 ? launch_reduce_t<__half, 128>(a, stream)
                           : launch_reduce_t<__half, 64>(a, stream);
  return head_dim == 128 ? launch_reduce_t<__nv_bfloat16, 128>(a, stream)
                         : launch_reduce_t<__nv_bfloat16, 64>(a, stream);
}

}  // namespace pa
