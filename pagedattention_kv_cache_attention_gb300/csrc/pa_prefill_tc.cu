// pa_prefill_tc.cu -- chunked-prefill attention on the fifth-generation tensor
// core (tcgen05: accumulators and P in tensor memory, operands staged by TMA).
//
// Chunked prefill ("Serving engines", How vLLM works: chunked prefill; chunk
// row t at position ctx - q_len + t attends causally to tokens 0..t's position
// through the block table), for head_dim 64 or 128 and every query group G
// from 1 to 8.  One kernel template, two shapes: two 128-row query tiles per
// CTA (one CTA per SM) for chunks longer than 128/G tokens, one tile per CTA
// (two CTAs per SM) for shorter ones.  The design and the measurements that
// shaped it are described above the kernel.
//
// The same kernel, with its shared-prefix flag, is the shared pass of
// pa_decode_shared_prefix: a tile's rows are then the (sequence, query head)
// pairs of the members of a group of sequences that share a prefix in the same
// physical blocks ("LLM Serving Engine Shootout", 3.2 Copy-on-Write), its keys
// one partition of that prefix with no causal limit, and its rows leave split
// partials (m, l, o) in the decode workspace for the decode kernel to join.

#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kTcRows = 128;     // query rows per tile = TMEM lanes
constexpr float kRescaleLog2 = 8.f;         // move the running max only past this growth
constexpr unsigned kFullMask = 0xffffffffu;

// D (TMEM) [+]= A (TMEM, K-major: lane = row, column c = elements 2c, 2c+1) * B (smem)
__device__ __forceinline__ void umma_f16_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t b_desc,
                                            uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1 : 0)
      : "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// Packed fp32 pairs (sm_100 and later): two IEEE fp32 operations per instruction,
// each rounded exactly as the scalar one.
// Non-blocking look at an mbarrier phase (acquire, CTA scope): true once the
// phase with the given parity has completed.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// ---------------------------------------------------------------------------
// Query tiles per CTA, 64-key steps, scores and P in separate TMEM columns.
//
// A CTA holds TILES (1 or 2) 128-row tiles of the same (sequence, KV head) --
// rows r = token (r / G) x head (r % G) of floor(128 TILES / G) tokens; when G
// does not divide 128 a token's heads may straddle the two tiles and the last
// 128 TILES mod G rows stay idle -- and streams 64-key K/V steps through two
// rings shared by its tiles (K and V apart, so a K stage is refilled as soon
// as the Q K^T products that read it are done).  Each tile owns 256 TMEM
// columns: scores (64, fp32), P (64: two 32-column fp16 buffers, or one bf16
// buffer of hi + lo parts) and O (head_dim, 64 or 128).  Two tiles take all
// 512 columns and one CTA per SM; one tile takes 256 and two CTAs share an SM.
// Q, K and V are staged as 64-dimension atoms of 128-byte rows (one atom at
// head_dim 64, two at 128).
// The softmax warps release the score columns as soon as they have loaded
// them, so Q K^T of step n + 1 runs while they work on step n, and P V of step
// n runs while they work on step n + 1.  Q is read from shared memory (one
// 32 KB tile per query tile).
//
// Warp roles (two tiles): warps 0-3 softmax for tile 0, 4-7 for tile 1
// (thread r of a tile owns its row r and TMEM lane r), warps 8-11 issue the
// MMAs (Q K^T of tile 0, P V of tile 0, Q K^T of tile 1, P V of tile 1),
// warps 12 and 13 load K and V; one tile has the same roles in warps 0-7.
// One thread issuing tcgen05.mma back to back gets about one instruction per
// 120 cycles whatever N is, and a warp issuing a step's TMA copies takes about
// as long as the step's softmax (measured on GB300), so every stream has its
// own warp.  V rows a product must not use (past the keys in use, or in a
// sub-tile whose block id is out of range) are zeroed by the V loader before
// the stage is handed over; the softmax warps mask those keys.
constexpr int kPairKeys = 64;                  // keys per step
constexpr int kPairQAtom = kTcRows * 128;      // one 64-dim atom of a Q tile (bytes)
constexpr int kPairKvAtom = kPairKeys * 128;   // one 64-dim atom of a K or V stage (bytes)

// TILES query tiles per CTA: softmax warps 0 .. 4 TILES - 1, issuing warps
// 4 TILES .. 6 TILES - 1 (Q K^T and P V of each tile), then the K and V warps.
// Over FP8 caches at head_dim 128 the two-tile kernel has two more warps that
// widen half of each step's K and V codes, so the widening is spread over all
// four schedulers of the SM.
template <int TILES, int D = 128, bool F8 = false>
__host__ __device__ constexpr bool f8_helpers() { return F8 && TILES == 2 && D == 128; }
template <int TILES, int D = 128, bool F8 = false>
constexpr int pair_threads() { return 32 * (6 * TILES + 2 + (f8_helpers<TILES, D, F8>() ? 2 : 0)); }

template <int SK, int SV, int TILES, int D>
struct PairLayout {
  static constexpr int kAtoms = D / 64;
  static constexpr int kQOff = 0;                                   // Q: [TILES][atoms]
  static constexpr int kKOff = TILES * kAtoms * kPairQAtom;         // K ring: [SK][atoms]
  static constexpr int kVOff = kKOff + SK * kAtoms * kPairKvAtom;   // V ring: [SV][atoms]
  static constexpr int kBarOff = kVOff + SV * kAtoms * kPairKvAtom;
  // + the FP8 landing barriers (SK + SV) and the V sub-tile masks (SV words)
  static constexpr int kBars = 2 * SK + 2 * SV + 1 + 2 + 2 + 4 + 4 + 1 + SK + SV;
  static constexpr size_t kSmem = 1024 + kBarOff + kBars * 8 + SV * 4 + 16;
};

// FP8 E4M3 caches: a step's codes (64 rows of D bytes, in the pool map's
// swizzle: 16-byte unit c of row r at unit c ^ (r & 7) for 128-byte rows,
// c ^ ((r >> 1) & 3) for 64-byte rows) are copied into the upper half of the
// fp16 stage and widened there to the fp16 tile the MMA reads (128-byte rows
// of 64 dims per atom, unit k of row r at k ^ (r & 7)); every code is exact
// in fp16.  A pass covers 1 KB of codes (8 rows at head_dim 128, 16 at 64);
// a warp widens passes [pass_begin, pass_end) (whole groups), reading kGroup
// passes into registers before it writes them.  At head_dim 128 the codes of
// row r share their 128 bytes with row r of the second atom only, and at
// head_dim 64 a group writes over codes of that group or of earlier ones
// only, so nothing is overwritten before it is read.
template <int D>
__device__ __forceinline__ void f8_stage_to_f16(uint8_t *st, int lane, int pass_begin,
                                                int pass_end) {
  constexpr int kRows = 1024 / D;      // rows per pass: 8 (d 128) or 16 (d 64)
  constexpr int kPerRow = 32 / kRows;  // lanes per row: 4 or 2
  constexpr int kPasses = kPairKeys / kRows;
  constexpr int kGroup = 4;            // passes read before the writes
  static_assert(kPasses % kGroup == 0, "whole groups");
  const uint8_t *codes = st + (D / 64) * kPairKvAtom / 2;
  const int c0 = 2 * (lane % kPerRow);  // this lane's 16-dim units c0 and c0 + 1
#pragma unroll 1
  for (int j0 = pass_begin; j0 < pass_end; j0 += kGroup) {
    uint4 x[kGroup][2];
#pragma unroll
    for (int g = 0; g < kGroup; ++g) {
      const int r = (j0 + g) * kRows + lane / kPerRow;
      const int sw = D == 128 ? (r & 7) : ((r >> 1) & 3);
      x[g][0] = *reinterpret_cast<const uint4 *>(codes + r * D + ((c0 ^ sw) << 4));
      x[g][1] = *reinterpret_cast<const uint4 *>(codes + r * D + (((c0 + 1) ^ sw) << 4));
    }
    __syncwarp();
    // At head_dim 128 the lanes of the second atom take their units in the
    // other order, so the eight lanes of each store phase (two rows, four
    // lanes each) write eight different 16-byte bank groups.
    const bool flip = D == 128 && (lane & 2);
#pragma unroll
    for (int g = 0; g < kGroup; ++g) {
      const int r = (j0 + g) * kRows + lane / kPerRow;
      const uint4 xa = flip ? x[g][1] : x[g][0], xb = flip ? x[g][0] : x[g][1];
      uint32_t h0[8], h1[8];
      e4m3x16_to_half(xa, h0);
      e4m3x16_to_half(xb, h1);
      // unit c (dims 16 c .. 16 c + 15) becomes fp16 units 2 (c & 3) and
      // 2 (c & 3) + 1 of atom c / 4; h0 holds unit c0 + flip, h1 the other
      uint8_t *row = st + (c0 >> 2) * kPairKvAtom + r * 128;
      const int ka = 2 * (c0 & 3) + (flip ? 2 : 0), kb = 2 * (c0 & 3) + (flip ? 0 : 2);
      const int sw = r & 7;
      *reinterpret_cast<uint4 *>(row + ((ka ^ sw) << 4)) = make_uint4(h0[0], h0[1], h0[2], h0[3]);
      *reinterpret_cast<uint4 *>(row + (((ka + 1) ^ sw) << 4)) =
          make_uint4(h0[4], h0[5], h0[6], h0[7]);
      *reinterpret_cast<uint4 *>(row + ((kb ^ sw) << 4)) = make_uint4(h1[0], h1[1], h1[2], h1[3]);
      *reinterpret_cast<uint4 *>(row + (((kb + 1) ^ sw) << 4)) =
          make_uint4(h1[4], h1[5], h1[6], h1[7]);
    }
    __syncwarp();
  }
}

// F8: the caches hold FP8 E4M3 codes, widened to fp16 in shared memory; the
// products then run in fp16 whatever T is (bf16 queries are carried in fp16,
// see the Q load).
template <typename T, int D, int SK, int SV, bool SPLIT, int TILES, bool PX, bool F8>
__global__ void __launch_bounds__(pair_threads<TILES, D, F8>(), TILES == 1 ? 2 : 1)
    pa_prefill_tc_pair_kernel(const __grid_constant__ CUtensorMap kmap,
                              const __grid_constant__ CUtensorMap vmap, const PrefillArgs a) {
  static_assert(TILES == 1 || TILES == 2, "one or two query tiles per CTA");
  static_assert(!PX || TILES == 1, "the shared-prefix pass runs one tile per CTA");
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static_assert(!F8 || !SPLIT, "FP8 caches: the products run in fp16 (no split P)");
  using L = PairLayout<SK, SV, TILES, D>;
  constexpr int kAtoms = L::kAtoms;
  constexpr int kIssue0 = 4 * TILES;      // first MMA-issuing warp
  constexpr int kLoad0 = 6 * TILES;       // K producer warp (V: kLoad0 + 1)
  // FP8 widening helpers (K: kLoad0 + 2, V: kLoad0 + 3); a stage is handed
  // over by every warp that widens part of it
  constexpr bool kHelpers = f8_helpers<TILES, D, F8>();
  constexpr int kWideners = kHelpers ? 2 : 1;
  constexpr int kSub = kPairKeys / 16;         // 16-row sub-tiles per step
  constexpr uint32_t kAllSub = (1u << kSub) - 1;
  constexpr bool kBf16 = sizeof(T) == 2 && !std::is_same<T, __half>::value;
  // MMA operand type (P included): T, or fp16 over FP8 caches
  using MT = typename std::conditional<F8, __half, T>::type;
  constexpr bool kMmaBf16 = kBf16 && !F8;
  // TMEM columns of a tile: scores 0..63, P 64..127, O from 128.  fp16 P: two
  // buffers of 32 columns (step n in buffer n % 2); bf16 P: one buffer, hi
  // parts in 64..95 and lo parts in 96..127.
  constexpr int kPBufs = SPLIT ? 1 : 2;
  constexpr int kPCol = 64, kOCol = 128;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *k_full = reinterpret_cast<uint64_t *>(smem + L::kBarOff);
  uint64_t *k_empty = k_full + SK;
  uint64_t *v_full = k_empty + SK;
  uint64_t *v_empty = v_full + SV;
  uint64_t *v_tail = v_empty + SV;     // the last step's V load, before its tail is zeroed
  uint64_t *s_full = v_tail + 1;       // [2 tiles]: scores computed
  uint64_t *s_free = s_full + 2;       // [2 tiles]: scores loaded by the softmax warps
  uint64_t *p_full = s_free + 2;       // [2 tiles][2 P buffers]
  uint64_t *pv_done = p_full + 4;      // [2 tiles][2 P buffers]
  uint64_t *q_ready = pv_done + 4;
  uint64_t *k_land = q_ready + 1;      // [SK] FP8: a K step's codes are in
  uint64_t *v_land = k_land + SK;      // [SV] FP8: a V step's codes are in
  uint32_t *v_masks = reinterpret_cast<uint32_t *>(v_land + SV);  // [SV] FP8: loaded sub-tiles
  uint32_t *tmem_slot = v_masks + SV;

  const int kvh = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.group;
  const int tpc = TILES * kTcRows / G; // tokens per CTA (members, in the shared-prefix pass)
  // shared-prefix pass: first_m of each member of the CTA, then the source
  // member, the member count and the first member's sequence
  int *px_first = reinterpret_cast<int *>(tmem_slot + 4);
  int *px_ctl = px_first + kTcRows;

  if (tid == 0) {
    for (int s = 0; s < SK; ++s) {
      mbar_init(&k_full[s], F8 ? kWideners : 1);
      mbar_init(&k_empty[s], TILES);  // released by every Q K^T issuer
    }
    for (int s = 0; s < SV; ++s) {
      mbar_init(&v_full[s], F8 ? kWideners : 1);
      mbar_init(&v_empty[s], TILES);  // and every P V issuer
    }
    mbar_init(v_tail, 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&s_free[t], kTcRows);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&p_full[i], kTcRows);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(q_ready, TILES * kTcRows);
    for (int s = 0; s < SK; ++s) mbar_init(&k_land[s], 1);
    for (int s = 0; s < SV; ++s) mbar_init(&v_land[s], 1);
    fence_barrier_init();
  }
  if (warp == kIssue0) tmem_alloc(tmem_slot, 256 * TILES);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dependency_wait();  // the chunk's K/V may come from the kernel before

  // Rows are (token, head) pairs of one chunk -- in the shared-prefix pass
  // (member, head) pairs of consecutive sequences, whose queries sit exactly
  // where a chunk's tokens would -- and keys run over [key_base, key_base +
  // n_keys) of the sequence's (the source member's) table.
  int q0, q_len, t_first, t_last, base_pos, n_keys, key_base = 0, px_p = 0;
  bool active = true;
  const int32_t *bt_row;
  if constexpr (PX) {
    // the decode grid after this one may start now: it streams the
    // sequences' own partitions meanwhile and waits for these partials only
    // before it joins them
    grid_launch_dependents();
    const int grp = blockIdx.z, chunk = blockIdx.x % a.chunks;
    px_p = blockIdx.x / a.chunks;
    const int P = a.part_tokens;
    if (warp == 0) {
      const int g0 = a.group_start[grp], g1 = a.group_start[grp + 1];
      const bool group_ok = g0 >= 0 && g1 >= g0 && g1 <= a.num_seqs &&
                            g1 - g0 <= a.max_group_size && (grp > 0 || g0 == 0) &&
                            (grp < a.num_groups - 1 || g1 == a.num_seqs);
      const bool reporter = px_p == 0 && kvh == 0;  // one CTA per chunk reports bad input
      if (!group_ok && reporter && chunk == 0 && lane == 0) atomicOr(a.err, kErrPrefix);
      const int m0 = g0 + chunk * a.members_per_cta;
      const int nm = group_ok ? max(0, min(a.members_per_cta, g1 - m0)) : 0;
      int src = -1;
      for (int i0 = 0; i0 < nm; i0 += 32) {
        const int i = i0 + lane;
        int first = 0;
        if (i < nm) {
          int c = a.context_lens[m0 + i];
          // the decode kernel flags a bad length; here it only means "nothing shared"
          if (c < 0 || c > (a.max_blocks_per_seq << a.bs_log2) || c > a.max_context_len) c = 0;
          const int np = c > 0 ? (c + P - 1) / P : 1;
          const int pl = a.prefix_lens[m0 + i];
          if (pl != a.prefix_lens[g0] && reporter) atomicOr(a.err, kErrPrefix);
          first = min(max(pl, 0) / P, np - 1);
          px_first[i] = first;
        }
        const unsigned takers = __ballot_sync(kFullMask, i < nm && px_p < first);
        if (src < 0 && takers) src = i0 + __ffs(takers) - 1;
      }
      if (lane == 0) {
        px_ctl[0] = src;
        px_ctl[1] = nm;
        px_ctl[2] = m0;
      }
    }
    __syncthreads();
    const int src = px_ctl[0], nm = px_ctl[1];
    q0 = px_ctl[2];
    active = src >= 0;  // some member takes this partition from here
    q_len = nm;
    t_first = 0;
    t_last = nm - 1;
    base_pos = 0;
    n_keys = P;
    key_base = px_p * P;
    // p < first_src <= np_src - 1: the partition ends inside the source's
    // context, so every table entry it needs is inside the source's row
    bt_row = a.block_tables + static_cast<int64_t>(q0 + max(src, 0)) * a.max_blocks_per_seq;
    if (active && kvh == 0) {
      // every other taker must reference the same blocks (checked once per
      // partition; it only sets a flag)
      const int lb0 = key_base >> a.bs_log2;
      const int nlb = ((key_base + P - 1) >> a.bs_log2) - lb0 + 1;
      for (int it = tid; it < nm * nlb; it += blockDim.x) {
        const int i = it / nlb, lb = lb0 + it % nlb;
        if (i != src && px_p < px_first[i] &&
            a.block_tables[static_cast<int64_t>(q0 + i) * a.max_blocks_per_seq + lb] !=
                bt_row[lb])
          atomicOr(a.err, kErrPrefix);
      }
    }
  } else {
    const int tile = blockIdx.x, seq = blockIdx.z;
    q0 = a.query_start[seq];
    q_len = a.query_start[seq + 1] - q0;
    const int ctx = a.context_lens[seq];
    if (q_len < 0 || ctx < q_len || ctx > (a.max_blocks_per_seq << a.bs_log2) ||
        q_len > a.max_q_len) {
      if (tid == 0 && tile == 0 && kvh == 0) atomicOr(a.err, kErrBadLen);
      active = false;
    }
    t_first = tile * tpc;
    if (t_first >= q_len) active = false;
    t_last = min(q_len, t_first + tpc) - 1;
    base_pos = ctx - q_len;
    n_keys = base_pos + t_last + 1;
    bt_row = a.block_tables + static_cast<int64_t>(seq) * a.max_blocks_per_seq;
  }
  // per tile: last token (-1 when the tile has no rows) and step count; tile 1
  // holds the later tokens, so it reads every step tile 0 reads.  Tile 0's
  // rows reach token (kTcRows - 1) / G; tile 1's begin at token kTcRows / G.
  // (The shared-prefix pass has no causal limit: every row sees all n_keys.)
  const int last0 = min(t_last, t_first + (kTcRows - 1) / G);
  const int last1 = TILES == 2 && t_first + kTcRows / G <= t_last ? t_last : -1;
  const int n_steps0 =
      active ? ((PX ? n_keys : base_pos + last0 + 1) + kPairKeys - 1) / kPairKeys : 0;
  const int n_steps1 = active && last1 >= 0 ? (n_keys + kPairKeys - 1) / kPairKeys : 0;
  const int n_steps = max(n_steps0, n_steps1);
  const int n_sub = (n_keys + 15) / 16;
  // table entry of the 16-key sub-tile u of the key range
  auto table_entry = [&](int u) { return bt_row[(key_base + u * 16) >> a.bs_log2]; };

  if (active && warp < kIssue0) {
    // ------------------------------------------------------------ softmax warps
    const int t = warp >> 2;
    const int r = tid & (kTcRows - 1);                 // row within the tile = TMEM lane
    const int rc = t * kTcRows + r;                    // row within the CTA
    const int tok = t_first + rc / G;
    const bool row_ok = tok <= t_last;
    const int pos = PX ? n_keys - 1 : base_pos + tok;  // keys up to pos are attended to
    const int my_steps = t == 0 ? n_steps0 : n_steps1;
    float sl2 = a.scale_log2;  // this row's softmax scale (base 2)
    {
      const T *qrow = static_cast<const T *>(a.query) +
                      (static_cast<int64_t>(q0 + (row_ok ? tok : 0)) * a.num_q_heads + kvh * G +
                       rc % G) * D;
      uint8_t *qt = smem + L::kQOff + t * kAtoms * kPairQAtom;
      // bf16 queries over FP8 caches: the row is scaled by 2^e so that its
      // largest magnitude lands in [2^14, 2^15), then rounded to fp16 (exact
      // for every value down to 2^-31 of the largest: bf16 carries 8
      // significant bits, and fp16 holds 8 bits at every magnitude from 2^-17
      // up), and 2^-e joins the row's softmax scale
      float qf = 1.f;
      if constexpr (F8 && kBf16) {
        float mx = 0.f;
        if (row_ok) {
#pragma unroll 4
          for (int ch = 0; ch < D / 8; ++ch) {
            const uint4 v = *reinterpret_cast<const uint4 *>(qrow + ch * 8);
#pragma unroll
            for (int w2 = 0; w2 < 4; ++w2) {
              const float2 f = Elem<T>::unpack(word_of(v, w2));
              mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
          }
        }
        const int ex = static_cast<int>((__float_as_uint(mx) >> 23) & 0xffu) - 127;
        const int e = min(120, 14 - ex);
        qf = ldexpf(1.f, e);
        sl2 = ldexpf(sl2, -e);
      }
#pragma unroll
      for (int ch = 0; ch < D / 8; ++ch) {
        uint4 v = row_ok ? *reinterpret_cast<const uint4 *>(qrow + ch * 8)
                         : make_uint4(0, 0, 0, 0);
        if constexpr (F8 && kBf16) {
          uint32_t w4[4];
#pragma unroll
          for (int w2 = 0; w2 < 4; ++w2) {
            const float2 f = Elem<T>::unpack(word_of(v, w2));
            w4[w2] = Elem<__half>::pack(f.x * qf, f.y * qf);
          }
          v = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
        *reinterpret_cast<uint4 *>(qt + (ch >> 3) * kPairQAtom + r * 128 +
                                   (((ch & 7) ^ (r & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();
      mbar_arrive(q_ready);
    }
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + t * 256;
    // sub-tile validity, as the producer decides it (lane h < kSub: sub-tile h of a step)
    auto step_mask = [&](int n) -> uint32_t {
      const int u = n * kSub + lane;
      bool ok = false;
      if (lane < kSub && u < n_sub) {
        const int phys = table_entry(u);
        ok = phys >= 0 && static_cast<int64_t>(phys) < a.num_blocks;
      }
      return __ballot_sync(kFullMask, ok) & kAllSub;
    };
    float m_ref = -INFINITY, l = 0.f;
    bool ok_run = true;
    uint32_t vmask_next = my_steps > 0 ? step_mask(0) : 0;
    for (int n = 0; n < my_steps && ok_run; ++n) {
      const uint32_t vmask = vmask_next;
      if (!__all_sync(kFullMask, mbar_wait_bounded(&s_full[t], n & 1))) {
        if (lane == 0) atomicOr(a.err, kErrTimeout);
        ok_run = false;
        break;
      }
      tc_fence_after();
      float sv[kPairKeys];
      static_assert(kPairKeys == 64, "two 32-column loads");
      {
        // both loads in flight before the one wait
        float t0[32], t1[32];
        tmem_ld32(lane_addr, t0);
        tmem_ld32(lane_addr + 32, t1);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          sv[i] = t0[i];
          sv[32 + i] = t1[i];
        }
      }
      // the score columns may now take the next step's Q K^T
      tc_fence_before();
      mbar_arrive(&s_free[t]);
      // block id of sub-tile `lane` of step n + 1: loaded now, used at the end
      // of the step, so its latency hides behind the softmax
      int bt_next = -1;
      {
        const int u = (n + 1) * kSub + lane;
        if (n + 1 < my_steps && lane < kSub && u < n_sub) bt_next = table_entry(u);
      }
      const int key0 = n * kPairKeys;
      const bool full_step = row_ok && key0 + kPairKeys - 1 <= pos && vmask == kAllSub;
      if (!full_step) {
#pragma unroll
        for (int c = 0; c < kPairKeys; ++c) {
          const int key = key0 + c;
          const bool ok = row_ok && key <= pos && ((vmask >> (c >> 4)) & 1u);
          sv[c] = ok ? sv[c] : -INFINITY;
        }
      }
      // row max: three-input max, 64 -> 22 -> 8 -> 3 -> 1
      static_assert(kPairKeys == 64, "max tree written for 64 keys");
      float t22[22], t8[8];
#pragma unroll
      for (int j = 0; j < 21; ++j) t22[j] = fmax3(sv[3 * j], sv[3 * j + 1], sv[3 * j + 2]);
      t22[21] = sv[63];
#pragma unroll
      for (int j = 0; j < 7; ++j) t8[j] = fmax3(t22[3 * j], t22[3 * j + 1], t22[3 * j + 2]);
      t8[7] = t22[21];
      const float tmax_raw = fmax3(fmax3(t8[0], t8[1], t8[2]), fmax3(t8[3], t8[4], t8[5]),
                                   fmaxf(t8[6], t8[7]));
      const float tmax = tmax_raw * sl2;  // the scale is positive: same order
      const float m_new = fmaxf(m_ref, tmax);
      const bool move = m_new > m_ref + kRescaleLog2;  // includes the first finite max
      const float alpha = !move ? 1.f : (m_ref == -INFINITY ? 0.f : ex2_approx(m_ref - m_new));
      if (move) {
        l *= alpha;
        m_ref = m_new;
      }
      const float neg_m = m_ref == -INFINITY ? 0.f : -m_ref;
      // P for the whole step in registers first (s scale - m and the row sum on
      // packed fp32 pairs), so the wait for its buffer below overlaps the math
      const uint64_t scale2 = f2_pack(sl2, sl2);
      const uint64_t negm2 = f2_pack(neg_m, neg_m);
      uint64_t ls2[4] = {0, 0, 0, 0};  // +0.0f pairs
      uint32_t ph[kPairKeys / 2], pl[SPLIT ? kPairKeys / 2 : 1];
#pragma unroll
      for (int e = 0; e < kPairKeys / 2; ++e) {
        const float2 x = f2_unpack(f2_fma(f2_pack(sv[2 * e], sv[2 * e + 1]), scale2, negm2));
        const float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
        ls2[e & 3] = f2_add(ls2[e & 3], f2_pack(p0, p1));
        ph[e] = Elem<MT>::pack(p0, p1);
        if constexpr (SPLIT) {
          const float2 h = Elem<MT>::unpack(ph[e]);
          pl[e] = Elem<MT>::pack(p0 - h.x, p1 - h.y);
        }
      }
      {
        const float2 sm = f2_unpack(f2_add(f2_add(ls2[0], ls2[1]), f2_add(ls2[2], ls2[3])));
        l += sm.x + sm.y;
      }
      // O must hold P V of every earlier step before it is rescaled; P's buffer
      // must have been read by the P V of step n - kPBufs.  Each pv_done
      // barrier belongs to one buffer, and P V of step n cannot start before
      // this warp arrives below, so no wait is more than one phase behind.
      const int pb = n % kPBufs;
      if (n > 0 && __any_sync(kFullMask, move)) {  // whole warp: rows that did not move use 1
        const int pp = (n - 1) % kPBufs;
        if (!__all_sync(kFullMask, mbar_wait_bounded(&pv_done[2 * t + pp], ((n - 1) / kPBufs) & 1))) {
          if (lane == 0) atomicOr(a.err, kErrTimeout);
          ok_run = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int cb = 0; cb < D / 32; ++cb) {
          float o[32];
          tmem_ld32(lane_addr + kOCol + cb * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(lane_addr + kOCol + cb * 32, o);
        }
      }
      if (n >= kPBufs &&
          !__all_sync(kFullMask, mbar_wait_bounded(&pv_done[2 * t + pb], ((n - kPBufs) / kPBufs) & 1))) {
        if (lane == 0) atomicOr(a.err, kErrTimeout);
        ok_run = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < kPairKeys / 32; ++c) {
        if constexpr (SPLIT) {
          tmem_st16(lane_addr + kPCol + 16 * c, ph + 16 * c);
          tmem_st16(lane_addr + kPCol + 32 + 16 * c, pl + 16 * c);
        } else {
          tmem_st16(lane_addr + kPCol + 32 * pb + 16 * c, ph + 16 * c);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[2 * t + pb]);
      vmask_next =
          __ballot_sync(kFullMask, bt_next >= 0 && static_cast<int64_t>(bt_next) < a.num_blocks) &
          kAllSub;
    }
    // ---- epilogue: O / l for this row
    if (ok_run && my_steps > 0) {
      const int last = my_steps - 1;
      if (__all_sync(kFullMask, mbar_wait_bounded(&pv_done[2 * t + last % kPBufs], (last / kPBufs) & 1))) {
        tc_fence_after();
        const float inv = l > 0.f ? a.out_scale / l : 0.f;  // times the V scale (FP8)
        const int64_t orow_idx = static_cast<int64_t>(q0 + tok) * a.num_q_heads + kvh * G + rc % G;
        if constexpr (PX) {
          // the partition's partial of this row, for a member that takes the
          // partition from here: (m, l) with the row's running reference
          // max and o = O / l
          // (the TMEM loads are warp-wide; only the stores depend on the row)
          const bool takes = row_ok && px_p < px_first[tok];
          const int64_t pr = orow_idx * a.num_parts + px_p;
          if (takes) {
            a.ws_m[pr] = m_ref;
            a.ws_l[pr] = l;
          }
#pragma unroll 1
          for (int cb = 0; cb < D / 32; ++cb) {
            float o[32];
            tmem_ld32(lane_addr + kOCol + cb * 32, o);
            tmem_wait_ld();
            if (takes) {
              float *orow = a.ws_o + pr * D + cb * 32;
#pragma unroll
              for (int q = 0; q < 8; ++q)
                *reinterpret_cast<float4 *>(orow + q * 4) =
                    make_float4(o[4 * q] * inv, o[4 * q + 1] * inv, o[4 * q + 2] * inv,
                                o[4 * q + 3] * inv);
            }
          }
        } else {
        T *orow = static_cast<T *>(a.out) + orow_idx * D;
#pragma unroll 1
        for (int cb = 0; cb < D / 32; ++cb) {
          float o[32];
          tmem_ld32(lane_addr + kOCol + cb * 32, o);
          tmem_wait_ld();
          if (row_ok) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 pk;
              pk.x = Elem<T>::pack(o[q * 8 + 0] * inv, o[q * 8 + 1] * inv);
              pk.y = Elem<T>::pack(o[q * 8 + 2] * inv, o[q * 8 + 3] * inv);
              pk.z = Elem<T>::pack(o[q * 8 + 4] * inv, o[q * 8 + 5] * inv);
              pk.w = Elem<T>::pack(o[q * 8 + 6] * inv, o[q * 8 + 7] * inv);
              *reinterpret_cast<uint4 *>(orow + cb * 32 + q * 8) = pk;
            }
          }
        }
        }
      } else if (lane == 0) {
        atomicOr(a.err, kErrTimeout);
      }
    }
  } else if (active && warp >= kIssue0 && warp < kLoad0) {
    // ------------------------------------------------------------ MMA issuers
    // Q K^T issuer of tile t: step n once the softmax warps have loaded the
    // scores of step n - 1 and K of step n is in.  P V issuer: step n once its
    // P and V are in place.  Each issuer releases every K (or V) stage once
    // (count-2 barriers); for steps its tile does not read it waits for the
    // stage to fill first, so its release lands in that step's phase.
    if (lane == 0) {
      const int t = (warp - kIssue0) >> 1;
      const bool qk_role = ((warp - kIssue0) & 1) == 0;
      const int nt = t == 0 ? n_steps0 : n_steps1;
      const uint32_t tt = tmem + t * 256;
      bool ok_run = true;
      if (qk_role) {
        const uint32_t id_qk = umma_idesc_f16(kMmaBf16 ? 1 : 0, false, kTcRows, kPairKeys);
        const uint32_t qb = smem_addr(smem + L::kQOff) + t * kAtoms * kPairQAtom;
        const uint32_t sk0 = smem_addr(smem + L::kKOff);
        // descriptors of the tile's Q and of K stage 0; every other operand
        // is these plus a byte offset / 16 in the address field (shared
        // memory lies below 2^18 bytes, so the 14-bit field never carries)
        const uint64_t dq0 = umma_desc_sw128(qb, 16, 1024);
        const uint64_t dk0 = umma_desc_sw128(sk0, 16, 1024);
        ok_run = mbar_wait_bounded(q_ready, 0);
        for (int n = 0; n < nt && ok_run; ++n) {
          // K is staged well ahead, so wait for it first: then only the
          // release of the score columns stands between the softmax and the
          // next product (that hand-off sets the step time)
          if (!mbar_wait_bounded(&k_full[n % SK], (n / SK) & 1) ||
              (n > 0 && !mbar_wait_bounded(&s_free[t], (n - 1) & 1))) {
            ok_run = false;
            break;
          }
          tc_fence_after();
          const uint64_t dkn = dk0 + static_cast<uint64_t>(((n % SK) * kAtoms * kPairKvAtom) >> 4);
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint64_t da = dq0 + static_cast<uint64_t>(((k >> 2) * kPairQAtom + (k & 3) * 32) >> 4);
            const uint64_t db = dkn + static_cast<uint64_t>(((k >> 2) * kPairKvAtom + (k & 3) * 32) >> 4);
            umma_f16(tt, da, db, id_qk, k > 0);
          }
          umma_commit(&s_full[t]);
          umma_commit(&k_empty[n % SK]);
        }
        for (int m = nt; m < n_steps && ok_run; ++m) {
          if (!mbar_wait_bounded(&k_full[m % SK], (m / SK) & 1)) {
            ok_run = false;
            break;
          }
          mbar_arrive(&k_empty[m % SK]);
        }
      } else {
        const uint32_t id_pv = umma_idesc_f16(kMmaBf16 ? 1 : 0, true, kTcRows, D);
        const uint32_t sv0 = smem_addr(smem + L::kVOff);
        const uint64_t dv0 = umma_desc_sw128(sv0, kPairKvAtom, 1024);  // V stage 0, as for K
        for (int n = 0; n < nt && ok_run; ++n) {
          const int s = n % SV, pb = n % kPBufs;
          if (!mbar_wait_bounded(&p_full[2 * t + pb], (n / kPBufs) & 1) ||
              !mbar_wait_bounded(&v_full[s], (n / SV) & 1)) {
            ok_run = false;
            break;
          }
          tc_fence_after();
          const uint64_t dvs = dv0 + static_cast<uint64_t>((s * kAtoms * kPairKvAtom) >> 4);
#pragma unroll
          for (int kk = 0; kk < kPairKeys / 16; ++kk) {
            const uint64_t dv = dvs + static_cast<uint64_t>((kk * 2048) >> 4);
            if constexpr (SPLIT) {
              umma_f16_ts(tt + kOCol, tt + kPCol + 8 * kk, dv, id_pv, n > 0 || kk > 0);
              umma_f16_ts(tt + kOCol, tt + kPCol + 32 + 8 * kk, dv, id_pv, true);
            } else {
              umma_f16_ts(tt + kOCol, tt + kPCol + 32 * pb + 8 * kk, dv, id_pv, n > 0 || kk > 0);
            }
          }
          umma_commit(&pv_done[2 * t + pb]);
          umma_commit(&v_empty[s]);
        }
        for (int m = nt; m < n_steps && ok_run; ++m) {
          if (!mbar_wait_bounded(&v_full[m % SV], (m / SV) & 1)) {
            ok_run = false;
            break;
          }
          mbar_arrive(&v_empty[m % SV]);
        }
      }
      if (!ok_run) atomicOr(a.err, kErrTimeout);
    }
  } else if (active && warp >= kLoad0) {
    // ---------------------------------------------------- TMA producers (K, V)
    // (and, over FP8 caches at head_dim 128 with two tiles, the K and V
    // widening helpers)
    const bool k_role = ((warp - kLoad0) & 1) == 0;
    const bool helper = warp - kLoad0 >= 2;
    const int bs_mask = (1 << a.bs_log2) - 1;
    auto block_of = [&](int u) -> int {
      if (u >= n_sub) return -1;
      const int phys = table_entry(u);
      if (phys < 0 || static_cast<int64_t>(phys) >= a.num_blocks) {
        atomicOr(a.err, kErrBadBlock);
        return -1;
      }
      return phys;
    };
    const uint64_t policy = l2_policy_evict_first();
    int win_base = 0;
    int win = helper ? -1 : block_of(lane);
    bool ok_run = true;
    if constexpr (F8) {
      // A step's copies (16 rows of head_dim codes per sub-tile) land in the
      // upper half of its stage; the warp widens them to fp16 there, clears
      // what V must not contribute and hands the stage over.  Copies and
      // widening each go ahead as soon as their own barrier allows (a stage
      // released by the MMAs, a step's codes in), so the widening of step m
      // waits for nothing later than the release of step m - S; the warp
      // polls both and gives up after kWaitLimitNs without progress.
      constexpr int kF8Sub = 16 * D;                // bytes of one sub-tile's codes
      constexpr int kStage = kAtoms * kPairKvAtom;  // bytes of one fp16 stage
      constexpr int kPassRows = 1024 / D;           // rows per 1 KB pass of codes
      constexpr int kPasses = kPairKeys / kPassRows;
      const int S = k_role ? SK : SV;
      uint64_t *land = k_role ? k_land : v_land;
      uint64_t *full = k_role ? k_full : v_full;
      uint64_t *empty = k_role ? k_empty : v_empty;
      uint8_t *ring = smem + (k_role ? L::kKOff : L::kVOff);
      const CUtensorMap *map = k_role ? &kmap : &vmap;
      // this warp's passes of every step: all of them, or with helpers the
      // first half (producer) or the second (helper)
      const int pass0 = kHelpers && helper ? kPasses / 2 : 0;
      const int pass1 = kHelpers && !helper ? kPasses / 2 : kPasses;
      // widen this warp's passes of step m (its codes are in), clear the V
      // rows among them that must not contribute, and hand the stage over
      auto widen = [&](int m) {
        const int s = m % S;
        uint8_t *st = ring + s * kStage;
        f8_stage_to_f16<D>(st, lane, pass0, pass1);
        if (!k_role) {
          // V rows past n_keys and of sub-tiles not loaded become zeros
          const uint32_t vm = v_masks[s];
          const int first = n_keys - m * kPairKeys;  // first row to clear
          if (vm != kAllSub || first < kPairKeys) {
            const int row0 = pass0 * kPassRows;
            for (int i = lane; i < (pass1 - pass0) * kPassRows * kAtoms * 8; i += 32) {
              const int row = row0 + i / (kAtoms * 8), b = (i >> 3) % kAtoms, u16 = i & 7;
              if (row >= first || !((vm >> (row >> 4)) & 1u))
                *reinterpret_cast<uint4 *>(st + b * kPairKvAtom + row * 128 + u16 * 16) =
                    make_uint4(0, 0, 0, 0);
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[s]);
      };
      if (helper) {
        // every step in order, once its codes are in (each lane observes it)
        for (int m = 0; m < n_steps; ++m) {
          if (!__all_sync(kFullMask, mbar_wait_bounded(&land[m % S], (m / S) & 1))) {
            ok_run = false;
            break;
          }
          widen(m);
        }
      } else {
        int n_issue = 0, n_conv = 0;
        uint64_t t_prog = global_timer_ns();
        while (n_conv < n_steps) {
          bool progressed = false;
          if (n_issue < n_steps) {
            const int n = n_issue, s = n % S;
            bool free_stage = true;
            if (lane == 0 && n >= S) free_stage = mbar_test_wait(&empty[s], ((n / S) - 1) & 1);
            if (__shfl_sync(kFullMask, free_stage ? 1 : 0, 0)) {
              if (n * kSub >= win_base + 32) {
                win_base += 32;
                win = block_of(win_base + lane);
              }
              const int my_phys =
                  __shfl_sync(kFullMask, win, n * kSub + (lane & (kSub - 1)) - win_base);
              const uint32_t mask =
                  __ballot_sync(kFullMask, lane < kSub && my_phys >= 0) & kAllSub;
              if (lane == 0) {
                if (!k_role) v_masks[s] = mask;
                if (mask == 0)
                  mbar_arrive(&land[s]);
                else
                  mbar_arrive_expect_tx(&land[s], __popc(mask) * kF8Sub);
              }
              __syncwarp();
              if (lane < kSub && my_phys >= 0) {
                const int u = n * kSub + lane;
                const int y = ((my_phys * a.num_kv_heads + kvh) << a.bs_log2) +
                              ((key_base + u * 16) & bs_mask);
                tma_load_2d(ring + s * kStage + kStage / 2 + lane * kF8Sub, map, 0, y, &land[s],
                            policy);
              }
              ++n_issue;
              progressed = true;
            }
          }
          // every lane observes the copies' completion before it reads them
          if (n_conv < n_issue &&
              __all_sync(kFullMask, mbar_test_wait(&land[n_conv % S], (n_conv / S) & 1))) {
            widen(n_conv);
            ++n_conv;
            progressed = true;
          }
          if (progressed) {
            t_prog = global_timer_ns();
          } else {
            if (global_timer_ns() - t_prog > kWaitLimitNs) {
              ok_run = false;
              break;
            }
            __nanosleep(32);
          }
        }
      }
    } else {
      for (int n = 0; n < n_steps && ok_run; ++n) {
        if (n * kSub >= win_base + 32) {
          win_base += 32;
          win = block_of(win_base + lane);
        }
        // lane h < kSub issues the copies of sub-tile h
        const int my_phys = __shfl_sync(kFullMask, win, n * kSub + (lane & (kSub - 1)) - win_base);
        const uint32_t mask = __ballot_sync(kFullMask, lane < kSub && my_phys >= 0) & kAllSub;
        const uint32_t bytes = __popc(mask) * kAtoms * 2048;
        auto load = [&](uint8_t *st, const CUtensorMap *map, uint64_t *bar) {
          if (lane < kSub && my_phys >= 0) {
            const int u = n * kSub + lane;
            const int y =
                ((my_phys * a.num_kv_heads + kvh) << a.bs_log2) + ((key_base + u * 16) & bs_mask);
  #pragma unroll
            for (int b = 0; b < kAtoms; ++b)
              tma_load_2d(st + b * kPairKvAtom + lane * 2048, map, b * 64, y, bar, policy);
          }
        };
        if (k_role) {
          // the expected bytes are posted (lane 0) before any lane issues a copy
          const int sk = n % SK;
          if (lane == 0) {
            if (n >= SK && !mbar_wait_bounded(&k_empty[sk], ((n / SK) - 1) & 1)) {
              ok_run = false;
            } else if (bytes == 0) {
              mbar_arrive(&k_full[sk]);
            } else {
              mbar_arrive_expect_tx(&k_full[sk], bytes);
            }
          }
          ok_run = __shfl_sync(kFullMask, ok_run ? 1 : 0, 0) != 0;
          if (!ok_run) break;
          __syncwarp();
          load(smem + L::kKOff + sk * kAtoms * kPairKvAtom, &kmap, &k_full[sk]);
          continue;
        }
        // V: rows past the keys in use and sub-tiles not loaded become zeros
        const int sv = n % SV;
        uint8_t *vst = smem + L::kVOff + sv * kAtoms * kPairKvAtom;
        if (lane == 0 && n >= SV && !mbar_wait_bounded(&v_empty[sv], ((n / SV) - 1) & 1))
          ok_run = false;
        ok_run = __shfl_sync(kFullMask, ok_run ? 1 : 0, 0) != 0;
        if (!ok_run) break;
        __syncwarp();
        const int key0 = n * kPairKeys;
        const bool tail = key0 + kPairKeys > n_keys;
        if (mask != kAllSub) {
          // sub-tiles with no load: zero every 64-dim atom of their 16 rows
          for (int i = lane; i < kSub * kAtoms * 16 * 8; i += 32) {  // 16-byte units
            const int h = i / (kAtoms * 128), b = (i >> 7) % kAtoms, row = (i >> 3) & 15,
                      u16 = i & 7;
            if (!((mask >> h) & 1u))
              *reinterpret_cast<uint4 *>(vst + b * kPairKvAtom + (h * 16 + row) * 128 + u16 * 16) =
                  make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (!tail) {
          if (lane == 0) {
            if (bytes == 0)
              mbar_arrive(&v_full[sv]);
            else
              mbar_arrive_expect_tx(&v_full[sv], bytes);
          }
          __syncwarp();
          load(vst, &vmap, &v_full[sv]);
        } else {
          // the last step: load, wait, zero the rows past n_keys, then hand over
          if (lane == 0 && bytes > 0) mbar_arrive_expect_tx(v_tail, bytes);
          __syncwarp();
          load(vst, &vmap, v_tail);
          bool got = true;
          if (lane == 0 && bytes > 0) got = mbar_wait_bounded(v_tail, 0);
          got = __shfl_sync(kFullMask, got ? 1 : 0, 0) != 0;
          if (!got) {
            ok_run = false;
            break;
          }
          __syncwarp();
          const int first = n_keys - key0;  // first row to clear
          for (int i = lane; i < kPairKeys * kAtoms * 8; i += 32) {
            const int row = i / (kAtoms * 8), b = (i >> 3) % kAtoms, u16 = i & 7;
            if (row >= first)
              *reinterpret_cast<uint4 *>(vst + b * kPairKvAtom + row * 128 + u16 * 16) =
                  make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&v_full[sv]);
        }
      }
    }
    if (!ok_run && lane == 0) atomicOr(a.err, kErrTimeout);
  }

  // ---- teardown: every tcgen05 operation is complete once each tile's last
  // P V has been observed by its softmax warps (its Q K^T products came
  // before it), or the tile had no work
  tc_fence_before();
  __syncthreads();
  if (warp == kIssue0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256 * TILES);
  }
  grid_launch_dependents();
}

template <typename T, int D, int SK, int SV, bool SPLIT, int TILES, bool PX = false,
          bool F8 = false>
cudaError_t launch_prefill_tc_pair_t(const PrefillArgs &a, const CUtensorMap &km,
                                     const CUtensorMap &vm, cudaStream_t stream) {
  // the shared-prefix pass keeps each member's first partition and the pass's
  // control words after the barriers
  constexpr size_t smem = PairLayout<SK, SV, TILES, D>::kSmem + (PX ? (kTcRows + 8) * 4 : 0);
  static_assert(smem <= (TILES == 1 ? 113 : 227) * 1024, "shared memory");
  auto kern = pa_prefill_tc_pair_kernel<T, D, SK, SV, SPLIT, TILES, PX, F8>;
  static SmemLimitOnce smem_limit;
  const cudaError_t e = smem_limit.ensure(kern, smem);
  if (e != cudaSuccess) return e;
  if constexpr (PX) {
    return launch_dependent(
        kern,
        dim3(static_cast<unsigned>(a.num_parts * a.chunks), static_cast<unsigned>(a.num_kv_heads),
             static_cast<unsigned>(a.num_groups)),
        dim3(pair_threads<TILES, D, F8>()), smem, stream, km, vm, a);
  }
  const int tpc = TILES * kTcRows / a.group;
  const int tiles = (a.max_q_len + tpc - 1) / tpc;
  return launch_dependent(kern, dim3(tiles, a.num_kv_heads, a.num_seqs),
                          dim3(pair_threads<TILES, D, F8>()), smem,
                          stream, km, vm, a);
}

}  // namespace

#ifndef PA_PREFILL_SOLO_KSTAGES
#define PA_PREFILL_SOLO_KSTAGES 2
#endif
#ifndef PA_PREFILL_SOLO_VSTAGES
#define PA_PREFILL_SOLO_VSTAGES 2
#endif
#ifndef PA_PREFILL_PAIR_KSTAGES
#define PA_PREFILL_PAIR_KSTAGES 4
#endif
#ifndef PA_PREFILL_PAIR_VSTAGES
#define PA_PREFILL_PAIR_VSTAGES 4
#endif

bool prefill_tc_supported(int head_dim, int group) {
  return (head_dim == 64 || head_dim == 128) && group >= 1 && group <= 8;
}

namespace {

template <int D>
cudaError_t launch_prefill_tc_d(const PrefillArgs &a, const CUtensorMap &km,
                                const CUtensorMap &vm, int dtype, bool kv_fp8,
                                cudaStream_t stream) {
  const bool pair = static_cast<int64_t>(a.max_q_len) * a.group > kTcRows;
  constexpr int PK = PA_PREFILL_PAIR_KSTAGES, PV = PA_PREFILL_PAIR_VSTAGES;
  constexpr int SK = PA_PREFILL_SOLO_KSTAGES, SV = PA_PREFILL_SOLO_VSTAGES;
  if (kv_fp8) {
    if (dtype == 0)
      return pair ? launch_prefill_tc_pair_t<__half, D, PK, PV, false, 2, false, true>(a, km, vm,
                                                                                       stream)
                  : launch_prefill_tc_pair_t<__half, D, SK, SV, false, 1, false, true>(a, km, vm,
                                                                                       stream);
    return pair ? launch_prefill_tc_pair_t<__nv_bfloat16, D, PK, PV, false, 2, false, true>(
                      a, km, vm, stream)
                : launch_prefill_tc_pair_t<__nv_bfloat16, D, SK, SV, false, 1, false, true>(
                      a, km, vm, stream);
  }
  if (dtype == 0) {
    if (pair)
      return launch_prefill_tc_pair_t<__half, D, PA_PREFILL_PAIR_KSTAGES, PA_PREFILL_PAIR_VSTAGES,
                                      false, 2>(a, km, vm, stream);
    return launch_prefill_tc_pair_t<__half, D, PA_PREFILL_SOLO_KSTAGES, PA_PREFILL_SOLO_VSTAGES,
                                    false, 1>(a, km, vm, stream);
  }
  if (pair)
    return launch_prefill_tc_pair_t<__nv_bfloat16, D, PA_PREFILL_PAIR_KSTAGES,
                                    PA_PREFILL_PAIR_VSTAGES, true, 2>(a, km, vm, stream);
  return launch_prefill_tc_pair_t<__nv_bfloat16, D, PA_PREFILL_SOLO_KSTAGES,
                                  PA_PREFILL_SOLO_VSTAGES, true, 1>(a, km, vm, stream);
}

}  // namespace

// Every shape pa_prefill accepts runs here.  Chunks that fill more than one
// 128-row tile run with two tiles per CTA (one CTA per SM); shorter ones
// (short chunks, decode-like rows) with one tile per CTA, two CTAs per SM.
cudaError_t launch_prefill(const PrefillArgs &a, const void *k_cache, const void *v_cache,
                           int64_t pool_rows, int head_dim, int dtype, bool kv_fp8,
                           cudaStream_t stream, bool *map_failed) {
  CUtensorMap km, vm;
  *map_failed = false;
  if (!encode_pool_map(&km, k_cache, pool_rows, head_dim, dtype, kv_fp8) ||
      !encode_pool_map(&vm, v_cache, pool_rows, head_dim, dtype, kv_fp8)) {
    *map_failed = true;
    return cudaErrorInvalidValue;
  }
  if (a.max_q_len == 0) return cudaSuccess;
  if (!prefill_tc_supported(head_dim, a.group)) return cudaErrorInvalidValue;
  return head_dim == 128 ? launch_prefill_tc_d<128>(a, km, vm, dtype, kv_fp8, stream)
                         : launch_prefill_tc_d<64>(a, km, vm, dtype, kv_fp8, stream);
}

// The shared-prefix pass of pa_decode_shared_prefix on the same kernel: one
// 128-row tile per CTA (two CTAs per SM) holding the (member, query head) rows
// of 128 / G members of a group, over one partition of the group's shared
// prefix.
int shared_prefix_members_per_cta(int group) { return kTcRows / group; }

cudaError_t launch_shared_prefix(const DecodeArgs &d, const void *k_cache, const void *v_cache,
                                 int64_t pool_rows, int head_dim, int dtype, bool kv_fp8,
                                 cudaStream_t stream, bool *map_failed) {
  CUtensorMap km, vm;
  *map_failed = false;
  if (!encode_pool_map(&km, k_cache, pool_rows, head_dim, dtype, kv_fp8) ||
      !encode_pool_map(&vm, v_cache, pool_rows, head_dim, dtype, kv_fp8)) {
    *map_failed = true;
    return cudaErrorInvalidValue;
  }
  PrefillArgs a{};
  a.query = d.query;
  a.block_tables = d.block_tables;
  a.context_lens = d.context_lens;
  a.max_blocks_per_seq = d.max_blocks_per_seq;
  a.num_seqs = d.num_seqs;
  a.num_q_heads = d.num_q_heads;
  a.num_kv_heads = d.num_kv_heads;
  a.group = d.group;
  a.bs_log2 = d.bs_log2;
  a.num_blocks = d.num_blocks;
  a.scale_log2 = d.scale_log2;
  a.out_scale = d.out_scale;
  a.err = d.err;
  a.ws_m = d.ws_m;
  a.ws_l = d.ws_l;
  a.ws_o = d.ws_o;
  a.prefix_lens = d.prefix_lens;
  a.group_start = d.group_start;
  a.num_groups = d.num_groups;
  a.max_group_size = d.max_group_size;
  a.members_per_cta = d.members_per_cta;
  a.chunks = d.chunks;
  a.part_tokens = d.part_tokens;
  a.num_parts = d.num_parts;
  a.max_context_len = d.max_context_len;
  constexpr int KS = PA_PREFILL_SOLO_KSTAGES, VS = PA_PREFILL_SOLO_VSTAGES;
  if (kv_fp8) {
    if (dtype == 0)
      return head_dim == 128
                 ? launch_prefill_tc_pair_t<__half, 128, KS, VS, false, 1, true, true>(a, km, vm,
                                                                                       stream)
                 : launch_prefill_tc_pair_t<__half, 64, KS, VS, false, 1, true, true>(a, km, vm,
                                                                                      stream);
    return head_dim == 128
               ? launch_prefill_tc_pair_t<__nv_bfloat16, 128, KS, VS, false, 1, true, true>(
                     a, km, vm, stream)
               : launch_prefill_tc_pair_t<__nv_bfloat16, 64, KS, VS, false, 1, true, true>(
                     a, km, vm, stream);
  }
  if (dtype == 0)
    return head_dim == 128
               ? launch_prefill_tc_pair_t<__half, 128, KS, VS, false, 1, true>(a, km, vm, stream)
               : launch_prefill_tc_pair_t<__half, 64, KS, VS, false, 1, true>(a, km, vm, stream);
  return head_dim == 128
             ? launch_prefill_tc_pair_t<__nv_bfloat16, 128, KS, VS, true, 1, true>(a, km, vm, stream)
             : launch_prefill_tc_pair_t<__nv_bfloat16, 64, KS, VS, true, 1, true>(a, km, vm, stream);
}

}  // namespace pa
