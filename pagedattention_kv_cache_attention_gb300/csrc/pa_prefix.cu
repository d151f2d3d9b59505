// pa_prefix.cu -- decode attention over the shared prefix of groups of
// sequences whose block tables point at the same physical blocks.
//
// Copy-on-write block sharing ("LLM Serving Engine Shootout", 3.2 Copy-on-Write
// and 4 RadixAttention; "Serving engines", How vLLM works) lets many sequences
// reference one copy of a prefix's K/V.  The plain decode kernel still reads
// those blocks once per sequence (the L2 serves the repeats when it can hold
// them).  Here each K/V sub-tile of a group's prefix leaves memory once per
// group: one CTA serves up to 32 query columns -- (member sequence, query head)
// pairs of one KV head -- so every staged tile feeds four MMA column tiles.
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
// CTA (partition p, KV head, chunk of a group): four warps; warp w owns MMA
// column tile w (columns 8w .. 8w+7, column = member * G + query head).  One
// ring of four shared-memory stages, two 16-token sub-tiles of K and V each,
// feeds all four warps.  A stage is refilled by the warp that releases it last
// (a counter per stage), so no warp ever waits for another.  The partition's
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

constexpr int kPxWarps = 4;                                // MMA column tiles per CTA
constexpr int kPxStages = 4;                               // ring stages
constexpr int kPxNsub = 2;                                 // sub-tiles per stage
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
  constexpr int NW = kPxWarps, S = kPxStages, NSUB = kPxNsub;
  constexpr int kStepBytes = 2 * NSUB * Sh::kTileBytes;  // K and V of one stage
  extern __shared__ uint8_t smem_raw[];
  // 128-byte swizzled TMA destinations need 1024-byte alignment.
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + S * kStepBytes);  // [S] data landed
  unsigned *released = reinterpret_cast<unsigned *>(full + S);          // [S] warps done
  int *last_issued = reinterpret_cast<int *>(released + S);  // [S] last step loaded per stage
  int *row_of = last_issued + S;       // [kPxMaxSub] pool row of each sub-tile, -1 = skip
  int *first_of = row_of + kPxMaxSub;  // [32] first_m of each member of this CTA
  int *ctl = first_of + 32;            // source member, member count, first member, timeout

  const int p = blockIdx.x, kvh = blockIdx.y;
  const int grp = blockIdx.z / a.chunks, chunk = blockIdx.z % a.chunks;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int G = a.group, P = a.part_tokens;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      released[s] = 0;
      last_issued[s] = -1;
    }
    ctl[3] = 0;
    fence_barrier_init();
  }

  // tables, lengths and the pool may come from the kernel launched just before
  grid_dependency_wait();

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
  __syncthreads();
  const int src = ctl[0];
  if (src < 0) return;  // no member takes this partition from here (uniform)
  const int nm = ctl[1], m0 = ctl[2];

  // ---- the partition's sub-tiles: pool rows from the source member's table.
  // p < first_src <= np_src - 1, so the partition ends inside the source's
  // context and every entry read is inside its table row.
  const int n_sub = P / kTile;
  const int t0 = p * P;
  const int bs_mask = (1 << a.bs_log2) - 1;
  const int32_t *src_row =
      a.block_tables + static_cast<int64_t>(m0 + src) * a.max_blocks_per_seq;
  for (int u = threadIdx.x; u < n_sub; u += NW * 32) {
    const int t = t0 + u * kTile;
    const int phys = src_row[t >> a.bs_log2];
    int row = -1;
    if (phys >= 0 && static_cast<int64_t>(phys) < a.num_blocks)
      row = ((phys * a.num_kv_heads + kvh) << a.bs_log2) + (t & bs_mask);
    else
      atomicOr(a.err, kErrBadBlock);
    row_of[u] = row;
  }
  // every other taker must reference the same blocks (checked once per partition)
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
  __syncthreads();

  const uint64_t policy = a.chunks > 1 ? l2_policy_evict_normal() : l2_policy_evict_first();
  const int n_steps = (n_sub + NSUB - 1) / NSUB;
  // start loading the sub-tiles of step k into stage s (one thread)
  auto issue = [&](int k, int s) {
    int rows[NSUB];
    uint32_t bytes = 0;
#pragma unroll
    for (int h = 0; h < NSUB; ++h) {
      const int u = k * NSUB + h;
      rows[h] = u < n_sub ? row_of[u] : -1;
      bytes += rows[h] >= 0 ? 2 * Sh::kTileBytes : 0;
    }
    last_issued[s] = k;
    if (bytes == 0) {
      mbar_arrive(&full[s]);  // nothing to load: complete the phase at once
      return;
    }
    mbar_arrive_expect_tx(&full[s], bytes);
    uint8_t *st = smem + s * kStepBytes;
#pragma unroll
    for (int h = 0; h < NSUB; ++h) {
      if (rows[h] < 0) continue;
#pragma unroll
      for (int b = 0; b < Sh::kBoxes; ++b) {
        tma_load_2d(st + h * Sh::kTileBytes + b * Sh::kBoxBytes, &kmap, b * Sh::kBoxElems,
                    rows[h], &full[s], policy);
        tma_load_2d(st + (NSUB + h) * Sh::kTileBytes + b * Sh::kBoxBytes, &vmap,
                    b * Sh::kBoxElems, rows[h], &full[s], policy);
      }
    }
  };
  if (threadIdx.x == 0) {
    for (int s = 0; s < S && s < n_steps; ++s) issue(s, s);
  }

  // query fragment of column g of this warp's tile (zero for padding columns)
  const int col = warp * 8 + g;
  const int mi = col / G;
  uint4 qf[Sh::kQChunks];
  load_q_16<T, D>(mi < nm ? static_cast<const T *>(a.query) +
                                (static_cast<int64_t>(m0 + mi) * a.num_q_heads + kvh * G +
                                 col % G) * D
                          : nullptr,
                  c, qf);

  float m0r = -INFINITY, m1r = -INFINITY, l0 = 0.f, l1 = 0.f;  // columns 2c, 2c+1
  float acc[Sh::kMTiles][4];
#pragma unroll
  for (int mt = 0; mt < Sh::kMTiles; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;

  bool timed_out = false;
#pragma unroll 1
  for (int k = 0; k < n_steps; ++k) {
    const int s = k % S;
    if (!__all_sync(kFull, mbar_wait_bounded(&full[s], (k / S) & 1))) {
      if (lane == 0) atomicOr(a.err, kErrTimeout);
      timed_out = true;
      break;
    }
    const uint8_t *stage = smem + s * kStepBytes;
    int nvalid[NSUB];
#pragma unroll
    for (int h = 0; h < NSUB; ++h) {
      const int u = k * NSUB + h;
      nvalid[h] = u < n_sub && row_of[u] >= 0 ? kTile : 0;
    }
    float sc[NSUB][4];
#pragma unroll
    for (int h = 0; h < NSUB; ++h) qk_subtile_16<T, D>(stage + h * Sh::kTileBytes, qf, g, c, sc[h]);
    float pr[NSUB][4];
    softmax_step<NSUB, Sh::kMTiles>(sc, nvalid, g, a.scale_log2, m0r, m1r, l0, l1, acc, pr);
#pragma unroll
    for (int h = 0; h < NSUB; ++h) {
      uint32_t pb0, pb1, pq0, pq1;
      p_operands<T>(pr[h], pb0, pb1, pq0, pq1);
      pv_subtile_16<T, D>(stage + (NSUB + h) * Sh::kTileBytes, nvalid[h], g, c, pb0, pb1, pq0,
                          pq1, acc);
    }

    // release the stage; the warp that releases it last refills it with step
    // k + S.  The fences order every warp's reads of the stage (made before
    // its release) before the refill's asynchronous-proxy writes.
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      const unsigned prev = atomicAdd(&released[s], 1u);
      if (prev == NW - 1) {
        released[s] = 0;
        __threadfence_block();
        if (k + S < n_steps) {
          fence_proxy_async_smem();
          issue(k + S, s);
        }
      }
    }
  }

  // ---- partials of the columns whose member takes this partition from here
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(kFull, l0, off);
    l1 += __shfl_xor_sync(kFull, l1, off);
  }
  const int cA = warp * 8 + 2 * c, cB = cA + 1;
  const int iA = cA / G, iB = cB / G;
  const bool okA = !timed_out && iA < nm && p < first_of[iA];
  const bool okB = !timed_out && iB < nm && p < first_of[iB];
  const int64_t prA =
      ((static_cast<int64_t>(m0 + iA) * a.num_q_heads + kvh * G + cA % G) * a.num_parts) + p;
  const int64_t prB =
      ((static_cast<int64_t>(m0 + iB) * a.num_q_heads + kvh * G + cB % G) * a.num_parts) + p;
  if (g == 0) {
    if (okA) {
      a.ws_m[prA] = m0r;
      a.ws_l[prA] = l0;
    }
    if (okB) {
      a.ws_m[prB] = m1r;
      a.ws_l[prB] = l1;
    }
  }
  const float invA = l0 > 0.f ? 1.f / l0 : 0.f;
  const float invB = l1 > 0.f ? 1.f / l1 : 0.f;
  store_partial_o<D, false>(okA ? a.ws_o + prA * D : nullptr, okB ? a.ws_o + prB * D : nullptr,
                            okA, okB, acc, invA, invB, g);
  grid_launch_dependents();

  if (timed_out && lane == 0) atomicOr(&ctl[3], 1);
  __syncthreads();
  if (ctl[3] && threadIdx.x == 0) {
    // a wait ran out: let every copy already issued land before the CTA
    // leaves (bounded again)
    for (int s = 0; s < S; ++s)
      if (last_issued[s] >= 0) (void)mbar_wait_bounded(&full[s], (last_issued[s] / S) & 1);
  }
}

template <typename T, int D>
cudaError_t launch_prefix_t(const DecodeArgs &a, const CUtensorMap &km, const CUtensorMap &vm,
                            cudaStream_t stream) {
  constexpr size_t step = 2 * kPxNsub * Shape<D, false>::kTileBytes;
  constexpr size_t smem =
      1024 + kPxStages * step + kPxStages * (8 + 4 + 4) + (kPxMaxSub + 32 + 4) * 4;
  auto kern = pa_shared_prefix_kernel<T, D>;
  static SmemLimitOnce smem_limit;
  const cudaError_t e = smem_limit.ensure(kern, smem);
  if (e != cudaSuccess) return e;
  return launch_dependent(
      kern,
      dim3(static_cast<unsigned>(a.num_parts), static_cast<unsigned>(a.num_kv_heads),
           static_cast<unsigned>(a.num_groups * a.chunks)),
      dim3(kPxWarps * 32), smem, stream, km, vm, a);
}

}  // namespace

int shared_prefix_members_per_cta(int group) { return 8 * kPxWarps / group; }

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
