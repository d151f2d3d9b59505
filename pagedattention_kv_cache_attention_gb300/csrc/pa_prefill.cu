// pa_prefill.cu -- chunked-prefill attention over the paged pool.
//
// What is computed ("Serving engines", How vLLM works: chunked prefill cuts a
// prompt into pieces that run alongside decode steps; "LLM Serving Engine
// Shootout", 1: prefill attends over every prompt token): sequence i appends
// a chunk of q_len_i tokens whose K/V are already in the cache; chunk row t
// sits at position p = ctx_i - q_len_i + t and attends causally to tokens
// 0..p, read through the block table exactly as decode reads them.
//
// How (sm_103a, warp-level tensor-core MMA):
//  * One CTA per (query tile, KV head, sequence).  Its 64 query rows are
//    (token, head) pairs of one KV head's group -- 64 / G tokens x G heads -- so
//    every K/V tile it stages serves the whole group.  Warp w owns rows
//    16w .. 16w+15.
//  * K/V 16-token sub-tiles move by 2-D TMA (128-byte swizzle) into a ring of
//    S stages shared by the CTA: a "full" mbarrier per stage counts the bytes,
//    an "empty" mbarrier per stage counts the four warps that are done with it;
//    thread 0 refills a stage once it is empty.  Block ids for the next 32
//    sub-tiles sit in warp 0's lanes.
//  * S = Q K^T per warp on mma.sync m16n8k16 (fp32 accumulate): Q rows are the
//    A operand (in registers for the whole kernel), each 8-key half of the
//    sub-tile the B operand, read from swizzled shared memory with the same
//    conflict-free chunk order the decode kernel uses.
//  * Causal mask and fp32 online softmax per row (two shuffles per row max);
//    the accumulator fragments of S are already the A-operand fragments of P,
//    carried as hi + lo parts for precision.  O += P V with V as the B
//    operand assembled by byte permutes from 16-byte shared loads.
//  * Keys past the context (tail slots) get a zero V row, so whatever they
//    hold cannot reach the output.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kTile = 16;
constexpr unsigned kFull = 0xffffffffu;

// chunk (8 elements) of a head_dim row that lane column c reads in k step pair i
__device__ __forceinline__ int k_chunk(int i, int c) { return 2 * c + (i & 1) + 8 * (i >> 1); }

template <typename T, int D, int NW, int S>
__global__ void __launch_bounds__(NW * 32)
    pa_prefill_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const PrefillArgs a) {
  constexpr int kBoxes = D / 64;
  constexpr int kBoxBytes = kTile * 128;
  constexpr int kTileBytes = kTile * D * 2;
  constexpr int kStageBytes = 2 * kTileBytes;
  constexpr int kChunks = D / 32;   // 16-byte chunk pairs per lane
  constexpr int kNTiles = D / 8;    // n8 tiles of the P.V product
  constexpr int kRows = NW * 16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + S * kStageBytes);
  uint64_t *empty = full + S;
  int *stage_valid = reinterpret_cast<int *>(empty + S);  // the stage's block id was valid

  const int tile = blockIdx.x, kvh = blockIdx.y, seq = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int G = a.group;
  const int tpc = kRows / G;  // query tokens per CTA

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NW);
    }
    fence_barrier_init();
  }
  __syncthreads();
  grid_dependency_wait();  // the pool (the chunk's K/V above all) may come from the kernel before

  const int q0 = a.query_start[seq];
  const int q_len = a.query_start[seq + 1] - q0;
  const int ctx = a.context_lens[seq];
  if (q_len < 0 || ctx < q_len || ctx > (a.max_blocks_per_seq << a.bs_log2) ||
      q_len > a.max_q_len) {
    if (threadIdx.x == 0 && tile == 0 && kvh == 0) atomicOr(a.err, kErrBadLen);
    return;
  }
  const int t_first = tile * tpc;
  if (t_first >= q_len) return;
  const int t_last = min(q_len, t_first + tpc) - 1;
  const int base_pos = ctx - q_len;                // position of chunk row 0
  const int n_keys = base_pos + t_last + 1;        // keys the CTA needs
  const int n_sub = (n_keys + kTile - 1) / kTile;

  // this thread's rows: A = 16w + g, B = A + 8
  auto row_token = [&](int r) { return t_first + r / G; };
  const int rA = warp * 16 + g, rB = rA + 8;
  const bool okA = rA < tpc * G && row_token(rA) <= t_last;
  const bool okB = rB < tpc * G && row_token(rB) <= t_last;
  const int posA = base_pos + row_token(rA), posB = base_pos + row_token(rB);
  // the warp's last position decides how many sub-tiles it computes on
  int wlast = -1;
  {
    const int r_hi = min(warp * 16 + 15, tpc * G - 1);
    if (warp * 16 <= r_hi) wlast = base_pos + min(row_token(r_hi), t_last);
  }
  const int w_sub = wlast >= 0 ? wlast / kTile + 1 : 0;

  // Q fragments (A operand): rows A and B, chunks k_chunk(i, c)
  uint4 qa[kChunks], qb[kChunks];
  {
    const T *qA = static_cast<const T *>(a.query) +
                  (static_cast<int64_t>(q0 + row_token(rA)) * a.num_q_heads + kvh * G + rA % G) * D;
    const T *qB = static_cast<const T *>(a.query) +
                  (static_cast<int64_t>(q0 + row_token(rB)) * a.num_q_heads + kvh * G + rB % G) * D;
#pragma unroll
    for (int i = 0; i < kChunks; ++i) {
      qa[i] = okA ? *reinterpret_cast<const uint4 *>(qA + k_chunk(i, c) * 8) : make_uint4(0, 0, 0, 0);
      qb[i] = okB ? *reinterpret_cast<const uint4 *>(qB + k_chunk(i, c) * 8) : make_uint4(0, 0, 0, 0);
    }
  }

  const int32_t *bt_row = a.block_tables + static_cast<int64_t>(seq) * a.max_blocks_per_seq;
  const int bs_mask = (1 << a.bs_log2) - 1;
  auto block_of = [&](int u) -> int {  // sub-tile u's physical block, -1 if invalid (flagged)
    if (u >= n_sub) return -1;
    const int phys = bt_row[(u * kTile) >> a.bs_log2];
    if (phys < 0 || static_cast<int64_t>(phys) >= a.num_blocks) {
      atomicOr(a.err, kErrBadBlock);
      return -1;
    }
    return phys;
  };
  const uint64_t policy = l2_policy_evict_first();
  auto issue = [&](int u, int phys, int s) {  // thread 0
    stage_valid[s] = phys >= 0;                // published by the barrier arrive below
    if (phys < 0) {
      mbar_arrive(&full[s]);
      return;
    }
    mbar_arrive_expect_tx(&full[s], kStageBytes);
    const int y = ((phys * a.num_kv_heads + kvh) << a.bs_log2) + ((u * kTile) & bs_mask);
    uint8_t *st = smem + s * kStageBytes;
#pragma unroll
    for (int b = 0; b < kBoxes; ++b) {
      tma_load_2d(st + b * kBoxBytes, &kmap, b * 64, y, &full[s], policy);
      tma_load_2d(st + kTileBytes + b * kBoxBytes, &vmap, b * 64, y, &full[s], policy);
    }
  };
  // warp 0 keeps the block ids of sub-tiles [win_base, win_base + 32)
  int win_base = 0, win = -1;
  if (warp == 0) {
    win = block_of(lane);
#pragma unroll
    for (int s = 0; s < S; ++s) {
      if (s < n_sub) {
        const int phys = __shfl_sync(kFull, win, s);
        if (lane == 0) issue(s, phys, s);
      }
    }
  }

  const float NEG_INF = -INFINITY;
  float mA = NEG_INF, mB = NEG_INF, lA = 0.f, lB = 0.f;
  float acc[kNTiles][4];
#pragma unroll
  for (int n = 0; n < kNTiles; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
  bool timed_out = false;
  int k_stop = n_sub;

#pragma unroll 1
  for (int k = 0; k < n_sub; ++k) {
    const int s = k % S;
    const uint32_t parity = (k / S) & 1;
    if (!__all_sync(kFull, mbar_wait_bounded(&full[s], parity))) {
      if (lane == 0) atomicOr(a.err, kErrTimeout);
      timed_out = true;
      k_stop = k;
      break;
    }
    const int key0 = k * kTile;
    if (k < w_sub) {
      const uint8_t *Ks = smem + s * kStageBytes;
      const uint8_t *Vs = Ks + kTileBytes;
      // a sub-tile whose block id was invalid was never loaded: its keys are masked
      const bool tile_ok = stage_valid[s] != 0;
      // ---- S = Q K^T for keys key0 + 0..7 (j = 0) and key0 + 8..15 (j = 1)
      float sc[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
        for (int i = 0; i < kChunks; ++i) {
          const int ch = k_chunk(i, c);
          const int row = j * 8 + g;  // key row; (row & 7) = g
          const uint4 kv = *reinterpret_cast<const uint4 *>(Ks + (ch >> 3) * kBoxBytes + row * 128 +
                                                            (((ch & 7) ^ g) << 4));
          Elem<T>::mma(sc[j], qa[i].x, qb[i].x, qa[i].y, qb[i].y, kv.x, kv.y);
          Elem<T>::mma(sc[j], qa[i].z, qb[i].z, qa[i].w, qb[i].w, kv.z, kv.w);
        }
      }
      // ---- causal mask + online softmax (rows A and B; keys 2c, 2c+1 of each half)
      float x[2][4];
      float mxA = NEG_INF, mxB = NEG_INF;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = key0 + j * 8 + 2 * c + e;
          x[j][e] = (okA && tile_ok && key <= posA) ? sc[j][e] * a.scale_log2 : NEG_INF;
          x[j][2 + e] = (okB && tile_ok && key <= posB) ? sc[j][2 + e] * a.scale_log2 : NEG_INF;
          mxA = fmaxf(mxA, x[j][e]);
          mxB = fmaxf(mxB, x[j][2 + e]);
        }
      }
#pragma unroll
      for (int off = 1; off < 4; off <<= 1) {
        mxA = fmaxf(mxA, __shfl_xor_sync(kFull, mxA, off));
        mxB = fmaxf(mxB, __shfl_xor_sync(kFull, mxB, off));
      }
      const float nA = fmaxf(mA, mxA), nB = fmaxf(mB, mxB);
      const float refA = nA == NEG_INF ? 0.f : nA, refB = nB == NEG_INF ? 0.f : nB;
      const float alA = exp2f(mA - refA), alB = exp2f(mB - refB);
      float p[2][4];
      float sA = 0.f, sB = 0.f;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        p[j][0] = exp2f(x[j][0] - refA);
        p[j][1] = exp2f(x[j][1] - refA);
        p[j][2] = exp2f(x[j][2] - refB);
        p[j][3] = exp2f(x[j][3] - refB);
        sA += p[j][0] + p[j][1];
        sB += p[j][2] + p[j][3];
      }
      lA = lA * alA + sA;
      lB = lB * alB + sB;
      mA = nA;
      mB = nB;
      if (__any_sync(kFull, alA != 1.f || alB != 1.f)) {
#pragma unroll
        for (int n = 0; n < kNTiles; ++n) {
          acc[n][0] *= alA;
          acc[n][1] *= alA;
          acc[n][2] *= alB;
          acc[n][3] *= alB;
        }
      }
      // P as the A operand (rows A/B x keys 2c,2c+1 | 8+2c, 8+2c+1), hi + lo parts
      uint32_t ph[4], pl[4];
      {
        const float v[4][2] = {{p[0][0], p[0][1]}, {p[0][2], p[0][3]},
                               {p[1][0], p[1][1]}, {p[1][2], p[1][3]}};
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          ph[r] = Elem<T>::pack(v[r][0], v[r][1]);
          const float2 f = Elem<T>::unpack(ph[r]);
          pl[r] = Elem<T>::pack(v[r][0] - f.x, v[r][1] - f.y);
        }
      }
      // ---- O += P V: V keys 2c, 2c+1, 2c+8, 2c+9 (zero past the keys the CTA needs)
      uint4 vv[4][kBoxes];
#pragma unroll
      for (int ri = 0; ri < 4; ++ri) {
        const int r = 2 * c + (ri & 1) + 8 * (ri >> 1);
        const bool keep = tile_ok && key0 + r < n_keys;
#pragma unroll
        for (int b = 0; b < kBoxes; ++b) {
          const uint4 xv = *reinterpret_cast<const uint4 *>(Vs + b * kBoxBytes + r * 128 +
                                                            ((g ^ (r & 7)) << 4));
          vv[ri][b] = keep ? xv : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int n = 0; n < kNTiles; ++n) {
        // n-tile n, column g: dim 8g + n (first 8 tiles) or 64 + 8g + (n - 8)
        const int b = n / 8, e = n % 8;
        const uint32_t b0 = pair_of(vv[0][b], vv[1][b], e);
        const uint32_t b1 = pair_of(vv[2][b], vv[3][b], e);
        Elem<T>::mma(acc[n], ph[0], ph[1], ph[2], ph[3], b0, b1);
        Elem<T>::mma(acc[n], pl[0], pl[1], pl[2], pl[3], b0, b1);
      }
    }
    // ---- release the stage; thread 0 refills it once every warp has
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (warp == 0) {
      const int nk = k + S;
      if (nk < n_sub) {
        if (nk >= win_base + 32) {
          win_base += 32;
          win = block_of(win_base + lane);
        }
        const int phys = __shfl_sync(kFull, win, nk - win_base);
        if (lane == 0) {
          if (mbar_wait_bounded(&empty[s], parity)) {
            fence_proxy_async_smem();
            issue(nk, phys, s);
          } else {
            atomicOr(a.err, kErrTimeout);
            mbar_arrive(&full[s]);  // let the consumers through; results are flagged
          }
        }
      }
    }
  }
  if (timed_out) {
    // let copies already in flight land before the CTA leaves (bounded again)
    for (int kk = k_stop; kk < min(k_stop + S, n_sub); ++kk)
      (void)mbar_wait_bounded(&full[kk % S], (kk / S) & 1);
  }

  // ---- row sums over the four lanes of a row, normalise, write
#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    lA += __shfl_xor_sync(kFull, lA, off);
    lB += __shfl_xor_sync(kFull, lB, off);
  }
  const float invA = lA > 0.f ? 1.f / lA : 0.f, invB = lB > 0.f ? 1.f / lB : 0.f;
  // output dims of this thread: n-tiles 0..7 give 16c + n (col 2c) and 16c + 8 + n (col 2c+1)
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const bool ok = half == 0 ? okA : okB;
    if (!ok) continue;
    const int r = half == 0 ? rA : rB;
    const float inv = half == 0 ? invA : invB;
    T *orow = static_cast<T *>(a.out) +
              (static_cast<int64_t>(q0 + row_token(r)) * a.num_q_heads + kvh * G + r % G) * D;
#pragma unroll
    for (int grp = 0; grp < kNTiles / 8; ++grp) {
      uint32_t w[8];
#pragma unroll
      for (int n = 0; n < 8; n += 2) {
        const float* a0 = acc[grp * 8 + n];
        const float* a1 = acc[grp * 8 + n + 1];
        w[n / 2] = Elem<T>::pack(a0[2 * half] * inv, a1[2 * half] * inv);          // dims 16c + n, +1
        w[4 + n / 2] = Elem<T>::pack(a0[2 * half + 1] * inv, a1[2 * half + 1] * inv);  // 16c + 8 + n
      }
      uint4 *dst = reinterpret_cast<uint4 *>(orow + grp * 64 + 16 * c);
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
  }
  grid_launch_dependents();
}

template <typename T, int D, int NW, int S>
cudaError_t launch_prefill_t(const PrefillArgs &a, const CUtensorMap &km, const CUtensorMap &vm,
                             cudaStream_t stream) {
  constexpr size_t smem = 1024 + static_cast<size_t>(S) * 2 * kTile * D * 2 + 2 * S * 8 + S * 4;
  auto kern = pa_prefill_kernel<T, D, NW, S>;
  static SmemLimitOnce smem_limit;
  const cudaError_t e = smem_limit.ensure(kern, smem);
  if (e != cudaSuccess) return e;
  const int tpc = NW * 16 / a.group;
  const int tiles = (a.max_q_len + tpc - 1) / tpc;
  return launch_dependent(kern, dim3(tiles, a.num_kv_heads, a.num_seqs), dim3(NW * 32), smem,
                          stream, km, vm, a);
}

}  // namespace

bool encode_pool_map(CUtensorMap *map, const void *pool, int64_t rows, int head_dim, int dtype,
                     bool fp8);
bool prefill_tc_supported(int head_dim, int group);
cudaError_t launch_prefill_tc(const PrefillArgs &a, const CUtensorMap &km, const CUtensorMap &vm,
                              int dtype, cudaStream_t stream);

constexpr int kPrefillWarps = 4;
constexpr int kPrefillStages = 4;

cudaError_t launch_prefill(const PrefillArgs &a, const void *k_cache, const void *v_cache,
                           int64_t pool_rows, int head_dim, int dtype, cudaStream_t stream,
                           bool *map_failed) {
  CUtensorMap km, vm;
  *map_failed = false;
  if (!encode_pool_map(&km, k_cache, pool_rows, head_dim, dtype, false) ||
      !encode_pool_map(&vm, v_cache, pool_rows, head_dim, dtype, false)) {
    *map_failed = true;
    return cudaErrorInvalidValue;
  }
  if (a.max_q_len == 0) return cudaSuccess;
  // head_dim 128 with a power-of-two group runs on the tcgen05 kernel
  if (a.use_tc && prefill_tc_supported(head_dim, a.group))
    return launch_prefill_tc(a, km, vm, dtype, stream);
  if (dtype == 0)
    return head_dim == 128
               ? launch_prefill_t<__half, 128, kPrefillWarps, kPrefillStages>(a, km, vm, stream)
               : launch_prefill_t<__half, 64, kPrefillWarps, kPrefillStages>(a, km, vm, stream);
  return head_dim == 128
             ? launch_prefill_t<__nv_bfloat16, 128, kPrefillWarps, kPrefillStages>(a, km, vm,
                                                                                   stream)
             : launch_prefill_t<__nv_bfloat16, 64, kPrefillWarps, kPrefillStages>(a, km, vm,
                                                                                  stream);
}

}  // namespace pa
