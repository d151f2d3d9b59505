// pa_internal.h -- argument blocks and launchers shared by the library's
// translation units (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

namespace pa {

constexpr int kMaxDevices = 64;

// Raises one kernel's dynamic shared-memory limit once per device.  Safe when
// several host threads make their first call at the same time: the attribute
// is set under a lock, and later calls only read an atomic flag.  Each
// launcher keeps one function-local static instance per kernel.
class SmemLimitOnce {
 public:
  template <typename Kern>
  cudaError_t ensure(Kern kern, size_t bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (done_[dev].load(std::memory_order_acquire)) return cudaSuccess;
    std::lock_guard<std::mutex> lk(mu_);
    if (!done_[dev].load(std::memory_order_relaxed)) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(bytes));
      if (e != cudaSuccess) return e;
      done_[dev].store(true, std::memory_order_release);
    }
    return cudaSuccess;
  }

 private:
  std::atomic<bool> done_[kMaxDevices]{};
  std::mutex mu_;
};

struct DecodeArgs {
  void *out;                    // [B, Hq, D] (used when num_parts == 1)
  const void *query;            // [B, Hq, D]
  const int32_t *block_tables;  // [B, max_blocks_per_seq]
  const int32_t *context_lens;  // [B]
  int max_blocks_per_seq;
  int num_seqs, num_q_heads, num_kv_heads, group, bs_log2;
  int64_t num_blocks;
  float scale_log2;             // scale * log2(e) (times the K dequantisation scale for FP8)
  float out_scale;              // V dequantisation scale for FP8, 1 otherwise
  int max_context_len;
  int part_tokens;              // tokens per partition (>= max_context_len when not split)
  int num_parts;
  float *ws_m, *ws_l, *ws_o;    // split partials (num_parts > 1)
  unsigned *ws_cnt;             // join counters, one per (sequence, KV head) (num_parts > 1)
  int fuse_join;                // 1: the last partition CTA of a (sequence, KV head) joins
  unsigned *err;                // device error word
  // Shared-prefix decode (nullptr / unused otherwise).  prefix_lens [B]:
  // leading tokens of each sequence held in the same physical blocks as the
  // rest of its group; group_start [num_groups + 1]: the groups are runs of
  // consecutive sequences.
  const int32_t *prefix_lens;
  const int32_t *group_start;
  int num_groups, max_group_size;
  int members_per_cta, chunks;  // sequences per shared-prefix CTA, CTAs per group
};

struct ReduceArgs {
  void *out;
  const float *ws_m, *ws_l, *ws_o;
  const int32_t *context_lens;
  int num_seqs, num_q_heads, num_parts, partition_size, max_context_len;
  // tokens the block table can address (max_blocks_per_seq * block_size); a
  // longer context is treated as invalid exactly as the decode kernel treats
  // it (INT32_MAX when the partials do not come from pa_decode)
  int64_t table_tokens;
  int warps_per_row;            // 1, 2 or 4 warps join one row
  unsigned *err;
};

struct ReshapeArgs {
  // FP8 caches: elements are stored as E4M3 codes of x / scale
  bool to_fp8;
  int src_dtype;                     // fp16 / bf16 source rows when to_fp8
  float k_scale, v_scale;
  const void *key, *value;
  int64_t key_stride, value_stride;  // elements
  void *k_cache, *v_cache;
  const int64_t *slot_mapping;
  int num_tokens, num_kv_heads, head_dim, block_size;
  int64_t num_blocks;
  unsigned *err;
};

struct PrefillArgs {
  void *out;                    // [total_q, Hq, D]
  const void *query;            // [total_q, Hq, D]
  const int32_t *query_start;   // [B + 1]
  const int32_t *block_tables;  // [B, max_blocks_per_seq]
  const int32_t *context_lens;  // [B], the chunk included
  int max_blocks_per_seq;
  int num_seqs, num_q_heads, num_kv_heads, group, bs_log2, max_q_len;
  int64_t num_blocks;
  float scale_log2;             // scale * log2(e) (times the K dequantisation scale for FP8)
  float out_scale;              // V dequantisation scale for FP8 caches, 1 otherwise
  unsigned *err;
  // The shared-prefix pass (the same kernel over a group's shared prefix):
  // rows are (member, query head) pairs of a group's sequences, keys the
  // partition [p part_tokens, (p + 1) part_tokens) read through the first
  // taking member's table, and each taking member's rows are written as split
  // partials (m, l, o) into the decode workspace.  Unused by pa_prefill.
  float *ws_m, *ws_l, *ws_o;
  const int32_t *prefix_lens, *group_start;
  int num_groups, max_group_size, members_per_cta, chunks;
  int part_tokens, num_parts, max_context_len;
};

struct BlockCopyArgs {
  const void *src[2];           // per tensor: source pool (device or mapped host memory)
  void *dst[2];                 // per tensor: destination pool
  const int64_t *mapping;       // [num_pairs, 2] (source block, destination block)
  int num_pairs;
  int64_t block_bytes;          // bytes of one block (multiple of 16)
  int64_t src_blocks, dst_blocks;
  unsigned *err;
};

// Launch `kern` on `stream` as a programmatic dependent of the work before it:
// it may start while the previous kernel finishes, and must call
// griddepcontrol.wait before reading anything that kernel writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// Largest partition size the shared-prefix kernel takes (its shared-memory
// table holds one pool row per 16-token sub-tile of a partition).
constexpr int kMaxSharedPrefixPartition = 8192;

// The pool viewed as a 2-D tensor [num_blocks * num_kv_heads * block_size
// rows, head_dim] for TMA loads of 16-row, 128-byte boxes (128-byte swizzle).
bool encode_pool_map(CUtensorMap *map, const void *pool, int64_t rows, int head_dim, int dtype,
                     bool fp8);

// kv_fp8: the caches hold FP8 E4M3 codes (queries and output fp16).
cudaError_t launch_decode(const DecodeArgs &a, const void *k_cache, const void *v_cache,
                          int64_t pool_rows, int head_dim, int dtype, bool kv_fp8,
                          cudaStream_t stream, bool *map_failed);
cudaError_t launch_reduce(const ReduceArgs &a, int head_dim, int dtype, cudaStream_t stream);
// The shared-prefix pass of pa_decode_shared_prefix (16-bit or FP8 caches);
// the decode launch with a.prefix_lens set follows it on the same stream.
cudaError_t launch_shared_prefix(const DecodeArgs &a, const void *k_cache, const void *v_cache,
                                 int64_t pool_rows, int head_dim, int dtype, bool kv_fp8,
                                 cudaStream_t stream, bool *map_failed);
// Sequences of one group that a shared-prefix CTA serves at query group size G.
int shared_prefix_members_per_cta(int group);
cudaError_t launch_reshape(const ReshapeArgs &a, cudaStream_t stream);
cudaError_t launch_block_copy(const BlockCopyArgs &a, int num_tensors, cudaStream_t stream);
cudaError_t launch_prefill(const PrefillArgs &a, const void *k_cache, const void *v_cache,
                           int64_t pool_rows, int head_dim, int dtype, bool kv_fp8,
                           cudaStream_t stream, bool *map_failed);

// The host-side checks of pa_decode that come before the workspace check;
// returns a pa_status value (PA_OK when pa_decode would go on to the workspace).
int32_t decode_check_args(const void *out, const void *query, const void *k_cache,
                          const void *v_cache, const int32_t *block_tables,
                          int32_t max_blocks_per_seq, const int32_t *context_lens,
                          int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                          int32_t head_dim, int32_t block_size, int64_t num_blocks, float scale,
                          int32_t max_context_len, int32_t partition_size, int32_t dtype);

// One CTA waiting on a barrier nothing completes (the wait-limit self-test).
cudaError_t launch_selftest_wait(unsigned *err, cudaStream_t stream);

}  // namespace pa
