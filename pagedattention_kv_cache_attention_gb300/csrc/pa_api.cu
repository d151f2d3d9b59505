// pa_api.cu -- the C ABI declared in include/pa.h: host-side argument checks,
// launch selection and the per-device error word.  Nothing here allocates
// device memory; every compute call only enqueues kernels on the caller's
// stream.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/pa.h"
#include "pa_internal.h"

// Device error word: kernels OR PA_DEVERR_* bits into it; pa_device_errors
// reads and clears it.  One copy per device that loads the library.
__device__ unsigned int g_pa_error_word;

namespace {

std::mutex g_err_mu;
unsigned int *g_err_ptr[pa::kMaxDevices] = {};

// Address of this device's error word, looked up once per device with that
// device current.
cudaError_t error_word(unsigned int **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= pa::kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_err_mu);
  if (!g_err_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_pa_error_word);
    if (e != cudaSuccess) return e;
    g_err_ptr[dev] = static_cast<unsigned int *>(p);
  }
  *out = g_err_ptr[dev];
  return cudaSuccess;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool dtype_ok(int32_t d) { return d == PA_FP16 || d == PA_BF16; }
bool fp8_scales_ok(float k_scale, float v_scale) {
  return std::isfinite(k_scale) && std::isfinite(v_scale) && k_scale > 0.f && v_scale > 0.f;
}
bool head_dim_ok(int32_t d) { return d == 64 || d == 128; }
bool block_size_ok(int32_t b) { return b == 16 || b == 32; }

int32_t num_partitions(int32_t max_context_len, int32_t partition_size) {
  if (partition_size <= 0 || max_context_len <= partition_size) return 1;
  return static_cast<int32_t>((static_cast<int64_t>(max_context_len) + partition_size - 1) /
                              partition_size);
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct WsLayout {
  size_t m_off, l_off, o_off, total;
};

// Split-context workspace: the join counters (PA_DECODE_COUNTER_BYTES, a fixed
// size so that no partial of any shape ever lands on them), then m, l, o.
WsLayout workspace_layout(int64_t rows, int64_t parts, int64_t head_dim) {
  WsLayout w;
  const size_t ml = static_cast<size_t>(rows * parts) * sizeof(float);
  w.m_off = PA_DECODE_COUNTER_BYTES;
  w.l_off = w.m_off + align256(ml);
  w.o_off = w.l_off + align256(ml);
  w.total = w.o_off + align256(static_cast<size_t>(rows * parts * head_dim) * sizeof(float));
  return w;
}

// Largest partition count whose join runs inside the decode kernel (by the
// last CTA of each sequence and KV head to finish); more partitions are
// joined by pa_decode_reduce_kernel, whose many CTAs share the longer join.
constexpr int32_t kMaxFusedParts = 32;

}  // namespace

extern "C" {

int32_t pa_version(void) { return 4; }

const char *pa_status_string(int32_t status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported shape";
    case PA_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

int32_t pa_decode_num_partitions(int32_t max_context_len, int32_t partition_size) {
  return num_partitions(max_context_len, partition_size);
}

size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                int32_t max_context_len, int32_t partition_size) {
  if (num_seqs <= 0 || num_q_heads <= 0 || head_dim <= 0 || max_context_len < 0) return 0;
  const int32_t P = num_partitions(max_context_len, partition_size);
  if (P <= 1) return 0;
  return workspace_layout(static_cast<int64_t>(num_seqs) * num_q_heads, P, head_dim).total;
}

pa_status pa_reshape_and_cache(const void *key, const void *value, int64_t key_stride,
                               int64_t value_stride, void *k_cache, void *v_cache,
                               const int64_t *slot_mapping, int32_t num_tokens,
                               int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                               int64_t num_blocks, int32_t dtype, void *stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks <= 0 || !dtype_ok(dtype))
    return PA_ERR_INVALID_ARG;
  if (!head_dim_ok(head_dim) || !block_size_ok(block_size)) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
  if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (key_stride < row || value_stride < row || key_stride % 8 || value_stride % 8)
    return PA_ERR_INVALID_ARG;
  if (num_tokens > 0x7fffffff) return PA_ERR_UNSUPPORTED;
  unsigned int *err = nullptr;
  if (error_word(&err) != cudaSuccess) return PA_ERR_CUDA;
  pa::ReshapeArgs a;
  a.to_fp8 = false;
  a.src_dtype = dtype;
  a.k_scale = a.v_scale = 1.f;
  a.key = key;
  a.value = value;
  a.key_stride = key_stride;
  a.value_stride = value_stride;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.slot_mapping = slot_mapping;
  a.num_tokens = num_tokens;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.err = err;
  return pa::launch_reshape(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK
                                                                                  : PA_ERR_CUDA;
}

}  // extern "C"

namespace {

// pa_decode_reduce with the number of tokens the block table can address:
// pa_decode passes its table's capacity so that a context length the decode
// kernel refused is refused here too; the exported call has no table.
pa_status reduce_impl(void *out, const void *workspace, const int32_t *context_lens,
                      int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                      int32_t max_context_len, int32_t partition_size, int32_t dtype,
                      int64_t table_tokens, void *stream) {
  if (num_seqs < 0 || num_q_heads <= 0 || max_context_len < 0 || partition_size <= 0 ||
      !dtype_ok(dtype))
    return PA_ERR_INVALID_ARG;
  if (!head_dim_ok(head_dim)) return PA_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PA_OK;
  if (!out || !workspace || !context_lens || !aligned16(out) || !aligned16(workspace))
    return PA_ERR_INVALID_ARG;
  // one CTA per output row
  if (num_seqs > 65535 || static_cast<int64_t>(num_seqs) * num_q_heads > 0x7fffffff)
    return PA_ERR_UNSUPPORTED;
  unsigned int *err = nullptr;
  if (error_word(&err) != cudaSuccess) return PA_ERR_CUDA;
  const int32_t P = num_partitions(max_context_len, partition_size);
  const WsLayout w = workspace_layout(static_cast<int64_t>(num_seqs) * num_q_heads, P, head_dim);
  const char *base = static_cast<const char *>(workspace);
  pa::ReduceArgs a;
  a.out = out;
  a.ws_m = reinterpret_cast<const float *>(base + w.m_off);
  a.ws_l = reinterpret_cast<const float *>(base + w.l_off);
  a.ws_o = reinterpret_cast<const float *>(base + w.o_off);
  a.context_lens = context_lens;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_parts = P;
  a.partition_size = partition_size;
  a.max_context_len = max_context_len;
  a.table_tokens = table_tokens;
  // more warps per row when rows hold many partitions (measured: one warp per
  // row up to 64 partitions; four for the 256 of a 131k-token context)
  a.warps_per_row = P > 128 ? 4 : (P > 64 ? 2 : 1);
  a.err = err;
  return pa::launch_reduce(a, head_dim, dtype, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

}  // namespace

extern "C" pa_status pa_decode_reduce(void *out, const void *workspace,
                                      const int32_t *context_lens, int32_t num_seqs,
                                      int32_t num_q_heads, int32_t head_dim,
                                      int32_t max_context_len, int32_t partition_size,
                                      int32_t dtype, void *stream) {
  return reduce_impl(out, workspace, context_lens, num_seqs, num_q_heads, head_dim,
                     max_context_len, partition_size, dtype, INT32_MAX, stream);
}

// Every host-side check pa_decode makes before it looks at the workspace, in
// the same order, so that a caller without a workspace gets the status
// pa_decode would return for the same arguments.
int32_t pa::decode_check_args(const void *out, const void *query, const void *k_cache,
                              const void *v_cache, const int32_t *block_tables,
                              int32_t max_blocks_per_seq, const int32_t *context_lens,
                              int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                              int32_t head_dim, int32_t block_size, int64_t num_blocks,
                              float scale, int32_t max_context_len, int32_t partition_size,
                              int32_t dtype) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_blocks <= 0 ||
      max_blocks_per_seq <= 0 || max_context_len < 0 || partition_size < 0 ||
      !dtype_ok(dtype) || !std::isfinite(scale))
    return PA_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads) return PA_ERR_INVALID_ARG;
  if (partition_size % 16) return PA_ERR_INVALID_ARG;
  const int32_t group = num_q_heads / num_kv_heads;
  if (!head_dim_ok(head_dim) || !block_size_ok(block_size) || group > 8)
    return PA_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PA_OK;
  if (!out || !query || !k_cache || !v_cache || !block_tables || !context_lens)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(query) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  // TMA row coordinates are 32-bit; grid y/z are 16-bit
  const int64_t pool_rows = num_blocks * num_kv_heads * block_size;
  if (pool_rows >= (int64_t(1) << 31) || num_seqs > 65535 || num_kv_heads > 65535)
    return PA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_blocks_per_seq) * block_size > 0x7fffffff)
    return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

namespace {

// The groups of pa_decode_shared_prefix (device arrays and their host-side bounds).
struct SharedPrefix {
  const int32_t *group_start, *prefix_lens;
  int32_t num_groups, max_group_size;
};

pa_status decode_impl(void *out, const void *query, const void *k_cache, const void *v_cache,
                      const int32_t *block_tables, int32_t max_blocks_per_seq,
                      const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                      int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                      int64_t num_blocks, float scale, int32_t max_context_len,
                      int32_t partition_size, void *workspace, size_t workspace_bytes,
                      int32_t dtype, bool kv_fp8, float k_scale, float v_scale, void *stream,
                      const SharedPrefix *sp = nullptr) {
  const int32_t st = pa::decode_check_args(
      out, query, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
      num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, max_context_len,
      partition_size, dtype);
  if (st != PA_OK) return static_cast<pa_status>(st);
  const int32_t group = num_q_heads / num_kv_heads;
  const int32_t P = num_partitions(max_context_len, partition_size);
  int32_t chunks = 0;
  if (sp) {
    if (!sp->group_start || !sp->prefix_lens || sp->num_groups < 1 || sp->max_group_size < 1 ||
        partition_size <= 0 || (num_seqs > 0 && (sp->num_groups > num_seqs ||
                                                 sp->max_group_size > num_seqs)))
      return PA_ERR_INVALID_ARG;
    if (partition_size > pa::kMaxSharedPrefixPartition) return PA_ERR_UNSUPPORTED;
    const int32_t mpc = pa::shared_prefix_members_per_cta(group);
    chunks = (sp->max_group_size + mpc - 1) / mpc;
    if (static_cast<int64_t>(P) * chunks > 0x7fffffff) return PA_ERR_UNSUPPORTED;
  }
  if (num_seqs == 0) return PA_OK;
  const int64_t pool_rows = num_blocks * num_kv_heads * block_size;
  WsLayout w{};
  if (P > 1) {
    w = workspace_layout(static_cast<int64_t>(num_seqs) * num_q_heads, P, head_dim);
    if (!workspace || workspace_bytes < w.total || !aligned16(workspace))
      return PA_ERR_INVALID_ARG;
  }
  const bool fuse = P > 1 && P <= kMaxFusedParts &&
                    static_cast<int64_t>(num_seqs) * num_kv_heads <= PA_DECODE_COUNTER_BYTES / 4;
  unsigned int *err = nullptr;
  if (error_word(&err) != cudaSuccess) return PA_ERR_CUDA;

  pa::DecodeArgs a{};
  a.out = out;
  a.query = query;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.group = group;
  a.bs_log2 = block_size == 16 ? 4 : 5;
  a.num_blocks = num_blocks;
  a.scale_log2 = scale * 1.4426950408889634f * k_scale;
  a.out_scale = v_scale;
  a.max_context_len = max_context_len;
  a.part_tokens = P > 1 ? partition_size : (max_context_len > 0 ? max_context_len : 1);
  a.num_parts = P;
  char *base = static_cast<char *>(workspace);
  a.ws_m = P > 1 ? reinterpret_cast<float *>(base + w.m_off) : nullptr;
  a.ws_l = P > 1 ? reinterpret_cast<float *>(base + w.l_off) : nullptr;
  a.ws_o = P > 1 ? reinterpret_cast<float *>(base + w.o_off) : nullptr;
  a.ws_cnt = P > 1 ? reinterpret_cast<unsigned *>(base) : nullptr;
  a.fuse_join = fuse ? 1 : 0;
  a.err = err;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  bool map_failed = false;
  if (sp && P > 1) {
    // the shared pass writes the partials of every member's shared partitions;
    // the decode launch below computes the rest and joins them all
    a.prefix_lens = sp->prefix_lens;
    a.group_start = sp->group_start;
    a.num_groups = sp->num_groups;
    a.max_group_size = sp->max_group_size;
    a.members_per_cta = pa::shared_prefix_members_per_cta(group);
    a.chunks = chunks;
    if (pa::launch_shared_prefix(a, k_cache, v_cache, pool_rows, head_dim, dtype, kv_fp8, cs,
                                 &map_failed) != cudaSuccess)
      return map_failed ? PA_ERR_INVALID_ARG : PA_ERR_CUDA;
  }
  if (pa::launch_decode(a, k_cache, v_cache, pool_rows, head_dim, dtype, kv_fp8, cs,
                        &map_failed) != cudaSuccess)
    return map_failed ? PA_ERR_INVALID_ARG : PA_ERR_CUDA;
  if (P > 1 && !fuse)
    return reduce_impl(out, workspace, context_lens, num_seqs, num_q_heads, head_dim,
                       max_context_len, partition_size, dtype,
                       static_cast<int64_t>(max_blocks_per_seq) * block_size, stream);
  return PA_OK;
}

}  // namespace

extern "C" {

pa_status pa_decode(void *out, const void *query, const void *k_cache, const void *v_cache,
                    const int32_t *block_tables, int32_t max_blocks_per_seq,
                    const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                    int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                    int64_t num_blocks, float scale, int32_t max_context_len,
                    int32_t partition_size, void *workspace, size_t workspace_bytes,
                    int32_t dtype, void *stream) {
  return decode_impl(out, query, k_cache, v_cache, block_tables, max_blocks_per_seq,
                     context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                     num_blocks, scale, max_context_len, partition_size, workspace,
                     workspace_bytes, dtype, false, 1.f, 1.f, stream);
}

pa_status pa_decode_shared_prefix(void *out, const void *query, const void *k_cache,
                                  const void *v_cache, const int32_t *block_tables,
                                  int32_t max_blocks_per_seq, const int32_t *context_lens,
                                  const int32_t *group_start, const int32_t *prefix_lens,
                                  int32_t num_groups, int32_t max_group_size, int32_t num_seqs,
                                  int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t block_size, int64_t num_blocks, float scale,
                                  int32_t max_context_len, int32_t partition_size,
                                  void *workspace, size_t workspace_bytes, int32_t dtype,
                                  void *stream) {
  const SharedPrefix sp{group_start, prefix_lens, num_groups, max_group_size};
  return decode_impl(out, query, k_cache, v_cache, block_tables, max_blocks_per_seq,
                     context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                     num_blocks, scale, max_context_len, partition_size, workspace,
                     workspace_bytes, dtype, false, 1.f, 1.f, stream, &sp);
}

pa_status pa_decode_shared_prefix_fp8(void *out, const void *query, const void *k_cache,
                                      const void *v_cache, const int32_t *block_tables,
                                      int32_t max_blocks_per_seq, const int32_t *context_lens,
                                      const int32_t *group_start, const int32_t *prefix_lens,
                                      int32_t num_groups, int32_t max_group_size,
                                      int32_t num_seqs, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                      int64_t num_blocks, float scale, float k_scale,
                                      float v_scale, int32_t max_context_len,
                                      int32_t partition_size, void *workspace,
                                      size_t workspace_bytes, int32_t dtype, void *stream) {
  if (!fp8_scales_ok(k_scale, v_scale) || !dtype_ok(dtype)) return PA_ERR_INVALID_ARG;
  const SharedPrefix sp{group_start, prefix_lens, num_groups, max_group_size};
  return decode_impl(out, query, k_cache, v_cache, block_tables, max_blocks_per_seq,
                     context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                     num_blocks, scale, max_context_len, partition_size, workspace,
                     workspace_bytes, dtype, true, k_scale, v_scale, stream, &sp);
}

pa_status pa_decode_fp8(void *out, const void *query, const void *k_cache, const void *v_cache,
                        const int32_t *block_tables, int32_t max_blocks_per_seq,
                        const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                        int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                        int64_t num_blocks, float scale, float k_scale, float v_scale,
                        int32_t max_context_len, int32_t partition_size, void *workspace,
                        size_t workspace_bytes, int32_t dtype, void *stream) {
  if (!std::isfinite(k_scale) || !std::isfinite(v_scale) || !(k_scale > 0.f) ||
      !(v_scale > 0.f) || dtype != PA_FP16 && dtype != PA_BF16)
    return PA_ERR_INVALID_ARG;
  return decode_impl(out, query, k_cache, v_cache, block_tables, max_blocks_per_seq,
                     context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                     num_blocks, scale, max_context_len, partition_size, workspace,
                     workspace_bytes, dtype, true, k_scale, v_scale, stream);
}

pa_status pa_reshape_and_cache_fp8(const void *key, const void *value, int64_t key_stride,
                                   int64_t value_stride, void *k_cache, void *v_cache,
                                   const int64_t *slot_mapping, int32_t num_tokens,
                                   int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                   int64_t num_blocks, int32_t src_dtype, float k_scale,
                                   float v_scale, void *stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks <= 0 || !dtype_ok(src_dtype) ||
      !std::isfinite(k_scale) || !std::isfinite(v_scale) || !(k_scale > 0.f) || !(v_scale > 0.f))
    return PA_ERR_INVALID_ARG;
  if (!head_dim_ok(head_dim) || !block_size_ok(block_size)) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
  if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (key_stride < row || value_stride < row || key_stride % 8 || value_stride % 8)
    return PA_ERR_INVALID_ARG;
  unsigned int *err = nullptr;
  if (error_word(&err) != cudaSuccess) return PA_ERR_CUDA;
  pa::ReshapeArgs a;
  a.to_fp8 = true;
  a.src_dtype = src_dtype;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.key = key;
  a.value = value;
  a.key_stride = key_stride;
  a.value_stride = value_stride;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.slot_mapping = slot_mapping;
  a.num_tokens = num_tokens;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.err = err;
  return pa::launch_reshape(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK
                                                                                  : PA_ERR_CUDA;
}

}  // extern "C"

namespace {

pa_status prefill_impl(void *out, const void *query, const int32_t *query_start,
                       const void *k_cache, const void *v_cache, const int32_t *block_tables,
                       int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                       int32_t max_q_len, int32_t num_q_heads, int32_t num_kv_heads,
                       int32_t head_dim, int32_t block_size, int64_t num_blocks, float scale,
                       int32_t dtype, bool kv_fp8, float k_scale, float v_scale, void *stream) {
  if (num_seqs < 0 || max_q_len < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      num_blocks <= 0 || max_blocks_per_seq <= 0 || !dtype_ok(dtype) || !std::isfinite(scale) ||
      !(scale > 0.f))
    return PA_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads) return PA_ERR_INVALID_ARG;
  const int32_t group = num_q_heads / num_kv_heads;
  if (!head_dim_ok(head_dim) || !block_size_ok(block_size) || group > 8)
    return PA_ERR_UNSUPPORTED;
  if (num_seqs == 0 || max_q_len == 0) return PA_OK;
  if (!out || !query || !query_start || !k_cache || !v_cache || !block_tables || !context_lens)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(query) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  const int64_t pool_rows = num_blocks * num_kv_heads * block_size;
  if (pool_rows >= (int64_t(1) << 31) || num_seqs > 65535 || num_kv_heads > 65535)
    return PA_ERR_UNSUPPORTED;
  unsigned int *err = nullptr;
  if (error_word(&err) != cudaSuccess) return PA_ERR_CUDA;
  pa::PrefillArgs a{};
  a.out = out;
  a.query = query;
  a.query_start = query_start;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.group = group;
  a.bs_log2 = block_size == 16 ? 4 : 5;
  a.max_q_len = max_q_len;
  a.num_blocks = num_blocks;
  a.scale_log2 = scale * 1.4426950408889634f * k_scale;
  a.out_scale = v_scale;
  a.err = err;
  bool map_failed = false;
  if (pa::launch_prefill(a, k_cache, v_cache, pool_rows, head_dim, dtype, kv_fp8,
                         static_cast<cudaStream_t>(stream), &map_failed) != cudaSuccess)
    return map_failed ? PA_ERR_INVALID_ARG : PA_ERR_CUDA;
  return PA_OK;
}

}  // namespace

extern "C" {

pa_status pa_prefill(void *out, const void *query, const int32_t *query_start,
                     const void *k_cache, const void *v_cache, const int32_t *block_tables,
                     int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                     int32_t max_q_len, int32_t num_q_heads, int32_t num_kv_heads,
                     int32_t head_dim, int32_t block_size, int64_t num_blocks, float scale,
                     int32_t dtype, void *stream) {
  return prefill_impl(out, query, query_start, k_cache, v_cache, block_tables, max_blocks_per_seq,
                      context_lens, num_seqs, max_q_len, num_q_heads, num_kv_heads, head_dim,
                      block_size, num_blocks, scale, dtype, false, 1.f, 1.f, stream);
}

pa_status pa_prefill_fp8(void *out, const void *query, const int32_t *query_start,
                         const void *k_cache, const void *v_cache, const int32_t *block_tables,
                         int32_t max_blocks_per_seq, const int32_t *context_lens,
                         int32_t num_seqs, int32_t max_q_len, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                         int64_t num_blocks, float scale, float k_scale, float v_scale,
                         int32_t dtype, void *stream) {
  if (!fp8_scales_ok(k_scale, v_scale)) return PA_ERR_INVALID_ARG;
  return prefill_impl(out, query, query_start, k_cache, v_cache, block_tables, max_blocks_per_seq,
                      context_lens, num_seqs, max_q_len, num_q_heads, num_kv_heads, head_dim,
                      block_size, num_blocks, scale, dtype, true, k_scale, v_scale, stream);
}

}  // extern "C"

namespace {

pa_status copy_blocks_impl(void *k_cache, void *v_cache, const int64_t *block_mapping,
                           int32_t num_pairs, int32_t num_kv_heads, int32_t head_dim,
                           int32_t block_size, int64_t num_blocks, int elem_bytes, void *stream) {
  if (num_pairs < 0 || num_kv_heads <= 0 || num_blocks <= 0) return PA_ERR_INVALID_ARG;
  if (!head_dim_ok(head_dim) || !block_size_ok(block_size)) return PA_ERR_UNSUPPORTED;
  if (num_pairs == 0) return PA_OK;
  if (!k_cache || !v_cache || !block_mapping || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  unsigned int *err = nullptr;
  if (error_word(&err) != cudaSuccess) return PA_ERR_CUDA;
  pa::BlockCopyArgs a;
  a.src[0] = k_cache;
  a.src[1] = v_cache;
  a.dst[0] = k_cache;
  a.dst[1] = v_cache;
  a.mapping = block_mapping;
  a.num_pairs = num_pairs;
  a.block_bytes = static_cast<int64_t>(num_kv_heads) * block_size * head_dim * elem_bytes;
  a.src_blocks = num_blocks;
  a.dst_blocks = num_blocks;
  a.err = err;
  return pa::launch_block_copy(a, 2, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

}  // namespace

extern "C" {

pa_status pa_copy_blocks(void *k_cache, void *v_cache, const int64_t *block_mapping,
                         int32_t num_pairs, int32_t num_kv_heads, int32_t head_dim,
                         int32_t block_size, int64_t num_blocks, void *stream) {
  return copy_blocks_impl(k_cache, v_cache, block_mapping, num_pairs, num_kv_heads, head_dim,
                          block_size, num_blocks, 2, stream);
}

pa_status pa_copy_blocks_fp8(void *k_cache, void *v_cache, const int64_t *block_mapping,
                             int32_t num_pairs, int32_t num_kv_heads, int32_t head_dim,
                             int32_t block_size, int64_t num_blocks, void *stream) {
  return copy_blocks_impl(k_cache, v_cache, block_mapping, num_pairs, num_kv_heads, head_dim,
                          block_size, num_blocks, 1, stream);
}

namespace {
// Device-usable address of device, managed or pinned host memory; null for
// memory the device cannot reach (pageable host memory that was not pinned).
const void *device_view(const void *p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  switch (at.type) {
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged:
      return p;
    case cudaMemoryTypeHost:
      return at.devicePointer;
    default:
      return nullptr;
  }
}
}  // namespace

pa_status pa_swap_blocks(const void *src, void *dst, const int64_t *block_mapping,
                         int32_t num_pairs, int64_t block_bytes, int64_t src_num_blocks,
                         int64_t dst_num_blocks, void *stream) {
  if (num_pairs < 0 || block_bytes <= 0 || block_bytes % 16 || src_num_blocks <= 0 ||
      dst_num_blocks <= 0)
    return PA_ERR_INVALID_ARG;
  if (num_pairs == 0) return PA_OK;
  if (!src || !dst || !block_mapping || !aligned16(src) || !aligned16(dst))
    return PA_ERR_INVALID_ARG;
  const void *s = device_view(src);
  void *d = const_cast<void *>(device_view(dst));
  const void *m = device_view(block_mapping);
  if (!s || !d || !m) return PA_ERR_INVALID_ARG;
  unsigned int *err = nullptr;
  if (error_word(&err) != cudaSuccess) return PA_ERR_CUDA;
  pa::BlockCopyArgs a;
  a.src[0] = a.src[1] = s;
  a.dst[0] = a.dst[1] = d;
  a.mapping = static_cast<const int64_t *>(m);
  a.num_pairs = num_pairs;
  a.block_bytes = block_bytes;
  a.src_blocks = src_num_blocks;
  a.dst_blocks = dst_num_blocks;
  a.err = err;
  return pa::launch_block_copy(a, 1, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

pa_status pa_selftest_bounded_wait(void *stream) {
  unsigned int *err = nullptr;
  if (error_word(&err) != cudaSuccess) return PA_ERR_CUDA;
  return pa::launch_selftest_wait(err, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

pa_status pa_device_errors(void *stream, uint32_t *flags) {
  if (!flags) return PA_ERR_INVALID_ARG;
  unsigned int *err = nullptr;
  if (error_word(&err) != cudaSuccess) return PA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned int host = 0;
  if (cudaStreamSynchronize(st) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaMemcpy(&host, err, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess)
    return PA_ERR_CUDA;
  if (host) {
    const unsigned int zero = 0;
    if (cudaMemcpy(err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return PA_ERR_CUDA;
  }
  *flags = host;
  return PA_OK;
}

}  // extern "C"
