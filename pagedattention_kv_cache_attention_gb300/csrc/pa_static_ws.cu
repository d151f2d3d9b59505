// pa_static_ws.cu -- pa_decode_static_workspace: paged decode for callers that
// cannot allocate device memory.
//
// Some callers of this library may not call cudaMalloc: a serving framework
// that has reserved nearly all device memory for its own KV pool and hands
// none of it to libraries, a plugin under a host runtime that owns every
// allocation on the device, or a real-time enqueue path that cannot risk the
// device-wide synchronisation an allocation may cause.  For them this entry
// point takes its split-context scratch (partials and join counters) from a
// fixed array in device memory that the library itself carries, instead of a
// caller-supplied workspace.
//
// The array is a file-scope __device__ variable: every device that loads the
// library holds PA_STATIC_WORKSPACE_BYTES of it until the process exits.  In
// host code its name only stands for the variable and is not a device
// address, so the address is looked up once per device, with that device
// current, by cudaGetSymbolAddress, and passed to the kernels.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/pa.h"
#include "pa_internal.h"

static __device__ __align__(256) unsigned char g_pa_static_workspace[PA_STATIC_WORKSPACE_BYTES];

namespace {

std::mutex g_ws_mu;
void *g_ws_ptr[pa::kMaxDevices] = {};

// Device address of this device's copy of the array (the first call per
// device does the lookup).
cudaError_t static_workspace(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= pa::kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_ws_mu);
  if (!g_ws_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_pa_static_workspace);
    if (e != cudaSuccess) return e;
    g_ws_ptr[dev] = p;
  }
  *out = g_ws_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" pa_status pa_decode_static_workspace(
    void *out, const void *query, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
    int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t block_size, int64_t num_blocks, float scale, int32_t max_context_len,
    int32_t partition_size, int32_t dtype, void *stream) {
  // the statuses pa_decode gives for bad arguments come first; only a valid
  // shape is measured against the array
  const int32_t st = pa::decode_check_args(
      out, query, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
      num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, max_context_len,
      partition_size, dtype);
  if (st != PA_OK || num_seqs == 0) return static_cast<pa_status>(st);
  const size_t need = pa_decode_workspace_size(num_seqs, num_q_heads, head_dim, max_context_len,
                                               partition_size);
  if (need > PA_STATIC_WORKSPACE_BYTES) return PA_ERR_UNSUPPORTED;
  void *ws = nullptr;
  if (need > 0) {
    if (static_workspace(&ws) != cudaSuccess) return PA_ERR_CUDA;
    // the array keeps whatever the previous call left: clear the join
    // counters this call uses (one per sequence and KV head, at the start of
    // the array); the partials are all written before they are read
    const size_t counters = static_cast<size_t>(num_seqs) * num_kv_heads * sizeof(uint32_t);
    const size_t clear = counters < PA_DECODE_COUNTER_BYTES ? counters : PA_DECODE_COUNTER_BYTES;
    if (cudaMemsetAsync(ws, 0, clear, static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return PA_ERR_CUDA;
  }
  return pa_decode(out, query, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                   num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                   max_context_len, partition_size, ws, need > 0 ? PA_STATIC_WORKSPACE_BYTES : 0,
                   dtype, stream);
}
