// pa_cache.cu -- reshape_and_cache: write each new token's K and V rows into
// its slot of the paged pool ("Serving engines", How vLLM works: the slot
// mapping gives, per new token, physical_block * block_size + offset).
//
// One CTA per token.  Each thread moves 16-byte chunks of the token's
// [num_kv_heads, head_dim] K and V rows to
// cache[slot / block_size, h, slot % block_size, :].  The copy is raw bytes,
// so it is bit-exact for either 16-bit dtype.  A negative slot is skipped; a
// slot past the pool is skipped and flagged.  It lets the next kernel in the
// stream (the decode) start launching as soon as it begins; that kernel waits
// for this one's writes before reading the pool.
#include <cuda_runtime.h>

#include <cstdint>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

__global__ void __launch_bounds__(128) reshape_and_cache_kernel(const ReshapeArgs a) {
  const int t = blockIdx.x;
  grid_dependency_wait();   // key/value/slots may come from the kernel before
  grid_launch_dependents();  // the next kernel (decode) may start its set-up now
  const int64_t slot = a.slot_mapping[t];
  if (slot < 0) return;
  if (slot >= a.num_blocks * a.block_size) {
    if (threadIdx.x == 0) atomicOr(a.err, kErrBadSlot);
    return;
  }
  const int64_t blk = slot / a.block_size;
  const int off = static_cast<int>(slot % a.block_size);
  const int chunks = a.head_dim / 8;  // 16-byte chunks per head row
  const int per_token = a.num_kv_heads * chunks;
  const uint4 *key = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.key) +
                                                     t * a.key_stride);
  const uint4 *value = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.value) +
                                                       t * a.value_stride);
  uint4 *kc = static_cast<uint4 *>(a.k_cache);
  uint4 *vc = static_cast<uint4 *>(a.v_cache);
  for (int i = threadIdx.x; i < per_token; i += blockDim.x) {
    const int h = i / chunks, ch = i % chunks;
    const int64_t dst = ((blk * a.num_kv_heads + h) * a.block_size + off) * chunks + ch;
    kc[dst] = key[i];
    vc[dst] = value[i];
  }
}

}  // namespace

cudaError_t launch_reshape(const ReshapeArgs &a, cudaStream_t stream) {
  return launch_dependent(reshape_and_cache_kernel, dim3(a.num_tokens), dim3(128), 0, stream, a);
}

}  // namespace pa
