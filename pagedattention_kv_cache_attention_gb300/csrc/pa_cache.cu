// pa_cache.cu -- reshape_and_cache: write each new token's K and V rows into
// its slot of the paged pool ("Serving engines", How vLLM works: the slot
// mapping gives, per new token, physical_block * block_size + offset).
//
// One CTA per token.  Each thread moves 16-byte chunks of the token's
// [num_kv_heads, head_dim] K and V rows to
// cache[slot / block_size, h, slot % block_size, :].  The copy is raw bytes,
// so it is bit-exact for either 16-bit dtype.  Into an FP8 cache each element
// is stored as the E4M3 code of x / scale (nearest even, saturating at 448).  A negative slot is skipped; a
// slot past the pool is skipped and flagged.  It lets the next kernel in the
// stream (the decode) start launching as soon as it begins; that kernel waits
// for this one's writes before reading the pool.
#include <cuda_runtime.h>

#include <cstdint>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

__device__ __forceinline__ float to_float(uint32_t w16, int dtype) {
  const uint16_t b = static_cast<uint16_t>(w16);
  if (dtype == 1) return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(&b));
  return __half2float(*reinterpret_cast<const __half *>(&b));
}

// 16 consecutive 16-bit elements at src -> 16 E4M3 codes of x / scale.
__device__ __forceinline__ uint4 quantize16(const uint4 *src, int dtype, float scale) {
  const uint4 x0 = src[0], x1 = src[1];
  const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
  uint32_t out[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t bytes = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t word = w[2 * k + h];
      const float2 f = make_float2(__fdiv_rn(to_float(word & 0xffffu, dtype), scale),
                                   __fdiv_rn(to_float(word >> 16, dtype), scale));
      const __nv_fp8x2_storage_t q = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
      bytes |= static_cast<uint32_t>(q) << (16 * h);
    }
    out[k] = bytes;
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

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
  if (!a.to_fp8) {
    for (int i = threadIdx.x; i < per_token; i += blockDim.x) {
      const int h = i / chunks, ch = i % chunks;
      const int64_t dst = ((blk * a.num_kv_heads + h) * a.block_size + off) * chunks + ch;
      kc[dst] = key[i];
      vc[dst] = value[i];
    }
    return;
  }
  // FP8 cache: 16 source elements (two 16-byte chunks) become one 16-byte
  // chunk of E4M3 codes of x / scale (IEEE division, nearest even, saturating)
  const int out_chunks = a.head_dim / 16;
  for (int i = threadIdx.x; i < a.num_kv_heads * out_chunks; i += blockDim.x) {
    const int h = i / out_chunks, ch = i % out_chunks;
    const int64_t dst = ((blk * a.num_kv_heads + h) * a.block_size + off) * out_chunks + ch;
    kc[dst] = quantize16(key + h * chunks + 2 * ch, a.src_dtype, a.k_scale);
    vc[dst] = quantize16(value + h * chunks + 2 * ch, a.src_dtype, a.v_scale);
  }
}

}  // namespace

cudaError_t launch_reshape(const ReshapeArgs &a, cudaStream_t stream) {
  return launch_dependent(reshape_and_cache_kernel, dim3(a.num_tokens), dim3(128), 0, stream, a);
}

}  // namespace pa
