// pa_blocks.cu -- whole-block moves of the paged pool ("Serving engines", How
// vLLM works):
//  * copy_blocks: copy-on-write fork.  Two sequences share a physical block
//    until one of them writes into it; then only that block is copied and the
//    writer's block table is pointed at the copy.
//  * swap_blocks: preemption by swapping.  When the pool runs dry a
//    sequence's blocks move to host memory and later come back, possibly to
//    other physical block ids.
//
// One kernel serves both: each CTA copies a slice of one (source block,
// destination block) pair with 16-byte loads and stores, four loads in flight
// per thread before the stores.  Host memory is reached directly through its
// unified (pinned, device-mapped) address, so a swap is one launch instead of
// one copy call per block.  A pair with an id outside its pool is skipped and
// flagged; the copy is bit-exact.
#include <cuda_runtime.h>

#include <cstdint>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kThreads) block_copy_kernel(const BlockCopyArgs a) {
  const int pair = blockIdx.x;
  const int tensor = blockIdx.z;  // 0: first (src, dst) pointer pair, 1: second
  grid_dependency_wait();         // the mapping and the pools may come from earlier kernels
  const int64_t src = a.mapping[2 * static_cast<int64_t>(pair)];
  const int64_t dst = a.mapping[2 * static_cast<int64_t>(pair) + 1];
  if (src < 0 || src >= a.src_blocks || dst < 0 || dst >= a.dst_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0 && tensor == 0) atomicOr(a.err, kErrBadBlock);
    return;
  }
  const int64_t n = a.block_bytes / 16;
  // select by value: indexing the parameter arrays would copy them to local memory
  const uint4 *s = static_cast<const uint4 *>(tensor == 0 ? a.src[0] : a.src[1]) + src * n;
  uint4 *d = static_cast<uint4 *>(tensor == 0 ? a.dst[0] : a.dst[1]) + dst * n;
  const int64_t stride = static_cast<int64_t>(gridDim.y) * kThreads;
  int64_t i = static_cast<int64_t>(blockIdx.y) * kThreads + threadIdx.x;
  for (; i + (kUnroll - 1) * stride < n; i += kUnroll * stride) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = s[i + u * stride];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) d[i + u * stride] = v[u];
  }
  for (; i < n; i += stride) d[i] = s[i];
}

}  // namespace

cudaError_t launch_block_copy(const BlockCopyArgs &a, int num_tensors, cudaStream_t stream) {
  const int64_t chunks = a.block_bytes / 16;
  // enough CTAs per pair that each thread moves ~kUnroll chunks of a block
  int64_t ys = (chunks + kThreads * kUnroll - 1) / (kThreads * kUnroll);
  if (ys < 1) ys = 1;
  if (ys > 65535) ys = 65535;
  return launch_dependent(block_copy_kernel, dim3(a.num_pairs, static_cast<unsigned>(ys),
                                                  num_tensors),
                          dim3(kThreads), 0, stream, a);
}

namespace {

// Waits on a barrier whose phase never completes: every thread's bounded wait
// gives up after kWaitLimitNs and the CTA reports it and exits.
__global__ void selftest_wait_kernel(unsigned *err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  const bool done = mbar_wait_bounded(&bar, 0);
  if (!done && threadIdx.x == 0) atomicOr(err, kErrTimeout);
}

}  // namespace

cudaError_t launch_selftest_wait(unsigned *err, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(err);
  return cudaGetLastError();
}

}  // namespace pa
