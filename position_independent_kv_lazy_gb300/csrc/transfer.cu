// Host-to-device copy driven by the SMs (lazy_copy_to_device).
//
// A serving step uploads about a megabyte of inputs (queries, the new tokens' K/V, page words,
// positions). A copy-engine transfer of that size is dominated by its start-up: on the GB300
// host link 921 KB took about 15 us. Here every SM reads the pinned, device-mapped host buffer
// directly, with a few 16-byte loads in flight per thread, so the transfer costs about one
// round trip over the link plus the bytes at link speed.
#include <algorithm>

#include "lazy_common.cuh"
#include "pool_internal.h"

namespace lazy {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;  // 16-byte loads in flight per thread

__global__ void __launch_bounds__(kCopyThreads) h2d_copy_kernel(uint4 *__restrict__ dst,
                                                                const uint4 *__restrict__ src,
                                                                size_t n16) {
  const size_t stride = (size_t)gridDim.x * kCopyThreads;
  size_t i = (size_t)blockIdx.x * kCopyThreads + threadIdx.x;
  for (; i + (kCopyUnroll - 1) * stride < n16; i += kCopyUnroll * stride) {
    uint4 v[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) v[u] = src[i + u * stride];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) dst[i + u * stride] = v[u];
  }
  for (; i < n16; i += stride) dst[i] = src[i];
}

}  // namespace
}  // namespace lazy

using namespace lazy;

extern "C" int lazy_copy_to_device(void *d_dst, const void *h_src, size_t bytes,
                                   lazy_stream_t stream) {
  if (bytes == 0) return LAZY_OK;
  if (!d_dst || !h_src || ((uintptr_t)d_dst & 15) || ((uintptr_t)h_src & 15) || (bytes & 15)) {
    record_msg("lazy_copy_to_device: pointers and size must be non-null multiples of 16 bytes");
    return LAZY_ERR_INVALID_ARG;
  }
  cudaPointerAttributes src_attr, dst_attr;
  if (cudaPointerGetAttributes(&src_attr, h_src) != cudaSuccess ||
      cudaPointerGetAttributes(&dst_attr, d_dst) != cudaSuccess) {
    cudaGetLastError();  // the failed query's error is not sticky; clear it
    record_msg("lazy_copy_to_device: pointer query failed");
    return LAZY_ERR_INVALID_ARG;
  }
  if (src_attr.type != cudaMemoryTypeHost || !src_attr.devicePointer) {
    record_msg("lazy_copy_to_device: the source must be pinned, device-mapped host memory");
    return LAZY_ERR_INVALID_ARG;
  }
  int dev = 0, sms = 0;
  LAZY_CUDA_TRY(cudaGetDevice(&dev));
  if (dst_attr.type != cudaMemoryTypeDevice || dst_attr.device != dev) {
    record_msg("lazy_copy_to_device: the destination must be memory of the current device");
    return LAZY_ERR_INVALID_ARG;
  }
  LAZY_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const size_t n16 = bytes / 16;
  // One 16-byte chunk per thread, spread over every SM (the link's throughput grows with the
  // SMs issuing, not with the loads one SM keeps in flight), at most 8 blocks per SM; larger
  // copies loop with 4 loads in flight per thread.
  const size_t want = (n16 + kCopyThreads - 1) / kCopyThreads;
  const int grid = (int)std::min<size_t>(want, (size_t)sms * 8);
  h2d_copy_kernel<<<grid, kCopyThreads, 0, (cudaStream_t)stream>>>(
      reinterpret_cast<uint4 *>(d_dst), reinterpret_cast<const uint4 *>(src_attr.devicePointer),
      n16);
  LAZY_CUDA_TRY(cudaGetLastError());
  return LAZY_OK;
}
