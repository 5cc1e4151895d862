// Read-back of results into page-locked host memory by a copy kernel.
//
// A copy-engine device-to-host transfer that runs beside a host-to-device one
// takes about half of the host link from it (measured on GB300: each
// direction ~170 GB/s instead of ~210 / ~190). Stores issued by a few SMs to
// the mapped address of pinned host memory travel over the same link but at a
// rate set by the number of CTAs (4-8 CTAs: ~90 GB/s beside the inflowing
// copy), and leave the copy engine's host-to-device bandwidth nearly whole.
// In a chunked decode, where inputs stream in while earlier results stream
// out, that is what bounds the chunk time.
#include <cuda_runtime.h>

#include <cstdint>

#include "cc.h"
#include "cc_host.h"

namespace cc {
namespace {

constexpr int kCopyThreads = 512;
constexpr int kCopyMaxCtas = 1024;

// Grid-stride copy in 16-byte vectors, four loads in flight per thread before
// their stores. The source is read once (streaming loads).
__global__ void __launch_bounds__(kCopyThreads) copy_to_host_kernel(const uint4* __restrict__ src,
                                                                    uint4* __restrict__ dst, size_t n16) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = __ldcs(src + i);
    const uint4 b = __ldcs(src + i + stride);
    const uint4 c = __ldcs(src + i + 2 * stride);
    const uint4 d = __ldcs(src + i + 3 * stride);
    dst[i] = a;
    dst[i + stride] = b;
    dst[i + 2 * stride] = c;
    dst[i + 3 * stride] = d;
  }
  for (; i < n16; i += stride) dst[i] = __ldcs(src + i);
}

// True when p and the last byte of the range are memory of `type` that the
// device addresses at the same pointer.
bool addressable_as(const void* p, size_t bytes, cudaMemoryType type) {
  const char* ends[2] = {static_cast<const char*>(p), static_cast<const char*>(p) + bytes - 1};
  for (const char* q : ends) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, q) != cudaSuccess) {
      (void)cudaGetLastError();
      return false;
    }
    if (at.type != type || at.devicePointer != q) return false;
  }
  return true;
}

}  // namespace
}  // namespace cc

using namespace cc;

extern "C" cc_status cc_copy_to_host(void* dst, const void* src, size_t bytes, int ctas, void* stream) {
  const char* what = "copy_to_host";
  if (bytes == 0) return CC_OK;
  if (!dst || !src) return fail(CC_ERR_INVALID, "%s: null pointer", what);
  if (!aligned16(dst) || !aligned16(src)) return fail(CC_ERR_INVALID, "%s: pointers must be 16-byte aligned", what);
  if (bytes % 16 != 0) return fail(CC_ERR_INVALID, "%s: bytes must be a multiple of 16 (got %zu)", what, bytes);
  if (ctas < 1 || ctas > kCopyMaxCtas)
    return fail(CC_ERR_INVALID, "%s: ctas must be in 1..%d (got %d)", what, kCopyMaxCtas, ctas);
  if (!addressable_as(dst, bytes, cudaMemoryTypeHost))
    return fail(CC_ERR_INVALID, "%s: dst must be page-locked host memory the device can address", what);
  if (!addressable_as(src, bytes, cudaMemoryTypeDevice))
    return fail(CC_ERR_INVALID, "%s: src must be device memory", what);
  DeviceInfo di;  // the same device check as every other entry point
  cc_status st = device_info(&di);
  if (st != CC_OK) return st;
  copy_to_host_kernel<<<ctas, kCopyThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(src), static_cast<uint4*>(dst), bytes / 16);
  return launch_status(what);
}
