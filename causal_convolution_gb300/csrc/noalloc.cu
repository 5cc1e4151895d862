// The output head for callers that cannot allocate device memory.
//
// cc_head_out needs a caller workspace for g, the 112-channel intermediate
// between its two stages. Some callers have no way to provide one: a host
// application or plugin framework that owns every device allocation and
// exposes no allocator to its plugins, or a latency-critical loop where a
// cudaMalloc (which can synchronise the whole device) is not allowed. For
// them, cc_head_out_noalloc keeps g in a fixed-size array in the library's
// own static device memory and runs the same two kernels as cc_head_out.
//
// Properties of the shared scratch array:
//  - It holds CC_HEAD_NOALLOC_SCRATCH_BYTES (64 MiB) on every GPU where this
//    library's device code is loaded, until the process exits.
//  - Every call on a device uses the same array and leaves its g behind.
//    Nothing in it has to start at zero: the temporal stage writes every
//    element of g that the stencil reads (all 112 channels of every
//    position) before the stencil runs.
//  - Two calls whose work overlaps on the GPU (different streams, or
//    different host threads without ordering) race on the array and
//    corrupt each other's results. Order such calls on one stream.
//  - Its device address is looked up on the first call on each device and
//    kept for the life of the process; a cudaDeviceReset() makes that address
//    stale, so the entry point is not to be used on a device after a reset.
#include <cuda_runtime.h>

#include <mutex>

#include "cc.h"
#include "cc_host.h"

namespace cc {
namespace {

static __device__ __align__(256) unsigned char g_head_scratch[CC_HEAD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// The device address of g_head_scratch on the current device. In host code
// the symbol itself is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
cc_status scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(CC_ERR_CUDA, "head_out_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(CC_ERR_UNSUPPORTED, "head_out_noalloc: device %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_head_scratch);
    if (e != cudaSuccess || !p)
      return fail(CC_ERR_CUDA, "head_out_noalloc: scratch address lookup failed: %s", cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return CC_OK;
}

}  // namespace
}  // namespace cc

using namespace cc;

extern "C" cc_status cc_head_out_noalloc(const cc_bf16* x, const cc_bf16* wp, const cc_bf16* bias, cc_bf16* out,
                                         int n, int d, int h, int w, int cin, int hist, void* stream) {
  const char* what = "head_out_noalloc";
  cc_status st;
  if (empty_request(what, {n, d, h, w}, &st)) return st;
  const long long positions = (long long)n * d * h * w;
  const long long max_positions = (long long)(CC_HEAD_NOALLOC_SCRATCH_BYTES / (CC_HEAD_G_CH * 2));
  if (positions > max_positions)
    return fail(CC_ERR_INVALID,
                "%s: %lld output positions need %lld bytes of scratch, but the built-in scratch holds %lld bytes "
                "(at most %lld positions); use cc_head_out with a workspace instead",
                what, positions, positions * CC_HEAD_G_CH * 2, (long long)CC_HEAD_NOALLOC_SCRATCH_BYTES,
                max_positions);
  void* g = nullptr;
  if ((st = scratch_address(&g)) != CC_OK) return st;
  if ((st = cc_head_temporal(x, wp, static_cast<cc_bf16*>(g), n, d, h, w, cin, hist, stream)) != CC_OK) return st;
  return cc_head_stencil(static_cast<const cc_bf16*>(g), bias, out, n, d, h, w, stream);
}
