// Library runtime: error reporting, per-device facts, tensor-map encoding and
// the self-test entry points of cc_debug.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <mutex>

#include "cc.h"
#include "cc_debug.h"
#include "cc_host.h"
#include "cc_ptx.cuh"

namespace cc {

// The device error word: kernels OR DEVERR_* bits into it; cc_check_device
// reads and clears it.
__device__ unsigned int g_err_word;

namespace {
thread_local char t_msg[512] = "";

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_ok[kMaxDevices] = {};

PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;
PFN_cuTensorMapEncodeIm2col_v12000 g_encode_im2col = nullptr;

cc_status load_driver_entry_points() {
  if (g_encode_tiled && g_encode_im2col) return CC_OK;
  cudaDriverEntryPointQueryResult q1 = cudaDriverEntryPointSymbolNotFound, q2 = cudaDriverEntryPointSymbolNotFound;
  void* f1 = nullptr;
  void* f2 = nullptr;
  cudaError_t e1 = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f1, 12000, cudaEnableDefault, &q1);
  cudaError_t e2 = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &f2, 12000, cudaEnableDefault, &q2);
  if (e1 != cudaSuccess || e2 != cudaSuccess || q1 != cudaDriverEntryPointSuccess ||
      q2 != cudaDriverEntryPointSuccess || !f1 || !f2)
    return fail(CC_ERR_CUDA, "driver entry points for tensor-map encoding not found (%s / %s)",
                cudaGetErrorString(e1), cudaGetErrorString(e2));
  g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f1);
  g_encode_im2col = reinterpret_cast<PFN_cuTensorMapEncodeIm2col_v12000>(f2);
  return CC_OK;
}
}  // namespace

cc_status fail(cc_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_msg, sizeof(t_msg), fmt, ap);
  va_end(ap);
  return st;
}

bool empty_request(const char* what, std::initializer_list<long long> counts, cc_status* st) {
  bool empty = false;
  for (long long c : counts) {
    if (c < 0) {
      *st = fail(CC_ERR_INVALID, "%s: sizes must not be negative", what);
      return true;
    }
    empty = empty || c == 0;
  }
  *st = CC_OK;
  return empty;
}

cc_status launch_status(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(CC_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
  return CC_OK;
}

cc_status device_info(DeviceInfo* out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(CC_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(CC_ERR_UNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_dev_ok[dev]) {
    DeviceInfo di{};
    di.device = dev;
    e = cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(CC_ERR_CUDA, "SM count: %s", cudaGetErrorString(e));
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3)
      return fail(CC_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only", dev, major,
                  minor);
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_err_word);
    if (e != cudaSuccess) return fail(CC_ERR_CUDA, "error word address: %s", cudaGetErrorString(e));
    di.err_word = static_cast<unsigned int*>(p);
    cc_status st = load_driver_entry_points();
    if (st != CC_OK) return st;
    g_dev[dev] = di;
    g_dev_ok[dev] = true;
  }
  *out = g_dev[dev];
  return CC_OK;
}

static cc_status encode_result(CUresult r, const char* what) {
  if (r != CUDA_SUCCESS) return fail(CC_ERR_CUDA, "%s: tensor-map encoding failed (CUresult %d)", what, (int)r);
  return CC_OK;
}

cc_status encode_im2col_5d(CUtensorMap* map, const void* base, int n, int d, int h, int w, int c, int lo_w, int lo_h,
                           int lo_d, int up_w, int up_h, int up_d, int pixels, int channels) {
  const cuuint64_t dims[5] = {(cuuint64_t)c, (cuuint64_t)w, (cuuint64_t)h, (cuuint64_t)d, (cuuint64_t)n};
  const cuuint64_t es = 2;
  const cuuint64_t strides[4] = {es * c, es * c * w, es * c * w * h, es * c * w * h * d};
  // Corner arrays are ordered innermost spatial dimension first (W, H, D),
  // like the dimension arrays.
  const int lower[3] = {lo_w, lo_h, lo_d};
  const int upper[3] = {up_w, up_h, up_d};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return encode_result(g_encode_im2col(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims,
                                       strides, lower, upper, (cuuint32_t)channels, (cuuint32_t)pixels, estr,
                                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE),
                       "im2col map");
}

cc_status encode_tiled_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                          uint32_t box_inner, uint32_t box_outer) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return encode_result(g_encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                                      box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE),
                       "2-D map");
}

cc_status encode_tiled_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t stride1,
                          uint64_t stride2, uint32_t box0, uint32_t box1) {
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {stride1, stride2};
  const cuuint32_t box[3] = {box0, box1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode_result(g_encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                                      box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE),
                       "3-D map");
}

cc_status encode_tiled_3d_f32_sw128(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                                    uint64_t stride1, uint64_t stride2, uint32_t box0, uint32_t box1) {
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {stride1, stride2};
  const cuuint32_t box[3] = {box0, box1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode_result(g_encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides,
                                      box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE),
                       "3-D fp32 map");
}

cc_status encode_tiled_5d(CUtensorMap* map, const void* base, const uint64_t dims[5], const uint64_t strides[4],
                          uint32_t box0, uint32_t box1, uint32_t box2) {
  const cuuint64_t d[5] = {dims[0], dims[1], dims[2], dims[3], dims[4]};
  const cuuint64_t st[4] = {strides[0], strides[1], strides[2], strides[3]};
  const cuuint32_t box[5] = {box0, box1, box2, 1, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return encode_result(g_encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), d, st, box,
                                      estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE),
                       "5-D map");
}

cc_status encode_tiled_4d_dense(CUtensorMap* map, const void* base, const uint64_t dims[4], const uint64_t strides[3],
                                uint32_t box0, uint32_t box1, uint32_t box2) {
  const cuuint64_t d[4] = {dims[0], dims[1], dims[2], dims[3]};
  const cuuint64_t st[3] = {strides[0], strides[1], strides[2]};
  const cuuint32_t box[4] = {box0, box1, box2, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return encode_result(g_encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), d, st, box,
                                      estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE),
                       "4-D map");
}

// ------------------------------------------------------- self-test kernels --

// One im2col load into a 1024-aligned shared tile, then every thread copies
// 16-byte chunks out, undoing the 128-byte swizzle (chunk j of row r sits at
// chunk j ^ (r & 7)).
__global__ void __launch_bounds__(128) im2col_probe_kernel(const __grid_constant__ CUtensorMap tm, __nv_bfloat16* out,
                                                           int c0, int cw, int ch, int cd, int cn, int ow, int oh,
                                                           int od, unsigned int* err) {
  __shared__ __align__(1024) uint8_t tile[128 * 128];
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(smem_u32(&bar), 128 * 128);
    tma_load_im2col_5d(smem_u32(tile), &tm, smem_u32(&bar), c0, cw, ch, cd, cn, (uint16_t)ow, (uint16_t)oh,
                       (uint16_t)od);
  }
  const bool ok = mbar_wait(smem_u32(&bar), 0, err, 1000000000ull);
  __syncthreads();
  if (!ok) return;
  for (int i = threadIdx.x; i < 128 * 8; i += blockDim.x) {
    const int r = i >> 3, j = i & 7;
    const uint4 v = *reinterpret_cast<const uint4*>(tile + r * 128 + ((j ^ (r & 7)) << 4));
    reinterpret_cast<uint4*>(out)[r * 8 + j] = v;
  }
}

__global__ void wait_timeout_kernel(unsigned long long limit_ns, unsigned int* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  // Nothing ever arrives on `bar`: the bounded wait must give up.
  (void)mbar_wait(smem_u32(&bar), 0, err, limit_ns);
}

}  // namespace cc

using namespace cc;

extern "C" const char* cc_last_error(void) { return t_msg; }

extern "C" int cc_version(void) { return 100; }

extern "C" cc_status cc_check_device(void* stream) {
  DeviceInfo di;
  cc_status st = device_info(&di);
  if (st != CC_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(CC_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
  unsigned int word = 0;
  e = cudaMemcpy(&word, di.err_word, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(CC_ERR_CUDA, "error word read: %s", cudaGetErrorString(e));
  if (word == 0) return CC_OK;
  const unsigned int zero = 0;
  e = cudaMemcpy(di.err_word, &zero, sizeof(zero), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return fail(CC_ERR_CUDA, "error word clear: %s", cudaGetErrorString(e));
  if (word & DEVERR_TIMEOUT) return fail(CC_ERR_TIMEOUT, "a kernel wait exceeded its time limit (word 0x%x)", word);
  return fail(CC_ERR_DEVICE, "a kernel index check failed (word 0x%x)", word);
}

extern "C" cc_status cc_debug_im2col_tile(const cc_bf16* x, cc_bf16* tile, int n, int d_in, int h, int w, int c,
                                          int lo_w, int lo_h, int lo_d, int up_w, int up_h, int up_d, int c0, int cw,
                                          int ch, int cd, int cn, int ow, int oh, int od, void* stream) {
  if (!x || !tile) return fail(CC_ERR_INVALID, "im2col probe: null pointer");
  if (!aligned16(x) || !aligned16(tile)) return fail(CC_ERR_INVALID, "im2col probe: pointers must be 16-byte aligned");
  if (n <= 0 || d_in <= 0 || h <= 0 || w <= 0 || c <= 0 || c % 64 != 0)
    return fail(CC_ERR_INVALID, "im2col probe: bad shape");
  if (c0 < 0 || c0 % 64 != 0 || c0 >= c) return fail(CC_ERR_INVALID, "im2col probe: c0 must be a multiple of 64 < C");
  const int corners[6] = {lo_w, lo_h, lo_d, up_w, up_h, up_d};
  for (int v : corners)
    if (v < -16 || v > 15) return fail(CC_ERR_INVALID, "im2col probe: corners must lie in [-16, 15]");
  if (ow < 0 || oh < 0 || od < 0 || ow > 255 || oh > 255 || od > 255)
    return fail(CC_ERR_INVALID, "im2col probe: offsets must lie in [0, 255]");
  DeviceInfo di;
  cc_status st = device_info(&di);
  if (st != CC_OK) return st;
  CUtensorMap tm;
  st = encode_im2col_5d(&tm, x, n, d_in, h, w, c, lo_w, lo_h, lo_d, up_w, up_h, up_d, 128, 64);
  if (st != CC_OK) return st;
  im2col_probe_kernel<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(
      tm, reinterpret_cast<__nv_bfloat16*>(tile), c0, cw, ch, cd, cn, ow, oh, od, di.err_word);
  return launch_status("im2col probe");
}

extern "C" cc_status cc_debug_wait_timeout(int64_t limit_ns, void* stream) {
  if (limit_ns <= 0 || limit_ns > 1000000000LL) return fail(CC_ERR_INVALID, "wait probe: limit must be in (0, 1 s]");
  DeviceInfo di;
  cc_status st = device_info(&di);
  if (st != CC_OK) return st;
  wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>((unsigned long long)limit_ns, di.err_word);
  return launch_status("wait probe");
}
