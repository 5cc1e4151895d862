// Bandwidth-bound passes: the resampler's interleave (phases + bias +
// shortcut -> high-resolution tensor) and the head's 3x3 stencil (g -> 12
// clamped channels), plus the composite resampler and head entry points.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "cc.h"
#include "cc_host.h"

namespace cc {
namespace {

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

__device__ __forceinline__ uint4 f32_to_bf16x8(const float (&f)[8]) {
  uint4 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return u;
}

// One thread per (low-resolution pixel, 8-channel vector): reads the four
// phase values, the shortcut source and the bias once and writes the 2x2
// output block. The grid carries the low-resolution row (y) and the position
// inside the row (x); each warp covers 32 consecutive 16-byte vectors, so
// every load and store is a contiguous 512-byte run.
__global__ void __launch_bounds__(256) interleave_kernel(const uint4* __restrict__ ph, const uint4* __restrict__ bias,
                                                         const uint4* __restrict__ skip, uint4* __restrict__ out,
                                                         int rows, int hl, int wl, int cv, long long phase_vecs) {
  const int per_row = wl * cv;
  for (int r = blockIdx.y; r < rows; r += gridDim.y) {
    const int i = r % hl;
    const long long frame = r / hl;
    const long long in_row = (long long)r * per_row;
    const long long out0 = ((frame * hl + i) * 2) * (long long)(2 * per_row);
    const long long out1 = out0 + 2LL * per_row;
    for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < per_row; idx += gridDim.x * blockDim.x) {
      const int j = idx / cv;
      const int c8 = idx - j * cv;
      const long long src = in_row + idx;
      const uint4 u00 = __ldcs(ph + src);
      const uint4 u01 = __ldcs(ph + phase_vecs + src);
      const uint4 u10 = __ldcs(ph + 2 * phase_vecs + src);
      const uint4 u11 = __ldcs(ph + 3 * phase_vecs + src);
      const uint4 us = __ldcs(skip + src);
      const uint4 ub = __ldg(bias + c8);
      float fb[8], fs[8], f[8];
      bf16x8_to_f32(ub, fb);
      bf16x8_to_f32(us, fs);
#pragma unroll
      for (int e = 0; e < 8; ++e) fs[e] += fb[e];
      const long long o = (long long)(2 * j) * cv + c8;
      bf16x8_to_f32(u00, f);
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] += fs[e];
      __stcs(out + out0 + o, f32_to_bf16x8(f));
      bf16x8_to_f32(u01, f);
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] += fs[e];
      __stcs(out + out0 + o + cv, f32_to_bf16x8(f));
      bf16x8_to_f32(u10, f);
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] += fs[e];
      __stcs(out + out1 + o, f32_to_bf16x8(f));
      bf16x8_to_f32(u11, f);
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] += fs[e];
      __stcs(out + out1 + o + cv, f32_to_bf16x8(f));
    }
  }
}

// One thread per output position: 12 fp32 accumulators start at the bias and
// take channel block (i, j) of g from the neighbour (h+i-1, w+j-1), skipping
// neighbours outside the plane; clamp, one bf16 rounding, 24-byte store.
__global__ void __launch_bounds__(128) head_stencil_kernel(const __nv_bfloat16* __restrict__ g,
                                                           const __nv_bfloat16* __restrict__ bias,
                                                           __nv_bfloat16* __restrict__ out, int rows, int h, int w) {
  float b[CC_HEAD_COUT];
#pragma unroll
  for (int c = 0; c < CC_HEAD_COUT; ++c) b[c] = __bfloat162float(bias[c]);
  for (int r = blockIdx.y; r < rows; r += gridDim.y) {
    const int hh = r % h;
    for (int x = blockIdx.x * blockDim.x + threadIdx.x; x < w; x += gridDim.x * blockDim.x) {
      float acc[CC_HEAD_COUT];
#pragma unroll
      for (int c = 0; c < CC_HEAD_COUT; ++c) acc[c] = b[c];
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        const int gh = hh + i - 1;
        if (gh < 0 || gh >= h) continue;
        const long long grow = (long long)(r + i - 1) * w;
#pragma unroll
        for (int j = 0; j < 3; ++j) {
          const int gw = x + j - 1;
          if (gw < 0 || gw >= w) continue;
          const uint2* src =
              reinterpret_cast<const uint2*>(g + (grow + gw) * CC_HEAD_G_CH + (i * 3 + j) * CC_HEAD_COUT);
#pragma unroll
          for (int k = 0; k < 3; ++k) {
            const uint2 u = __ldg(src + k);
            const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&u);
            const float2 f0 = __bfloat1622float2(hv[0]);
            const float2 f1 = __bfloat1622float2(hv[1]);
            acc[4 * k] += f0.x;
            acc[4 * k + 1] += f0.y;
            acc[4 * k + 2] += f1.x;
            acc[4 * k + 3] += f1.y;
          }
        }
      }
      uint2* dst = reinterpret_cast<uint2*>(out + ((long long)r * w + x) * CC_HEAD_COUT);
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(fminf(1.f, fmaxf(-1.f, acc[4 * k])), fminf(1.f, fmaxf(-1.f, acc[4 * k + 1])));
        __nv_bfloat162 hi =
            __floats2bfloat162_rn(fminf(1.f, fmaxf(-1.f, acc[4 * k + 2])), fminf(1.f, fmaxf(-1.f, acc[4 * k + 3])));
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&lo);
        u.y = *reinterpret_cast<uint32_t*>(&hi);
        dst[k] = u;
      }
    }
  }
}

cc_status check_ptr(const char* what, const void* p) {
  if (!p) return fail(CC_ERR_INVALID, "%s: null pointer", what);
  if (!aligned16(p)) return fail(CC_ERR_INVALID, "%s: pointers must be 16-byte aligned", what);
  return CC_OK;
}

}  // namespace
}  // namespace cc

using namespace cc;

extern "C" size_t cc_resample_workspace_bytes(int n, int d, int hl, int wl, int cout) {
  if (n <= 0 || d <= 0 || hl <= 0 || wl <= 0 || cout <= 0) return 0;
  return 4ull * n * d * hl * wl * cout * 2;
}

extern "C" cc_status cc_resample_interleave(const cc_bf16* phases, const cc_bf16* bias, const cc_bf16* skip,
                                            cc_bf16* out, int n, int d, int hl, int wl, int c, void* stream) {
  const char* what = "resample_interleave";
  cc_status st;
  if ((st = check_ptr(what, phases)) != CC_OK || (st = check_ptr(what, bias)) != CC_OK ||
      (st = check_ptr(what, skip)) != CC_OK || (st = check_ptr(what, out)) != CC_OK)
    return st;
  if (n <= 0 || d <= 0 || hl <= 0 || wl <= 0 || c <= 0) return fail(CC_ERR_INVALID, "%s: sizes must be positive", what);
  if (c % 8 != 0) return fail(CC_ERR_UNSUPPORTED, "%s: C must be a multiple of 8 (got %d)", what, c);
  const long long rows = (long long)n * d * hl;
  const long long per_row = (long long)wl * (c / 8);
  if (rows > (1LL << 31) - 1 || per_row > (1LL << 30)) return fail(CC_ERR_UNSUPPORTED, "%s: tensor too large", what);
  DeviceInfo di;
  if ((st = device_info(&di)) != CC_OK) return st;
  const int threads = 256;
  const unsigned gx = (unsigned)std::min<long long>((per_row + threads - 1) / threads, 65535);
  const unsigned gy = (unsigned)std::min<long long>(rows, 65535);
  interleave_kernel<<<dim3(gx, gy), threads, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(phases), reinterpret_cast<const uint4*>(bias),
      reinterpret_cast<const uint4*>(skip), reinterpret_cast<uint4*>(out), (int)rows, hl, wl, c / 8,
      rows * per_row);
  return launch_status(what);
}

extern "C" cc_status cc_resample_up2(const cc_bf16* x, const cc_bf16* pw, const cc_bf16* bias, const cc_bf16* skip,
                                     cc_bf16* out, int n, int d, int hl, int wl, int cin, int cout, int hist,
                                     void* ws, size_t ws_bytes, void* stream) {
  const char* what = "resample_up2";
  cc_status st = check_ptr(what, ws);
  if (st != CC_OK) return st;
  const size_t need = cc_resample_workspace_bytes(n, d, hl, wl, cout);
  if (need == 0) return fail(CC_ERR_INVALID, "%s: sizes must be positive", what);
  if (ws_bytes < need) return fail(CC_ERR_INVALID, "%s: workspace of %zu bytes, need %zu", what, ws_bytes, need);
  cc_bf16* phases = static_cast<cc_bf16*>(ws);
  if ((st = cc_resample_phase_conv(x, pw, phases, n, d, hl, wl, cin, cout, hist, stream)) != CC_OK) return st;
  return cc_resample_interleave(phases, bias, skip, out, n, d, hl, wl, cout, stream);
}

extern "C" size_t cc_head_workspace_bytes(int n, int d, int h, int w) {
  if (n <= 0 || d <= 0 || h <= 0 || w <= 0) return 0;
  return (size_t)n * d * h * w * CC_HEAD_G_CH * 2;
}

extern "C" cc_status cc_head_stencil(const cc_bf16* g, const cc_bf16* bias, cc_bf16* out, int n, int d, int h, int w,
                                     void* stream) {
  const char* what = "head_stencil";
  cc_status st;
  if ((st = check_ptr(what, g)) != CC_OK || (st = check_ptr(what, bias)) != CC_OK ||
      (st = check_ptr(what, out)) != CC_OK)
    return st;
  if (n <= 0 || d <= 0 || h <= 0 || w <= 0) return fail(CC_ERR_INVALID, "%s: sizes must be positive", what);
  const long long rows = (long long)n * d * h;
  if (rows > (1LL << 31) - 1 || (long long)rows * w > (1LL << 40))
    return fail(CC_ERR_UNSUPPORTED, "%s: tensor too large", what);
  DeviceInfo di;
  if ((st = device_info(&di)) != CC_OK) return st;
  const int threads = 128;
  const unsigned gx = (unsigned)std::min<long long>((w + threads - 1) / threads, 65535);
  const unsigned gy = (unsigned)std::min<long long>(rows, 65535);
  head_stencil_kernel<<<dim3(gx, gy), threads, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const __nv_bfloat16*>(g), reinterpret_cast<const __nv_bfloat16*>(bias),
      reinterpret_cast<__nv_bfloat16*>(out), (int)rows, h, w);
  return launch_status(what);
}

extern "C" cc_status cc_head_out(const cc_bf16* x, const cc_bf16* wp, const cc_bf16* bias, cc_bf16* out, int n, int d,
                                 int h, int w, int cin, int hist, void* ws, size_t ws_bytes, void* stream) {
  const char* what = "head_out";
  cc_status st = check_ptr(what, ws);
  if (st != CC_OK) return st;
  const size_t need = cc_head_workspace_bytes(n, d, h, w);
  if (need == 0) return fail(CC_ERR_INVALID, "%s: sizes must be positive", what);
  if (ws_bytes < need) return fail(CC_ERR_INVALID, "%s: workspace of %zu bytes, need %zu", what, ws_bytes, need);
  cc_bf16* g = static_cast<cc_bf16*>(ws);
  if ((st = cc_head_temporal(x, wp, g, n, d, h, w, cin, hist, stream)) != CC_OK) return st;
  return cc_head_stencil(g, bias, out, n, d, h, w, stream);
}
