// Bandwidth-bound passes: the resampler's interleave (phases + bias +
// shortcut -> high-resolution tensor) and the head's 3x3 stencil (g -> 12
// clamped channels), plus the composite resampler and head entry points.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "cc.h"
#include "cc_host.h"
#include "cc_ptx.cuh"

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

// Head stencil, persistent. A tile is 8 output rows x 32 output positions of
// one frame; it needs the g window of rows h0-1 .. h0+8 and positions
// w0-1 .. w0+32 with all 112 channels, which one rank-4 TMA box copies into
// shared memory (zero-filled outside the plane, so the plane's zero padding
// costs nothing). Each CTA walks tiles with a 3-deep ring of windows: while it
// sums one tile, the next two are in flight. Three threads share an output
// position, each summing 4 of its 12 channels over the nine (i, j) blocks
// (8-byte shared reads), adding the bias, clamping and storing 8 bytes, so a
// warp's stores form one contiguous run.
constexpr int kStTW = 32;                                  // output positions per tile row
constexpr int kStTH = 8;                                   // output rows per tile
constexpr int kStPos = kStTW + 2;                          // positions held (with halo)
constexpr int kStRows = kStTH + 2;                         // rows held (with halo)
constexpr int kStBox = kStRows * kStPos * CC_HEAD_G_CH * 2;  // 76,160 bytes per window
constexpr int kStStages = 3;
constexpr int kStThreads = kStTW * kStTH * 3;
constexpr int kStSmem = 1024 + kStStages * kStBox + 64;

struct StencilArgs {
  int h, w;
  int strips, hblocks, tiles;
  const __nv_bfloat16* bias;
  __nv_bfloat16* out;
  unsigned int* err;
  unsigned long long timeout_ns;
};

__device__ __forceinline__ void stencil_tile_coords(const StencilArgs& a, int t, int& frame, int& hb, int& wb) {
  wb = t % a.strips;
  const int r = t / a.strips;
  hb = r % a.hblocks;
  frame = r / a.hblocks;
}

__global__ void __launch_bounds__(kStThreads, 1)
    head_stencil_kernel(const __grid_constant__ CUtensorMap tmG, const __grid_constant__ StencilArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStStages * kStBox);
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < kStStages; ++s) mbar_init(smem_u32(&full[s]), 1);
    fence_mbar_init();
    tma_prefetch_map(&tmG);
  }
  __syncthreads();
  // set up: let the next kernel on the stream be scheduled, then wait for the
  // previous one before the first global access
  pdl_launch_dependents();
  pdl_wait();

  auto issue = [&](int t, int s) {
    int frame, hb, wb;
    stencil_tile_coords(a, t, frame, hb, wb);
    const uint32_t bar = smem_u32(&full[s]);
    mbar_arrive_expect_tx(bar, kStBox);
    tma_load_4d(smem_u32(smem + s * kStBox), &tmG, bar, 0, wb * kStTW - 1, hb * kStTH - 1, frame);
  };
  // Tile iteration j of this CTA is tile blockIdx.x + j*gridDim.x, held in
  // stage j % kStStages; its load is issued kStStages - 1 iterations early.
  const int iters = (a.tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
  if (tid == 0)
    for (int j = 0; j < kStStages - 1 && j < iters; ++j) issue(blockIdx.x + j * gridDim.x, j);
  const int cg = tid % 3;     // channels 4*cg .. 4*cg+3
  const int pix = tid / 3;
  const int p = pix % kStTW;
  const int r = pix / kStTW;
  float b4[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) b4[e] = __bfloat162float(a.bias[cg * 4 + e]);

  int k = 0;
  for (int t = blockIdx.x; t < a.tiles; t += gridDim.x, ++k) {
    const int stage = k % kStStages;
    const bool ok = mbar_wait(smem_u32(&full[stage]), (k / kStStages) & 1, a.err, a.timeout_ns);
    // one barrier per tile: every thread is done with tile k-1 here, so its
    // window's stage may be refilled; a failed wait stops the whole CTA
    if (__syncthreads_or(!ok)) break;
    if (tid == 0 && k + kStStages - 1 < iters) issue(t + (kStStages - 1) * gridDim.x, (k + kStStages - 1) % kStStages);
    int frame, hb, wb;
    stencil_tile_coords(a, t, frame, hb, wb);
    const int oh = hb * kStTH + r;
    const int ow = wb * kStTW + p;
    const uint8_t* win = smem + stage * kStBox;
    float acc[4] = {b4[0], b4[1], b4[2], b4[3]};
#pragma unroll
    for (int i = 0; i < 3; ++i) {
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        // g at (oh + i - 1, ow + j - 1) is held at row r + i, position p + j
        const uint2 u = *reinterpret_cast<const uint2*>(
            win + (((r + i) * kStPos + p + j) * CC_HEAD_G_CH + (i * 3 + j) * CC_HEAD_COUT + cg * 4) * 2);
        const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&u);
        const float2 f0 = __bfloat1622float2(hv[0]);
        const float2 f1 = __bfloat1622float2(hv[1]);
        acc[0] += f0.x;
        acc[1] += f0.y;
        acc[2] += f1.x;
        acc[3] += f1.y;
      }
    }
    if (oh < a.h && ow < a.w) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(fminf(1.f, fmaxf(-1.f, acc[0])), fminf(1.f, fmaxf(-1.f, acc[1])));
      __nv_bfloat162 hi = __floats2bfloat162_rn(fminf(1.f, fmaxf(-1.f, acc[2])), fminf(1.f, fmaxf(-1.f, acc[3])));
      uint2 u;
      u.x = *reinterpret_cast<uint32_t*>(&lo);
      u.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(a.out + (((long long)frame * a.h + oh) * a.w + ow) * CC_HEAD_COUT + cg * 4) = u;
    }
  }
  if (tid == 0) {
    // after a failed wait, let the copies still in flight (iterations k ..
    // k + kStStages - 2) land before the CTA exits
    for (int j = k; j < iters && j < k + kStStages - 1; ++j)
      (void)mbar_wait(smem_u32(&full[j % kStStages]), (j / kStStages) & 1, a.err, 200000000ull);
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
  if (empty_request(what, {n, d, hl, wl}, &st)) return st;
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
  cc_status st;
  if (empty_request(what, {n, d, hl, wl}, &st)) return st;
  if ((st = check_ptr(what, ws)) != CC_OK) return st;
  const size_t need = cc_resample_workspace_bytes(n, d, hl, wl, cout);
  if (need == 0) return fail(CC_ERR_INVALID, "%s: channel counts must be positive", what);
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
  if (empty_request(what, {n, d, h, w}, &st)) return st;
  if ((st = check_ptr(what, g)) != CC_OK || (st = check_ptr(what, bias)) != CC_OK ||
      (st = check_ptr(what, out)) != CC_OK)
    return st;
  if (n <= 0 || d <= 0 || h <= 0 || w <= 0) return fail(CC_ERR_INVALID, "%s: sizes must be positive", what);
  const long long frames = (long long)n * d;
  const long long strips = (w + kStTW - 1) / kStTW, hblocks = (h + kStTH - 1) / kStTH;
  if (frames * strips * hblocks > (1LL << 31) - 1 || frames * h * w > (1LL << 40))
    return fail(CC_ERR_UNSUPPORTED, "%s: tensor too large", what);
  DeviceInfo di;
  if ((st = device_info(&di)) != CC_OK) return st;
  CUtensorMap tm;
  const uint64_t dims[4] = {CC_HEAD_G_CH, (uint64_t)w, (uint64_t)h, (uint64_t)frames};
  const uint64_t strides[3] = {CC_HEAD_G_CH * 2ull, CC_HEAD_G_CH * 2ull * w, CC_HEAD_G_CH * 2ull * w * h};
  if ((st = encode_tiled_4d_dense(&tm, g, dims, strides, CC_HEAD_G_CH, kStPos, kStRows)) != CC_OK) return st;
  StencilArgs a{};
  a.h = h;
  a.w = w;
  a.strips = (int)strips;
  a.hblocks = (int)hblocks;
  a.tiles = (int)(frames * strips * hblocks);
  a.bias = reinterpret_cast<const __nv_bfloat16*>(bias);
  a.out = reinterpret_cast<__nv_bfloat16*>(out);
  a.err = di.err_word;
  a.timeout_ns = kWaitLimitNs;
  cudaError_t e = cudaFuncSetAttribute(head_stencil_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kStSmem);
  if (e != cudaSuccess) return fail(CC_ERR_CUDA, "%s: shared-memory attribute: %s", what, cudaGetErrorString(e));
  e = launch_pdl(head_stencil_kernel, dim3(std::min(a.tiles, di.sm_count)), dim3(kStThreads), kStSmem,
                 static_cast<cudaStream_t>(stream), tm, a);
  if (e != cudaSuccess) return fail(CC_ERR_CUDA, "%s: launch: %s", what, cudaGetErrorString(e));
  return launch_status(what);
}

extern "C" cc_status cc_head_out(const cc_bf16* x, const cc_bf16* wp, const cc_bf16* bias, cc_bf16* out, int n, int d,
                                 int h, int w, int cin, int hist, void* ws, size_t ws_bytes, void* stream) {
  const char* what = "head_out";
  cc_status st;
  if (empty_request(what, {n, d, h, w}, &st)) return st;
  if ((st = check_ptr(what, ws)) != CC_OK) return st;
  const size_t need = cc_head_workspace_bytes(n, d, h, w);
  if (ws_bytes < need) return fail(CC_ERR_INVALID, "%s: workspace of %zu bytes, need %zu", what, ws_bytes, need);
  cc_bf16* g = static_cast<cc_bf16*>(ws);
  if ((st = cc_head_temporal(x, wp, g, n, d, h, w, cin, hist, stream)) != CC_OK) return st;
  return cc_head_stencil(g, bias, out, n, d, h, w, stream);
}
