// The convolutions: the causal 3x3x3 conv and the resampler's four phase
// convs -- one tcgen05 implicit GEMM fed by an im2col TMA map over the
// channels-last input -- and their weight repacks.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "cc.h"
#include "cc_gemm_launch.cuh"
#include "cc_host.h"

namespace cc {
namespace {

constexpr long long kMaxPositions = (1LL << 31) - 1024;

__device__ __forceinline__ float bf(const __nv_bfloat16* p, long long i) { return __bfloat162float(p[i]); }

// wp[tap][co][ci] = w[co][ci][tap], tap = kt*9 + kh*3 + kw.
__global__ void conv_prepare_kernel(const __nv_bfloat16* __restrict__ w, __nv_bfloat16* __restrict__ wp, int cout,
                                    int cin) {
  const long long total = 27LL * cout * cin;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
    const int ci = static_cast<int>(i % cin);
    const long long r = i / cin;
    const int co = static_cast<int>(r % cout);
    const int tap = static_cast<int>(r / cout);
    wp[i] = w[((long long)co * cin + ci) * 27 + tap];
  }
}

// Phase kernels: for output parity p and phase tap a the 3x3 rows that land on
// low-resolution row i + p - 1 + a are {0} / {1,2} (p = 0) and {0,1} / {2}
// (p = 1); columns likewise. Sums in fp32, one rounding.
__global__ void resample_prepare_kernel(const __nv_bfloat16* __restrict__ w, __nv_bfloat16* __restrict__ pw, int cout,
                                        int cin) {
  const long long total = 48LL * cout * cin;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
    const int ci = static_cast<int>(i % cin);
    long long r = i / cin;
    const int co = static_cast<int>(r % cout);
    r /= cout;
    const int tap = static_cast<int>(r % 12);
    const int phase = static_cast<int>(r / 12);
    const int p = phase >> 1, q = phase & 1;
    const int kt = tap >> 2, a = (tap >> 1) & 1, b = tap & 1;
    const int r_lo = (p == 0) ? (a == 0 ? 0 : 1) : (a == 0 ? 0 : 2);
    const int r_hi = (p == 0) ? (a == 0 ? 0 : 2) : (a == 0 ? 1 : 2);
    const int c_lo = (q == 0) ? (b == 0 ? 0 : 1) : (b == 0 ? 0 : 2);
    const int c_hi = (q == 0) ? (b == 0 ? 0 : 2) : (b == 0 ? 1 : 2);
    const long long base = ((long long)co * cin + ci) * 27 + kt * 9;
    float s = 0.f;
    for (int kh = r_lo; kh <= r_hi; ++kh)
      for (int kw = c_lo; kw <= c_hi; ++kw) s += bf(w, base + kh * 3 + kw);
    pw[i] = __float2bfloat16_rn(s);
  }
}

// Temporal variant: 8 phases (s, p, q) x 8 taps (a, b, c). Taps kt of output
// frame 2t+s that land on low-resolution frame t-1+a are {0,1} / {2} (s = 0)
// and {0} / {1,2} (s = 1) -- causal alignment; rows and columns as above.
__global__ void resample_prepare_temporal_kernel(const __nv_bfloat16* __restrict__ w, __nv_bfloat16* __restrict__ pw,
                                                 int cout, int cin) {
  const long long total = 64LL * cout * cin;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
    const int ci = static_cast<int>(i % cin);
    long long r = i / cin;
    const int co = static_cast<int>(r % cout);
    r /= cout;
    const int tap = static_cast<int>(r % 8);
    const int phase = static_cast<int>(r / 8);
    const int s = phase >> 2, p = (phase >> 1) & 1, q = phase & 1;
    const int a = tap >> 2, b = (tap >> 1) & 1, c = tap & 1;
    const int t_lo = (s == 0) ? (a == 0 ? 0 : 2) : (a == 0 ? 0 : 1);
    const int t_hi = (s == 0) ? (a == 0 ? 1 : 2) : (a == 0 ? 0 : 2);
    const int r_lo = (p == 0) ? (b == 0 ? 0 : 1) : (b == 0 ? 0 : 2);
    const int r_hi = (p == 0) ? (b == 0 ? 0 : 2) : (b == 0 ? 1 : 2);
    const int c_lo = (q == 0) ? (c == 0 ? 0 : 1) : (c == 0 ? 0 : 2);
    const int c_hi = (q == 0) ? (c == 0 ? 0 : 2) : (c == 0 ? 1 : 2);
    const long long base = ((long long)co * cin + ci) * 27;
    float acc = 0.f;
    for (int kt = t_lo; kt <= t_hi; ++kt)
      for (int kh = r_lo; kh <= r_hi; ++kh)
        for (int kw = c_lo; kw <= c_hi; ++kw) acc += bf(w, base + kt * 9 + kh * 3 + kw);
    pw[i] = __float2bfloat16_rn(acc);
  }
}

cc_status check_ptrs(const char* what, std::initializer_list<const void*> ptrs) {
  for (const void* p : ptrs) {
    if (!p) return fail(CC_ERR_INVALID, "%s: null pointer", what);
    if (!aligned16(p)) return fail(CC_ERR_INVALID, "%s: pointers must be 16-byte aligned", what);
  }
  return CC_OK;
}

cc_status check_grid(const char* what, int n, int d, int h, int w, int hist) {
  if (n <= 0 || d <= 0 || h <= 0 || w <= 0) return fail(CC_ERR_INVALID, "%s: sizes must be positive", what);
  if (hist != 0 && hist != 2) return fail(CC_ERR_INVALID, "%s: hist must be 0 or 2", what);
  if ((long long)n * d * h * w > kMaxPositions) return fail(CC_ERR_UNSUPPORTED, "%s: too many positions", what);
  return CC_OK;
}

int prep_grid(long long total) { return static_cast<int>(std::min<long long>((total + 255) / 256, 8192)); }

}  // namespace
}  // namespace cc

using namespace cc;

extern "C" cc_status cc_conv3d_prepare(const cc_bf16* w, cc_bf16* wp, int cout, int cin, void* stream) {
  cc_status st = check_ptrs("conv3d_prepare", {w, wp});
  if (st != CC_OK) return st;
  if (cout <= 0 || cin <= 0) return fail(CC_ERR_INVALID, "conv3d_prepare: sizes must be positive");
  DeviceInfo di;
  if ((st = device_info(&di)) != CC_OK) return st;
  conv_prepare_kernel<<<prep_grid(27LL * cout * cin), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const __nv_bfloat16*>(w), reinterpret_cast<__nv_bfloat16*>(wp), cout, cin);
  return launch_status("conv3d_prepare");
}

namespace cc {
namespace {

// The causal conv; bad_entry >= 0 (self test only) replaces that entry of the
// pair tiles' walking order by one past every row tile.
cc_status conv3d_causal_impl(const char* what, const cc_bf16* x, const cc_bf16* wp, const cc_bf16* bias, cc_bf16* y,
                             int n, int d, int h, int w, int cin, int cout, int hist, void* stream, int bad_entry) {
  cc_status st;
  if (empty_request(what, {n, d, h, w}, &st)) return st;
  if ((st = check_ptrs(what, {x, wp, y})) != CC_OK) return st;
  if (bias && !aligned16(bias)) return fail(CC_ERR_INVALID, "%s: bias must be 16-byte aligned", what);
  if ((st = check_grid(what, n, d, h, w, hist)) != CC_OK) return st;
  if (cin <= 0 || cout <= 0) return fail(CC_ERR_INVALID, "%s: channel counts must be positive", what);
  if (cin % 64 != 0) return fail(CC_ERR_UNSUPPORTED, "%s: C_in must be a multiple of 64 (got %d)", what, cin);
  if (cout % 16 != 0) return fail(CC_ERR_UNSUPPORTED, "%s: C_out must be a multiple of 16 (got %d)", what, cout);
  DeviceInfo di;
  if ((st = device_info(&di)) != CC_OK) return st;

  const int lo_d = hist ? 0 : -2;
  CUtensorMap ta, tb;
  if ((st = encode_im2col_5d(&ta, x, n, d + hist, h, w, cin, -1, -1, lo_d, -1, -1, -2, kBlockM, kBlockK)) != CC_OK)
    return st;
  const long long m = (long long)n * d * h * w;
  // two or more 128-row tiles: 256 x 256 tiles on CTA pairs, each CTA
  // loading half of B (128 rows per box)
  const bool pair = m > kBlockM;
  if ((st = encode_tiled_2d(&tb, wp, cin, 27ull * cout, 2ull * cin, kBlockK, pair ? 128 : 256)) != CC_OK) return st;

  GemmArgs a{};
  a.m_total = static_cast<int>(m);
  a.n_total = cout;
  a.m_tiles = ceil_div(m, kBlockM);
  a.n_tiles = ceil_div(cout, 256);
  a.batches = 1;
  a.num_tiles = a.m_tiles * a.n_tiles;
  a.taps = 27;
  a.kb_per_tap = cin / kBlockK;
  a.img_w = w;
  a.img_h = h;
  a.img_d = d;
  a.lo_w = -1;
  a.lo_h = -1;
  a.lo_d = lo_d;
  for (int kt = 0; kt < 3; ++kt)
    for (int kh = 0; kh < 3; ++kh)
      for (int kw = 0; kw < 3; ++kw) a.tap_off[kt * 9 + kh * 3 + kw] = kw | (kh << 8) | (kt << 16);
  a.b_rows_per_tap = cout;
  a.b_rows_per_batch = 0;
  a.out = y;
  a.out_ld = cout;
  a.out_batch = 0;
  a.bias = reinterpret_cast<const __nv_bfloat16*>(bias);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (pair) {
    set_frame_interleaved_order(a);
    if (bad_entry >= 0) {
      if (bad_entry >= a.mp_perm_n) return fail(CC_ERR_INVALID, "%s: no walking-order entry %d", what, bad_entry);
      a.mp_perm[bad_entry] = 0xFFFF;
    }
    if (bias) return launch_tc_gemm_pair<256, kAIm2col, false, false, true>(ta, tb, a, di, s, what);
    return launch_tc_gemm_pair<256, kAIm2col, false, false, false>(ta, tb, a, di, s, what);
  }
  if (bad_entry >= 0) return fail(CC_ERR_INVALID, "%s: one row tile has no walking order", what);
  if (bias) return launch_tc_gemm<256, kAIm2col, false, false, true>(ta, tb, a, di, s, what);
  return launch_tc_gemm<256, kAIm2col, false, false, false>(ta, tb, a, di, s, what);
}

}  // namespace
}  // namespace cc

extern "C" cc_status cc_conv3d_causal(const cc_bf16* x, const cc_bf16* wp, const cc_bf16* bias, cc_bf16* y, int n,
                                      int d, int h, int w, int cin, int cout, int hist, void* stream) {
  return conv3d_causal_impl("conv3d_causal", x, wp, bias, y, n, d, h, w, cin, cout, hist, stream, -1);
}

extern "C" cc_status cc_debug_conv_bad_tile_order(const cc_bf16* x, const cc_bf16* wp, cc_bf16* y, int n, int d,
                                                  int h, int w, int cin, int cout, int entry, void* stream) {
  if (entry < 0) return fail(CC_ERR_INVALID, "conv bad-order probe: entry must be >= 0");
  return conv3d_causal_impl("conv bad-order probe", x, wp, nullptr, y, n, d, h, w, cin, cout, 0, stream, entry);
}

extern "C" cc_status cc_resample_prepare(const cc_bf16* w, cc_bf16* pw, int cout, int cin, void* stream) {
  cc_status st = check_ptrs("resample_prepare", {w, pw});
  if (st != CC_OK) return st;
  if (cout <= 0 || cin <= 0) return fail(CC_ERR_INVALID, "resample_prepare: sizes must be positive");
  DeviceInfo di;
  if ((st = device_info(&di)) != CC_OK) return st;
  resample_prepare_kernel<<<prep_grid(48LL * cout * cin), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const __nv_bfloat16*>(w), reinterpret_cast<__nv_bfloat16*>(pw), cout, cin);
  return launch_status("resample_prepare");
}

extern "C" cc_status cc_resample_prepare_temporal(const cc_bf16* w, cc_bf16* pw, int cout, int cin, void* stream) {
  cc_status st = check_ptrs("resample_prepare_temporal", {w, pw});
  if (st != CC_OK) return st;
  if (cout <= 0 || cin <= 0) return fail(CC_ERR_INVALID, "resample_prepare_temporal: sizes must be positive");
  DeviceInfo di;
  if ((st = device_info(&di)) != CC_OK) return st;
  resample_prepare_temporal_kernel<<<prep_grid(64LL * cout * cin), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const __nv_bfloat16*>(w), reinterpret_cast<__nv_bfloat16*>(pw), cout, cin);
  return launch_status("resample_prepare_temporal");
}

extern "C" cc_status cc_resample_phase_conv(const cc_bf16* x, const cc_bf16* pw, cc_bf16* phases, int n, int d,
                                            int hl, int wl, int cin, int cout, int hist, void* stream) {
  const char* what = "resample_phase_conv";
  cc_status st;
  if (empty_request(what, {n, d, hl, wl}, &st)) return st;
  if ((st = check_ptrs(what, {x, pw, phases})) != CC_OK) return st;
  if ((st = check_grid(what, n, d, hl, wl, hist)) != CC_OK) return st;
  if (cin <= 0 || cout <= 0) return fail(CC_ERR_INVALID, "%s: channel counts must be positive", what);
  if (cin % 64 != 0) return fail(CC_ERR_UNSUPPORTED, "%s: C_in must be a multiple of 64 (got %d)", what, cin);
  if (cout % 16 != 0) return fail(CC_ERR_UNSUPPORTED, "%s: C_out must be a multiple of 16 (got %d)", what, cout);
  DeviceInfo di;
  if ((st = device_info(&di)) != CC_OK) return st;

  const int lo_d = hist ? 0 : -2;
  CUtensorMap ta, tb;
  if ((st = encode_im2col_5d(&ta, x, n, d + hist, hl, wl, cin, -1, -1, lo_d, -1, -1, -2, kBlockM, kBlockK)) != CC_OK)
    return st;
  const long long m = (long long)n * d * hl * wl;
  const bool pair = m > kBlockM;
  if ((st = encode_tiled_2d(&tb, pw, cin, 48ull * cout, 2ull * cin, kBlockK, pair ? 128 : 256)) != CC_OK) return st;

  GemmArgs a{};
  a.m_total = static_cast<int>(m);
  a.n_total = cout;
  a.m_tiles = ceil_div(m, kBlockM);
  a.n_tiles = ceil_div(cout, 256);
  a.batches = 4;
  a.num_tiles = a.m_tiles * a.n_tiles * 4;
  a.taps = 12;
  a.kb_per_tap = cin / kBlockK;
  a.img_w = wl;
  a.img_h = hl;
  a.img_d = d;
  a.lo_w = -1;
  a.lo_h = -1;
  a.lo_d = lo_d;
  // Phase (p, q), tap (kt, a, b) reads low-resolution pixel
  // (t + kt - 2, i + p - 1 + a, j + q - 1 + b): offsets from the box corner
  // are (q + b, p + a, kt).
  for (int ph = 0; ph < 4; ++ph) {
    const int p = ph >> 1, q = ph & 1;
    for (int kt = 0; kt < 3; ++kt)
      for (int aa = 0; aa < 2; ++aa)
        for (int bb = 0; bb < 2; ++bb) a.tap_off[ph * 12 + (kt * 2 + aa) * 2 + bb] = (q + bb) | ((p + aa) << 8) | (kt << 16);
  }
  a.b_rows_per_tap = cout;
  a.b_rows_per_batch = 12 * cout;
  a.out = phases;
  a.out_ld = cout;
  a.out_batch = m * cout;
  a.bias = nullptr;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (pair) {
    set_frame_interleaved_order(a);
    return launch_tc_gemm_pair<256, kAIm2col, false, false, false>(ta, tb, a, di, s, what);
  }
  return launch_tc_gemm<256, kAIm2col, false, false, false>(ta, tb, a, di, s, what);
}

extern "C" cc_status cc_resample_up2_fused(const cc_bf16* x, const cc_bf16* pw, const cc_bf16* bias,
                                           const cc_bf16* skip, cc_bf16* out, int n, int d, int hl, int wl, int cin,
                                           int cout, int hist, int temporal, void* stream) {
  const char* what = "resample_up2_fused";
  cc_status st;
  if (empty_request(what, {n, d, hl, wl}, &st)) return st;
  if ((st = check_ptrs(what, {x, pw, bias, skip, out})) != CC_OK) return st;
  if ((st = check_grid(what, n, d, hl, wl, hist)) != CC_OK) return st;
  if (temporal != 0 && temporal != 1) return fail(CC_ERR_INVALID, "%s: temporal must be 0 or 1", what);
  if (cin <= 0 || cout <= 0) return fail(CC_ERR_INVALID, "%s: channel counts must be positive", what);
  if (cin % 64 != 0) return fail(CC_ERR_UNSUPPORTED, "%s: C_in must be a multiple of 64 (got %d)", what, cin);
  if (cout % 16 != 0) return fail(CC_ERR_UNSUPPORTED, "%s: C_out must be a multiple of 16 (got %d)", what, cout);
  if ((long long)n * d * 4 * hl * wl > kMaxPositions * 4LL)
    return fail(CC_ERR_UNSUPPORTED, "%s: too many positions", what);
  DeviceInfo di;
  if ((st = device_info(&di)) != CC_OK) return st;

  const int lo_d = hist ? 0 : -2;
  CUtensorMap ta, tb;
  if ((st = encode_im2col_5d(&ta, x, n, d + hist, hl, wl, cin, -1, -1, lo_d, -1, -1, -2, kBlockM, kBlockK)) != CC_OK)
    return st;
  const long long m = (long long)n * d * hl * wl;
  const bool pair = m > kBlockM;
  const int phases = temporal ? 8 : 4, taps = temporal ? 8 : 12;
  if ((st = encode_tiled_2d(&tb, pw, cin, (uint64_t)phases * taps * cout, 2ull * cin, kBlockK, pair ? 128 : 256)) !=
      CC_OK)
    return st;

  GemmArgs a{};
  a.m_total = static_cast<int>(m);
  a.n_total = cout;
  a.m_tiles = ceil_div(m, kBlockM);
  a.n_tiles = ceil_div(cout, 256);
  a.batches = phases;
  a.num_tiles = a.m_tiles * a.n_tiles * phases;
  a.taps = taps;
  a.kb_per_tap = cin / kBlockK;
  a.img_w = wl;
  a.img_h = hl;
  a.img_d = d;
  a.lo_w = -1;
  a.lo_h = -1;
  a.lo_d = lo_d;
  if (temporal) {
    // phase (s, p, q), tap (a, b, c) reads frame t-1+a, row i+p-1+b, column
    // j+q-1+c: offsets from the box corner (q + c, p + b, 1 + a)
    for (int ph = 0; ph < 8; ++ph) {
      const int p = (ph >> 1) & 1, q = ph & 1;
      for (int at = 0; at < 2; ++at)
        for (int bb = 0; bb < 2; ++bb)
          for (int cc = 0; cc < 2; ++cc)
            a.tap_off[ph * 8 + (at * 2 + bb) * 2 + cc] = (q + cc) | ((p + bb) << 8) | ((1 + at) << 16);
    }
  } else {
    for (int ph = 0; ph < 4; ++ph) {
      const int p = ph >> 1, q = ph & 1;
      for (int kt = 0; kt < 3; ++kt)
        for (int aa = 0; aa < 2; ++aa)
          for (int bb = 0; bb < 2; ++bb)
            a.tap_off[ph * 12 + (kt * 2 + aa) * 2 + bb] = (q + bb) | ((p + aa) << 8) | (kt << 16);
    }
  }
  a.b_rows_per_tap = cout;
  a.b_rows_per_batch = taps * cout;
  a.out = out;
  a.out_ld = cout;  // also the shortcut's row stride
  a.out_batch = 0;
  a.bias = reinterpret_cast<const __nv_bfloat16*>(bias);
  a.skip = reinterpret_cast<const __nv_bfloat16*>(skip);
  a.epi_tscale = temporal ? 2 : 1;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (pair) {
    set_frame_interleaved_order(a);
    return launch_tc_gemm_pair<256, kAIm2col, false, false, true, kEpiResample>(ta, tb, a, di, s, what);
  }
  return launch_tc_gemm<256, kAIm2col, false, false, true, kEpiResample>(ta, tb, a, di, s, what);
}
