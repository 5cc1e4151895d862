// Mid-block per-frame single-head attention, two ways:
//  - three passes: S = q k^T (tcgen05, fp32 out) -> P = softmax(scale * S)
//    (bf16) -> O = P v (tcgen05, v read as stored through an MN-major B
//    operand, no transpose);
//  - through key-tile numerators: the scores kernel's epilogue turns each
//    TMEM tile of S into E = exp2(kx*s - c_t) (bf16) and row statistics, a
//    bandwidth pass moves every tile of a row onto the row's largest c_t by
//    exact powers of two, and the PV epilogue divides each row by its sum --
//    no fp32 S in memory and no softmax pass.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "cc.h"
#include "cc_gemm_launch.cuh"
#include "cc_host.h"

namespace cc {
namespace {

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ uint2 pack4_bf16(float a, float b, float c, float d) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(a, b);
  __nv_bfloat162 hi = __floats2bfloat162_rn(c, d);
  uint2 r;
  r.x = *reinterpret_cast<uint32_t*>(&lo);
  r.y = *reinterpret_cast<uint32_t*>(&hi);
  return r;
}

constexpr int kSoftmaxWarps = 8;

// One warp per row; the row stays in registers (NV float4 per lane, columns
// (j*32 + lane)*4), so S is read once and P written once. k2 = scale*log2(e):
// exp(scale*(s - max)) is computed as exp2((s - max) * k2).
template <int NV>
__global__ void __launch_bounds__(kSoftmaxWarps * 32) softmax_rows_kernel(const float* __restrict__ s,
                                                                           __nv_bfloat16* __restrict__ p,
                                                                           long long rows, int hw, long long ld_s,
                                                                           long long ld_p, float k2) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * kSoftmaxWarps + warp;
  if (row >= rows) return;
  const float* sr = s + row * ld_s;
  float4 v[NV];
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int c = (j * 32 + lane) * 4;
    if (c + 3 < hw) {
      v[j] = __ldcs(reinterpret_cast<const float4*>(sr + c));
    } else {
      v[j].x = c < hw ? sr[c] : -INFINITY;
      v[j].y = c + 1 < hw ? sr[c + 1] : -INFINITY;
      v[j].z = c + 2 < hw ? sr[c + 2] : -INFINITY;
      v[j].w = -INFINITY;
    }
    m = fmaxf(m, fmaxf(fmaxf(v[j].x, v[j].y), fmaxf(v[j].z, v[j].w)));
  }
  m = warp_max(m);
  float sum = 0.f;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    v[j].x = exp2f((v[j].x - m) * k2);
    v[j].y = exp2f((v[j].y - m) * k2);
    v[j].z = exp2f((v[j].z - m) * k2);
    v[j].w = exp2f((v[j].w - m) * k2);
    sum += (v[j].x + v[j].y) + (v[j].z + v[j].w);
  }
  sum = warp_sum(sum);
  const float inv = 1.f / sum;
  __nv_bfloat16* pr = p + row * ld_p;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int c = (j * 32 + lane) * 4;
    if (c + 3 < hw) {
      *reinterpret_cast<uint2*>(pr + c) = pack4_bf16(v[j].x * inv, v[j].y * inv, v[j].z * inv, v[j].w * inv);
    } else if (c < hw) {
      const float t[3] = {v[j].x, v[j].y, v[j].z};
      for (int e = 0; e < 3 && c + e < hw; ++e) pr[c + e] = __float2bfloat16_rn(t[e] * inv);
    }
  }
  for (long long c = hw + lane; c < ld_p; c += 32) pr[c] = __float2bfloat16_rn(0.f);
}

// Rows longer than the register-resident kernel covers: an online pass for
// (max, sum), then a second pass that writes P (the row is still in L2).
__global__ void __launch_bounds__(kSoftmaxWarps * 32) softmax_rows_long_kernel(const float* __restrict__ s,
                                                                                __nv_bfloat16* __restrict__ p,
                                                                                long long rows, int hw,
                                                                                long long ld_s, long long ld_p,
                                                                                float k2) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * kSoftmaxWarps + warp;
  if (row >= rows) return;
  const float* sr = s + row * ld_s;
  float m = -INFINITY, l = 0.f;
  for (int c = lane; c < hw; c += 32) {
    const float x = sr[c];
    if (x > m) {
      l = l * exp2f((m - x) * k2) + 1.f;
      m = x;
    } else {
      l += exp2f((x - m) * k2);
    }
  }
  const float mw = warp_max(m);
  l = (m == -INFINITY) ? 0.f : l * exp2f((m - mw) * k2);
  l = warp_sum(l);
  const float inv = 1.f / l;
  __nv_bfloat16* pr = p + row * ld_p;
  for (int c = lane; c < hw; c += 32) pr[c] = __float2bfloat16_rn(exp2f((sr[c] - mw) * k2) * inv);
  for (long long c = hw + lane; c < ld_p; c += 32) pr[c] = __float2bfloat16_rn(0.f);
}

// Per-frame GEMMs: 128-row tiles of the HW queries times 256-column tiles of
// the keys (or channels), for every frame, must be countable in an int.
cc_status check_tiles(const char* what, int t, int rows, int cols) {
  if ((long long)((rows + 127) / 128) * ((cols + 255) / 256) * t > 0x7fffffffLL)
    return fail(CC_ERR_UNSUPPORTED, "%s: too many output tiles", what);
  return CC_OK;
}

cc_status check_ptr(const char* what, const void* p) {
  if (!p) return fail(CC_ERR_INVALID, "%s: null pointer", what);
  if (!aligned16(p)) return fail(CC_ERR_INVALID, "%s: pointers must be 16-byte aligned", what);
  return CC_OK;
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace
}  // namespace cc

using namespace cc;

// Rows of S, P and E start on 32-byte boundaries (16 bf16 or 8 fp32 columns),
// so the numerators' epilogue can write whole 32-byte sectors.
extern "C" int64_t cc_attn_ld(int hw) { return hw <= 0 ? 0 : (int64_t)round_up((size_t)hw, 16); }

extern "C" size_t cc_attn_workspace_bytes(int t, int hw) {
  if (t <= 0 || hw <= 0) return 0;
  const size_t ld = (size_t)cc_attn_ld(hw);
  return round_up((size_t)t * hw * ld * 4, 256) + round_up((size_t)t * hw * ld * 2, 256);
}

extern "C" cc_status cc_attn_scores(const cc_bf16* q, const cc_bf16* k, float* s, int t, int hw, int c, int64_t ld_q,
                                    int64_t ld_k, int64_t ld_s, void* stream) {
  const char* what = "attn_scores";
  cc_status st;
  if (empty_request(what, {t, hw}, &st)) return st;
  if ((st = check_ptr(what, q)) != CC_OK || (st = check_ptr(what, k)) != CC_OK || (st = check_ptr(what, s)) != CC_OK)
    return st;
  if (t <= 0 || hw <= 0 || c <= 0) return fail(CC_ERR_INVALID, "%s: sizes must be positive", what);
  if (c % 64 != 0) return fail(CC_ERR_UNSUPPORTED, "%s: C must be a multiple of 64 (got %d)", what, c);
  if ((st = check_tiles(what, t, hw, hw)) != CC_OK) return st;
  if (ld_q < c || ld_k < c || ld_s < hw) return fail(CC_ERR_INVALID, "%s: row strides too small", what);
  if (ld_q % 8 || ld_k % 8 || ld_s % 4)
    return fail(CC_ERR_INVALID, "%s: ld_q, ld_k must be multiples of 8 and ld_s of 4", what);
  DeviceInfo di;
  if ((st = device_info(&di)) != CC_OK) return st;
  CUtensorMap ta, tb;
  if ((st = encode_tiled_3d(&ta, q, c, hw, t, 2ull * ld_q, 2ull * ld_q * hw, kBlockK, kBlockM)) != CC_OK) return st;
  const bool pair = hw > kBlockM;
  if ((st = encode_tiled_3d(&tb, k, c, hw, t, 2ull * ld_k, 2ull * ld_k * hw, kBlockK, pair ? 128 : 256)) != CC_OK)
    return st;
  GemmArgs a{};
  a.m_total = hw;
  a.n_total = hw;
  a.m_tiles = ceil_div(hw, kBlockM);
  a.n_tiles = ceil_div(hw, 256);
  a.batches = t;
  a.num_tiles = a.m_tiles * a.n_tiles * t;
  a.taps = 1;
  a.kb_per_tap = c / kBlockK;
  a.out = s;
  a.out_ld = ld_s;
  a.out_batch = (long long)hw * ld_s;
  cudaStream_t s_ = static_cast<cudaStream_t>(stream);
  if (pair) {
    // S leaves through TMA tensor stores of 32-column x 128-row fp32 boxes
    CUtensorMap tc;
    if ((st = encode_tiled_3d_f32_sw128(&tc, s, hw, hw, t, 4ull * ld_s, 4ull * ld_s * hw, 32, kBlockM)) != CC_OK)
      return st;
    return launch_tc_gemm_pair<256, kATiled3d, false, true, false, kEpiStoreF32>(ta, tb, a, di, s_, what, &tc);
  }
  return launch_tc_gemm<256, kATiled3d, false, true, false>(ta, tb, a, di, s_, what);
}

extern "C" cc_status cc_attn_softmax(const float* s, cc_bf16* p, int t, int hw, int64_t ld_s, int64_t ld_p,
                                     float scale, void* stream) {
  const char* what = "attn_softmax";
  cc_status st;
  if (empty_request(what, {t, hw}, &st)) return st;
  if ((st = check_ptr(what, s)) != CC_OK || (st = check_ptr(what, p)) != CC_OK) return st;
  if (t <= 0 || hw <= 0) return fail(CC_ERR_INVALID, "%s: sizes must be positive", what);
  if (ld_s < hw || ld_p < hw || ld_s % 4 || ld_p % 8)
    return fail(CC_ERR_INVALID, "%s: need ld_s >= HW, ld_p >= HW, ld_s %% 4 == 0, ld_p %% 8 == 0", what);
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(CC_ERR_INVALID, "%s: scale must be finite and > 0", what);
  DeviceInfo di;
  if ((st = device_info(&di)) != CC_OK) return st;
  const long long rows = (long long)t * hw;
  const unsigned grid = (unsigned)((rows + kSoftmaxWarps - 1) / kSoftmaxWarps);
  const float k2 = scale * 1.4426950408889634f;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const float* sp = s;
  __nv_bfloat16* pp = reinterpret_cast<__nv_bfloat16*>(p);
  const int need = (hw + 127) / 128;
  if (need <= 4)
    softmax_rows_kernel<4><<<grid, kSoftmaxWarps * 32, 0, cs>>>(sp, pp, rows, hw, ld_s, ld_p, k2);
  else if (need <= 8)
    softmax_rows_kernel<8><<<grid, kSoftmaxWarps * 32, 0, cs>>>(sp, pp, rows, hw, ld_s, ld_p, k2);
  else if (need <= 16)
    softmax_rows_kernel<16><<<grid, kSoftmaxWarps * 32, 0, cs>>>(sp, pp, rows, hw, ld_s, ld_p, k2);
  else if (need <= 28)
    softmax_rows_kernel<28><<<grid, kSoftmaxWarps * 32, 0, cs>>>(sp, pp, rows, hw, ld_s, ld_p, k2);
  else
    softmax_rows_long_kernel<<<grid, kSoftmaxWarps * 32, 0, cs>>>(sp, pp, rows, hw, ld_s, ld_p, k2);
  return launch_status(what);
}

extern "C" cc_status cc_attn_pv(const cc_bf16* p, const cc_bf16* v, cc_bf16* o, int t, int hw, int c, int64_t ld_p,
                                int64_t ld_v, int64_t ld_o, void* stream) {
  const char* what = "attn_pv";
  cc_status st;
  if (empty_request(what, {t, hw}, &st)) return st;
  if ((st = check_ptr(what, p)) != CC_OK || (st = check_ptr(what, v)) != CC_OK || (st = check_ptr(what, o)) != CC_OK)
    return st;
  if (t <= 0 || hw <= 0 || c <= 0) return fail(CC_ERR_INVALID, "%s: sizes must be positive", what);
  if (c % 64 != 0) return fail(CC_ERR_UNSUPPORTED, "%s: C must be a multiple of 64 (got %d)", what, c);
  if ((st = check_tiles(what, t, hw, c)) != CC_OK) return st;
  if (ld_p < hw || ld_v < c || ld_o < c) return fail(CC_ERR_INVALID, "%s: row strides too small", what);
  if (ld_p % 8 || ld_v % 8 || ld_o % 8) return fail(CC_ERR_INVALID, "%s: row strides must be multiples of 8", what);
  DeviceInfo di;
  if ((st = device_info(&di)) != CC_OK) return st;
  CUtensorMap ta, tb;
  // A = P (keys innermost; the map ends at HW so the padded tail is never read)
  if ((st = encode_tiled_3d(&ta, p, hw, hw, t, 2ull * ld_p, 2ull * ld_p * hw, kBlockK, kBlockM)) != CC_OK) return st;
  // B = v as stored: channels innermost, 64 channels x 64 keys per box
  if ((st = encode_tiled_3d(&tb, v, c, hw, t, 2ull * ld_v, 2ull * ld_v * hw, 64, kBlockK)) != CC_OK) return st;
  GemmArgs a{};
  a.m_total = hw;
  a.n_total = c;
  a.m_tiles = ceil_div(hw, kBlockM);
  a.n_tiles = ceil_div(c, 256);
  a.batches = t;
  a.num_tiles = a.m_tiles * a.n_tiles * t;
  a.taps = 1;
  a.kb_per_tap = ceil_div(hw, kBlockK);
  a.out = o;
  a.out_ld = ld_o;
  a.out_batch = (long long)hw * ld_o;
  cudaStream_t s_ = static_cast<cudaStream_t>(stream);
  if (hw > kBlockM) return launch_tc_gemm_pair<256, kATiled3d, true, false, false>(ta, tb, a, di, s_, what);
  return launch_tc_gemm<256, kATiled3d, true, false, false>(ta, tb, a, di, s_, what);
}

extern "C" cc_status cc_attn_frame(const cc_bf16* q, const cc_bf16* k, const cc_bf16* v, cc_bf16* o, int t, int hw,
                                   int c, int64_t ld_q, int64_t ld_k, int64_t ld_v, int64_t ld_o, float scale,
                                   void* ws, size_t ws_bytes, void* stream) {
  const char* what = "attn_frame";
  cc_status st;
  if (empty_request(what, {t, hw}, &st)) return st;
  if ((st = check_ptr(what, ws)) != CC_OK) return st;
  const size_t need = cc_attn_workspace_bytes(t, hw);
  if (ws_bytes < need) return fail(CC_ERR_INVALID, "%s: workspace of %zu bytes, need %zu", what, ws_bytes, need);
  const int64_t ld = cc_attn_ld(hw);
  float* s = static_cast<float*>(ws);
  cc_bf16* p = reinterpret_cast<cc_bf16*>(static_cast<char*>(ws) + round_up((size_t)t * hw * ld * 4, 256));
  if ((st = cc_attn_scores(q, k, s, t, hw, c, ld_q, ld_k, ld, stream)) != CC_OK) return st;
  if ((st = cc_attn_softmax(s, p, t, hw, ld, ld, scale, stream)) != CC_OK) return st;
  return cc_attn_pv(p, v, o, t, hw, c, ld, ld_v, ld_o, stream);
}

// ------------------------------------------- numerators in key tiles (E) --

namespace cc {
namespace {
constexpr int kKeyTile = 256;  // keys per statistics tile = the scores kernel's BN
constexpr int kRescaleWarps = 8;

// Rescale of one row by the whole warp: every key tile with c_t < c_row is
// multiplied in place by 2^(c_t - c_row), an exact power of two (lane j takes
// keys 8j .. 8j+7 of the tile, one 16-byte vector), and its statistics become
// (c_row, 2^(c_t - c_row) l_t). Tiles already at c_row are not touched. Lane
// i reads the statistics of tile t0 + i, so the tiles to rescale are known at
// once and up to kRescaleBatch of them are loaded before any is written.
constexpr int kRescaleBatch = 8;

__device__ void rescale_row(__nv_bfloat16* __restrict__ er, float2* __restrict__ st, int hw, int tiles, float c_row,
                            int lane) {
  for (int t0 = 0; t0 < tiles; t0 += 32) {
    const int tl = t0 + lane;
    const float2 mine = tl < tiles ? st[tl] : make_float2(c_row, 0.f);
    const float my_al = pow2_nonpos(mine.x - c_row);
    unsigned todo = __ballot_sync(0xffffffffu, mine.x != c_row);
    if (mine.x != c_row) st[tl] = make_float2(c_row, mine.y * my_al);
    while (todo) {  // the same for every lane
      int tb[kRescaleBatch];
      uint4 x[kRescaleBatch];
#pragma unroll
      for (int i = 0; i < kRescaleBatch; ++i) {
        tb[i] = -1;
        if (todo) {
          tb[i] = __ffs(todo) - 1;
          todo &= todo - 1;
        }
        const int k0 = (t0 + tb[i]) * kKeyTile + 8 * lane;
        if (tb[i] >= 0 && k0 + 8 <= hw) x[i] = *reinterpret_cast<const uint4*>(er + k0);
      }
#pragma unroll
      for (int i = 0; i < kRescaleBatch; ++i) {
        const float al = __shfl_sync(0xffffffffu, my_al, tb[i] < 0 ? 0 : tb[i]);
        if (tb[i] < 0) continue;
        const int k0 = (t0 + tb[i]) * kKeyTile + 8 * lane;
        if (k0 + 8 <= hw) {
          const __nv_bfloat162 al2 = __float2bfloat162_rn(al);
          __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&x[i]);
#pragma unroll
          for (int j = 0; j < 4; ++j) h[j] = __hmul2(h[j], al2);
          *reinterpret_cast<uint4*>(er + k0) = x[i];
        } else {
          for (int j = 0; j < 8 && k0 + j < hw; ++j)
            er[k0 + j] = __float2bfloat16_rn(__bfloat162float(er[k0 + j]) * al);
        }
      }
    }
  }
}

// One warp per 32 rows: lane l checks row r0 + l (c_row = max_t c_t over its
// statistics, all loads in flight at once), and the warp rescales together
// the rows that hold a tile below their c_row -- with key-tile exponents on
// a grain of 32 those are rare, so the pass is mostly one read of the
// statistics.
__global__ void __launch_bounds__(kRescaleWarps * 32) exp_rescale_kernel(__nv_bfloat16* __restrict__ e,
                                                                          float2* __restrict__ stats,
                                                                          long long rows, int hw, long long ld_e,
                                                                          int tiles) {
  // launched after the scores kernel that writes e and stats; the grid is one
  // wave (32 rows per warp), so the next kernel may be scheduled at once: its
  // CTAs take the idle SMs and do their set-up, then wait for this grid to
  // complete before they read e
  pdl_launch_dependents();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long r0 = ((long long)blockIdx.x * kRescaleWarps + warp) * 32;
  if (r0 >= rows) return;
  const long long row = r0 + lane;
  float c_row = __int_as_float(0xff800000u);  // -inf
  bool need = false;
  if (row < rows) {
    const float2* st = stats + row * tiles;
    float c_min = __int_as_float(0x7f800000u);  // +inf
    for (int t = 0; t < tiles; ++t) {
      const float c = st[t].x;
      c_row = fmaxf(c_row, c);
      c_min = fminf(c_min, c);
    }
    need = c_min != c_row;
  }
  unsigned todo = __ballot_sync(0xffffffffu, need);
  while (todo) {
    const int l = __ffs(todo) - 1;
    todo &= todo - 1;
    const float c = __shfl_sync(0xffffffffu, c_row, l);
    rescale_row(e + (r0 + l) * ld_e, stats + (r0 + l) * tiles, hw, tiles, c, lane);
  }
}
}  // namespace
}  // namespace cc

extern "C" int cc_attn_exp_key_tiles(int hw) { return hw <= 0 ? 0 : ceil_div(hw, kKeyTile); }

extern "C" size_t cc_attn_exp_workspace_bytes(int t, int hw) {
  if (t <= 0 || hw <= 0) return 0;
  const size_t ld = (size_t)cc_attn_ld(hw);
  return round_up((size_t)t * hw * ld * 2, 256) + round_up((size_t)t * hw * cc_attn_exp_key_tiles(hw) * 8, 256);
}

extern "C" cc_status cc_attn_scores_exp(const cc_bf16* q, const cc_bf16* k, cc_bf16* e, float* stats, int t, int hw,
                                        int c, int64_t ld_q, int64_t ld_k, int64_t ld_e, float scale, void* stream) {
  const char* what = "attn_scores_exp";
  cc_status st;
  if (empty_request(what, {t, hw}, &st)) return st;
  if ((st = check_ptr(what, q)) != CC_OK || (st = check_ptr(what, k)) != CC_OK || (st = check_ptr(what, e)) != CC_OK ||
      (st = check_ptr(what, stats)) != CC_OK)
    return st;
  if (t <= 0 || hw <= 0 || c <= 0) return fail(CC_ERR_INVALID, "%s: sizes must be positive", what);
  if (c % 64 != 0) return fail(CC_ERR_UNSUPPORTED, "%s: C must be a multiple of 64 (got %d)", what, c);
  if ((st = check_tiles(what, t, hw, hw)) != CC_OK) return st;
  if (ld_q < c || ld_k < c || ld_e < hw) return fail(CC_ERR_INVALID, "%s: row strides too small", what);
  if (ld_q % 8 || ld_k % 8 || ld_e % 8) return fail(CC_ERR_INVALID, "%s: row strides must be multiples of 8", what);
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(CC_ERR_INVALID, "%s: scale must be finite and > 0", what);
  DeviceInfo di;
  if ((st = device_info(&di)) != CC_OK) return st;
  CUtensorMap ta, tb, tc;
  if ((st = encode_tiled_3d(&ta, q, c, hw, t, 2ull * ld_q, 2ull * ld_q * hw, kBlockK, kBlockM)) != CC_OK) return st;
  if ((st = encode_tiled_3d(&tb, k, c, hw, t, 2ull * ld_k, 2ull * ld_k * hw, kBlockK, 128)) != CC_OK) return st;
  // E leaves through TMA tensor stores of 64-key x 128-row bf16 boxes
  if ((st = encode_tiled_3d(&tc, e, hw, hw, t, 2ull * ld_e, 2ull * ld_e * hw, kBlockK, kBlockM)) != CC_OK) return st;
  GemmArgs a{};
  a.m_total = hw;
  a.n_total = hw;
  a.m_tiles = ceil_div(hw, kBlockM);
  a.n_tiles = ceil_div(hw, kKeyTile);
  a.batches = t;
  a.num_tiles = a.m_tiles * a.n_tiles * t;
  a.taps = 1;
  a.kb_per_tap = c / kBlockK;
  a.out = e;
  a.out_ld = ld_e;
  a.out_batch = (long long)hw * ld_e;
  a.stats = reinterpret_cast<float2*>(stats);
  a.stat_tiles = a.n_tiles;
  a.exp_k = scale * 1.4426950408889634f;
  return launch_tc_gemm_pair<kKeyTile, kATiled3d, false, false, false, kEpiExpBf16>(
      ta, tb, a, di, static_cast<cudaStream_t>(stream), what, &tc);
}

extern "C" cc_status cc_attn_scores_stats(const cc_bf16* q, const cc_bf16* k, float* stats, int t, int hw, int c,
                                          int64_t ld_q, int64_t ld_k, float scale, void* stream) {
  const char* what = "attn_scores_stats";
  cc_status st;
  if (empty_request(what, {t, hw}, &st)) return st;
  if ((st = check_ptr(what, q)) != CC_OK || (st = check_ptr(what, k)) != CC_OK ||
      (st = check_ptr(what, stats)) != CC_OK)
    return st;
  if (t <= 0 || hw <= 0 || c <= 0) return fail(CC_ERR_INVALID, "%s: sizes must be positive", what);
  if (c % 64 != 0) return fail(CC_ERR_UNSUPPORTED, "%s: C must be a multiple of 64 (got %d)", what, c);
  if ((st = check_tiles(what, t, hw, hw)) != CC_OK) return st;
  if (ld_q < c || ld_k < c) return fail(CC_ERR_INVALID, "%s: row strides too small", what);
  if (ld_q % 8 || ld_k % 8) return fail(CC_ERR_INVALID, "%s: row strides must be multiples of 8", what);
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(CC_ERR_INVALID, "%s: scale must be finite and > 0", what);
  DeviceInfo di;
  if ((st = device_info(&di)) != CC_OK) return st;
  CUtensorMap ta, tb;
  if ((st = encode_tiled_3d(&ta, q, c, hw, t, 2ull * ld_q, 2ull * ld_q * hw, kBlockK, kBlockM)) != CC_OK) return st;
  if ((st = encode_tiled_3d(&tb, k, c, hw, t, 2ull * ld_k, 2ull * ld_k * hw, kBlockK, 128)) != CC_OK) return st;
  GemmArgs a{};
  a.m_total = hw;
  a.n_total = hw;
  a.m_tiles = ceil_div(hw, kBlockM);
  a.n_tiles = ceil_div(hw, kKeyTile);
  a.batches = t;
  a.num_tiles = a.m_tiles * a.n_tiles * t;
  a.taps = 1;
  a.kb_per_tap = c / kBlockK;
  a.out = nullptr;  // the numerators' epilogue then writes the statistics only
  a.stats = reinterpret_cast<float2*>(stats);
  a.stat_tiles = a.n_tiles;
  a.exp_k = scale * 1.4426950408889634f;
  return launch_tc_gemm_pair<kKeyTile, kATiled3d, false, false, false, kEpiExpBf16>(
      ta, tb, a, di, static_cast<cudaStream_t>(stream), what, &tb);
}

extern "C" cc_status cc_attn_exp_rescale(cc_bf16* e, float* stats, int t, int hw, int64_t ld_e, void* stream) {
  const char* what = "attn_exp_rescale";
  cc_status st;
  if (empty_request(what, {t, hw}, &st)) return st;
  if ((st = check_ptr(what, e)) != CC_OK || (st = check_ptr(what, stats)) != CC_OK) return st;
  if (t <= 0 || hw <= 0) return fail(CC_ERR_INVALID, "%s: sizes must be positive", what);
  if (ld_e < hw || ld_e % 8) return fail(CC_ERR_INVALID, "%s: need ld_e >= HW and ld_e %% 8 == 0", what);
  DeviceInfo di;
  if ((st = device_info(&di)) != CC_OK) return st;
  const long long rows = (long long)t * hw;
  const unsigned grid = (unsigned)((rows + 32LL * kRescaleWarps - 1) / (32LL * kRescaleWarps));
  const cudaError_t err = launch_pdl(exp_rescale_kernel, dim3(grid), dim3(kRescaleWarps * 32), 0,
                                     static_cast<cudaStream_t>(stream), reinterpret_cast<__nv_bfloat16*>(e),
                                     reinterpret_cast<float2*>(stats), rows, hw, (long long)ld_e,
                                     cc_attn_exp_key_tiles(hw));
  if (err != cudaSuccess) return fail(CC_ERR_CUDA, "%s: launch: %s", what, cudaGetErrorString(err));
  return launch_status(what);
}

extern "C" cc_status cc_attn_pv_exp(const cc_bf16* e, const float* stats, const cc_bf16* v, cc_bf16* o, int t, int hw,
                                    int c, int64_t ld_e, int64_t ld_v, int64_t ld_o, void* stream) {
  const char* what = "attn_pv_exp";
  cc_status st;
  if (empty_request(what, {t, hw}, &st)) return st;
  if ((st = check_ptr(what, e)) != CC_OK || (st = check_ptr(what, stats)) != CC_OK ||
      (st = check_ptr(what, v)) != CC_OK || (st = check_ptr(what, o)) != CC_OK)
    return st;
  if (t <= 0 || hw <= 0 || c <= 0) return fail(CC_ERR_INVALID, "%s: sizes must be positive", what);
  if (c % 64 != 0) return fail(CC_ERR_UNSUPPORTED, "%s: C must be a multiple of 64 (got %d)", what, c);
  if ((st = check_tiles(what, t, hw, c)) != CC_OK) return st;
  if (ld_e < hw || ld_v < c || ld_o < c) return fail(CC_ERR_INVALID, "%s: row strides too small", what);
  if (ld_e % 8 || ld_v % 8 || ld_o % 8) return fail(CC_ERR_INVALID, "%s: row strides must be multiples of 8", what);
  DeviceInfo di;
  if ((st = device_info(&di)) != CC_OK) return st;
  CUtensorMap ta, tb;
  if ((st = encode_tiled_3d(&ta, e, hw, hw, t, 2ull * ld_e, 2ull * ld_e * hw, kBlockK, kBlockM)) != CC_OK) return st;
  if ((st = encode_tiled_3d(&tb, v, c, hw, t, 2ull * ld_v, 2ull * ld_v * hw, 64, kBlockK)) != CC_OK) return st;
  GemmArgs a{};
  a.m_total = hw;
  a.n_total = c;
  a.m_tiles = ceil_div(hw, kBlockM);
  a.n_tiles = ceil_div(c, 256);
  a.batches = t;
  a.num_tiles = a.m_tiles * a.n_tiles * t;
  a.taps = 1;
  a.kb_per_tap = ceil_div(hw, kBlockK);
  a.out = o;
  a.out_ld = ld_o;
  a.out_batch = (long long)hw * ld_o;
  a.stats = const_cast<float2*>(reinterpret_cast<const float2*>(stats));
  a.stat_tiles = cc_attn_exp_key_tiles(hw);
  a.batch_outer = 1;  // frame by frame: one frame's v (7 MB at C=1024) serves every concurrent tile
  // O leaves through TMA tensor stores of 64-channel x 128-row bf16 boxes
  CUtensorMap tc;
  if ((st = encode_tiled_3d(&tc, o, c, hw, t, 2ull * ld_o, 2ull * ld_o * hw, kBlockK, kBlockM)) != CC_OK) return st;
  return launch_tc_gemm_pair<256, kATiled3d, true, false, false, kEpiRowScale>(
      ta, tb, a, di, static_cast<cudaStream_t>(stream), what, &tc);
}

extern "C" cc_status cc_attn_frame_exp(const cc_bf16* q, const cc_bf16* k, const cc_bf16* v, cc_bf16* o, int t, int hw,
                                       int c, int64_t ld_q, int64_t ld_k, int64_t ld_v, int64_t ld_o, float scale,
                                       void* ws, size_t ws_bytes, void* stream) {
  const char* what = "attn_frame_exp";
  cc_status st;
  if (empty_request(what, {t, hw}, &st)) return st;
  if ((st = check_ptr(what, ws)) != CC_OK) return st;
  const size_t need = cc_attn_exp_workspace_bytes(t, hw);
  if (ws_bytes < need) return fail(CC_ERR_INVALID, "%s: workspace of %zu bytes, need %zu", what, ws_bytes, need);
  const int64_t ld = cc_attn_ld(hw);
  cc_bf16* e = static_cast<cc_bf16*>(ws);
  float* stats = reinterpret_cast<float*>(static_cast<char*>(ws) + round_up((size_t)t * hw * ld * 2, 256));
  if ((st = cc_attn_scores_exp(q, k, e, stats, t, hw, c, ld_q, ld_k, ld, scale, stream)) != CC_OK) return st;
  if ((st = cc_attn_exp_rescale(e, stats, t, hw, ld, stream)) != CC_OK) return st;
  return cc_attn_pv_exp(e, stats, v, o, t, hw, c, ld, ld_v, ld_o, stream);
}
