// Mid-block attention with the softmax numerators kept on chip: per frame
// O = softmax(q k^T * scale) v ([ATTN]: attn_forward's scores, row softmax and
// PV), with neither S nor P nor E in memory. Two launches:
//  1. cc_attn_scores_stats: the key-tile scores kernel (attn.cu) writing only
//     the row statistics (c_t, l_t) per 256-key tile;
//  2. attn_fused_kernel: per work item -- one frame, 256 query rows (a CTA
//     pair, 128 rows each) and one 256-channel chunk of O -- for each 256-key
//     tile it computes S in tensor memory (K = C), turns it into
//     E = bf16(exp2(kx * S - c_row)) in shared memory (c_row = the row's
//     largest c_t, so every tile is on the row's final scale and nothing is
//     rescaled), and multiplies E by the tile's values into O in tensor
//     memory; after the last tile O is divided by l_row = sum_t
//     2^(c_t - c_row) l_t and rounded once.
// E is rounded once, as P is in the three-pass path. S is computed once per
// 256-channel chunk of O (four times at C = 1024, plus once for the
// statistics): O for all C channels of a 128-row block would need 1024
// tensor-memory columns where a CTA has 512, so this is the fused form that
// fits; it trades the numerators' HBM round trip for recomputed scores.
//
// Per CTA: warp 0 streams q/k k-blocks (a 4-stage ring, 32 KB each) and value
// blocks (2 stages, 16 KB) with TMA; warp 1 of the even CTA issues the MMAs
// (whole warp, elected lane): S (M = 256, N = 256 keys, K = C) into TMEM
// columns 0-255, PV (M = 256, N = 256 channels, K = 256 keys, A = E from
// shared memory, B = v read as stored through an MN-major descriptor) into
// columns 256-511; warps 2-5 of both CTAs turn S into E and finish O. The
// MMA order S(t), PV(t-1), S(t+1), ... lets the epilogue work on S(t) while
// the tensor pipe runs PV(t-1) and S(t+1). Every wait is bounded.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "cc.h"
#include "cc_gemm_launch.cuh"
#include "cc_host.h"
#include "cc_ptx.cuh"

namespace cc {
namespace {

constexpr int kFaKeys = 256;   // keys per S tile = the statistics' key tile
constexpr int kFaChunk = 256;  // O channels per work item
constexpr int kFaSStages = 4;
constexpr int kFaVStages = 2;
constexpr int kFaABytes = kBlockM * kBlockK * 2;                // q: 128 rows x 64 channels
constexpr int kFaSStageBytes = 2 * kFaABytes;                   // + k: 128 keys x 64 channels
constexpr int kFaVStageBytes = (kFaChunk / 2) * kBlockK * 2;    // v: 64 keys x 128 channels
constexpr int kFaEBlock = kBlockM * kBlockK * 2;                // E: 128 rows x 64 keys
constexpr int kFaEBytes = (kFaKeys / kBlockK) * kFaEBlock;      // 64 KB
constexpr int kFaSmem = 1024 + kFaSStages * kFaSStageBytes + kFaVStages * kFaVStageBytes + kFaEBytes + 256;
static_assert(kFaSmem <= 232448, "shared memory budget");
constexpr uint32_t kFaSCol = 0;    // TMEM columns of S
constexpr uint32_t kFaOCol = 256;  // TMEM columns of O

struct FaArgs {
  int hw;         // query rows = keys per frame
  int frames;
  int m_pairs;    // 256-row blocks per frame
  int chunks;     // C / 256
  int key_tiles;  // ceil(hw / 256)
  int kb_s;       // C / 64: k-blocks of one S tile
  int items;      // frames x m_pairs x chunks
  float exp_k;    // scale * log2(e)
  const float2* stats;  // [frames][hw][key_tiles] (c_t, l_t)
  __nv_bfloat16* out;
  long long ld_o;
  unsigned int* err;
  unsigned long long timeout_ns;
};

// item -> (frame, 256-row block, channel chunk), chunks fastest: neighbouring
// pairs share the row block's q from L2.
__device__ __forceinline__ void fa_decode(const FaArgs& a, int item, int& f, int& mp, int& cc) {
  cc = item % a.chunks;
  const int r = item / a.chunks;
  mp = r % a.m_pairs;
  f = r / a.m_pairs;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    attn_fused_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ FaArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sS = smem;                                      // q/k stages
  uint8_t* sV = sS + kFaSStages * kFaSStageBytes;          // value stages
  uint8_t* sE = sV + kFaVStages * kFaVStageBytes;          // E, 4 blocks of 64 keys
  uint64_t* bars = reinterpret_cast<uint64_t*>(sE + kFaEBytes);
  uint64_t* sfull = bars;
  uint64_t* sempty = sfull + kFaSStages;
  uint64_t* vfull = sempty + kFaSStages;
  uint64_t* vempty = vfull + kFaVStages;
  uint64_t* s_ready = vempty + kFaVStages;  // S in TMEM complete
  uint64_t* s_free = s_ready + 1;           // both CTAs' epilogues have read S
  uint64_t* e_ready = s_free + 1;           // both CTAs' E written
  uint64_t* e_free = e_ready + 1;           // PV has read E
  uint64_t* o_ready = e_free + 1;           // O complete
  uint64_t* o_free = o_ready + 1;           // both CTAs' epilogues have read O
  uint64_t* done = o_free + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kFaSStages; ++s) {
      mbar_init(smem_u32(&sfull[s]), 1);
      mbar_init(smem_u32(&sempty[s]), 1);
    }
    for (int s = 0; s < kFaVStages; ++s) {
      mbar_init(smem_u32(&vfull[s]), 1);
      mbar_init(smem_u32(&vempty[s]), 1);
    }
    mbar_init(smem_u32(s_ready), 1);
    mbar_init(smem_u32(s_free), 2 * 4);
    mbar_init(smem_u32(e_ready), 2 * 4);
    mbar_init(smem_u32(e_free), 1);
    mbar_init(smem_u32(o_ready), 1);
    mbar_init(smem_u32(o_free), 2 * 4);
    mbar_init(smem_u32(done), 1);
    fence_mbar_init();
    tma_prefetch_map(&tmQ);
    tma_prefetch_map(&tmK);
    tma_prefetch_map(&tmV);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_launch_dependents();
  pdl_wait();
  const uint64_t tlim = a.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      int ss = 0, vs = 0;
      uint32_t sph = 0, vph = 0;
      bool ok = true;
      auto load_v = [&](int f, int cc, int t) {
        for (int vb = 0; ok && vb < kFaKeys / kBlockK; ++vb) {
          if (!mbar_wait(smem_u32(&vempty[vs]), vph ^ 1u, a.err, tlim)) {
            ok = false;
            return;
          }
          const uint32_t fb_local = smem_u32(&vfull[vs]);
          if (leader) mbar_arrive_expect_tx(fb_local, 2 * kFaVStageBytes);
          const uint32_t fb = mapa_shared(fb_local, 0);
          const uint32_t dst = smem_u32(sV + vs * kFaVStageBytes);
#pragma unroll
          for (int j = 0; j < kFaChunk / 2 / 64; ++j)
            tma_load_3d_pair(dst + j * 8192, &tmV, fb, cc * kFaChunk + static_cast<int>(rank) * (kFaChunk / 2) + 64 * j,
                             t * kFaKeys + vb * kBlockK, f);
          if (++vs == kFaVStages) {
            vs = 0;
            vph ^= 1u;
          }
        }
      };
      for (int item = pair; ok && item < a.items; item += npairs) {
        int f, mp, cc;
        fa_decode(a, item, f, mp, cc);
        const int m0 = (2 * mp + static_cast<int>(rank)) * kBlockM;
        for (int t = 0; ok && t < a.key_tiles; ++t) {
          for (int kb = 0; kb < a.kb_s; ++kb) {
            if (!mbar_wait(smem_u32(&sempty[ss]), sph ^ 1u, a.err, tlim)) {
              ok = false;
              break;
            }
            const uint32_t fb_local = smem_u32(&sfull[ss]);
            if (leader) mbar_arrive_expect_tx(fb_local, 2 * kFaSStageBytes);
            const uint32_t fb = mapa_shared(fb_local, 0);
            const uint32_t dst = smem_u32(sS + ss * kFaSStageBytes);
            tma_load_3d_pair(dst, &tmQ, fb, kb * kBlockK, m0, f);
            tma_load_3d_pair(dst + kFaABytes, &tmK, fb, kb * kBlockK,
                             t * kFaKeys + static_cast<int>(rank) * (kFaKeys / 2), f);
            if (++ss == kFaSStages) {
              ss = 0;
              sph ^= 1u;
            }
          }
          if (ok && t >= 1) load_v(f, cc, t - 1);
        }
        if (ok) load_v(f, cc, a.key_tiles - 1);
      }
      if (!ok && leader) {
        for (int s = 0; s < kFaSStages; ++s)
          (void)mbar_wait(smem_u32(&sfull[s]), (s < ss) ? sph : (sph ^ 1u), a.err, 200000000ull);
        for (int s = 0; s < kFaVStages; ++s)
          (void)mbar_wait(smem_u32(&vfull[s]), (s < vs) ? vph : (vph ^ 1u), a.err, 200000000ull);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------- MMA issuer (even CTA's warp) --
    if (leader) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(2 * kBlockM, kFaKeys, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(2 * kBlockM, kFaChunk, true);
      const uint64_t sa0 = sdesc_sw128(smem_u32(sS), 16, 1024);
      const uint64_t sb0 = sdesc_sw128(smem_u32(sS + kFaABytes), 16, 1024);
      const uint64_t ea0 = sdesc_sw128(smem_u32(sE), 16, 1024);
      const uint64_t vb0 = sdesc_sw128(smem_u32(sV), 8192, 1024);
      int ss = 0, vs = 0;
      uint32_t sph = 0, vph = 0;
      int g = 0;  // tiles issued so far (S buffer / E buffer phases)
      int it = 0; // items so far (O phases)
      bool ok = true;
      // PV of tile number gt (E in shared memory) into O
      auto pv = [&](int gt, bool first) {
        if (!__all_sync(0xffffffffu, mbar_wait_cluster(smem_u32(e_ready), gt & 1, a.err, tlim))) {
          ok = false;
          return;
        }
        if (first && !__all_sync(0xffffffffu, mbar_wait(smem_u32(o_free), (it & 1) ^ 1u, a.err, tlim))) {
          ok = false;
          return;
        }
        tc_fence_after();
        for (int vb = 0; vb < kFaKeys / kBlockK; ++vb) {
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&vfull[vs]), vph, a.err, tlim))) {
            ok = false;
            return;
          }
          tc_fence_after();
          const uint64_t ad = ea0 + static_cast<uint64_t>(vb) * (kFaEBlock >> 4);
          const uint64_t bd = vb0 + static_cast<uint64_t>(vs) * (kFaVStageBytes >> 4);
          if (elect_one()) {
#pragma unroll
            for (int k = 0; k < kBlockK / kUmmaK; ++k)
              mma_bf16_pair(tmem_base + kFaOCol, ad + 2 * k, bd + 128 * k, idesc_o,
                            (first && vb == 0 && k == 0) ? 0u : 1u);
            mma_commit_pair_both(smem_u32(&vempty[vs]));
          }
          __syncwarp();
          if (++vs == kFaVStages) {
            vs = 0;
            vph ^= 1u;
          }
        }
        if (elect_one()) mma_commit_pair_both(smem_u32(e_free));
        __syncwarp();
      };
      for (int item = pair; ok && item < a.items; item += npairs, ++it) {
        for (int t = 0; ok && t < a.key_tiles; ++t, ++g) {
          // S(t): the S columns must have been read by both epilogues
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(s_free), (g & 1) ^ 1u, a.err, tlim))) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int kb = 0; kb < a.kb_s; ++kb) {
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sfull[ss]), sph, a.err, tlim))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t ad = sa0 + static_cast<uint64_t>(ss) * (kFaSStageBytes >> 4);
            const uint64_t bd = sb0 + static_cast<uint64_t>(ss) * (kFaSStageBytes >> 4);
            if (elect_one()) {
#pragma unroll
              for (int k = 0; k < kBlockK / kUmmaK; ++k)
                mma_bf16_pair(tmem_base + kFaSCol, ad + 2 * k, bd + 2 * k, idesc_s, (kb != 0 || k != 0) ? 1u : 0u);
              mma_commit_pair_both(smem_u32(&sempty[ss]));
            }
            __syncwarp();
            if (++ss == kFaSStages) {
              ss = 0;
              sph ^= 1u;
            }
          }
          if (!ok) break;
          if (elect_one()) mma_commit_pair_both(smem_u32(s_ready));
          __syncwarp();
          if (t >= 1) pv(g - 1, t == 1);
        }
        if (!ok) break;
        pv(g - 1, a.key_tiles == 1);
        if (!ok) break;
        if (elect_one()) mma_commit_pair_both(smem_u32(o_ready));
        __syncwarp();
      }
      if (elect_one()) mma_commit_pair_both(smem_u32(done));
      __syncwarp();
      (void)mbar_wait(smem_u32(done), 0, a.err, tlim);
    }
  } else {
    // -------------------------------------------------------- epilogue --
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const float kx = a.exp_k;
    const uint32_t lanes = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t e_ready_leader = mapa_shared(smem_u32(e_ready), 0);
    const uint32_t s_free_leader = mapa_shared(smem_u32(s_free), 0);
    const uint32_t o_free_leader = mapa_shared(smem_u32(o_free), 0);
    int g = 0, it = 0;
    bool ok = true;
    for (int item = pair; ok && item < a.items; item += npairs, ++it) {
      int f, mp, cc;
      fa_decode(a, item, f, mp, cc);
      const int m = (2 * mp + static_cast<int>(rank)) * kBlockM + row;
      const bool row_ok = m < a.hw;
      // the row's scale: c_row = max_t c_t, l_row = sum_t 2^(c_t - c_row) l_t
      float c_row = 0.f, l_row = 1.f;
      if (row_ok) {
        const float2* st = a.stats + (static_cast<long long>(f) * a.hw + m) * a.key_tiles;
        c_row = __int_as_float(0xff800000u);
        for (int t = 0; t < a.key_tiles; ++t) c_row = fmaxf(c_row, st[t].x);
        l_row = 0.f;
        for (int t = 0; t < a.key_tiles; ++t) {
          const float2 v = st[t];
          l_row += v.y * pow2_nonpos(v.x - c_row);
        }
      }
      for (int t = 0; ok && t < a.key_tiles; ++t, ++g) {
        if (!named_barrier_and(1, 128, mbar_wait(smem_u32(s_ready), g & 1, a.err, tlim))) {
          ok = false;
          break;
        }
        tc_fence_after();
        // E = exp2(kx*s - c_row) for this row's 256 keys, packed to bf16;
        // keys past HW and rows past HW are zero
        uint32_t pk[4][32];
        const int n0 = t * kFaKeys;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r0[32], r1[32];
          tmem_ld32_wait(tmem_base + lanes + kFaSCol + c * 64, r0);
          tmem_ld32_wait(tmem_base + lanes + kFaSCol + c * 64 + 32, r1);
          const int nb = n0 + c * 64;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const uint32_t s0 = j < 16 ? r0[2 * j] : r1[2 * j - 32];
            const uint32_t s1 = j < 16 ? r0[2 * j + 1] : r1[2 * j - 31];
            float e0 = ex2_approx(fmaf(__uint_as_float(s0), kx, -c_row));
            float e1 = ex2_approx(fmaf(__uint_as_float(s1), kx, -c_row));
            e0 = (row_ok && nb + 2 * j < a.hw) ? e0 : 0.f;
            e1 = (row_ok && nb + 2 * j + 1 < a.hw) ? e1 : 0.f;
            __nv_bfloat162 b = __floats2bfloat162_rn(e0, e1);
            pk[c][j] = *reinterpret_cast<uint32_t*>(&b);
          }
        }
        // S read: the next tile's S may overwrite it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(s_free_leader);
        // the previous tile's PV must have read E before it is replaced
        if (!named_barrier_and(1, 128, mbar_wait(smem_u32(e_free), (g & 1) ^ 1u, a.err, tlim))) {
          ok = false;
          break;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint8_t* rowp = sE + c * kFaEBlock + row * 128;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<uint4*>(rowp + ((j ^ (row & 7)) << 4)) =
                make_uint4(pk[c][4 * j], pk[c][4 * j + 1], pk[c][4 * j + 2], pk[c][4 * j + 3]);
        }
        // make the rows visible to the (leader's) tensor-core reads
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_release(e_ready_leader);
      }
      if (!ok) break;
      // O: divide by l_row, one rounding, 16-byte stores of 8 channels
      if (!named_barrier_and(1, 128, mbar_wait(smem_u32(o_ready), it & 1, a.err, tlim))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float inv = 1.f / l_row;
      __nv_bfloat16* orow = a.out + (static_cast<long long>(f) * a.hw + m) * a.ld_o + cc * kFaChunk;
#pragma unroll 1
      for (int c = 0; c < kFaChunk / 32; ++c) {
        uint32_t r[32];
        tmem_ld32_wait(tmem_base + lanes + kFaOCol + c * 32, r);
        if (row_ok) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              __nv_bfloat162 b = __floats2bfloat162_rn(__uint_as_float(r[8 * q + 2 * j]) * inv,
                                                       __uint_as_float(r[8 * q + 2 * j + 1]) * inv);
              w[j] = *reinterpret_cast<uint32_t*>(&b);
            }
            *reinterpret_cast<uint4*>(orow + c * 32 + 8 * q) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(o_free_leader);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 512);
  }
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

extern "C" size_t cc_attn_fused_workspace_bytes(int t, int hw) {
  if (t <= 0 || hw <= 0) return 0;
  return round_up((size_t)t * hw * cc_attn_exp_key_tiles(hw) * 8, 256);
}

extern "C" cc_status cc_attn_frame_fused(const cc_bf16* q, const cc_bf16* k, const cc_bf16* v, cc_bf16* o, int t,
                                         int hw, int c, int64_t ld_q, int64_t ld_k, int64_t ld_v, int64_t ld_o,
                                         float scale, void* ws, size_t ws_bytes, void* stream) {
  const char* what = "attn_frame_fused";
  cc_status st;
  if (empty_request(what, {t, hw}, &st)) return st;
  if ((st = check_ptr(what, q)) != CC_OK || (st = check_ptr(what, k)) != CC_OK || (st = check_ptr(what, v)) != CC_OK ||
      (st = check_ptr(what, o)) != CC_OK || (st = check_ptr(what, ws)) != CC_OK)
    return st;
  if (t <= 0 || hw <= 0 || c <= 0) return fail(CC_ERR_INVALID, "%s: sizes must be positive", what);
  if (c % kFaChunk != 0) return fail(CC_ERR_UNSUPPORTED, "%s: C must be a multiple of 256 (got %d)", what, c);
  if (ld_q < c || ld_k < c || ld_v < c || ld_o < c) return fail(CC_ERR_INVALID, "%s: row strides too small", what);
  if (ld_q % 8 || ld_k % 8 || ld_v % 8 || ld_o % 8)
    return fail(CC_ERR_INVALID, "%s: row strides must be multiples of 8", what);
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(CC_ERR_INVALID, "%s: scale must be finite and > 0", what);
  const size_t need = cc_attn_fused_workspace_bytes(t, hw);
  if (ws_bytes < need) return fail(CC_ERR_INVALID, "%s: workspace of %zu bytes, need %zu", what, ws_bytes, need);
  const long long items = (long long)t * ((hw + 2 * kBlockM - 1) / (2 * kBlockM)) * (c / kFaChunk);
  if (items > 0x7fffffffLL) return fail(CC_ERR_UNSUPPORTED, "%s: too many work items", what);
  DeviceInfo di;
  if ((st = device_info(&di)) != CC_OK) return st;
  float* stats = static_cast<float*>(ws);
  if ((st = cc_attn_scores_stats(q, k, stats, t, hw, c, ld_q, ld_k, scale, stream)) != CC_OK) return st;
  CUtensorMap tq, tk, tv;
  if ((st = encode_tiled_3d(&tq, q, c, hw, t, 2ull * ld_q, 2ull * ld_q * hw, kBlockK, kBlockM)) != CC_OK) return st;
  if ((st = encode_tiled_3d(&tk, k, c, hw, t, 2ull * ld_k, 2ull * ld_k * hw, kBlockK, kFaKeys / 2)) != CC_OK)
    return st;
  // v as stored: channels innermost, 64 channels x 64 keys per box (MN-major B)
  if ((st = encode_tiled_3d(&tv, v, c, hw, t, 2ull * ld_v, 2ull * ld_v * hw, 64, kBlockK)) != CC_OK) return st;
  FaArgs a{};
  a.hw = hw;
  a.frames = t;
  a.m_pairs = (hw + 2 * kBlockM - 1) / (2 * kBlockM);
  a.chunks = c / kFaChunk;
  a.key_tiles = cc_attn_exp_key_tiles(hw);
  a.kb_s = c / kBlockK;
  a.items = static_cast<int>(items);
  a.exp_k = scale * 1.4426950408889634f;
  a.stats = reinterpret_cast<const float2*>(stats);
  a.out = reinterpret_cast<__nv_bfloat16*>(o);
  a.ld_o = ld_o;
  a.err = di.err_word;
  a.timeout_ns = kWaitLimitNs;
  cudaError_t e = cudaFuncSetAttribute(attn_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kFaSmem);
  if (e != cudaSuccess) return fail(CC_ERR_CUDA, "%s: shared-memory attribute: %s", what, cudaGetErrorString(e));
  const int pairs = std::min(a.items, di.sm_count / 2);
  e = launch_pdl(attn_fused_kernel, dim3(2 * pairs), dim3(kGemmThreads), kFaSmem, static_cast<cudaStream_t>(stream),
                 tq, tk, tv, a);
  if (e != cudaSuccess) return fail(CC_ERR_CUDA, "%s: launch: %s", what, cudaGetErrorString(e));
  return launch_status(what);
}
