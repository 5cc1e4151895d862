// Output head, stage A: the temporal-only (3x1x1) part of conv_out, written as
// g[n,t,p,(i*3+j)*12+c] = sum_{ci,kt} wp[kt][(i*3+j)*12+c][ci] x~[n,t+kt-2,p,ci]
// (p = in-plane position), and the weight repack that feeds it.
//
// The operation is HBM-bound (a 256-channel input read once, 112 channels
// written), so the kernel is organised around reading x exactly once:
//  - the whole repacked weight (3 taps x 112 rows x C_in, 172 KB at C_in=256)
//    is loaded into shared memory once per CTA and stays resident;
//  - a CTA owns a 128-position in-plane tile of one image and walks its frames
//    in order; each input frame tile (128 x C_in) is loaded once and feeds the
//    three outputs that read it -- frame f is tap kt of output f - hist + 2 - kt
//    -- through three of four TMEM accumulators (4 x 128 columns), so an
//    output is complete, and drained by the epilogue warps, as soon as its
//    last (kt = 2) frame has been multiplied in.
//  - CTAs work in pairs (cta_group::2): a pair owns two neighbouring tiles,
//    each CTA streams its own tile and keeps half of the weight's rows
//    (56 of each tap's 112, 86 KB), so 6 A stages (96 KB) fit beside it and
//    enough input is in flight to run at the copy bandwidth; one
//    tcgen05.mma.cta_group::2 (M=256, N=112) from the even CTA covers both.
//  - The work is the sequence of (tile pair, output frame) items, split into
//    equal contiguous shares, one per CTA pair: a share may start or end in
//    the middle of a tile pair's frames (a segment), and a segment that starts
//    at output u0 re-reads the (up to two) input frames before it that
//    output u0 needs. Whole tile pairs per CTA pair would leave the last
//    wave a quarter full at the bench size (858 tile pairs on 76 CTA pairs).
// Warp 0 streams A with TMA, warp 1 of the even CTA issues the MMAs (the whole
// warp runs the loop, one elected lane issues), warps 2-5 of both CTAs drain
// accumulators to bf16 g. Every wait is bounded.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "cc.h"
#include "cc_gemm_launch.cuh"
#include "cc_host.h"
#include "cc_ptx.cuh"

namespace cc {
namespace {

constexpr int kHeadN = CC_HEAD_G_CH;  // 112 output channels of stage A
constexpr int kHeadAccCols = 128;     // TMEM columns per accumulator slot
constexpr int kHeadSlots = 4;         // outputs t, t+1, t+2 accumulating + one draining
constexpr int kSmemBudget = 232448;

struct HeadArgs {
  int plane;        // positions per frame (H*W)
  int plane_tiles;  // 128-position tiles per frame
  int pair_tiles;   // pairs of tiles per frame: ceil(plane_tiles / 2)
  int units;        // images x pair_tiles
  long long work;   // units x d_out: (tile pair, output frame) items
  int d_in;         // frames of x per image (D + hist)
  int d_out;        // output frames per image
  int hist;         // 0 or 2
  __nv_bfloat16* g;
  unsigned int* err;
  unsigned long long timeout_ns;
};

template <int CB>  // C_in / 64
struct HeadShape {
  static constexpr int kHalfN = kHeadN / 2;              // weight rows per CTA of the pair
  static constexpr int kBBlock = kHalfN * kBlockK * 2;   // one tap x 64 channels, this CTA's half: 7168 B
  static constexpr int kBBytes = 3 * CB * kBBlock;
  static constexpr int kABytes = kBlockM * kBlockK * 2;
  static constexpr int kOutBytes = kBlockM * kHeadN * 2;  // one output tile staged for a bulk store: 28 KB
  static constexpr int kAStagesFit = (kSmemBudget - 1024 - 256 - kBBytes - kOutBytes) / kABytes;
  static constexpr int kAStages = kAStagesFit > 6 ? 6 : kAStagesFit;
  static constexpr int kSmemBytes = 1024 + kBBytes + kAStages * kABytes + kOutBytes + 256;
  static_assert(kBBlock % 1024 == 0, "weight blocks must keep 1024-byte swizzle atoms aligned");
  static_assert(kAStages >= 2, "at least two A stages");
  static_assert(kSmemBytes <= kSmemBudget, "shared memory budget");
};

// First frame of x that contributes to output u.
__device__ __forceinline__ int first_frame(int u, int hist) { return max(0, u + hist - 2); }

// The next segment of this CTA pair's share [*g, end) of the work items:
// outputs u0 .. u1-1 of tile pair `unit`. False when the share is done.
__device__ __forceinline__ bool next_segment(const HeadArgs& a, long long& g, long long end, int& unit, int& u0,
                                             int& u1) {
  if (g >= end) return false;
  unit = static_cast<int>(g / a.d_out);
  u0 = static_cast<int>(g - static_cast<long long>(unit) * a.d_out);
  u1 = static_cast<int>(min(static_cast<long long>(a.d_out), u0 + (end - g)));
  g += u1 - u0;
  return true;
}

template <int CB>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    head_temporal_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                         const __grid_constant__ HeadArgs a) {
  using S = HeadShape<CB>;
  constexpr int AST = S::kAStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sB = smem;
  uint8_t* sA = smem + S::kBBytes;
  uint8_t* sOut = sA + AST * S::kABytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sOut + S::kOutBytes);
  uint64_t* afull = bars;
  uint64_t* aempty = bars + AST;
  uint64_t* bfull = bars + 2 * AST;
  uint64_t* tfull = bfull + 1;
  uint64_t* tempty = tfull + kHeadSlots;
  uint64_t* done = tempty + kHeadSlots;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;
  const long long share_begin = a.work * pair / npairs;
  const long long share_end = a.work * (pair + 1) / npairs;
  if (threadIdx.x == 0) {
    for (int s = 0; s < AST; ++s) {
      mbar_init(smem_u32(&afull[s]), 1);
      mbar_init(smem_u32(&aempty[s]), 1);
    }
    mbar_init(smem_u32(bfull), 1);
    for (int i = 0; i < kHeadSlots; ++i) {
      mbar_init(smem_u32(&tfull[i]), 1);
      mbar_init(smem_u32(&tempty[i]), 2 * 4);  // one arrival per epilogue warp of each CTA
    }
    mbar_init(smem_u32(done), 1);
    fence_mbar_init();
    tma_prefetch_map(&tmX);
    tma_prefetch_map(&tmW);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), kHeadSlots * kHeadAccCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // set up: let the next kernel on the stream be scheduled, then wait for the
  // previous one before the first global access
  pdl_launch_dependents();
  pdl_wait();
  const uint64_t tlim = a.timeout_ns;

  if (warp == 0) {
    // ---------------------------------------------------- TMA producer --
    if (lane == 0) {
      // this CTA's half of the weight: rows rank*56 .. rank*56+55 of each tap
      const uint32_t bb_local = smem_u32(bfull);
      const uint32_t bb = mapa_shared(bb_local, 0);
      if (leader) mbar_arrive_expect_tx(bb_local, 2 * S::kBBytes);
      for (int tap = 0; tap < 3; ++tap)
        for (int kb = 0; kb < CB; ++kb)
          tma_load_2d_pair(smem_u32(sB + (tap * CB + kb) * S::kBBlock), &tmW, bb, kb * kBlockK,
                           tap * kHeadN + static_cast<int>(rank) * S::kHalfN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      long long gi = share_begin;
      int unit, u0, u1;
      while (ok && next_segment(a, gi, share_end, unit, u0, u1)) {
        const int img = unit / a.pair_tiles;
        const int m0 = (2 * (unit - img * a.pair_tiles) + static_cast<int>(rank)) * kBlockM;
        for (int f = first_frame(u0, a.hist); ok && f < u1 + a.hist; ++f) {
          for (int kb = 0; kb < CB; ++kb) {
            if (!mbar_wait(smem_u32(&aempty[stage]), phase ^ 1u, a.err, tlim)) {
              ok = false;
              break;
            }
            const uint32_t fb_local = smem_u32(&afull[stage]);
            if (leader) mbar_arrive_expect_tx(fb_local, 2 * S::kABytes);
            tma_load_3d_pair(smem_u32(sA + stage * S::kABytes), &tmX, mapa_shared(fb_local, 0), kb * kBlockK, m0,
                             img * a.d_in + f);
            if (++stage == AST) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (leader) {
        // copies of both CTAs complete on the even CTA's barriers
        if (!ok)
          for (int s = 0; s < AST; ++s)
            (void)mbar_wait(smem_u32(&afull[s]), (s < stage) ? phase : (phase ^ 1u), a.err, 200000000ull);
        (void)mbar_wait(bb_local, 0, a.err, 200000000ull);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------- MMA issuer (even CTA's warp) --
    // The whole warp runs the loop (waits and descriptors stay warp-uniform);
    // the elected lane issues the MMAs and the commits that track them.
    if (leader) {
      constexpr uint32_t idesc = idesc_bf16_f32(2 * kBlockM, kHeadN, false);
      // descriptors of A stage 0 and weight block 0; the others differ only in
      // the start-address field (all blocks are 1024-byte aligned)
      const uint64_t a_desc0 = sdesc_sw128(smem_u32(sA), 16, 1024);
      const uint64_t b_desc0 = sdesc_sw128(smem_u32(sB), 16, 1024);
      bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(bfull), 0, a.err, tlim));
      tc_fence_after();
      int stage = 0;
      uint32_t phase = 0;
      int q_base = 0;  // sequence number of the segment's output u0 among this CTA's outputs, minus u0
      long long gi = share_begin;
      int unit, u0, u1;
      while (ok && next_segment(a, gi, share_end, unit, u0, u1)) {
        q_base -= u0;
        for (int f = first_frame(u0, a.hist); ok && f < u1 + a.hist; ++f) {
          // Outputs this frame starts must have their accumulator slot drained.
          for (int kt = 0; kt < 3; ++kt) {
            const int u = f - a.hist + 2 - kt;
            if (u < u0 || u >= u1 || f != first_frame(u, a.hist)) continue;
            const int q = q_base + u;
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&tempty[q & 3]), ((q >> 2) & 1) ^ 1u, a.err, tlim))) {
              ok = false;
              break;
            }
          }
          if (!ok) break;
          tc_fence_after();
          // per frame: which of the three taps feed a live output, into which
          // accumulator, and whether this frame starts that output
          uint32_t d_col[3];
          bool live[3], starts[3];
#pragma unroll
          for (int kt = 0; kt < 3; ++kt) {
            const int u = f - a.hist + 2 - kt;
            live[kt] = u >= u0 && u < u1;
            starts[kt] = live[kt] && f == first_frame(u, a.hist);
            d_col[kt] = tmem_base + ((q_base + u) & 3) * kHeadAccCols;
          }
          for (int kb = 0; kb < CB; ++kb) {
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&afull[stage]), phase, a.err, tlim))) {
              ok = false;
              break;
            }
            tc_fence_after();
            // K advances by 16 bf16 = 32 bytes = 2 in the descriptor's address field
            const uint64_t ad = a_desc0 + static_cast<uint64_t>(stage) * (S::kABytes >> 4);
            if (elect_one()) {
#pragma unroll
              for (int kt = 0; kt < 3; ++kt) {
                if (!live[kt]) continue;
                const uint64_t bd = b_desc0 + static_cast<uint64_t>((kt * CB + kb) * (S::kBBlock >> 4));
                const uint32_t acc0 = (starts[kt] && kb == 0) ? 0u : 1u;
#pragma unroll
                for (int k = 0; k < kBlockK / kUmmaK; ++k)
                  mma_bf16_pair(d_col[kt], ad + 2 * k, bd + 2 * k, idesc, k == 0 ? acc0 : 1u);
              }
              mma_commit_pair_both(smem_u32(&aempty[stage]));
            }
            __syncwarp();
            if (++stage == AST) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          const int u_done = f - a.hist;  // its kt = 2 frame was the last one
          if (u_done >= u0 && u_done < u1) {
            if (elect_one()) mma_commit_pair_both(smem_u32(&tfull[(q_base + u_done) & 3]));
            __syncwarp();
          }
        }
        q_base += u1;
      }
      if (elect_one()) mma_commit_pair_both(smem_u32(done));
      __syncwarp();
      (void)mbar_wait(smem_u32(done), 0, a.err, tlim);
    }
  } else {
    // -------------------------------------------------------- epilogue --
    // Per output: all 112 columns of this thread's row come out of TMEM in
    // one go, the slot is released at once, and the 128 x 112 bf16 tile --
    // contiguous in g -- leaves through shared memory as one bulk copy.
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const bool issuer = (warp == 2 && lane == 0);
    uint8_t* my_row = sOut + row * (kHeadN * 2);
    int q = 0;
    bool ok = true;
    long long gi = share_begin;
    int unit, u0, u1;
    while (ok && next_segment(a, gi, share_end, unit, u0, u1)) {
      const int img = unit / a.pair_tiles;
      const int m0 = (2 * (unit - img * a.pair_tiles) + static_cast<int>(rank)) * kBlockM;
      const int rows = min(kBlockM, a.plane - m0);  // may be <= 0 for the odd CTA of the last pair
      for (int u = u0; u < u1; ++u, ++q) {
        const int slot = q & 3;
        // uniform over the four epilogue warps: they leave together, since
        // they share .sync.aligned TMEM loads and named barriers
        if (!named_barrier_and(1, 128, mbar_wait(smem_u32(&tfull[slot]), (q >> 2) & 1, a.err, tlim))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + slot * kHeadAccCols;
        uint32_t r[7][16];
#pragma unroll
        for (int c = 0; c < 7; ++c) tmem_ld16(tbase + c * 16, r[c]);
#pragma unroll
        for (int c = 0; c < 7; ++c) tmem_wait16(r[c]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[slot]), 0));
        // the previous output's bulk store must have read the staging tile
        if (issuer) bulk_wait_read_all();
        named_barrier_sync(1, 128);
#pragma unroll
        for (int c = 0; c < 7; ++c) {
          uint4 pk[2];
          __nv_bfloat162* p2 = reinterpret_cast<__nv_bfloat162*>(pk);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            p2[j] = __floats2bfloat162_rn(__uint_as_float(r[c][2 * j]), __uint_as_float(r[c][2 * j + 1]));
          reinterpret_cast<uint4*>(my_row + c * 32)[0] = pk[0];
          reinterpret_cast<uint4*>(my_row + c * 32)[1] = pk[1];
        }
        fence_proxy_async_smem();
        named_barrier_sync(1, 128);
        if (issuer && rows > 0) {
          bulk_store(a.g + ((long long)(img * a.d_out + u) * a.plane + m0) * kHeadN, smem_u32(sOut),
                     static_cast<uint32_t>(rows) * kHeadN * 2);
          bulk_commit();
        }
      }
    }
    if (issuer) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kHeadSlots * kHeadAccCols);
  }
}

// wp[kt][(i*3+j)*12 + c][ci] = w[c][ci][kt][i][j]; rows 108..111 zero.
__global__ void head_prepare_kernel(const __nv_bfloat16* __restrict__ w, __nv_bfloat16* __restrict__ wp, int cin) {
  const long long total = 3LL * CC_HEAD_G_CH * cin;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
    const int ci = static_cast<int>(i % cin);
    const long long r = i / cin;
    const int row = static_cast<int>(r % CC_HEAD_G_CH);
    const int kt = static_cast<int>(r / CC_HEAD_G_CH);
    __nv_bfloat16 v = __float2bfloat16_rn(0.f);
    if (row < 9 * CC_HEAD_COUT) {
      const int c = row % CC_HEAD_COUT, tap = row / CC_HEAD_COUT;  // tap = i*3 + j
      v = w[((long long)c * cin + ci) * 27 + kt * 9 + tap];
    }
    wp[i] = v;
  }
}

cc_status check_ptr(const char* what, const void* p) {
  if (!p) return fail(CC_ERR_INVALID, "%s: null pointer", what);
  if (!aligned16(p)) return fail(CC_ERR_INVALID, "%s: pointers must be 16-byte aligned", what);
  return CC_OK;
}

template <int CB>
cc_status launch_head_temporal(const CUtensorMap& tx, const CUtensorMap& tw, HeadArgs& a, const DeviceInfo& di,
                               cudaStream_t stream) {
  using S = HeadShape<CB>;
  auto kern = head_temporal_kernel<CB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
  if (e != cudaSuccess) return fail(CC_ERR_CUDA, "head_temporal: shared-memory attribute: %s", cudaGetErrorString(e));
  a.err = di.err_word;
  a.timeout_ns = kWaitLimitNs;
  e = launch_pdl(kern, dim3(2 * static_cast<int>(std::min<long long>(a.work, di.sm_count / 2))), dim3(kGemmThreads),
                 S::kSmemBytes, stream, tx, tw, a);
  if (e != cudaSuccess) return fail(CC_ERR_CUDA, "head_temporal: launch: %s", cudaGetErrorString(e));
  return launch_status("head_temporal");
}

}  // namespace
}  // namespace cc

using namespace cc;

extern "C" cc_status cc_head_prepare(const cc_bf16* w, cc_bf16* wp, int cin, void* stream) {
  cc_status st;
  if ((st = check_ptr("head_prepare", w)) != CC_OK || (st = check_ptr("head_prepare", wp)) != CC_OK) return st;
  if (cin <= 0) return fail(CC_ERR_INVALID, "head_prepare: C_in must be positive");
  DeviceInfo di;
  if ((st = device_info(&di)) != CC_OK) return st;
  const long long total = 3LL * CC_HEAD_G_CH * cin;
  head_prepare_kernel<<<(unsigned)std::min<long long>((total + 255) / 256, 8192), 256, 0,
                        static_cast<cudaStream_t>(stream)>>>(reinterpret_cast<const __nv_bfloat16*>(w),
                                                             reinterpret_cast<__nv_bfloat16*>(wp), cin);
  return launch_status("head_prepare");
}

extern "C" cc_status cc_head_temporal(const cc_bf16* x, const cc_bf16* wp, cc_bf16* g, int n, int d, int h, int w,
                                      int cin, int hist, void* stream) {
  const char* what = "head_temporal";
  cc_status st;
  if (empty_request(what, {n, d, h, w}, &st)) return st;
  if ((st = check_ptr(what, x)) != CC_OK || (st = check_ptr(what, wp)) != CC_OK || (st = check_ptr(what, g)) != CC_OK)
    return st;
  if (n <= 0 || d <= 0 || h <= 0 || w <= 0) return fail(CC_ERR_INVALID, "%s: sizes must be positive", what);
  if (hist != 0 && hist != 2) return fail(CC_ERR_INVALID, "%s: hist must be 0 or 2", what);
  if (cin <= 0 || cin % 64 != 0 || cin > 256)
    return fail(CC_ERR_UNSUPPORTED, "%s: C_in must be 64, 128, 192 or 256 (got %d)", what, cin);
  const long long plane = (long long)h * w;
  if (plane * n * (d + hist) > (1LL << 31) - 1) return fail(CC_ERR_UNSUPPORTED, "%s: too many positions", what);
  DeviceInfo di;
  if ((st = device_info(&di)) != CC_OK) return st;
  CUtensorMap tx, tw;
  // x as [frames = N*(D+hist)][plane][C_in]; rows past the plane are zero-filled
  if ((st = encode_tiled_3d(&tx, x, cin, plane, (uint64_t)n * (d + hist), 2ull * cin, 2ull * cin * plane, kBlockK,
                            kBlockM)) != CC_OK)
    return st;
  if ((st = encode_tiled_2d(&tw, wp, cin, 3ull * CC_HEAD_G_CH, 2ull * cin, kBlockK, CC_HEAD_G_CH / 2)) != CC_OK)
    return st;
  HeadArgs a{};
  a.plane = static_cast<int>(plane);
  a.plane_tiles = ceil_div(plane, kBlockM);
  a.pair_tiles = (a.plane_tiles + 1) / 2;
  a.units = n * a.pair_tiles;
  a.work = static_cast<long long>(a.units) * d;
  a.d_in = d + hist;
  a.d_out = d;
  a.hist = hist;
  a.g = reinterpret_cast<__nv_bfloat16*>(g);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (cin / 64) {
    case 1: return launch_head_temporal<1>(tx, tw, a, di, s);
    case 2: return launch_head_temporal<2>(tx, tw, a, di, s);
    case 3: return launch_head_temporal<3>(tx, tw, a, di, s);
    default: return launch_head_temporal<4>(tx, tw, a, di, s);
  }
}
