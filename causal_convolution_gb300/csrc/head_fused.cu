// Output head in ONE kernel: causal conv_out (3x3x3, C_in -> 12) + bias +
// clamp to [-1, 1], with the regrouping of [HEAD]'s header comment -- a
// temporal-only 3x1x1 conv into 9 x 12 channels g (spatial tap (i, j) of
// output channel c in channel (i*3+j)*12 + c), then the 3x3 stencil
//   out[t,h,w,c] = clamp(b[c] + sum_{i,j} g[t, h+i-1, w+j-1, (i*3+j)*12+c])
// -- done on chip: g stays in fp32 (TMEM, then registers) and never reaches
// memory, so the head reads x once and writes the 12-channel output, and its
// only rounding is the output's.
//
// Tiles. A CTA's 128 accumulator rows are a 4-row x 32-column block of one
// frame: column 0 and 31 are the halo columns of a strip of 30 interior
// columns (strips overlap by the two halo columns, whose g is recomputed), and
// a TMA box [64 channels, 32 columns, 4 rows] loads the block's x, zero-filled
// outside the plane (which is the stencil's zero padding). TMEM lane 32r + l
// holds row r, column l: epilogue warp r (by TMEM lane quarter) owns row r.
//
// Time. As in the two-stage head's first kernel (head.cu): each input frame
// tile is loaded once and multiplied into the (up to) three outputs that read
// it, through four rotating TMEM accumulators of 112 columns; a CTA pair
// (cta_group::2, M = 256, N = 112) shares one MMA, each CTA keeping half of
// the weight rows resident (86 KB at C_in = 256).
//
// Space. A CTA walks the row blocks of a strip downwards (a segment of output
// rows [a, b) of one strip), all output frames of a block before the next.
// For each output frame the epilogue
//  - sums each g row horizontally: r_i[w] = g[w-1](i,0) + g[w](i,1) + g[w+1](i,2)
//    (12 channels each), the neighbours' values by warp shuffles;
//  - sums vertically: out[row] = r_0[row-1] + r_1[row] + r_2[row+1], the
//    neighbour rows' r_0 / r_2 exchanged through shared memory between the
//    four warps;
//  - carries to the next row block, per column and frame, the partial sums of
//    the two outputs it cannot finish yet (the block's last row, which needs
//    the next block's first, and the next block's first row, which needs this
//    block's last): 24 fp32 values, 49 KB of shared memory for 16 frames.
// A segment's first block starts one row above a (its own first output row
// needs that row's r_0), so each segment recomputes two g rows: one above and
// one below its outputs.
//
// Work: the strip-rows of all images and strips, cut into equal contiguous
// shares, one per CTA (a share may span strips: several segments). The two
// CTAs of a pair run in lockstep through the shared MMA; the one with fewer
// blocks loads out-of-plane boxes (zero fill, nothing read) for the rest and
// stores nothing for them. Every wait is bounded.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "cc.h"
#include "cc_gemm_launch.cuh"
#include "cc_host.h"
#include "cc_ptx.cuh"

namespace cc {
namespace {

constexpr int kHeadN = CC_HEAD_G_CH;  // 112 accumulator columns (108 used)
constexpr int kAccCols = 128;         // TMEM columns per accumulator slot
constexpr int kSlots = 4;
constexpr int kTR = 4;                // block rows: one epilogue warp each
constexpr int kTC = 32;               // block columns: one lane each
constexpr int kTI = kTC - 2;          // interior columns per strip
constexpr int kMaxD = 16;             // output frames per pass (carried state)
constexpr int kMaxCtas = 256;         // shares the host can hand out
constexpr int kPrefetchFrames = 1;    // x frames requested into L2 ahead of their loads
constexpr int kSmemBudget = 232448;

struct FusedArgs {
  int h, w;          // plane
  int strips;        // ceil(w / 30)
  int d_out;         // output frames per image in this pass (<= kMaxD)
  int hist;          // 0 or 2
  int d_in;          // input frames of x per image in this pass: d_out + hist
  long long units;   // strip-rows: images x strips x h
  long long out_img; // elements between images of out
  // CTA i takes strip-rows [share[i], share[i+1]); at most kMaxCtas CTAs
  long long share[kMaxCtas + 1];
  const __nv_bfloat16* bias;
  __nv_bfloat16* out;
  unsigned int* err;
  unsigned long long timeout_ns;
};

template <int CB>  // C_in / 64
struct FusedShape {
  static constexpr int kHalfN = kHeadN / 2;              // weight rows per CTA of the pair
  static constexpr int kBBlock = kHalfN * kBlockK * 2;   // one tap x 64 channels: 7168 B
  static constexpr int kBBytes = 3 * CB * kBBlock;
  static constexpr int kABytes = kBlockM * kBlockK * 2;  // one block of 128 positions x 64 channels
  static constexpr int kStateBytes = kMaxD * 6 * kTC * 16;  // [frame][6 float4][column]
  static constexpr int kXBytes = 6 * kBlockM * 16;          // [6 float4][thread]: r_0 and r_2
  static constexpr int kFixed = 1024 + kBBytes + kStateBytes + kXBytes + 256;
  static constexpr int kAStagesFit = (kSmemBudget - kFixed) / kABytes;
  static constexpr int kAStages = kAStagesFit > 6 ? 6 : kAStagesFit;
  static constexpr int kSmemBytes = kFixed + kAStages * kABytes;
  static_assert(kBBlock % 1024 == 0, "weight blocks must keep 1024-byte swizzle atoms aligned");
  static_assert(kAStages >= 3, "at least three A stages");
  static_assert(kSmemBytes <= kSmemBudget, "shared memory budget");
};

// First input frame (index into x's frames) that output u reads.
__device__ __forceinline__ int first_frame(int u, int hist) { return max(0, u + hist - 2); }

// The row blocks of one CTA's share of strip-rows, in order. A segment is the
// output rows [a, b) of strip `strip_id` (image * strips + strip); its blocks
// start at g rows a-1, a+3, ... until the block covering output b-1.
struct BlockIter {
  long long pos, end;
  int strip_id, a, b, h0;
  bool valid;
};

__device__ __forceinline__ void seg_start(const FusedArgs& A, BlockIter& it) {
  it.strip_id = static_cast<int>(it.pos / A.h);
  it.a = static_cast<int>(it.pos - static_cast<long long>(it.strip_id) * A.h);
  it.b = static_cast<int>(min(static_cast<long long>(A.h), it.a + (it.end - it.pos)));
  it.h0 = it.a - 1;
}
__device__ __forceinline__ void iter_init(const FusedArgs& A, BlockIter& it, long long begin, long long end) {
  it.pos = begin;
  it.end = end;
  it.valid = begin < end;
  if (it.valid) seg_start(A, it);
}
// A block starting at g row h0 finishes outputs h0-1 .. h0+2.
__device__ __forceinline__ void iter_next(const FusedArgs& A, BlockIter& it) {
  if (it.h0 + 2 < it.b - 1) {
    it.h0 += kTR;
    return;
  }
  it.pos += it.b - it.a;
  it.valid = it.pos < it.end;
  if (it.valid) seg_start(A, it);
}
__device__ __forceinline__ long long share_begin(const FusedArgs& A, int cta, int) { return A.share[cta]; }
__device__ int count_blocks(const FusedArgs& A, int cta, int ctas) {
  BlockIter it;
  iter_init(A, it, share_begin(A, cta, ctas), share_begin(A, cta + 1, ctas));
  int n = 0;
  while (it.valid) {
    ++n;
    iter_next(A, it);
  }
  return n;
}

template <int CB>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    head_fused_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                      const __grid_constant__ FusedArgs a) {
  using S = FusedShape<CB>;
  constexpr int AST = S::kAStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sB = smem;
  uint8_t* sA = smem + S::kBBytes;
  float4* sState = reinterpret_cast<float4*>(sA + AST * S::kABytes);
  float4* sX = reinterpret_cast<float4*>(reinterpret_cast<uint8_t*>(sState) + S::kStateBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(sX) + S::kXBytes);
  uint64_t* afull = bars;
  uint64_t* aempty = bars + AST;
  uint64_t* bfull = bars + 2 * AST;
  uint64_t* tfull = bfull + 1;
  uint64_t* tempty = tfull + kSlots;
  uint64_t* done = tempty + kSlots;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int ctas = gridDim.x;
  const int cta = blockIdx.x;
  if (threadIdx.x == 0) {
    for (int s = 0; s < AST; ++s) {
      mbar_init(smem_u32(&afull[s]), 1);
      mbar_init(smem_u32(&aempty[s]), 1);
    }
    mbar_init(smem_u32(bfull), 1);
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(smem_u32(&tfull[i]), 1);
      mbar_init(smem_u32(&tempty[i]), 2 * 4);  // one arrival per epilogue warp of each CTA
    }
    mbar_init(smem_u32(done), 1);
    fence_mbar_init();
    tma_prefetch_map(&tmX);
    tma_prefetch_map(&tmW);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), kSlots * kAccCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_launch_dependents();
  pdl_wait();
  const uint64_t tlim = a.timeout_ns;
  // both CTAs of the pair run the larger of their two block counts
  const int pair0 = cta & ~1;
  const int nblocks = max(count_blocks(a, pair0, ctas), count_blocks(a, pair0 + 1, ctas));

  if (warp == 0) {
    // ---------------------------------------------------- TMA producer --
    if (lane == 0) {
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
      BlockIter it;
      iter_init(a, it, share_begin(a, cta, ctas), share_begin(a, cta + 1, ctas));
      const int f_first = first_frame(0, a.hist);
      for (int blk = 0; ok && blk < nblocks; ++blk) {
        int img = 0, col = -1, row = a.h;  // past the pair's own blocks: an out-of-plane box (zero fill)
        if (it.valid) {
          img = it.strip_id / a.strips;
          col = (it.strip_id - img * a.strips) * kTI - 1;
          row = it.h0;
        }
        // the block after this one, for prefetches that run past its last frame
        BlockIter nx = it;
        if (nx.valid) iter_next(a, nx);
        for (int f = f_first; ok && f < a.d_in; ++f) {
          // ask L2 for the frame kPrefetchFrames ahead: the stage ring alone
          // holds too few bytes to cover the DRAM latency at this rate
          if (it.valid) {
            const int pf = f + kPrefetchFrames;
            if (pf < a.d_in) {
              for (int kb = 0; kb < CB; ++kb) tma_prefetch_5d(&tmX, kb * kBlockK, col, row, pf, img);
            } else if (nx.valid) {
              const int nimg = nx.strip_id / a.strips;
              const int ncol = (nx.strip_id - nimg * a.strips) * kTI - 1;
              for (int kb = 0; kb < CB; ++kb)
                tma_prefetch_5d(&tmX, kb * kBlockK, ncol, nx.h0, f_first + pf - a.d_in, nimg);
            }
          }
          for (int kb = 0; kb < CB; ++kb) {
            if (!mbar_wait(smem_u32(&aempty[stage]), phase ^ 1u, a.err, tlim)) {
              ok = false;
              break;
            }
            const uint32_t fb_local = smem_u32(&afull[stage]);
            if (leader) mbar_arrive_expect_tx(fb_local, 2 * S::kABytes);
            tma_load_5d_pair(smem_u32(sA + stage * S::kABytes), &tmX, mapa_shared(fb_local, 0), kb * kBlockK, col,
                             row, f, img);
            if (++stage == AST) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        if (it.valid) iter_next(a, it);
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
      const uint64_t a_desc0 = sdesc_sw128(smem_u32(sA), 16, 1024);
      const uint64_t b_desc0 = sdesc_sw128(smem_u32(sB), 16, 1024);
      bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(bfull), 0, a.err, tlim));
      tc_fence_after();
      int stage = 0;
      uint32_t phase = 0;
      int q_base = 0;  // sequence number of the block's output 0 among this pair's outputs
      for (int blk = 0; ok && blk < nblocks; ++blk) {
        for (int f = first_frame(0, a.hist); ok && f < a.d_in; ++f) {
          // outputs this frame starts must have their accumulator slot drained
          for (int kt = 0; kt < 3; ++kt) {
            const int u = f - a.hist + 2 - kt;
            if (u < 0 || u >= a.d_out || f != first_frame(u, a.hist)) continue;
            const int q = q_base + u;
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&tempty[q & 3]), ((q >> 2) & 1) ^ 1u, a.err, tlim))) {
              ok = false;
              break;
            }
          }
          if (!ok) break;
          tc_fence_after();
          uint32_t d_col[3];
          bool live[3], starts[3];
#pragma unroll
          for (int kt = 0; kt < 3; ++kt) {
            const int u = f - a.hist + 2 - kt;
            live[kt] = u >= 0 && u < a.d_out;
            starts[kt] = live[kt] && f == first_frame(u, a.hist);
            d_col[kt] = tmem_base + ((q_base + u) & 3) * kAccCols;
          }
          for (int kb = 0; kb < CB; ++kb) {
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&afull[stage]), phase, a.err, tlim))) {
              ok = false;
              break;
            }
            tc_fence_after();
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
          if (u_done >= 0 && u_done < a.d_out) {
            if (elect_one()) mma_commit_pair_both(smem_u32(&tfull[(q_base + u_done) & 3]));
            __syncwarp();
          }
        }
        q_base += a.d_out;
      }
      if (elect_one()) mma_commit_pair_both(smem_u32(done));
      __syncwarp();
      (void)mbar_wait(smem_u32(done), 0, a.err, tlim);
    }
  } else {
    // -------------------------------------------------------- epilogue --
    const int r = warp & 3;  // block row = TMEM lane quarter
    const int tid = r * 32 + lane;
    float bias[CC_HEAD_COUT];
#pragma unroll
    for (int c = 0; c < CC_HEAD_COUT; ++c) bias[c] = __bfloat162float(a.bias[c]);
    BlockIter it;
    iter_init(a, it, share_begin(a, cta, ctas), share_begin(a, cta + 1, ctas));
    int q = 0;
    bool ok = true;
    for (int blk = 0; ok && blk < nblocks; ++blk) {
      const bool real = it.valid;
      int img = 0, wcol = -1, h0 = 0, seg_a = 0, seg_b = 0;
      if (real) {
        img = it.strip_id / a.strips;
        wcol = (it.strip_id - img * a.strips) * kTI - 1 + lane;  // this lane's plane column
        h0 = it.h0;
        seg_a = it.a;
        seg_b = it.b;
      }
      // interior lanes inside the plane store; rows are checked per output
      const bool col_ok = real && lane >= 1 && lane <= kTI && wcol < a.w;
      __nv_bfloat16* out_img = a.out + static_cast<long long>(img) * a.out_img;
      for (int u = 0; u < a.d_out; ++u, ++q) {
        const int slot = q & 3;
        if (!named_barrier_and(1, 128, mbar_wait(smem_u32(&tfull[slot]), (q >> 2) & 1, a.err, tlim))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(r * 32) << 16) + slot * kAccCols;
        uint32_t g[7][16];
#pragma unroll
        for (int c = 0; c < 7; ++c) tmem_ld16(tbase + c * 16, g[c]);
#pragma unroll
        for (int c = 0; c < 7; ++c) tmem_wait16(g[c]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[slot]), 0));
        // horizontal sums: r_i[c] = g[w-1](i,0,c) + g[w](i,1,c) + g[w+1](i,2,c);
        // lanes 0 and 31 (halo columns) get values that are never used
        float rs[3][CC_HEAD_COUT];
#pragma unroll
        for (int i = 0; i < 3; ++i) {
#pragma unroll
          for (int c = 0; c < CC_HEAD_COUT; ++c) {
            const int c0 = (i * 3 + 0) * CC_HEAD_COUT + c;
            const int c1 = c0 + CC_HEAD_COUT;
            const int c2 = c1 + CC_HEAD_COUT;
            const float left = __shfl_up_sync(0xffffffffu, __uint_as_float(g[c0 >> 4][c0 & 15]), 1);
            const float right = __shfl_down_sync(0xffffffffu, __uint_as_float(g[c2 >> 4][c2 & 15]), 1);
            rs[i][c] = left + __uint_as_float(g[c1 >> 4][c1 & 15]) + right;
          }
        }
        // publish r_0 and r_2 for the rows below and above
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          sX[k * kBlockM + tid] = make_float4(rs[0][4 * k], rs[0][4 * k + 1], rs[0][4 * k + 2], rs[0][4 * k + 3]);
          sX[(3 + k) * kBlockM + tid] =
              make_float4(rs[2][4 * k], rs[2][4 * k + 1], rs[2][4 * k + 2], rs[2][4 * k + 3]);
        }
        // row 0 takes the carried sums of this frame before row 3 replaces them
        float carry[2 * CC_HEAD_COUT];
        float4* st = sState + (u * 6) * kTC + lane;
        if (r == 0) {
#pragma unroll
          for (int k = 0; k < 6; ++k) {
            const float4 v = st[k * kTC];
            carry[4 * k] = v.x;
            carry[4 * k + 1] = v.y;
            carry[4 * k + 2] = v.z;
            carry[4 * k + 3] = v.w;
          }
        }
        named_barrier_sync(1, 128);
        // the row above's r_0 (row 0: the carried r_0 of the block above) and
        // the row below's r_2
        float above[CC_HEAD_COUT], below[CC_HEAD_COUT];
        if (r > 0) {
#pragma unroll
          for (int k = 0; k < 3; ++k) {
            const float4 v = sX[k * kBlockM + tid - 32];
            above[4 * k] = v.x;
            above[4 * k + 1] = v.y;
            above[4 * k + 2] = v.z;
            above[4 * k + 3] = v.w;
          }
        }
        if (r < kTR - 1) {
#pragma unroll
          for (int k = 0; k < 3; ++k) {
            const float4 v = sX[(3 + k) * kBlockM + tid + 32];
            below[4 * k] = v.x;
            below[4 * k + 1] = v.y;
            below[4 * k + 2] = v.z;
            below[4 * k + 3] = v.w;
          }
        }
        auto store_row = [&](int y, const float (&v)[CC_HEAD_COUT]) {
          if (!col_ok || y < seg_a || y >= seg_b) return;
          uint32_t pk[CC_HEAD_COUT / 2];
#pragma unroll
          for (int c = 0; c < CC_HEAD_COUT / 2; ++c) {
            const float v0 = fminf(1.f, fmaxf(-1.f, bias[2 * c] + v[2 * c]));
            const float v1 = fminf(1.f, fmaxf(-1.f, bias[2 * c + 1] + v[2 * c + 1]));
            __nv_bfloat162 b2 = __floats2bfloat162_rn(v0, v1);
            pk[c] = *reinterpret_cast<uint32_t*>(&b2);
          }
          uint2* o = reinterpret_cast<uint2*>(
              out_img + ((static_cast<long long>(u) * a.h + y) * a.w + wcol) * CC_HEAD_COUT);
          o[0] = make_uint2(pk[0], pk[1]);
          o[1] = make_uint2(pk[2], pk[3]);
          o[2] = make_uint2(pk[4], pk[5]);
        };
        float v[CC_HEAD_COUT];
        if (r == 0) {
          // the block above's last row: carried r_0[h0-2] + r_1[h0-1], plus r_2 of row 0
#pragma unroll
          for (int c = 0; c < CC_HEAD_COUT; ++c) v[c] = carry[c] + rs[2][c];
          store_row(h0 - 1, v);
          // row 0: carried r_0[h0-1] + r_1 + the row below's r_2
#pragma unroll
          for (int c = 0; c < CC_HEAD_COUT; ++c) v[c] = carry[CC_HEAD_COUT + c] + rs[1][c] + below[c];
          store_row(h0, v);
        } else if (r < kTR - 1) {
#pragma unroll
          for (int c = 0; c < CC_HEAD_COUT; ++c) v[c] = above[c] + rs[1][c] + below[c];
          store_row(h0 + r, v);
        } else {
          // last row: carry r_0[row 2] + r_1 (for this row) and r_0 (for the next block's row 0)
#pragma unroll
          for (int k = 0; k < 3; ++k) {
            st[k * kTC] = make_float4(above[4 * k] + rs[1][4 * k], above[4 * k + 1] + rs[1][4 * k + 1],
                                      above[4 * k + 2] + rs[1][4 * k + 2], above[4 * k + 3] + rs[1][4 * k + 3]);
            st[(3 + k) * kTC] = make_float4(rs[0][4 * k], rs[0][4 * k + 1], rs[0][4 * k + 2], rs[0][4 * k + 3]);
          }
        }
        // sX is rewritten for the next frame only after every warp has read it
        named_barrier_sync(1, 128);
      }
      if (real) iter_next(a, it);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kSlots * kAccCols);
  }
}

cc_status check_ptr(const char* what, const void* p) {
  if (!p) return fail(CC_ERR_INVALID, "%s: null pointer", what);
  if (!aligned16(p)) return fail(CC_ERR_INVALID, "%s: pointers must be 16-byte aligned", what);
  return CC_OK;
}

// Blocks a share [p, p + rows) of strip-rows costs, and how far a share that
// starts at p may reach with at most `cap` blocks: a segment of L output rows
// of one strip costs floor((L + 1) / 4) + 1 blocks (its g rows a-1 .. b).
long long share_reach(long long p, long long units, int h, int cap) {
  int left = cap;
  while (p < units && left > 0) {
    const long long rest = h - p % h;         // rows left in this strip
    const long long fit = 4LL * left - 2;     // longest segment `left` blocks cover
    if (rest <= fit) {
      left -= static_cast<int>((rest + 1) / 4 + 1);
      p += rest;
    } else {
      p += fit;
      left = 0;
    }
  }
  return std::min(p, units);
}

// Cuts the strip-rows into at most `max_ctas` contiguous shares of at most
// `cap` blocks each, with the smallest cap that fits; returns the number of
// shares (the rest of a.share is units).
int split_shares(FusedArgs& a, int max_ctas) {
  const long long per = (a.units + 4LL * max_ctas - 1) / (4LL * max_ctas);
  for (int cap = static_cast<int>(std::max<long long>(1, per));; ++cap) {
    long long p = 0;
    int used = 0;
    a.share[0] = 0;
    while (p < a.units && used < max_ctas) {
      p = share_reach(p, a.units, a.h, cap);
      a.share[++used] = p;
    }
    if (p >= a.units) {
      for (int i = used + 1; i <= kMaxCtas; ++i) a.share[i] = a.units;
      return used;
    }
  }
}

template <int CB>
cc_status launch_head_fused(const CUtensorMap& tx, const CUtensorMap& tw, FusedArgs& a, const DeviceInfo& di,
                            cudaStream_t stream) {
  using S = FusedShape<CB>;
  auto kern = head_fused_kernel<CB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
  if (e != cudaSuccess) return fail(CC_ERR_CUDA, "head_out_fused: shared-memory attribute: %s", cudaGetErrorString(e));
  a.err = di.err_word;
  a.timeout_ns = kWaitLimitNs;
  // at least ~16 strip-rows per CTA, at most one CTA per SM, an even count;
  // shares of equal block counts (the two CTAs of a pair run in lockstep)
  const long long want = (a.units + 15) / 16;
  const int max_ctas = 2 * static_cast<int>(std::max<long long>(
                               1, std::min<long long>(std::min(di.sm_count, kMaxCtas) / 2, (want + 1) / 2)));
  const int used = split_shares(a, max_ctas);
  const int pairs = (used + 1) / 2;
  e = launch_pdl(kern, dim3(2 * pairs), dim3(kGemmThreads), S::kSmemBytes, stream, tx, tw, a);
  if (e != cudaSuccess) return fail(CC_ERR_CUDA, "head_out_fused: launch: %s", cudaGetErrorString(e));
  return launch_status("head_out_fused");
}

}  // namespace
}  // namespace cc

using namespace cc;

extern "C" cc_status cc_head_out_fused(const cc_bf16* x, const cc_bf16* wp, const cc_bf16* bias, cc_bf16* out, int n,
                                       int d, int h, int w, int cin, int hist, void* stream) {
  const char* what = "head_out_fused";
  cc_status st;
  if (empty_request(what, {n, d, h, w}, &st)) return st;
  if ((st = check_ptr(what, x)) != CC_OK || (st = check_ptr(what, wp)) != CC_OK ||
      (st = check_ptr(what, bias)) != CC_OK || (st = check_ptr(what, out)) != CC_OK)
    return st;
  if (n <= 0 || d <= 0 || h <= 0 || w <= 0) return fail(CC_ERR_INVALID, "%s: sizes must be positive", what);
  if (hist != 0 && hist != 2) return fail(CC_ERR_INVALID, "%s: hist must be 0 or 2", what);
  if (cin <= 0 || cin % 64 != 0 || cin > 256)
    return fail(CC_ERR_UNSUPPORTED, "%s: C_in must be 64, 128, 192 or 256 (got %d)", what, cin);
  const long long strips = (w + kTI - 1) / kTI;
  if ((long long)n * strips > (1LL << 30) || (long long)n * strips * h > (1LL << 40) ||
      (long long)n * (d + hist) * h * w > (1LL << 40) || h > (1 << 30) || w > (1 << 30))
    return fail(CC_ERR_UNSUPPORTED, "%s: tensor too large", what);
  DeviceInfo di;
  if ((st = device_info(&di)) != CC_OK) return st;
  CUtensorMap tw;
  if ((st = encode_tiled_2d(&tw, wp, cin, 3ull * CC_HEAD_G_CH, 2ull * cin, kBlockK, CC_HEAD_G_CH / 2)) != CC_OK)
    return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint64_t plane = (uint64_t)h * w;
  // one pass per group of at most 16 output frames; a later group reads its
  // two preceding input frames as carried history
  for (int u0 = 0; u0 < d; u0 += kMaxD) {
    const int dg = std::min(kMaxD, d - u0);
    const int hg = u0 == 0 ? hist : 2;
    const long long f0 = u0 == 0 ? 0 : (long long)u0 + hist - 2;  // first input frame of the group
    CUtensorMap tx;
    const uint64_t dims[5] = {(uint64_t)cin, (uint64_t)w, (uint64_t)h, (uint64_t)(dg + hg), (uint64_t)n};
    const uint64_t strides[4] = {2ull * cin, 2ull * cin * w, 2ull * cin * plane, 2ull * cin * plane * (d + hist)};
    if ((st = encode_tiled_5d(&tx, x + f0 * plane * cin, dims, strides, kBlockK, kTC, kTR)) != CC_OK) return st;
    FusedArgs a{};
    a.h = h;
    a.w = w;
    a.strips = static_cast<int>(strips);
    a.d_out = dg;
    a.hist = hg;
    a.d_in = dg + hg;
    a.units = (long long)n * strips * h;
    a.out_img = (long long)d * plane * CC_HEAD_COUT;
    a.bias = reinterpret_cast<const __nv_bfloat16*>(bias);
    a.out = reinterpret_cast<__nv_bfloat16*>(out) + (long long)u0 * plane * CC_HEAD_COUT;
    switch (cin / 64) {
      case 1: st = launch_head_fused<1>(tx, tw, a, di, s); break;
      case 2: st = launch_head_fused<2>(tx, tw, a, di, s); break;
      case 3: st = launch_head_fused<3>(tx, tw, a, di, s); break;
      default: st = launch_head_fused<4>(tx, tw, a, di, s); break;
    }
    if (st != CC_OK) return st;
  }
  return CC_OK;
}
