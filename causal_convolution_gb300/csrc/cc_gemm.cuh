// Persistent, warp-specialised tcgen05 implicit GEMM for sm_103a.
//
//   C[m, n] = sum_tap sum_k A_tap[m, k] * B_tap[n, k]      (fp32 in TMEM)
//
// One CTA per SM walks output tiles of 128 rows x BN columns. Warp 0 (one
// lane) streams A and B k-blocks of 64 bf16 (one 128-byte swizzle row) into a
// STAGES-deep shared-memory ring with TMA; warp 1 (the whole warp runs the
// loop, one elected lane issues) issues tcgen05.mma (M=128, N=BN, K=16) into
// one of two TMEM accumulators; warps 2-5
// drain the other accumulator (tcgen05.ld -> +bias -> bf16/fp32 -> global), so
// the epilogue of tile i overlaps the main loop of tile i+1.
//
// A comes either from an im2col TMA map over a channels-last activation (the
// convolutions: every tap is the same map read at a different pixel offset,
// with the causal and spatial zero padding produced by the map's bounding box
// and out-of-range fill) or from a tiled rank-3 map (the attention products).
// B is K-major (weights [rows][C_in], keys [j][C]) or MN-major (values
// [j][C], read without a transpose).
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "cc_ptx.cuh"

namespace cc {

constexpr int kBlockM = 128;
constexpr int kBlockK = 64;   // bf16 elements per 128-byte swizzle row
constexpr int kUmmaK = 16;
constexpr int kGemmThreads = 192;
constexpr int kMaxTapEntries = 64;

enum AMode : int { kAIm2col = 0, kATiled3d = 1 };

struct GemmArgs {
  int m_total;       // valid rows per batch
  int n_total;       // valid columns
  int m_tiles;       // row tiles per batch
  int n_tiles;
  int batches;       // attention: frames; resampler: phases; otherwise 1
  int num_tiles;     // m_tiles * n_tiles * batches
  int taps;          // taps per batch
  int kb_per_tap;    // 64-wide k-blocks per tap
  // Row-tile order: when frame_tiles > 0, consecutive tiles walk the frames of
  // one in-plane tile before moving on (temporal taps then hit L2).
  int frame_tiles;   // row tiles per frame (0 = plain order)
  int frames;        // frames (images x depth) when frame_tiles > 0
  // Pair kernel: nonzero walks all row tiles of one batch before the next
  // batch (the batch's B operand stays hot in L2); zero puts the batch
  // inside the row tile (a row tile's A is shared by every batch at once).
  int batch_outer;
  // im2col traversal: output grid and the bounding box's lower corner
  int img_w, img_h, img_d;
  int lo_w, lo_h, lo_d;
  // per (batch, tap): pixel offsets packed as ow | oh << 8 | od << 16
  int tap_off[kMaxTapEntries];
  int b_rows_per_tap;    // B rows between taps (2-D B map)
  int b_rows_per_batch;  // B rows between batches (2-D B map)
  // output
  void* out;
  long long out_ld;      // elements between rows
  long long out_batch;   // elements between batches
  const __nv_bfloat16* bias;  // per column, or nullptr
  const __nv_bfloat16* skip;  // resampler epilogue: shortcut rows (row m at m * out_ld)
  int epi_tscale;             // resampler epilogue: 2 when the output is also x2 in time
  // 1 when every bf16 output row piece (and shortcut row piece) of 16
  // columns starts on a 32-byte boundary: the epilogue then moves it with one
  // 32-byte access instead of two 16-byte ones (set by the launcher)
  int vec32;
  // softmax numerators in key tiles (kEpiExpBf16 writes them, kEpiRowScale
  // reads them to divide each output row by its sum): per (batch, row, key
  // tile) the pair (c_t, l_t)
  float2* stats;
  int stat_tiles;   // key tiles per row
  float exp_k;      // scale * log2(e): exp(scale * s) = exp2(exp_k * s)
  // Pair kernel: when mp_perm_n > 0, the k-th 256-row pair tile in walking
  // order is mp_perm[k] (set by the launcher for im2col convolutions over
  // several frames: tiles at the same position inside a frame, one per
  // frame, come one after another, so the rows a tile's temporal taps read
  // were loaded moments before by its neighbours and are still in L2)
  int mp_perm_n;
  unsigned short mp_perm[512];
  unsigned int* err;
  unsigned long long timeout_ns;
};

template <int BN>
struct GemmShape {
  static constexpr int kABytes = kBlockM * kBlockK * 2;
  static constexpr int kBBytes = BN * kBlockK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = BN >= 256 ? 4 : (232448 - 4096) / kStageBytes > 8 ? 8 : (232448 - 4096) / kStageBytes;
  static constexpr uint32_t kAccCols = BN <= 32 ? 32 : BN <= 64 ? 64 : BN <= 128 ? 128 : 256;
  static constexpr uint32_t kTmemCols = 2 * kAccCols;
  static constexpr int kBarBytes = 256;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kBarBytes;
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M=128 must be a multiple of 16 in [16,256]");
  static_assert(kBBytes % 1024 == 0, "B stage must be a whole number of 1024-byte swizzle atoms");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

__device__ __forceinline__ void gemm_decode_tile(const GemmArgs& a, int tile, int& batch, int& mt, int& nt) {
  nt = tile % a.n_tiles;
  int r = tile / a.n_tiles;
  batch = r % a.batches;
  r /= a.batches;
  if (a.frame_tiles > 0) {
    const int frame = r % a.frames;
    mt = frame * a.frame_tiles + r / a.frames;
  } else {
    mt = r;
  }
}

// Epilogue modes. Plain: row m of batch b goes to out + b*out_batch + m*out_ld.
// Resample: the accumulator rows are low-resolution positions (frame f, row i,
// column j) of output parity batch = 4s + 2p + q; the row is written, with the
// bias and the shortcut row m added, to high-resolution position
// (f*epi_tscale + s, 2i+p, 2j+q) of out [frames, 2*img_h, 2*img_w, out_ld] --
// the interleave done in registers (s = 0 unless the output is x2 in time).
// StoreF32: fp32 rows leave in 32-column chunks through a swizzled shared
// staging buffer and TMA tensor stores (pair kernel only).
// ExpBf16 (pair kernel only): the tile holds scores s of one row against BN
// keys; per row, with c_t = kExpGrain * ceil(exp_k * max over the tile's valid
// keys / kExpGrain), e = exp2(exp_k * s - c_t) in (0, 1] leaves as bf16 through the same staged
// TMA stores, and (c_t, l_t = sum of the fp32 e) goes to stats.
// RowScale: plain rows multiplied by 1 / l_row, l_row = sum_t 2^(c_t - c_row) l_t.
// Granularity (log2 units) of the key-tile exponents c_t: a power of two, so
// the rounding is exact; 32 keeps the numerators at the row maximum within
// (2^-32, 1], far above bf16's smallest normal (2^-126).
constexpr float kExpGrain = 32.f;

enum EpiMode : int { kEpiPlain = 0, kEpiResample = 1, kEpiStoreF32 = 2, kEpiExpBf16 = 3, kEpiRowScale = 4 };

// 2^e for an integer-valued e <= 0, exactly (0 below the normal range).
__device__ __forceinline__ float pow2_nonpos(float e) {
  return e <= -127.f ? 0.f : __int_as_float((127 + static_cast<int>(e)) << 23);
}

// max_t c_t over a row's key-tile statistics (four loads in flight).
__device__ __forceinline__ float row_max_c(const float2* st, int tiles) {
  float m[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) m[i] = __int_as_float(0xff800000u);  // -inf
  int t = 0;
  for (; t + 4 <= tiles; t += 4) {
#pragma unroll
    for (int i = 0; i < 4; ++i) m[i] = fmaxf(m[i], st[t + i].x);
  }
  for (; t < tiles; ++t) m[0] = fmaxf(m[0], st[t].x);
  return fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
}

// c_row and l_row of one row from its key-tile statistics.
__device__ __forceinline__ void row_stats(const GemmArgs& a, int batch, int m, float& c_row, float& l_row) {
  const float2* st = a.stats + (static_cast<long long>(batch) * a.m_total + m) * a.stat_tiles;
  c_row = row_max_c(st, a.stat_tiles);
  l_row = 0.f;
  for (int t = 0; t < a.stat_tiles; ++t) {
    const float2 v = st[t];
    l_row += v.y * pow2_nonpos(v.x - c_row);
  }
}

template <int EPI>
__device__ __forceinline__ long long epi_row_offset(const GemmArgs& a, int batch, int m) {
  if (EPI == kEpiResample) {
    const int j = m % a.img_w;
    const int r = m / a.img_w;
    const int i = r % a.img_h;
    const long long f = r / a.img_h;
    const int q = batch & 1, p = (batch >> 1) & 1, s = batch >> 2;
    const long long fo = a.epi_tscale == 2 ? 2 * f + s : f;
    return ((fo * (2 * a.img_h) + 2 * i + p) * (2LL * a.img_w) + 2 * j + q) * a.out_ld;
  }
  return static_cast<long long>(batch) * a.out_batch + static_cast<long long>(m) * a.out_ld;
}

__device__ __forceinline__ void add_bf16x16(float (&v)[16], const __nv_bfloat16* src) {
  const uint4* sp = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint4 bb = __ldg(sp + h);
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&bb);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __bfloat1622float2(b2[j]);
      v[8 * h + 2 * j] += f.x;
      v[8 * h + 2 * j + 1] += f.y;
    }
  }
}

// Stores accumulator columns n .. n+15 (r) of one row at element offset roff
// (skip row at soff): + bias, + shortcut, one rounding (or fp32 as is).
template <bool OUT_F32, bool HAS_BIAS, int EPI>
__device__ __forceinline__ void epi_store16(const GemmArgs& a, long long roff, long long soff, int n,
                                            const uint32_t (&r)[16]) {
  const bool full_chunk = n + 16 <= a.n_total;
  if constexpr (OUT_F32) {
    float* o = static_cast<float*>(a.out) + roff + n;
    if (full_chunk) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        reinterpret_cast<float4*>(o)[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                                      __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (n + j < a.n_total) o[j] = __uint_as_float(r[j]);
    }
  } else {
  float v[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) + roff + n;
  if (full_chunk) {
    if (HAS_BIAS) add_bf16x16(v, a.bias + n);
    if (EPI == kEpiResample) {
      if (a.vec32) {
        uint32_t s8[8];
        ld_global_nc_v8(a.skip + soff + n, s8);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&s8[j]));
          v[2 * j] += f.x;
          v[2 * j + 1] += f.y;
        }
      } else {
        add_bf16x16(v, a.skip + soff + n);
      }
    }
    uint4 pk[2];
    __nv_bfloat162* p2 = reinterpret_cast<__nv_bfloat162*>(pk);
#pragma unroll
    for (int j = 0; j < 8; ++j) p2[j] = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
    // one 32-byte store per row piece where aligned: half as many, whole-sector
    // L2 writes from a warp whose 32 lanes write 32 different rows
    if (a.vec32) {
      st_global_v8(o, pk);
    } else {
      reinterpret_cast<uint4*>(o)[0] = pk[0];
      reinterpret_cast<uint4*>(o)[1] = pk[1];
    }
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (n + j >= a.n_total) continue;
      float t = v[j];
      if (HAS_BIAS) t += __bfloat162float(a.bias[n + j]);
      if (EPI == kEpiResample) t += __bfloat162float(a.skip[soff + n + j]);
      o[j] = __float2bfloat16_rn(t);
    }
  }
  }
}

template <int BN, int AMODE, bool B_MN, bool OUT_F32, bool HAS_BIAS, int EPI = kEpiPlain>
__global__ void __launch_bounds__(kGemmThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ GemmArgs args) {
  using S = GemmShape<BN>;
  constexpr int STAGES = S::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * S::kABytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * S::kBBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&tfull[i]), 1);
      mbar_init(smem_u32(&tempty[i]), 128);
    }
    mbar_init(smem_u32(done), 1);
    fence_mbar_init();
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), S::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // set up: let the next kernel on the stream be scheduled, then wait for the
  // previous one before the first global access
  pdl_launch_dependents();
  pdl_wait();
  const uint64_t tlim = args.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      // number of loads armed per stage, to drain in-flight copies on abort
      for (int tile = blockIdx.x; ok && tile < args.num_tiles; tile += gridDim.x) {
        int batch, mt, nt;
        gemm_decode_tile(args, tile, batch, mt, nt);
        const int m0 = mt * kBlockM;
        const int n0 = nt * BN;
        int cw = 0, ch = 0, cd = 0, cn = 0;
        if (AMODE == kAIm2col) {
          int q = m0;
          cw = q % args.img_w;
          q /= args.img_w;
          ch = q % args.img_h;
          q /= args.img_h;
          cd = q % args.img_d;
          cn = q / args.img_d;
          cw += args.lo_w;
          ch += args.lo_h;
          cd += args.lo_d;
        }
        for (int tap = 0; ok && tap < args.taps; ++tap) {
          const int off = (AMODE == kAIm2col) ? args.tap_off[batch * args.taps + tap] : 0;
          const int brow = batch * args.b_rows_per_batch + tap * args.b_rows_per_tap + n0;
          for (int kb = 0; kb < args.kb_per_tap; ++kb) {
            if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, args.err, tlim)) {
              ok = false;
              break;
            }
            const uint32_t fb = smem_u32(&full[stage]);
            mbar_arrive_expect_tx(fb, S::kStageBytes);
            const uint32_t dA = smem_u32(sA + stage * S::kABytes);
            const uint32_t dB = smem_u32(sB + stage * S::kBBytes);
            if (AMODE == kAIm2col) {
              tma_load_im2col_5d(dA, &tmA, fb, kb * kBlockK, cw, ch, cd, cn, uint16_t(off & 0xff),
                                 uint16_t((off >> 8) & 0xff), uint16_t((off >> 16) & 0xff));
              tma_load_2d(dB, &tmB, fb, kb * kBlockK, brow);
            } else {
              tma_load_3d(dA, &tmA, fb, kb * kBlockK, m0, batch);
              if (B_MN) {
#pragma unroll
                for (int j = 0; j < BN / 64; ++j) tma_load_3d(dB + j * 8192, &tmB, fb, n0 + 64 * j, kb * kBlockK, batch);
              } else {
                tma_load_3d(dB, &tmB, fb, kb * kBlockK, n0, batch);
              }
            }
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (!ok) {
        // Let every copy already issued land before the CTA can exit: the
        // last armed phase of each stage is the only one that may be open.
        // Copies land within microseconds; 200 ms per stage is ample.
        for (int s = 0; s < STAGES; ++s) {
          (void)mbar_wait(smem_u32(&full[s]), (s < stage) ? phase : (phase ^ 1u), args.err, 200000000ull);
        }
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer --
    // The whole warp runs the loop (waits and descriptors stay warp-uniform);
    // the elected lane issues the MMAs and the commits that track them.
    {
      constexpr uint32_t idesc = idesc_bf16_f32(kBlockM, BN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      const int kblocks = args.taps * args.kb_per_tap;
      // 8-row groups are 1024 bytes apart; MN-major 64-column blocks 8192 bytes
      const uint64_t a_desc0 = sdesc_sw128(smem_u32(sA), 16, 1024);
      const uint64_t b_desc0 = B_MN ? sdesc_sw128(smem_u32(sB), 8192, 1024) : sdesc_sw128(smem_u32(sB), 16, 1024);
      for (int tile = blockIdx.x; ok && tile < args.num_tiles; tile += gridDim.x) {
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&tempty[acc]), acc_phase ^ 1u, args.err, tlim))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * S::kAccCols;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&full[stage]), phase, args.err, tlim))) {
            ok = false;
            break;
          }
          tc_fence_after();
          // stage and K offsets only move the descriptors' start-address field
          // (16-byte units): K-major, the next 16 elements are 32 bytes on
          // inside the 128-byte swizzle row; MN-major B (values), 16 keys are
          // two 8-row groups of 128 bytes = 2048 bytes on.
          const uint64_t ad = a_desc0 + static_cast<uint64_t>(stage) * (S::kABytes >> 4);
          const uint64_t bd = b_desc0 + static_cast<uint64_t>(stage) * (S::kBBytes >> 4);
          if (elect_one()) {
#pragma unroll
            for (int k = 0; k < kBlockK / kUmmaK; ++k)
              mma_bf16(d_tmem, ad + 2 * k, bd + (B_MN ? 128 : 2) * k, idesc, (kb | k) != 0 ? 1u : 0u);
            mma_commit(smem_u32(&empty[stage]));
          }
          __syncwarp();
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (elect_one()) mma_commit(smem_u32(&tfull[acc]));
        __syncwarp();
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // No MMA may still be running when TMEM is released.
      if (elect_one()) mma_commit(smem_u32(done));
      __syncwarp();
      (void)mbar_wait(smem_u32(done), 0, args.err, tlim);
    }
  } else {
    // ---------------------------------------------------------- epilogue --
    const int quarter = warp & 3;  // TMEM lanes this warp may read
    const int row = quarter * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < args.num_tiles; tile += gridDim.x) {
      int batch, mt, nt;
      gemm_decode_tile(args, tile, batch, mt, nt);
      // warp-uniform: the lanes leave together (they share .sync.aligned ops)
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&tfull[acc]), acc_phase, args.err, tlim))) break;
      tc_fence_after();
      const int m = mt * kBlockM + row;
      const int n0 = nt * BN;
      const bool row_ok = m < args.m_total;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * S::kAccCols;
      const long long roff = row_ok ? epi_row_offset<EPI>(args, batch, m) : 0;
      const long long soff = static_cast<long long>(m) * args.out_ld;
#pragma unroll 1
      for (int c = 0; c < BN; c += 16) {
        uint32_t r[16];
        __syncwarp();
        tmem_ld16(tbase + c, r);
        tmem_wait16(r);
        const int n = n0 + c;
        if (row_ok && n < args.n_total) epi_store16<OUT_F32, HAS_BIAS, EPI>(args, roff, soff, n, r);
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&tempty[acc]));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, S::kTmemCols);
  }
}

}  // namespace cc
