// The same implicit GEMM on CTA pairs: one tcgen05.mma.cta_group::2 computes
// a 256 x BN tile across two SMs. CTA rank r of the pair streams its own A
// tile (rows 128r .. 128r+127 of the pair tile) and its half of B (BN/2 rows)
// into its own shared memory; the MMAs that the even CTA's MMA warp issues
// (from one elected lane) read both CTAs' operands and write each CTA's 128
// accumulator rows into that CTA's TMEM. Per k-block each SM now loads 16 KB of A and 16 KB of B for a 128 x BN
// share of the tile (the single-CTA kernel loads 16 KB + 32 KB), which lowers
// both the L2 traffic and the shared-memory reads per MMA.
//
// Synchronisation across the pair: both producers complete their copies on
// the even CTA's `full` barrier (the even producer alone declares the bytes
// of both); MMA completion is multicast to the `empty` / `tfull` barriers of
// both CTAs; both epilogues arrive on the even CTA's `tempty`. Every wait is
// bounded, and a cluster barrier at the end keeps each CTA's shared memory
// alive until its peer is done with it.
#pragma once

#include "cc_gemm.cuh"

namespace cc {

template <int BN, int STAGING = 0>  // STAGING: bytes of output staging (TMA-store epilogue)
struct PairShape {
  static constexpr int kHalfN = BN / 2;
  static constexpr int kABytes = kBlockM * kBlockK * 2;
  static constexpr int kBBytes = kHalfN * kBlockK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;  // per CTA
  static constexpr int kStagesFit = (232448 - 1024 - 256 - STAGING) / kStageBytes;
  static constexpr int kStages = kStagesFit > 8 ? 8 : kStagesFit;
  static constexpr uint32_t kAccCols = BN <= 128 ? 128 : 256;
  static constexpr uint32_t kTmemCols = 2 * kAccCols;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + STAGING + 256;
  static_assert(BN % 128 == 0 && BN <= 256, "pair tiles split B into halves of whole 64-column blocks");
  static_assert(kBBytes % 1024 == 0, "B stage must be a whole number of 1024-byte swizzle atoms");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// tile -> (batch, pair row tile, column tile); the CTA of rank r takes row
// tile 2 * mp + r. False when the host-made row-tile order maps the tile
// outside the pair row tiles: every role then skips the tile, and the
// producers record DEVERR_BOUNDS (CC_ERR_DEVICE at the next device check).
__device__ __forceinline__ bool pair_decode_tile(const GemmArgs& a, int tile, int& batch, int& mp, int& nt) {
  const int mpt = (a.m_tiles + 1) / 2;
  nt = tile % a.n_tiles;
  const int r = tile / a.n_tiles;
  if (a.batch_outer) {
    mp = r % mpt;
    batch = r / mpt;
  } else {
    batch = r % a.batches;
    mp = r / a.batches;
  }
  if (a.mp_perm_n > 0) {
    if (mp >= a.mp_perm_n) return false;
    mp = a.mp_perm[mp];
  }
  return mp < mpt;
}

// Taps are ordered by their temporal offset. With zero frames before frame 0
// (lo_d < 0), a tap whose input frame t + od + lo_d is negative for every row
// of the pair tile multiplies only the causal zero padding: its exact-zero
// products are skipped, and the tile's k-loop starts at the first tap that
// reads a real frame for some row. The last tap (od = -lo_d) always does.
template <int AMODE>
__device__ __forceinline__ int tile_first_tap(const GemmArgs& a, int batch, int mp) {
  if (AMODE != kAIm2col || a.lo_d >= 0) return 0;
  // 32-bit arithmetic (m_total < 2^31 - 1024): the MMA warp runs this
  // between two tiles, where 64-bit divisions showed up as idle tensor cycles
  const unsigned plane = static_cast<unsigned>(a.img_h) * a.img_w;
  const unsigned per_image = plane * a.img_d;
  const unsigned m0 = static_cast<unsigned>(mp) * 2 * kBlockM;
  const unsigned m1 = min(m0 + 2 * kBlockM, static_cast<unsigned>(a.m_total)) - 1;
  // the latest frame any row of the tile lies in (a tile across an image
  // boundary holds the previous image's last frame)
  const int t_max = m0 / per_image != m1 / per_image ? a.img_d - 1 : static_cast<int>((m1 / plane) % a.img_d);
  int tap = 0;
  while (tap < a.taps - 1 && t_max + ((a.tap_off[batch * a.taps + tap] >> 16) & 0xff) + a.lo_d < 0) ++tap;
  return tap;
}

// The k-th tile of a CTA pair: waves of npairs consecutive tiles, walked
// forward in even waves and backward in odd ones, so a pair that gets a
// short tile (leading zero taps skipped) early gets a long one next. -1 when
// the pair has no tile in that (last, partial) wave; num_tiles when done.
__device__ __forceinline__ int pair_tile(const GemmArgs& a, int pair, int npairs, int k) {
  const int base = k * npairs;
  if (base >= a.num_tiles) return a.num_tiles;
  const int tile = (k & 1) ? base + npairs - 1 - pair : base + pair;
  return tile < a.num_tiles ? tile : -1;
}

constexpr int kStoreChunk = 32;  // fp32 columns per staged TMA store (64 bf16 columns in the exp-tile epilogue)
constexpr int kStoreBufBytes = kBlockM * kStoreChunk * 4;  // 16 KB: 128 rows x 128 bytes

template <int EPI>
constexpr int pair_staging_bytes() {
  return (EPI == kEpiStoreF32 || EPI == kEpiExpBf16 || EPI == kEpiRowScale) ? 2 * kStoreBufBytes : 0;
}

template <int BN, int AMODE, bool B_MN, bool OUT_F32, bool HAS_BIAS, int EPI = kEpiPlain>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const __grid_constant__ GemmArgs args) {
  using S = PairShape<BN, pair_staging_bytes<EPI>()>;
  constexpr int STAGES = S::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * S::kABytes;
  uint8_t* sStage = sB + STAGES * S::kBBytes;  // output staging (TMA-store epilogue only)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStage + pair_staging_bytes<EPI>());
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&tfull[i]), 1);
      mbar_init(smem_u32(&tempty[i]), 2 * 4);  // one arrival per epilogue warp of each CTA
    }
    mbar_init(smem_u32(done), 1);
    fence_mbar_init();
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
    if (pair_staging_bytes<EPI>() > 0) tma_prefetch_map(&tmC);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), S::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers exist before any cross-CTA signal
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
      for (int k = 0, tile; ok && (tile = pair_tile(args, pair, npairs, k)) < args.num_tiles; ++k) {
        if (tile < 0) continue;
        int batch, mp, nt;
        if (!pair_decode_tile(args, tile, batch, mp, nt)) {
          atomicOr(args.err, DEVERR_BOUNDS);
          continue;
        }
        const int m0 = (2 * mp + static_cast<int>(rank)) * kBlockM;
        const int nb0 = nt * BN + static_cast<int>(rank) * S::kHalfN;  // this CTA's half of the columns
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
        for (int tap = tile_first_tap<AMODE>(args, batch, mp); ok && tap < args.taps; ++tap) {
          const int off = (AMODE == kAIm2col) ? args.tap_off[batch * args.taps + tap] : 0;
          const int brow = batch * args.b_rows_per_batch + tap * args.b_rows_per_tap + nb0;
          for (int kb = 0; kb < args.kb_per_tap; ++kb) {
            if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, args.err, tlim)) {
              ok = false;
              break;
            }
            const uint32_t fb_local = smem_u32(&full[stage]);
            const uint32_t fb = mapa_shared(fb_local, 0);
            if (leader) mbar_arrive_expect_tx(fb_local, 2 * S::kStageBytes);
            const uint32_t dA = smem_u32(sA + stage * S::kABytes);
            const uint32_t dB = smem_u32(sB + stage * S::kBBytes);
            if (AMODE == kAIm2col) {
              tma_load_im2col_5d_pair(dA, &tmA, fb, kb * kBlockK, cw, ch, cd, cn, uint16_t(off & 0xff),
                                      uint16_t((off >> 8) & 0xff), uint16_t((off >> 16) & 0xff));
              tma_load_2d_pair(dB, &tmB, fb, kb * kBlockK, brow);
            } else {
              tma_load_3d_pair(dA, &tmA, fb, kb * kBlockK, m0, batch);
              if (B_MN) {
#pragma unroll
                for (int j = 0; j < S::kHalfN / 64; ++j)
                  tma_load_3d_pair(dB + j * 8192, &tmB, fb, nb0 + 64 * j, kb * kBlockK, batch);
              } else {
                tma_load_3d_pair(dB, &tmB, fb, kb * kBlockK, nb0, batch);
              }
            }
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      if (!ok && leader) {
        // copies of both CTAs complete on the even CTA's barriers; let the
        // armed ones land (200 ms each at most) before the pair winds down
        for (int s = 0; s < STAGES; ++s)
          (void)mbar_wait(smem_u32(&full[s]), (s < stage) ? phase : (phase ^ 1u), args.err, 200000000ull);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------- MMA issuer (even CTA only) --
    // The whole warp runs the loop (waits and descriptors stay warp-uniform);
    // the elected lane issues the MMAs and the commits that track them.
    if (leader) {
      constexpr uint32_t idesc = idesc_bf16_f32(2 * kBlockM, BN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      const int kblocks = args.taps * args.kb_per_tap;
      // 8-row groups are 1024 bytes apart; MN-major 64-column blocks 8192 bytes
      const uint64_t a_desc0 = sdesc_sw128(smem_u32(sA), 16, 1024);
      const uint64_t b_desc0 = B_MN ? sdesc_sw128(smem_u32(sB), 8192, 1024) : sdesc_sw128(smem_u32(sB), 16, 1024);
      for (int k = 0, tile; ok && (tile = pair_tile(args, pair, npairs, k)) < args.num_tiles; ++k) {
        if (tile < 0) continue;
        int batch, mp, nt;
        if (!pair_decode_tile(args, tile, batch, mp, nt)) continue;
        const int kb0 = tile_first_tap<AMODE>(args, batch, mp) * args.kb_per_tap;
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&tempty[acc]), acc_phase ^ 1u, args.err, tlim))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * S::kAccCols;
        for (int kb = kb0; kb < kblocks; ++kb) {
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
              mma_bf16_pair(d_tmem, ad + 2 * k, bd + (B_MN ? 128 : 2) * k, idesc, (kb != kb0 || k != 0) ? 1u : 0u);
            mma_commit_pair_both(smem_u32(&empty[stage]));
          }
          __syncwarp();
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (elect_one()) mma_commit_pair_both(smem_u32(&tfull[acc]));
        __syncwarp();
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (elect_one()) mma_commit_pair_both(smem_u32(done));
      __syncwarp();
      (void)mbar_wait(smem_u32(done), 0, args.err, tlim);
    }
  } else if constexpr (EPI == kEpiExpBf16) {
    // ------------- epilogue: softmax numerators per key tile (both CTAs) --
    // Two passes over the row's BN accumulator columns: the max over the
    // valid keys, then e = exp2(exp_k * s - c_t) packed to bf16 in 64-column
    // chunks through the swizzled staging buffers and TMA stores (as in
    // StoreF32), with l_t summed from the fp32 e.
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const bool issuer = (warp == 2 && lane == 0);
    const float kx = args.exp_k;
    int acc = 0;
    uint32_t acc_phase = 0;
    int chunk = 0;
    for (int k = 0, tile; (tile = pair_tile(args, pair, npairs, k)) < args.num_tiles; ++k) {
      if (tile < 0) continue;
      int batch, mp, nt;
      if (!pair_decode_tile(args, tile, batch, mp, nt)) continue;
      if (!named_barrier_and(1, 128, mbar_wait(smem_u32(&tfull[acc]), acc_phase, args.err, tlim))) break;
      tc_fence_after();
      const int m0 = (2 * mp + static_cast<int>(rank)) * kBlockM;
      const int n0 = nt * BN;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * S::kAccCols;
      // chunks holding at least one valid key (the same for every thread)
      const int valid = args.n_total - n0;
      const int c32_end = valid >= BN ? BN / 32 : (valid + 31) / 32;
      const int c64_end = valid >= BN ? BN / 64 : (valid + 63) / 64;
      float m4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) m4[i] = __int_as_float(0xff800000u);
#pragma unroll 1
      for (int c = 0; c < c32_end; ++c) {
        uint32_t r[32];
        tmem_ld32_wait(tbase + c * 32, r);
        const int nb = n0 + c * 32;
        if (nb + 32 <= args.n_total) {
#pragma unroll
          for (int j = 0; j < 32; ++j) m4[j & 3] = fmaxf(m4[j & 3], __uint_as_float(r[j]));
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (nb + j < args.n_total) m4[j & 3] = fmaxf(m4[j & 3], __uint_as_float(r[j]));
        }
      }
      // c_t: the tile's scaled max rounded up to a multiple of kExpGrain, so
      // that the tiles of one row nearly always share it and the rescale pass
      // has little to move (every e stays in (2^-kExpGrain, 1] at the max
      // and keeps bf16's relative precision far above the normal range)
      const float ct =
          ceilf(fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * kx * (1.f / kExpGrain)) * kExpGrain;
      float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
      for (int c = 0; c < c64_end; ++c, ++chunk) {
        uint32_t r0[32], r1[32];
        tmem_ld32_wait(tbase + c * 64, r0);
        tmem_ld32_wait(tbase + c * 64 + 32, r1);
        if (c == c64_end - 1) {  // accumulator fully read: release it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));
        }
        const int nb = n0 + c * 64;
        const bool full_chunk = nb + 64 <= args.n_total;
        uint32_t pk[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const uint32_t s0 = j < 16 ? r0[2 * j] : r1[2 * j - 32];
          const uint32_t s1 = j < 16 ? r0[2 * j + 1] : r1[2 * j - 31];
          float e0 = ex2_approx(fmaf(__uint_as_float(s0), kx, -ct));
          float e1 = ex2_approx(fmaf(__uint_as_float(s1), kx, -ct));
          if (!full_chunk) {
            e0 = nb + 2 * j < args.n_total ? e0 : 0.f;
            e1 = nb + 2 * j + 1 < args.n_total ? e1 : 0.f;
          }
          l4[j & 3] += e0 + e1;
          __nv_bfloat162 b = __floats2bfloat162_rn(e0, e1);
          pk[j] = *reinterpret_cast<uint32_t*>(&b);
        }
        if (args.out == nullptr) {
          // statistics only: E is not written
        } else if (args.vec32) {
          // rows start on 32-byte boundaries: each 16-key piece leaves the
          // registers as one whole 32-byte sector, and shared memory -- whose
          // bandwidth the main loop's operand traffic already uses up -- is
          // not touched
          const int m = m0 + row;
          if (m < args.m_total) {
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(args.out) + batch * args.out_batch +
                                 static_cast<long long>(m) * args.out_ld + nb;
#pragma unroll
            for (int p = 0; p < 4; ++p) {
              if (nb + 16 * p + 16 <= args.n_total) {
                const uint4 v[2] = {make_uint4(pk[8 * p], pk[8 * p + 1], pk[8 * p + 2], pk[8 * p + 3]),
                                    make_uint4(pk[8 * p + 4], pk[8 * p + 5], pk[8 * p + 6], pk[8 * p + 7])};
                st_global_v8(dst + 16 * p, v);
              } else {
                uint16_t* d16 = reinterpret_cast<uint16_t*>(dst);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                  const int e = 16 * p + j;
                  if (nb + e < args.n_total) d16[e] = static_cast<uint16_t>(pk[e >> 1] >> ((e & 1) * 16));
                }
              }
            }
          }
        } else {
          uint8_t* buf = sStage + (chunk & 1) * kStoreBufBytes;
          if (issuer) bulk_wait_read_1();  // the store two chunks back has read this buffer
          named_barrier_sync(1, 128);
          uint8_t* rowp = buf + row * 128;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<uint4*>(rowp + ((j ^ (row & 7)) << 4)) =
                make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
          fence_proxy_async_smem();
          named_barrier_sync(1, 128);
          if (issuer) {
            tma_store_3d(&tmC, smem_u32(buf), nb, m0, batch);
            bulk_commit();
          }
        }
      }
      const float l = (l4[0] + l4[1]) + (l4[2] + l4[3]);
      const int m = m0 + row;
      if (m < args.m_total)
        args.stats[(static_cast<long long>(batch) * args.m_total + m) * args.stat_tiles + nt] = make_float2(ct, l);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (issuer) bulk_wait_all();
  } else if constexpr (EPI == kEpiRowScale) {
    // -------- epilogue: row-scaled bf16 through staged TMA stores (both CTAs) --
    // Each row's BN columns times 1 / l_row, packed to bf16 in 64-column
    // chunks through the two swizzled staging buffers and one TMA tensor
    // store per chunk (clipped at the last row), as in the numerators'
    // epilogue: whole 128-byte row pieces leave the SM instead of 32-byte
    // pieces of 128 rows, which held up the operand loads.
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const bool issuer = (warp == 2 && lane == 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    int chunk = 0;
    for (int k = 0, tile; (tile = pair_tile(args, pair, npairs, k)) < args.num_tiles; ++k) {
      if (tile < 0) continue;
      int batch, mp, nt;
      if (!pair_decode_tile(args, tile, batch, mp, nt)) continue;
      if (!named_barrier_and(1, 128, mbar_wait(smem_u32(&tfull[acc]), acc_phase, args.err, tlim))) break;
      tc_fence_after();
      const int m0 = (2 * mp + static_cast<int>(rank)) * kBlockM;
      const int n0 = nt * BN;
      const int m = m0 + row;
      float rscale = 0.f;  // rows past the end are staged but clipped by the store
      if (m < args.m_total) {
        float c_row, l_row;
        row_stats(args, batch, m, c_row, l_row);
        rscale = 1.f / l_row;
      }
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * S::kAccCols;
      const int valid = args.n_total - n0;
      const int c64_end = valid >= BN ? BN / 64 : (valid + 63) / 64;
#pragma unroll 1
      for (int c = 0; c < c64_end; ++c, ++chunk) {
        uint32_t r0[32], r1[32];
        tmem_ld32_wait(tbase + c * 64, r0);
        tmem_ld32_wait(tbase + c * 64 + 32, r1);
        if (c == c64_end - 1) {  // accumulator fully read: release it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));
        }
        uint32_t pk[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const uint32_t s0 = j < 16 ? r0[2 * j] : r1[2 * j - 32];
          const uint32_t s1 = j < 16 ? r0[2 * j + 1] : r1[2 * j - 31];
          __nv_bfloat162 b = __floats2bfloat162_rn(__uint_as_float(s0) * rscale, __uint_as_float(s1) * rscale);
          pk[j] = *reinterpret_cast<uint32_t*>(&b);
        }
        uint8_t* buf = sStage + (chunk & 1) * kStoreBufBytes;
        if (issuer) bulk_wait_read_1();  // the store two chunks back has read this buffer
        named_barrier_sync(1, 128);
        uint8_t* rowp = buf + row * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<uint4*>(rowp + ((j ^ (row & 7)) << 4)) =
              make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
        fence_proxy_async_smem();
        named_barrier_sync(1, 128);
        if (issuer) {
          tma_store_3d(&tmC, smem_u32(buf), n0 + c * 64, m0, batch);
          bulk_commit();
        }
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (issuer) bulk_wait_all();
  } else if constexpr (EPI == kEpiStoreF32) {
    // ------------------------------ epilogue: staged TMA stores (both CTAs) --
    // Each 32-column chunk of the 128 x BN fp32 tile goes to one of two
    // swizzled 16 KB shared buffers (row r's 16-byte piece j at j ^ (r & 7)),
    // then one thread stores it with a TMA tensor store (clipped at the
    // tensor's edge), so global writes are whole 128-byte rows.
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const bool issuer = (warp == 2 && lane == 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    int chunk = 0;
    for (int k = 0, tile; (tile = pair_tile(args, pair, npairs, k)) < args.num_tiles; ++k) {
      if (tile < 0) continue;
      int batch, mp, nt;
      if (!pair_decode_tile(args, tile, batch, mp, nt)) continue;
      // uniform over the four epilogue warps (shared named barriers below)
      if (!named_barrier_and(1, 128, mbar_wait(smem_u32(&tfull[acc]), acc_phase, args.err, tlim))) break;
      tc_fence_after();
      const int m0 = (2 * mp + static_cast<int>(rank)) * kBlockM;
      const int n0 = nt * BN;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * S::kAccCols;
#pragma unroll 1
      for (int c = 0; c < BN / kStoreChunk; ++c, ++chunk) {
        uint32_t r[32];
        tmem_ld32_wait(tbase + c * kStoreChunk, r);
        if (c == BN / kStoreChunk - 1) {  // accumulator fully read: release it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));
        }
        uint8_t* buf = sStage + (chunk & 1) * kStoreBufBytes;
        if (issuer) bulk_wait_read_1();  // the store two chunks back has read this buffer
        named_barrier_sync(1, 128);
        uint8_t* rowp = buf + row * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<float4*>(rowp + ((j ^ (row & 7)) << 4)) =
              make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]), __uint_as_float(r[4 * j + 2]),
                          __uint_as_float(r[4 * j + 3]));
        fence_proxy_async_smem();
        named_barrier_sync(1, 128);
        if (issuer) {
          tma_store_3d(&tmC, smem_u32(buf), n0 + c * kStoreChunk, m0, batch);
          bulk_commit();
        }
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (issuer) bulk_wait_all();
  } else {
    // --------------------------------------------- epilogue (both CTAs) --
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int k = 0, tile; (tile = pair_tile(args, pair, npairs, k)) < args.num_tiles; ++k) {
      if (tile < 0) continue;
      int batch, mp, nt;
      if (!pair_decode_tile(args, tile, batch, mp, nt)) continue;
      // warp-uniform: the lanes leave together (they share .sync.aligned ops)
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&tfull[acc]), acc_phase, args.err, tlim))) break;
      tc_fence_after();
      const int m = (2 * mp + static_cast<int>(rank)) * kBlockM + row;
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
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer no longer reads this CTA's shared memory or signals its barriers
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, S::kTmemCols);
  }
}

}  // namespace cc
