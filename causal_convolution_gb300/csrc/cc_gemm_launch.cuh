// Host-side launch of the tcgen05 implicit GEMM (one persistent CTA per SM).
#pragma once

#include <algorithm>

#include "cc_gemm.cuh"
#include "cc_gemm_pair.cuh"
#include "cc_host.h"

namespace cc {

// Whether the direct-store epilogue may use 32-byte accesses: every bf16 row
// piece of 16 columns (output and shortcut) then starts on a 32-byte boundary.
inline int epi_vec32(const GemmArgs& a, bool out_f32) {
  const uintptr_t bases = reinterpret_cast<uintptr_t>(a.out) | reinterpret_cast<uintptr_t>(a.skip);
  return !out_f32 && (bases & 31u) == 0 && a.out_ld % 16 == 0 && a.out_batch % 16 == 0;
}

template <int BN, int AMODE, bool B_MN, bool OUT_F32, bool HAS_BIAS, int EPI = kEpiPlain>
cc_status launch_tc_gemm(const CUtensorMap& ta, const CUtensorMap& tb, GemmArgs& args, const DeviceInfo& di,
                         cudaStream_t stream, const char* what) {
  using S = GemmShape<BN>;
  if ((long long)args.m_tiles * args.n_tiles * args.batches > 0x7fffffffLL)
    return fail(CC_ERR_UNSUPPORTED, "%s: too many output tiles", what);
  if (args.num_tiles <= 0) return CC_OK;
  auto kern = tc_gemm_kernel<BN, AMODE, B_MN, OUT_F32, HAS_BIAS, EPI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
  if (e != cudaSuccess) return fail(CC_ERR_CUDA, "%s: shared-memory attribute: %s", what, cudaGetErrorString(e));
  args.err = di.err_word;
  args.timeout_ns = kWaitLimitNs;
  args.vec32 = epi_vec32(args, OUT_F32);
  const int grid = std::min(args.num_tiles, di.sm_count);
  e = launch_pdl(kern, dim3(grid), dim3(kGemmThreads), S::kSmemBytes, stream, ta, tb, args);
  if (e != cudaSuccess) return fail(CC_ERR_CUDA, "%s: launch: %s", what, cudaGetErrorString(e));
  return launch_status(what);
}

// Pair kernel: args.m_tiles counts 128-row tiles; args.num_tiles is
// overwritten with the number of 256-row pair tiles.
template <int BN, int AMODE, bool B_MN, bool OUT_F32, bool HAS_BIAS, int EPI = kEpiPlain>
cc_status launch_tc_gemm_pair(const CUtensorMap& ta, const CUtensorMap& tb, GemmArgs& args, const DeviceInfo& di,
                              cudaStream_t stream, const char* what, const CUtensorMap* tc = nullptr) {
  using S = PairShape<BN, pair_staging_bytes<EPI>()>;
  if (pair_staging_bytes<EPI>() > 0 && !tc)
    return fail(CC_ERR_INVALID, "%s: output tensor map missing", what);
  const long long tiles = ((args.m_tiles + 1LL) / 2) * args.n_tiles * args.batches;
  if (tiles > 0x7fffffffLL) return fail(CC_ERR_UNSUPPORTED, "%s: too many output tiles", what);
  args.num_tiles = static_cast<int>(tiles);
  if (args.num_tiles <= 0) return CC_OK;
  auto kern = tc_gemm_pair_kernel<BN, AMODE, B_MN, OUT_F32, HAS_BIAS, EPI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
  if (e != cudaSuccess) return fail(CC_ERR_CUDA, "%s: shared-memory attribute: %s", what, cudaGetErrorString(e));
  args.err = di.err_word;
  args.timeout_ns = kWaitLimitNs;
  args.vec32 = epi_vec32(args, OUT_F32);
  const int pairs = std::min(args.num_tiles, di.sm_count / 2);
  e = launch_pdl(kern, dim3(2 * pairs), dim3(kGemmThreads), S::kSmemBytes, stream, ta, tb, tc ? *tc : tb, args);
  if (e != cudaSuccess) return fail(CC_ERR_CUDA, "%s: launch: %s", what, cudaGetErrorString(e));
  return launch_status(what);
}

inline int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// Walking order of the 256-row pair tiles of an im2col convolution over
// [N, D, H, W] positions. With zero frames before frame 0 (lo_d < 0) the
// tiles whose rows lie in the first -lo_d frames skip their leading taps and
// are short: they go first, in plain order (the snake then evens out their
// cost across CTA pairs, as before). The full tiles follow, sorted by
// (image, position of the tile's first row inside its frame, tile): the
// tiles at one place of the plane, one per frame, follow each other, so a
// tile's earlier-frame taps find their rows in L2 instead of DRAM. Left as
// the identity (mp_perm_n = 0) for a single frame or more pair tiles than
// the table holds.
inline void set_frame_interleaved_order(GemmArgs& a) {
  a.mp_perm_n = 0;
  const long long mpt = (a.m_tiles + 1LL) / 2;
  const long long plane = static_cast<long long>(a.img_h) * a.img_w;
  const long long image = plane * a.img_d;
  constexpr long long kMax = sizeof(a.mp_perm) / sizeof(a.mp_perm[0]);
  if (a.img_d <= 1 || mpt <= 1 || mpt > kMax || plane <= 0) return;
  long long key[kMax];
  for (long long mp = 0; mp < mpt; ++mp) {
    const long long r0 = mp * 2 * kBlockM;
    const long long r1 = std::min(r0 + 2 * kBlockM, static_cast<long long>(a.m_total)) - 1;
    // the latest frame a row of the tile lies in (the tile_first_tap rule)
    const long long t_max = r0 / image != r1 / image ? a.img_d - 1 : (r1 % image) / plane;
    const bool short_tile = a.lo_d < 0 && t_max + a.lo_d < 0;
    const long long order = short_tile ? mp : mpt + (r0 / image) * image + (r0 % image) % plane;
    key[mp] = order * kMax + mp;
  }
  std::sort(key, key + mpt);
  for (long long i = 0; i < mpt; ++i) a.mp_perm[i] = static_cast<unsigned short>(key[i] % kMax);
  a.mp_perm_n = static_cast<int>(mpt);
}

}  // namespace cc
