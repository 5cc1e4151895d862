// Host-side helpers shared by the translation units of the library: the
// thread-local error message, argument checks, tensor-map encoding through
// the driver entry points, and per-device facts (SM count, error word).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstddef>
#include <cstdint>
#include <initializer_list>
#include <utility>

#include "cc.h"

namespace cc {

// Records a printf-style message as the calling thread's last error and
// returns `st` so call sites can `return fail(CC_ERR_INVALID, "...")`.
cc_status fail(cc_status st, const char* fmt, ...);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A request whose output covers no position (a zero batch, frame, row,
// column or per-frame position count) has nothing to compute: it succeeds
// before any other check, launching nothing and reading no pointer. A
// negative count is invalid. Returns true when the caller is to return *st.
bool empty_request(const char* what, std::initializer_list<long long> counts, cc_status* st);

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel on the stream is still finishing (its CTAs take
// SMs as that kernel's CTAs exit), do its setup, and then block in
// griddepcontrol.wait until the previous kernel has completed and its writes
// are visible -- the same ordering as a plain launch, with the setup hidden.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Per-device facts, cached on first use.
struct DeviceInfo {
  int device;
  int sm_count;
  unsigned int* err_word;  // device address of the library's error word
};
cc_status device_info(DeviceInfo* out);

// Kernel launch wrapper: maps cudaGetLastError into a status.
cc_status launch_status(const char* what);

// Tensor maps (bf16 elements unless stated).
cc_status encode_im2col_5d(CUtensorMap* map, const void* base, int n, int d, int h, int w, int c, int lo_w, int lo_h,
                           int lo_d, int up_w, int up_h, int up_d, int pixels, int channels);
cc_status encode_tiled_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                          uint32_t box_inner, uint32_t box_outer);
cc_status encode_tiled_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t stride1,
                          uint64_t stride2, uint32_t box0, uint32_t box1);
// Rank-3 fp32 map with 128-byte swizzle, box {box0, box1, 1} (box0 * 4 <= 128).
cc_status encode_tiled_3d_f32_sw128(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                                    uint64_t stride1, uint64_t stride2, uint32_t box0, uint32_t box1);
// Rank-5 map with 128-byte swizzle, box {box0, box1, box2, 1, 1}; strides[i]
// is the byte stride of dimension i + 1.
cc_status encode_tiled_5d(CUtensorMap* map, const void* base, const uint64_t dims[5], const uint64_t strides[4],
                          uint32_t box0, uint32_t box1, uint32_t box2);
// Rank-4 map without swizzle (dense box in shared memory), box {b0, b1, b2, 1}.
cc_status encode_tiled_4d_dense(CUtensorMap* map, const void* base, const uint64_t dims[4], const uint64_t strides[3],
                                uint32_t box0, uint32_t box1, uint32_t box2);

// Upper bound on one mbarrier wait inside the library's kernels.
constexpr unsigned long long kWaitLimitNs = 4000000000ull;

}  // namespace cc
