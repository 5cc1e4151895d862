/*
 * cc_debug.h -- self-test entry points of libcc.so.
 *
 * These exercise building blocks of the kernels in isolation so that the
 * test suite can check them against the definitions. They are not part of
 * the decoder's path. Conventions as in cc.h (device pointers, 16-byte
 * alignment, asynchronous on `stream`, host-side argument checks).
 */
#ifndef CC_DEBUG_H_
#define CC_DEBUG_H_

#include "cc.h"

#ifdef __cplusplus
extern "C" {
#endif

/* One im2col TMA load exactly as the convolution kernels issue it, written
 * out un-swizzled: tile[p][c] for 128 pixels p and 64 channels c.
 * x: [N, D_in, H, W, C] bf16 with C % 64 == 0. The map's bounding box has
 * lower corner (lo_w, lo_h, lo_d) and upper corner (up_w, up_h, up_d) relative
 * to the far edge; the load starts at pixel (cw, ch, cd, cn) of the box, at
 * channel c0, with pixel offsets (ow, oh, od). tile: 128*64 elements. */
cc_status cc_debug_im2col_tile(const cc_bf16* x, cc_bf16* tile, int n, int d_in, int h, int w, int c, int lo_w,
                               int lo_h, int lo_d, int up_w, int up_h, int up_d, int c0, int cw, int ch, int cd,
                               int cn, int ow, int oh, int od, void* stream);

/* Launches one CTA that waits on an mbarrier nothing ever arrives at, with a
 * time limit of `limit_ns` (at most 1 s). The wait gives up, the kernel
 * returns normally and the device error word records a timeout, which the
 * next cc_check_device() reports as CC_ERR_TIMEOUT. Tests the failure path
 * without hanging or faulting the GPU. */
cc_status cc_debug_wait_timeout(int64_t limit_ns, void* stream);

/* cc_conv3d_causal (no bias, zero history) with entry `entry` of the CTA
 * pairs' walking order over the 256-row tiles replaced by a row tile that does
 * not exist. The kernel's own check of the order finds it: that tile is
 * skipped by every role (its 256 output rows are not written), the other
 * tiles are computed as usual, and the device error word records an index
 * failure, which the next cc_check_device() reports as CC_ERR_DEVICE. Needs a
 * shape whose conv walks an explicit order (two or more frames, 2 to 512
 * pair row tiles) and 0 <= entry < its pair row tiles; CC_ERR_INVALID
 * otherwise. Tests that failure path without any
 * out-of-range access. */
cc_status cc_debug_conv_bad_tile_order(const cc_bf16* x, const cc_bf16* wp, cc_bf16* y, int n, int d, int h, int w,
                                       int cin, int cout, int entry, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* CC_DEBUG_H_ */
