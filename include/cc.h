/*
 * cc.h -- C ABI of the GB300 causal-convolution library (libcc.so).
 *
 * The bf16 causal 3-D convolution stack of the Wan2.2 (TI2V-5B style) video
 * VAE decoder: the causal 3x3x3 convolution, the nearest-x2 spatial
 * resampler (four pre-summed phase convolutions + one interleave pass), the
 * mid-block per-frame single-head attention and the output head (conv_out to
 * 12 channels, bias, clamp). All compute runs in the library's own sm_103a
 * kernels; nothing here falls back to the CPU.
 *
 * Conventions shared by every entry point
 *  - Pointers are DEVICE pointers owned by the caller. The library allocates
 *    no device memory: intermediates live in a caller-provided workspace
 *    whose size the matching *_workspace_bytes() function returns.
 *  - bf16 tensors are passed as raw 16-bit patterns (cc_bf16 = uint16_t).
 *  - Activations are channels-last: [N, D, H, W, C] contiguous, C fastest.
 *    Convolution weights keep the PyTorch Conv3d order [C_out, C_in, 3, 3, 3]
 *    until a *_prepare() call repacks them.
 *  - Every pointer must be 16-byte aligned.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream). Calls are
 *    asynchronous on it; the caller keeps every buffer alive until the work
 *    on the stream is done.
 *  - Arguments are checked on the host before any launch. A rejected call
 *    launches nothing and returns CC_ERR_INVALID or CC_ERR_UNSUPPORTED;
 *    cc_last_error() then describes the reason. No C++ exception crosses
 *    the ABI.
 *  - A request whose output covers no position (a count of images, frames,
 *    rows, columns or per-frame positions is 0) succeeds at once: it
 *    launches nothing and reads none of its pointers, which may be NULL.
 *    Negative counts are CC_ERR_INVALID; channel counts must be positive.
 *  - Kernels never trap. A pipeline wait that runs past its time limit makes
 *    the kernel wind down and set a device error word, which
 *    cc_check_device() reports as CC_ERR_TIMEOUT.
 *  - `hist` selects what precedes frame 0 in time: 0 = two zero frames (the
 *    causal zero padding), x then holds D frames; 2 = x holds two history
 *    frames in front of its D frames (D + 2 frames in total), so a chunked
 *    decode can carry the previous chunk's last two frames.
 *
 * Sources for the definitions (pages of the reference material):
 *  [ATTN] FastVideo wan22_vae_decode solution/attn.cu -- header comment and
 *         attn_forward: per-frame softmax(q k^T / sqrt(C)) v, no mask.
 *  [RES]  FastVideo wan22_vae_decode solution/resample.h -- header comment
 *         (four-phase decomposition, interleave pass) and the comment on
 *         resample_upsample (history frames, phase order 2*row_parity +
 *         col_parity).
 *  [HEAD] FastVideo wan22_vae_decode solution/head.cu -- header comment
 *         (conv_out folded into a 3x1x1 conv with 9x12 output channels, then
 *         a 3x3 stencil, bias and clamp) and head_stencil_kernel.
 *  [STACK] the stack's definition: causal 3x3x3 conv with two history frames,
 *         zeros before frame 0, spatial zero padding 1, fp32 accumulation.
 *  [HOST] no page: a transfer helper for the chunk-by-chunk decode loop.
 */
#ifndef CC_H_
#define CC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t cc_bf16;

typedef enum cc_status {
  CC_OK = 0,
  CC_ERR_INVALID = 1,     /* null/misaligned pointer, bad size or shape     */
  CC_ERR_UNSUPPORTED = 2, /* valid request outside what the kernels cover  */
  CC_ERR_CUDA = 3,        /* a CUDA runtime/driver call or launch failed    */
  CC_ERR_TIMEOUT = 4,     /* a kernel wait ran past its limit (see above)  */
  CC_ERR_DEVICE = 5       /* a kernel-side index check failed              */
} cc_status;

/* Message describing the calling thread's most recent failure ("" if none). */
const char* cc_last_error(void);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int cc_version(void);

/* Synchronises `stream`, then reads and clears the current device's error
 * word. Returns CC_OK, CC_ERR_TIMEOUT, CC_ERR_DEVICE or CC_ERR_CUDA. */
cc_status cc_check_device(void* stream);

/* ------------------------------------------------ causal 3x3x3 conv [STACK] */

/* Repacks w [C_out, C_in, 3, 3, 3] into wp [27][C_out][C_in] (tap-major,
 * tap = kt*9 + kh*3 + kw, each row K-major), the B operand of the implicit
 * GEMM. wp holds 27*C_out*C_in elements. */
cc_status cc_conv3d_prepare(const cc_bf16* w, cc_bf16* wp, int cout, int cin, void* stream);

/* y[n,t,h,w,co] = bias[co] + sum_{ci,kt,kh,kw} W[co,ci,kt,kh,kw]
 *                          * x~[n, t+kt-2, h+kh-1, w+kw-1, ci]
 * with x~ zero outside the plane and before frame 0 as `hist` says; fp32
 * accumulation, one rounding to bf16. x: [N, D+hist, H, W, C_in]; wp from
 * cc_conv3d_prepare; bias [C_out] or NULL; y: [N, D, H, W, C_out].
 * Needs C_in % 64 == 0 and C_out % 16 == 0. */
cc_status cc_conv3d_causal(const cc_bf16* x, const cc_bf16* wp, const cc_bf16* bias, cc_bf16* y, int n, int d,
                           int h, int w, int cin, int cout, int hist, void* stream);

/* ------------------------------------------------ spatial resampler [RES] */

/* Pre-sums the taps that nearest-x2 makes coincide. For output parity
 * (p, q) and phase tap (kt, a, b), rows {0} | {1,2} (p=0, a=0|1) or {0,1} | {2}
 * (p=1) and the same for columns are summed in fp32 and rounded once:
 * pw[(2p+q)][(kt*2+a)*2+b][co][ci]; 48*C_out*C_in elements. */
cc_status cc_resample_prepare(const cc_bf16* w, cc_bf16* pw, int cout, int cin, void* stream);

/* Bytes of workspace cc_resample_up2 needs: the four phase tensors. */
size_t cc_resample_workspace_bytes(int n, int d, int hl, int wl, int cout);

/* The four phase convolutions at low resolution (no bias):
 * phases[2p+q][n,t,i,j,co] = sum_{ci,kt,a,b} pw[2p+q][(kt*2+a)*2+b][co][ci]
 *                            * x~[n, t+kt-2, i+p-1+a, j+q-1+b, ci].
 * x: [N, D+hist, HL, WL, C_in]; phases: 4 x [N, D, HL, WL, C_out] back to back.
 * Needs C_in % 64 == 0 and C_out % 16 == 0. */
cc_status cc_resample_phase_conv(const cc_bf16* x, const cc_bf16* pw, cc_bf16* phases, int n, int d, int hl,
                                 int wl, int cin, int cout, int hist, void* stream);

/* The interleave pass: out[n,t,2i+p,2j+q,c] = phases[2p+q][n,t,i,j,c] + bias[c]
 * + skip[n,t,i,j,c], summed in fp32 and rounded once. skip: [N, D, HL, WL, C];
 * out: [N, D, 2HL, 2WL, C]. Needs C % 8 == 0. */
cc_status cc_resample_interleave(const cc_bf16* phases, const cc_bf16* bias, const cc_bf16* skip, cc_bf16* out,
                                 int n, int d, int hl, int wl, int c, void* stream);

/* Whole resampler: nearest x2 in space, causal 3x3x3 conv, bias, plus the
 * nearest-duplicated shortcut `skip` (same channel count as the output).
 * out: [N, D, 2HL, 2WL, C_out]. ws: at least cc_resample_workspace_bytes(). */
cc_status cc_resample_up2(const cc_bf16* x, const cc_bf16* pw, const cc_bf16* bias, const cc_bf16* skip,
                          cc_bf16* out, int n, int d, int hl, int wl, int cin, int cout, int hist, void* ws,
                          size_t ws_bytes, void* stream);

/* Temporal variant's pre-summed kernels ([RES]: for up_blocks 0 and 1 the
 * phase kernels and the shortcut are nearest-x2 in time as well). Output
 * frame 2t+s, row 2i+p, column 2j+q; phase tap (a, b, c) reads low-resolution
 * frame t-1+a, row i+p-1+b, column j+q-1+c. Causal tap kt of up-sampled frame
 * 2t+s lands on frame t-1+a for kt in {0,1} | {2} (s=0) or {0} | {1,2} (s=1);
 * rows/columns as in cc_resample_prepare. Sums in fp32, rounded once:
 * pw[(4s+2p+q)][(a*2+b)*2+c][co][ci]; 64*C_out*C_in elements. */
cc_status cc_resample_prepare_temporal(const cc_bf16* w, cc_bf16* pw, int cout, int cin, void* stream);

/* The whole resampler in ONE kernel, no workspace: the phase-convolution
 * epilogue adds the bias and the shortcut to each accumulator row in fp32 and
 * writes it, rounded once, straight to its interleaved high-resolution
 * position (the interleave pass of [RES] done in registers, so the phase
 * tensors never reach memory). temporal = 0: pw from cc_resample_prepare, out
 * [N, D, 2HL, 2WL, C_out], same result as cc_resample_up2 up to rounding (one
 * bf16 rounding instead of two). temporal = 1: pw from
 * cc_resample_prepare_temporal, nearest x2 in time as well -- out
 * [N, 2D, 2HL, 2WL, C_out], shortcut duplicated in time too; with hist = 2
 * only the last history frame matters (it fills both up-sampled frames
 * before frame 0). skip: [N, D, HL, WL, C_out]. */
cc_status cc_resample_up2_fused(const cc_bf16* x, const cc_bf16* pw, const cc_bf16* bias, const cc_bf16* skip,
                                cc_bf16* out, int n, int d, int hl, int wl, int cin, int cout, int hist, int temporal,
                                void* stream);

/* ------------------------------------------------ per-frame attention [ATTN] */

/* Row stride (elements) used for S (fp32), P and E (bf16) inside the
 * workspaces: HW rounded up to a multiple of 16, so rows start on 32-byte
 * boundaries. */
int64_t cc_attn_ld(int hw);

/* Bytes of workspace cc_attn_frame needs: S fp32 and P bf16, T*HW rows each. */
size_t cc_attn_workspace_bytes(int t, int hw);

/* S[f,i,j] = sum_c q[f,i,c] k[f,j,c] in fp32 (unscaled). q, k: T frames of HW
 * rows with row strides ld_q, ld_k elements (frame stride HW*ld); s: row
 * stride ld_s floats. Needs C % 64 == 0, ld_q and ld_k % 8 == 0,
 * ld_s % 4 == 0, ld_s >= HW. S leaves through TMA tensor stores, which end
 * each row on a 16-byte boundary: when HW % 4 != 0, columns HW .. (the next
 * multiple of 4) - 1 may be written (with zeros); nothing past them is. */
cc_status cc_attn_scores(const cc_bf16* q, const cc_bf16* k, float* s, int t, int hw, int c, int64_t ld_q,
                         int64_t ld_k, int64_t ld_s, void* stream);

/* P[f,i,j] = bf16( exp(scale*S[f,i,j] - m_i) / sum_j exp(scale*S[f,i,j] - m_i) ),
 * m_i = max_j scale*S[f,i,j]; columns HW..ld_p-1 of P are written as zero.
 * Needs ld_s % 4 == 0, ld_p % 8 == 0, ld_p >= HW, scale > 0. */
cc_status cc_attn_softmax(const float* s, cc_bf16* p, int t, int hw, int64_t ld_s, int64_t ld_p, float scale,
                          void* stream);

/* O[f,i,c] = sum_j P[f,i,j] v[f,j,c], fp32 accumulation, bf16 out. v is read
 * as stored ([j][c], no transpose). Needs C % 64 == 0, ld_p, ld_v, ld_o % 8 == 0. */
cc_status cc_attn_pv(const cc_bf16* p, const cc_bf16* v, cc_bf16* o, int t, int hw, int c, int64_t ld_p,
                     int64_t ld_v, int64_t ld_o, void* stream);

/* Whole attention: O = softmax(q k^T * scale) v per frame, no mask (scale is
 * 1/sqrt(C) in the decoder). Packed qkv [T, HW, 3C] works with
 * ld_q = ld_k = ld_v = 3C and k = q + C, v = q + 2C.
 * ws: at least cc_attn_workspace_bytes(). */
cc_status cc_attn_frame(const cc_bf16* q, const cc_bf16* k, const cc_bf16* v, cc_bf16* o, int t, int hw, int c,
                        int64_t ld_q, int64_t ld_k, int64_t ld_v, int64_t ld_o, float scale, void* ws,
                        size_t ws_bytes, void* stream);

/* Attention without the fp32 S round trip and the softmax pass, for the same
 * result as cc_attn_frame (softmax per row, [ATTN]), in three launches:
 *  1. cc_attn_scores_exp keeps each 128 x 256 tile of S in TMEM and writes,
 *     per row i and key tile t = j / 256, the numerators
 *     E[f,i,j] = bf16( exp2(kx * S[f,i,j] - c_t) ), kx = scale * log2(e),
 *     c_t = 32 * ceil(kx * max of the row's S over the tile / 32), so every
 *     E is in (0, 1] and the tile's largest E is above 2^-32; and the row
 *     statistics (c_t, l_t), l_t = sum over the tile of the unrounded
 *     exponentials. The coarse grain makes the tiles of a row share c_t in
 *     all but rare cases, which leaves step 2 little to move.
 *  2. cc_attn_exp_rescale puts every row on one scale: c_row = max_t c_t, and
 *     each tile with c_t < c_row is multiplied in place by the exact power of
 *     two 2^(c_t - c_row), its statistics becoming (c_row, 2^(c_t - c_row) l_t).
 *  3. cc_attn_pv_exp computes O = E v with fp32 accumulation and scales each
 *     output row by 1 / l_row, l_row = sum_t l_t.
 * P = E / l_row is then the softmax of the row; E is rounded once, as P is in
 * cc_attn_softmax. */

/* Key tiles per row: ceil(HW / 256). */
int cc_attn_exp_key_tiles(int hw);

/* Bytes of workspace cc_attn_frame_exp needs: E bf16 [T, HW, cc_attn_ld(HW)]
 * and the statistics, float pairs [T, HW, cc_attn_exp_key_tiles(HW)]. */
size_t cc_attn_exp_workspace_bytes(int t, int hw);

/* Step 1 from q, k [T, HW, C] (row strides ld_q, ld_k elements). e: row
 * stride ld_e elements (ld_e >= HW, % 8 == 0); keys HW .. ld_e-1 are not
 * written when e is 32-byte aligned and ld_e % 16 == 0 (E leaves from
 * registers in 32-byte pieces), otherwise E leaves through TMA tensor stores,
 * which end each row on a 16-byte boundary and may write keys HW .. (the next
 * multiple of 8) - 1 with zeros, nothing past them; stats:
 * T*HW*cc_attn_exp_key_tiles(HW) pairs (c_t, l_t), row-major [T][HW][tiles].
 * Needs C % 64 == 0, scale finite and > 0. */
cc_status cc_attn_scores_exp(const cc_bf16* q, const cc_bf16* k, cc_bf16* e, float* stats, int t, int hw, int c,
                             int64_t ld_q, int64_t ld_k, int64_t ld_e, float scale, void* stream);

/* Step 2, in place on e and stats (as written by step 1). */
cc_status cc_attn_exp_rescale(cc_bf16* e, float* stats, int t, int hw, int64_t ld_e, void* stream);

/* Step 3: O[f,i,:] = sum_j E[f,i,j] v[f,j,:] / l_row for E and statistics on
 * one scale per row (after step 2); v read as stored ([j][c]). Needs
 * C % 64 == 0, ld_e, ld_v, ld_o % 8 == 0. */
cc_status cc_attn_pv_exp(const cc_bf16* e, const float* stats, const cc_bf16* v, cc_bf16* o, int t, int hw, int c,
                         int64_t ld_e, int64_t ld_v, int64_t ld_o, void* stream);

/* Steps 1-3: the same contract as cc_attn_frame with a workspace of
 * cc_attn_exp_workspace_bytes(). */
cc_status cc_attn_frame_exp(const cc_bf16* q, const cc_bf16* k, const cc_bf16* v, cc_bf16* o, int t, int hw, int c,
                            int64_t ld_q, int64_t ld_k, int64_t ld_v, int64_t ld_o, float scale, void* ws,
                            size_t ws_bytes, void* stream);

/* Step 1 alone, statistics only: the (c_t, l_t) of cc_attn_scores_exp for
 * every row and key tile, E not written. stats: T*HW*cc_attn_exp_key_tiles(HW)
 * pairs. Needs C % 64 == 0, ld_q and ld_k % 8 == 0, scale finite and > 0. */
cc_status cc_attn_scores_stats(const cc_bf16* q, const cc_bf16* k, float* stats, int t, int hw, int c, int64_t ld_q,
                               int64_t ld_k, float scale, void* stream);

/* Attention with the numerators kept on chip ([ATTN]'s scores, row softmax
 * and PV with nothing between them in memory): cc_attn_scores_stats, then
 * one kernel that, per frame, 256 query rows and 256 channels of O, walks the
 * 256-key tiles, computes S in tensor memory, turns it into
 * E = bf16(exp2(kx * S - c_row)) in shared memory (c_row = the row's largest
 * c_t, so no tile is rescaled) and accumulates E v into O, divided by
 * l_row = sum_t 2^(c_t - c_row) l_t and rounded once at the end. S is
 * computed once per 256-channel chunk of O (O for all C channels of a row
 * block would not fit in tensor memory): C / 256 + 1 times the scores work.
 * Same contract as cc_attn_frame with C % 256 == 0 and a workspace of
 * cc_attn_fused_workspace_bytes() (the statistics only). */
size_t cc_attn_fused_workspace_bytes(int t, int hw);
cc_status cc_attn_frame_fused(const cc_bf16* q, const cc_bf16* k, const cc_bf16* v, cc_bf16* o, int t, int hw, int c,
                              int64_t ld_q, int64_t ld_k, int64_t ld_v, int64_t ld_o, float scale, void* ws,
                              size_t ws_bytes, void* stream);

/* ------------------------------------------------------ output head [HEAD] */

#define CC_HEAD_COUT 12
#define CC_HEAD_G_CH 112 /* 9 spatial taps x 12 channels, padded to 112 */

/* Repacks conv_out's w [12, C_in, 3, 3, 3] into wp [3][112][C_in]:
 * wp[kt][(i*3+j)*12 + c][ci] = w[c][ci][kt][i][j]; rows 108..111 are zero. */
cc_status cc_head_prepare(const cc_bf16* w, cc_bf16* wp, int cin, void* stream);

/* Bytes of workspace cc_head_out needs: g, [N, D, H, W, 112] bf16. */
size_t cc_head_workspace_bytes(int n, int d, int h, int w);

/* Stage A, the temporal-only part of conv_out:
 * g[n,t,h,w,r] = sum_{ci,kt} wp[kt][r][ci] x~[n, t+kt-2, h, w, ci] (fp32 acc,
 * bf16 out). x: [N, D+hist, H, W, C_in], C_in % 64 == 0. */
cc_status cc_head_temporal(const cc_bf16* x, const cc_bf16* wp, cc_bf16* g, int n, int d, int h, int w, int cin,
                           int hist, void* stream);

/* Stage B: out[n,t,h,w,c] = clamp(bias[c] + sum_{i,j} g[n,t,h+i-1,w+j-1,(i*3+j)*12+c],
 * -1, 1), zero outside the plane, fp32 sum, one bf16 rounding.
 * g: [N, D, H, W, 112]; out: [N, D, H, W, 12]. */
cc_status cc_head_stencil(const cc_bf16* g, const cc_bf16* bias, cc_bf16* out, int n, int d, int h, int w,
                          void* stream);

/* Whole head: causal conv_out 3x3x3 C_in -> 12, bias, clamp to [-1, 1].
 * out: [N, D, H, W, 12]; ws: at least cc_head_workspace_bytes(). */
cc_status cc_head_out(const cc_bf16* x, const cc_bf16* wp, const cc_bf16* bias, cc_bf16* out, int n, int d, int h,
                      int w, int cin, int hist, void* ws, size_t ws_bytes, void* stream);

/* The whole head in ONE kernel, no workspace: the same result as
 * cc_head_out (causal conv_out 3x3x3 C_in -> 12, bias, clamp to [-1, 1]) with
 * [HEAD]'s regrouping done on chip. g (the 3x1x1 conv into 9 x 12 channels)
 * stays in fp32 in tensor memory and registers, the 3x3 stencil sums it there,
 * and only the output is rounded to bf16 (cc_head_out also rounds g to bf16).
 * A CTA owns 4-row x 32-column blocks (30 interior columns plus one recomputed
 * halo column on each side) and walks down a strip of the plane, carrying the
 * stencil's partial sums of the rows it cannot finish yet. More than 16
 * output frames run as several passes of at most 16 frames. x: [N, D+hist, H,
 * W, C_in], C_in one of 64, 128, 192, 256; wp from cc_head_prepare; out:
 * [N, D, H, W, 12]. */
cc_status cc_head_out_fused(const cc_bf16* x, const cc_bf16* wp, const cc_bf16* bias, cc_bf16* out, int n, int d,
                            int h, int w, int cin, int hist, void* stream);

/* Size of the library's built-in scratch for cc_head_out_noalloc: 64 MiB,
 * i.e. at most 64 MiB / (112 * 2 B) = 299,593 output positions per call. */
#define CC_HEAD_NOALLOC_SCRATCH_BYTES (64u << 20)

/* The whole head, like cc_head_out, for callers that cannot allocate device
 * memory and so cannot pass a workspace -- for example a plugin inside a host
 * framework that owns every device allocation and exposes no allocator, or a
 * latency-critical loop where cudaMalloc (which may synchronise the device) is
 * not allowed. The source pages have no counterpart to this entry point; it
 * is an addition of this library. g lives in a fixed 64 MiB array in the
 * library's static device memory, which every GPU that loads the library
 * holds until the process exits; this function allocates nothing.
 *  - The first call on a device looks up the array's device address (no
 *    allocation) with that device current. The address is kept for the life
 *    of the process, so after cudaDeviceReset() on a device this function
 *    must not be called again in that process (it would hand the kernels a
 *    stale address).
 *  - More than CC_HEAD_NOALLOC_SCRATCH_BYTES / 224 positions (N*D*H*W):
 *    CC_ERR_INVALID with a message naming the limit; nothing is launched.
 *  - All calls on a device share the array and leave their g in it; nothing
 *    in it needs to start at zero (every element read is written first in the
 *    same call). Calls whose GPU work overlaps (other streams or threads
 *    without ordering) race on it: order them on one stream.
 * Other arguments, layouts and errors as cc_head_out. */
cc_status cc_head_out_noalloc(const cc_bf16* x, const cc_bf16* wp, const cc_bf16* bias, cc_bf16* out, int n, int d,
                              int h, int w, int cin, int hist, void* stream);

/* ------------------------------------------------- result read-back [HOST] */

/* Copies `bytes` from device memory at `src` to page-locked host memory at
 * `dst` with a copy kernel of `ctas` thread blocks on `stream`, for a chunked
 * decode whose outputs go back to the host while the next chunk's inputs
 * come in. Not part of the method: a transfer helper. A copy-engine read-back
 * (cudaMemcpyAsync) beside a host-to-device copy takes about half of the host
 * link from it; the SMs' stores to the mapped host address run at a rate set
 * by `ctas` (4-8: ~90 GB/s measured on GB300) and leave the inflowing copy
 * nearly its whole bandwidth.
 *  - dst: page-locked host memory (cudaHostAlloc, cudaHostRegister) that the
 *    device addresses at the same pointer (unified addressing); src: device
 *    memory; both 16-byte aligned, `bytes` a multiple of 16, 1 <= ctas <= 1024.
 *    Both ends of each range are checked with cudaPointerGetAttributes;
 *    anything else is CC_ERR_INVALID and nothing is launched. bytes == 0
 *    succeeds at once.
 *  - Asynchronous on `stream`; `dst` holds the data once the stream's work up
 *    to this call is done. The caller keeps both buffers alive until then. */
cc_status cc_copy_to_host(void* dst, const void* src, size_t bytes, int ctas, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* CC_H_ */
