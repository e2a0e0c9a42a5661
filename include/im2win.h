/*
 * im2win.h -- C ABI of the GB300 (sm_103a) im2win convolution library.
 *
 * The method is the im2win convolution of
 *   [SIMD] "Im2win: Memory Efficient Convolution On SIMD Architectures" (Abstract), and
 *   [GPU]  "Enabling Memory-efficient Im2win Convolution with Multi-precision Support
 *           on GPU CUDA and Tensor Cores" (Abstract, Fig. 1, Tables I and II).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Shapes: N images, C_i input channels of H_i x W_i, C_o filters of C_i x H_f x W_f,
 *    strides s_h, s_w; "valid" convolution with no padding or dilation, so
 *    H_o = (H_i - H_f)/s_h + 1 and W_o = (W_i - W_f)/s_w + 1 (floor), which every
 *    layer of [GPU] Table I satisfies. All sizes are int64_t and must be >= 1
 *    (N may be 0: the call then does nothing), with H_f <= H_i and W_f <= W_i.
 *    Each tensor a call touches (input, window tensor, output, filter) must hold
 *    at most 2^50 elements; larger shapes return IM2WIN_ERR_UNSUPPORTED from
 *    every call, the workspace queries included, so a size these return never
 *    wraps around.
 *  - Layouts are dense and row-major: x[N][C_i][H_i][W_i] (NCHW),
 *    filt[C_o][C_i][H_f][W_f], out[N][C_o][H_o][W_o], and the window tensor
 *    win[N][C_i][H_o][W_i*H_f].
 *  - dtype is one of im2win_dtype. x, filt, win and out all have that dtype.
 *    F16/BF16 convolutions multiply on the tensor cores with fp32 accumulation and
 *    round the result to the input dtype (round-to-nearest-even); F32
 *    convolutions run on the CUDA cores in fp32.
 *  - Every pointer argument except `bytes` is a DEVICE pointer on the current
 *    CUDA device, allocated and owned by the caller; the library never allocates,
 *    frees or synchronises (except im2win_device_status, which synchronises the
 *    given stream). Pointers must be 16-byte aligned.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    All work is enqueued asynchronously on it; calls on different streams that
 *    share a workspace race.
 *  - Return value: an im2win_status. Argument errors are reported before any work
 *    is enqueued. IM2WIN_ERR_CUDA means a launch failed (cudaGetLastError).
 *    Kernels that wait on in-kernel barriers give up after a bounded time and
 *    record IM2WIN_ERR_TIMEOUT in the workspace's status word, which
 *    im2win_device_status reads back.
 */
#ifndef IM2WIN_H
#define IM2WIN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    IM2WIN_F32 = 0,
    IM2WIN_F16 = 1,
    IM2WIN_BF16 = 2
} im2win_dtype;

typedef enum {
    IM2WIN_OK = 0,
    IM2WIN_ERR_INVALID_ARG = 1, /* bad shape, null pointer, unknown dtype or op */
    IM2WIN_ERR_UNSUPPORTED = 2, /* well-formed but outside what the kernels handle */
    IM2WIN_ERR_MISALIGNED = 3,  /* a pointer is not 16-byte aligned */
    IM2WIN_ERR_WORKSPACE = 4,   /* ws is NULL or ws_bytes is below the required size */
    IM2WIN_ERR_CUDA = 5,        /* a CUDA call or kernel launch failed */
    IM2WIN_ERR_TIMEOUT = 6      /* an in-kernel barrier wait gave up (device status only) */
} im2win_status;

/* Which call a workspace size is asked for. */
typedef enum {
    IM2WIN_OP_TRANSFORM = 0,       /* bytes of the window tensor `win` that im2win_transform or
                                      im2win_transform_nhwc writes (the same count) */
    IM2WIN_OP_CONV = 1,            /* workspace of im2win_conv (status block + re-laid filter) */
    IM2WIN_OP_CONV_FUSED = 2,      /* workspace of im2win_conv_fused (status block + re-laid filter) */
    IM2WIN_OP_CONV_NHWC = 3,       /* workspace of im2win_conv_nhwc */
    IM2WIN_OP_CONV_FUSED_NHWC = 4  /* workspace of im2win_conv_fused_nhwc */
} im2win_op;

/*
 * Bytes needed for `op` on this problem, written to *bytes (a HOST pointer).
 * Pure host arithmetic: no device call. For IM2WIN_OP_TRANSFORM this is
 * N*C_i*H_o*W_i*H_f*esz, the size of the window tensor ([SIMD] Abstract: one row of
 * W_i*H_f unique elements per channel and output row). For the two convolutions it
 * is a 256-byte status block plus the filter re-laid for the kernel that runs, each
 * part rounded up to 256 bytes; the fused convolution needs no window tensor.
 * Errors: INVALID_ARG for a bad shape, dtype or op, or bytes == NULL;
 * UNSUPPORTED for a shape beyond the 2^50-element limit above.
 */
im2win_status im2win_workspace_size(int op, int64_t N, int64_t C_i, int64_t H_i, int64_t W_i,
                                    int64_t C_o, int64_t H_f, int64_t W_f, int64_t s_h,
                                    int64_t s_w, int dtype, size_t *bytes);

/*
 * The im2win transformation ([SIMD] Abstract; [GPU] Fig. 1, middle column):
 *   win[n][ci][ho][w*H_f + r] = x[n][ci][ho*s_h + r][w]   for w < W_i, r < H_f,
 * i.e. the H_f input rows under output row ho are flattened column by column into
 * one contiguous window row; all W_i columns are kept. A bit-exact copy of
 * esz-byte elements. Reads x (N*C_i*H_i*W_i elements), writes exactly
 * N*C_i*H_o*W_i*H_f elements at win; C_o, W_f and s_w are validated but do not
 * change the result. x and win must not overlap.
 */
im2win_status im2win_transform(const void *x, void *win, int64_t N, int64_t C_i, int64_t H_i,
                               int64_t W_i, int64_t C_o, int64_t H_f, int64_t W_f,
                               int64_t s_h, int64_t s_w, int dtype, void *stream);

/*
 * Convolution over a window tensor ([GPU] Abstract: full precision on CUDA cores,
 * half precision on tensor cores; [SIMD] Abstract):
 *   out[n][co][ho][wo] = sum_ci sum_{k < W_f*H_f} win[n][ci][ho][wo*s_w*H_f + k] * filt'[co][ci][k],
 *   filt'[co][ci][j*H_f + r] = filt[co][ci][r][j],
 * which equals the direct valid cross-correlation of x with filt. `win` is the
 * output of im2win_transform for the same shape. The filter is re-laid into `ws`
 * on every call (ws_bytes >= im2win_workspace_size(IM2WIN_OP_CONV, ...)).
 * Errors: INVALID_ARG, MISALIGNED, WORKSPACE, UNSUPPORTED (shape beyond the
 * kernels' index range), CUDA.
 */
im2win_status im2win_conv(const void *win, const void *filt, void *out, void *ws,
                          size_t ws_bytes, int64_t N, int64_t C_i, int64_t H_i, int64_t W_i,
                          int64_t C_o, int64_t H_f, int64_t W_f, int64_t s_h, int64_t s_w,
                          int dtype, void *stream);

/*
 * Fused im2win convolution: the same result as im2win_transform followed by
 * im2win_conv, computed straight from the NCHW input. The kernel stages, in
 * shared memory only, the unique input elements of the windows of the output
 * tile it computes, so the window tensor is never written to device memory;
 * the workspace holds only the re-laid filter and the status block
 * (ws_bytes >= im2win_workspace_size(IM2WIN_OP_CONV_FUSED, ...)).
 * Errors as for im2win_conv.
 */
im2win_status im2win_conv_fused(const void *x, const void *filt, void *out, void *ws,
                                size_t ws_bytes, int64_t N, int64_t C_i, int64_t H_i,
                                int64_t W_i, int64_t C_o, int64_t H_f, int64_t W_f,
                                int64_t s_h, int64_t s_w, int dtype, void *stream);

/*
 * Channels-last (NHWC) layouts
 * ----------------------------
 * [SIMD] names, as a title only, a successor work that carries im2win to three
 * tensor layouts; these calls take its plainest reading: the NCHW window row
 * keeps its order and each of its elements becomes the C_i channels of that
 * position, innermost. Layouts:
 *   x[N][H_i][W_i][C_i], win[N][H_o][W_i*H_f][C_i], out[N][H_o][W_o][C_o];
 *   the filter keeps filt[C_o][C_i][H_f][W_f].
 * Arguments, dtypes, alignment, streams, workspaces and errors are as for the
 * NCHW calls above; each convolution's workspace is sized by its own op
 * (IM2WIN_OP_CONV_NHWC, IM2WIN_OP_CONV_FUSED_NHWC). F16/BF16 convolutions need
 * one of: C_i a multiple of 8 (16-byte channel groups), or a window step
 * s_w*H_f*C_i (window tensor) / s_w*C_i (fused) that the tensor-core tiling
 * accepts; otherwise they return IM2WIN_ERR_UNSUPPORTED.
 */

/*
 * Channels-last im2win transformation:
 *   win[n][ho][w*H_f + r][c] = x[n][ho*s_h + r][w][c]   for w < W_i, r < H_f, c < C_i.
 * A bit-exact copy; writes exactly N*H_o*W_i*H_f*C_i elements at win.
 */
im2win_status im2win_transform_nhwc(const void *x, void *win, int64_t N, int64_t C_i, int64_t H_i,
                                    int64_t W_i, int64_t C_o, int64_t H_f, int64_t W_f,
                                    int64_t s_h, int64_t s_w, int dtype, void *stream);

/*
 * Convolution over the channels-last window tensor: the window row of (n, ho)
 * is one run of W_i*H_f*C_i elements and
 *   out[n][ho][wo][co] = sum_{k < W_f*H_f*C_i} win[n][ho][wo*s_w*H_f*C_i + k] * filt''[co][k],
 *   filt''[co][(j*H_f + r)*C_i + c] = filt[co][c][r][j],
 * which equals the direct valid cross-correlation of the NHWC input with filt.
 * ws_bytes >= im2win_workspace_size(IM2WIN_OP_CONV_NHWC, ...).
 */
im2win_status im2win_conv_nhwc(const void *win, const void *filt, void *out, void *ws,
                               size_t ws_bytes, int64_t N, int64_t C_i, int64_t H_i, int64_t W_i,
                               int64_t C_o, int64_t H_f, int64_t W_f, int64_t s_h, int64_t s_w,
                               int dtype, void *stream);

/*
 * Fused channels-last convolution: the result of im2win_transform_nhwc followed
 * by im2win_conv_nhwc, computed straight from the NHWC input without writing the
 * window tensor. ws_bytes >= im2win_workspace_size(IM2WIN_OP_CONV_FUSED_NHWC, ...).
 */
im2win_status im2win_conv_fused_nhwc(const void *x, const void *filt, void *out, void *ws,
                                     size_t ws_bytes, int64_t N, int64_t C_i, int64_t H_i,
                                     int64_t W_i, int64_t C_o, int64_t H_f, int64_t W_f,
                                     int64_t s_h, int64_t s_w, int dtype, void *stream);

/*
 * Zero padding, dilation and the layout as arguments
 * --------------------------------------------------
 * The pages' layers are valid convolutions; these calls add the two usual CNN
 * options (neither is on the pages, so this is the usual definition):
 *   out[n][co][ho][wo] = sum_ci sum_r sum_j xpad[n][ci][ho*s_h + r*d_h][wo*s_w + j*d_w] * filt[co][ci][r][j],
 * where xpad is x with p_h zero rows above and below and p_w zero columns on
 * each side, and
 *   H_o = (H_i + 2 p_h - d_h (H_f - 1) - 1) / s_h + 1,  W_o likewise (floor).
 * Requirements: p_h, p_w >= 0; d_h, d_w >= 1; d_h (H_f - 1) + 1 <= H_i + 2 p_h and
 * d_w (W_f - 1) + 1 <= W_i + 2 p_w (else IM2WIN_ERR_INVALID_ARG).
 * The window tensor runs over the W_p = W_i + 2 p_w padded columns and holds the
 * dilated rows:
 *   NCHW: win[n][ci][ho][w*H_f + r] = xpad[n][ci][ho*s_h + r*d_h][w],
 *   NHWC: win[n][ho][w*H_f + r][ci] = xpad[n][ci][ho*s_h + r*d_h][w],   w < W_p,
 * N*C_i*H_o*W_p*H_f elements; the convolution from it sums, per filter column j,
 * the run of H_f window elements starting at (wo*s_w + j*d_w)*H_f.
 * `layout` is an im2win_layout and applies to x, win and out (the filter is
 * always filt[C_o][C_i][H_f][W_f]). With p = 0 and d = 1 each call equals its
 * counterpart above. Other arguments, dtypes and errors as above; a workspace
 * comes from im2win_workspace_size_ex with the same padding, dilation and
 * layout (op IM2WIN_OP_TRANSFORM, IM2WIN_OP_CONV or IM2WIN_OP_CONV_FUSED).
 * F16/BF16 convolutions with padding or dilation run the channel-group tensor-core
 * kernel only and return IM2WIN_ERR_UNSUPPORTED where it has no tiling.
 */
typedef enum {
    IM2WIN_LAYOUT_NCHW = 0,
    IM2WIN_LAYOUT_NHWC = 1
} im2win_layout;

im2win_status im2win_workspace_size_ex(int op, int64_t N, int64_t C_i, int64_t H_i, int64_t W_i,
                                       int64_t C_o, int64_t H_f, int64_t W_f, int64_t s_h, int64_t s_w,
                                       int64_t p_h, int64_t p_w, int64_t d_h, int64_t d_w, int layout,
                                       int dtype, size_t *bytes);

im2win_status im2win_transform_ex(const void *x, void *win, int64_t N, int64_t C_i, int64_t H_i, int64_t W_i,
                                  int64_t C_o, int64_t H_f, int64_t W_f, int64_t s_h, int64_t s_w,
                                  int64_t p_h, int64_t p_w, int64_t d_h, int64_t d_w, int layout, int dtype,
                                  void *stream);

im2win_status im2win_conv_ex(const void *win, const void *filt, void *out, void *ws, size_t ws_bytes,
                             int64_t N, int64_t C_i, int64_t H_i, int64_t W_i, int64_t C_o, int64_t H_f,
                             int64_t W_f, int64_t s_h, int64_t s_w, int64_t p_h, int64_t p_w, int64_t d_h,
                             int64_t d_w, int layout, int dtype, void *stream);

im2win_status im2win_conv_fused_ex(const void *x, const void *filt, void *out, void *ws, size_t ws_bytes,
                                   int64_t N, int64_t C_i, int64_t H_i, int64_t W_i, int64_t C_o, int64_t H_f,
                                   int64_t W_f, int64_t s_h, int64_t s_w, int64_t p_h, int64_t p_w, int64_t d_h,
                                   int64_t d_w, int layout, int dtype, void *stream);

/*
 * Plan query (host only: no GPU work, usable without a device). Reports which
 * kernel a convolution call with these arguments would launch and, for the
 * tensor-core tap kernel, its tiling. op is IM2WIN_OP_CONV (from the window
 * tensor) or IM2WIN_OP_CONV_FUSED; the shape, padding, dilation, layout and
 * dtype are those of im2win_conv_ex / im2win_conv_fused_ex; sms is the SM count
 * the persistent grid is planned for, or <= 0 for the current device's (148
 * when no device is visible). Returns INVALID_ARG or UNSUPPORTED where the call
 * would, else fills *info (every field zero where it does not apply).
 */
typedef enum {
    IM2WIN_KERNEL_F32 = 0,      /* fp32 CUDA-core convolution */
    IM2WIN_KERNEL_TAP = 1,      /* tensor-core tap kernel (tcgen05, persistent) */
    IM2WIN_KERNEL_EXPAND = 2    /* tensor-core expand kernel (fallback, NCHW without padding) */
} im2win_kernel;

typedef struct {
    int32_t kernel;             /* im2win_kernel */
    int32_t tap_mode;           /* tap kernel: 0 channel slab (NCHW input, or window tensor read as an
                                   input), 1 window rows of one channel from the input, 2 window rows
                                   from the window tensor, 3 channel slab of a channels-last tensor;
                                   -1 for the other kernels */
    int32_t stacked;            /* C_o <= 64: two filter taps per MMA; 1: along M, 2: along N
                                   with the output positions along M (TMEM double-buffered) */
    int32_t rows_per_tile;      /* output rows per tile */
    int32_t pitch;              /* accumulator columns per output row */
    int32_t tmem_columns;       /* accumulator columns of the widest tile (<= 512; stacked 2: one
                                   past the last column of the second buffer) */
    int32_t tmem_read_end;      /* one past the highest accumulator column the epilogue reads */
    int32_t smem_bytes;         /* dynamic shared memory per CTA */
    int32_t filter_stage_taps;  /* filter taps per shared-memory stage */
    int32_t filter_stages;      /* filter stages */
    int32_t slab_stages;        /* input slab stages */
    int32_t reserved;
    int64_t tiles;              /* tiles of the launch: N * ceil(C_o / 128) * ceil(H_o / rows_per_tile) */
    int64_t grid;               /* CTAs launched: min(sms, tiles) */
} im2win_plan_info;

im2win_status im2win_plan(int op, int64_t N, int64_t C_i, int64_t H_i, int64_t W_i, int64_t C_o,
                          int64_t H_f, int64_t W_f, int64_t s_h, int64_t s_w, int64_t p_h, int64_t p_w,
                          int64_t d_h, int64_t d_w, int layout, int dtype, int sms, im2win_plan_info *info);

/* Static, NUL-terminated description of a status code (never NULL). */
const char *im2win_status_string(int status);

/*
 * Synchronises `stream`, then reads the status word that the last convolution
 * enqueued with workspace `ws` left in it: IM2WIN_OK, or IM2WIN_ERR_TIMEOUT if
 * one of its in-kernel waits gave up. ws_bytes must cover the 256-byte status
 * block. Returns IM2WIN_ERR_CUDA if the synchronisation or the copy fails.
 */
im2win_status im2win_device_status(const void *ws, size_t ws_bytes, void *stream);

/* Size of the scratch array built into the library for im2win_conv_fused_noalloc. */
#define IM2WIN_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

/*
 * im2win_conv_fused for callers that cannot allocate a workspace. The pages
 * have no counterpart to this call: it exists for callers that only hold the
 * input and output buffers -- a plugin slot that is handed tensor pointers and
 * nothing else, or code that must not call cudaMalloc because it may
 * synchronise the device. Same arguments and result as im2win_conv_fused,
 * minus ws/ws_bytes: the scratch lives in one array of
 * IM2WIN_NOALLOC_SCRATCH_BYTES compiled into the library (device memory of
 * every GPU that loads it, held until the process exits). A problem whose
 * fused workspace (im2win_workspace_size(IM2WIN_OP_CONV_FUSED, ...)) exceeds
 * that size is rejected with IM2WIN_ERR_WORKSPACE before any work is queued.
 * Every call looks up the array's device address on the current device
 * (cudaGetSymbolAddress), so a device reset, which may move the array, does
 * not leave a stale address; the first call on a device loads the library's
 * module there, so make one call before any stream capture.
 * All calls share the array and it keeps the last call's contents (each call
 * re-lays the filter and clears the status word itself): calls whose work can
 * overlap on the GPU race and may return wrong results. Calls no cudaMalloc,
 * cudaFree or other allocating routine. An in-kernel wait that gives up is
 * recorded in the shared array, which im2win_device_status cannot read; use
 * im2win_conv_fused with a workspace when that check is needed.
 */
im2win_status im2win_conv_fused_noalloc(const void *x, const void *filt, void *out, int64_t N,
                                        int64_t C_i, int64_t H_i, int64_t W_i, int64_t C_o,
                                        int64_t H_f, int64_t W_f, int64_t s_h, int64_t s_w,
                                        int dtype, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* IM2WIN_H */
