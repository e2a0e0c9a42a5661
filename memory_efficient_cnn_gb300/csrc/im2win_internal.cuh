// Internal declarations shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "im2win.h"

namespace im2win {

// Problem shape with the output extents derived. Table I of the GPU im2win
// paper has valid convolutions (no padding, floor division); the optional zero
// padding p_h, p_w and dilation d_h, d_w follow the usual CNN definitions:
//   H_o = (H_i + 2 p_h - d_h (H_f - 1) - 1) / s_h + 1   (likewise W_o),
// input element (ho*s_h + r*d_h - p_h, wo*s_w + j*d_w - p_w), zero outside.
// g_w > 1 only in the virtual shape of a window tensor read as an input with
// column dilation: filter column j there sits at input column
// (j / g_w)*d_w*g_w + j % g_w (runs of g_w = H_f window elements).
struct Shape {
    int64_t N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, H_o, W_o;
    int64_t p_h = 0, p_w = 0, d_h = 1, d_w = 1, g_w = 1;
};

// No padding, no dilation: the pages' valid convolution.
inline bool plain(const Shape &s) { return s.p_h == 0 && s.p_w == 0 && s.d_h == 1 && s.d_w == 1 && s.g_w == 1; }
// Padded input width.
inline int64_t padded_w(const Shape &s) { return s.W_i + 2 * s.p_w; }

// Status block at the start of every convolution workspace (256 bytes).
// word 0: im2win_status of the last call; word 1: wait site that gave up;
// word 2: block index that gave up.
constexpr size_t kStatusBytes = 256;

inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline int elem_size(int dtype) {
    switch (dtype) {
        case IM2WIN_F32: return 4;
        case IM2WIN_F16: return 2;
        case IM2WIN_BF16: return 2;
        default: return 0;
    }
}

// 32-bit division by a run-time constant through a multiply-high
// (Granlund & Montgomery, "Division by invariant integers using
// multiplication", 1994): q = (umulhi(n, m) + n) >> l with
// l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1, exact for n < 2^31.
struct FastDiv {
    uint32_t d, m, l;
};

inline FastDiv make_fastdiv(uint32_t d) {
    FastDiv f;
    f.d = d;
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;
    f.l = l;
    f.m = (uint32_t)(((1ull << 32) * ((1ull << l) - d)) / d + 1);
    return f;
}

__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv &f) {
    return (__umulhi(n, f.m) + n) >> f.l;
}

// A kernel computes the convolution of a (virtual) shape whose filter is a
// re-ordering of the caller's filter w[C_o][C][H_f][W_f]. The view names the
// re-ordering: a virtual filter element (ci_v, r_v, j_v) is the caller's
// element (c, r, j) with
//   VIEW_IDENT     (ci_v, r_v, j_v)                              the shape itself
//   VIEW_WIN       (ci_v, j_v % H_f, j_v / H_f)                  NCHW window tensor as the input,
//                                                                 one row of W_f*H_f taps
//   VIEW_CL_X      (j_v % C, r_v, j_v / C)                       NHWC input as one channel of
//                                                                 H_i x W_i*C (columns (w, c))
//   VIEW_CL_WIN    (j_v % C, (j_v / C) % H_f, j_v / C / H_f)     NHWC window tensor as one channel,
//                                                                 one row of W_f*H_f*C taps
//   VIEW_CL_ROWS   (j_v % C, ci_v, j_v / C)                      NHWC input, filter rows as channels,
//                                                                 one row of W_f*C taps each
enum FilterView { VIEW_IDENT = 0, VIEW_WIN = 1, VIEW_CL_X = 2, VIEW_CL_WIN = 3, VIEW_CL_ROWS = 4 };

// Offset of virtual filter element (ci_v, r_v, j_v) within the caller's filter
// row w[co][:][:][:] (C x H_f x W_f are the caller's extents).
__host__ __device__ inline int64_t filter_src_offset(int view, int ci_v, int r_v, int j_v, int C, int H_f,
                                                     int W_f) {
    int c = ci_v, r = r_v, j = j_v;
    switch (view) {
        case VIEW_WIN: r = j_v % H_f; j = j_v / H_f; break;
        case VIEW_CL_X: c = j_v % C; j = j_v / C; break;
        case VIEW_CL_WIN: c = j_v % C; r = (j_v / C) % H_f; j = j_v / C / H_f; break;
        case VIEW_CL_ROWS: c = j_v % C; r = ci_v; j = j_v / C; break;
        default: break;
    }
    return ((int64_t)c * H_f + r) * W_f + j;
}

// Tensor layouts of the convolution entry points.
enum Layout { LAYOUT_NCHW = 0, LAYOUT_NHWC = 1 };

// ---- launchers (each returns cudaSuccess or the launch error) ----

// Window transform of esz-byte elements (NCHW), and its channels-last form
// win[n][ho][w*H_f + r][c] = x[n][ho*s_h + r][w][c]; the padded/dilated form
// (either layout) runs over the W_i + 2 p_w padded columns and rows
// ho*s_h + r*d_h - p_h, zero outside x.
cudaError_t launch_transform(const void *x, void *win, const Shape &s, int esz, cudaStream_t st);
bool transform_supported(const Shape &s, int esz);
cudaError_t launch_transform_nhwc(const void *x, void *win, const Shape &s, int esz, cudaStream_t st);
bool transform_nhwc_supported(const Shape &s, int esz);
cudaError_t launch_transform_pd(const void *x, void *win, const Shape &s, int esz, int layout, cudaStream_t st);
bool transform_pd_supported(const Shape &s, int esz);

// fp32 CUDA-core convolution; from_x selects the fused variant that gathers
// from the input instead of the window tensor; layout is NCHW or NHWC for the
// input, window tensor and output alike. ws holds the status block followed
// by the re-laid filter.
size_t conv_f32_filter_bytes(const Shape &s, bool from_x, int layout);
bool conv_f32_supported(const Shape &s, bool from_x, int layout);
cudaError_t launch_conv_f32(const void *src, const void *filt, void *out, void *ws,
                            const Shape &s, bool from_x, int layout, cudaStream_t st);

// fp16/bf16 tensor-core convolution (tcgen05): from the window tensor or fused
// from the input, in either layout.
size_t conv_tc_filter_bytes(const Shape &s, bool fused, int layout);
bool conv_tc_supported(const Shape &s, bool fused, int layout);

// What a tensor-core convolution launches (host only; the plan query).
// kernel 1: tap kernel, 2: expand kernel; the other fields describe the tap
// kernel (zero for the expand kernel). tmem_read_end is one past the highest
// accumulator column the epilogue reads, as its drain walks the columns.
struct TcPlanInfo {
    int kernel, tap_mode, stacked, rows_per_tile, pitch, tmem_columns, tmem_read_end, smem_bytes;
    int filter_stage_taps, filter_stages, slab_stages;
    int64_t tiles, grid;
};
// false: no tensor-core kernel covers the shape. sms <= 0: the current device's.
bool conv_tc_plan_info(const Shape &s, bool fused, int layout, int64_t sms, TcPlanInfo &info);
cudaError_t launch_conv_tc(const void *src, const void *filt, void *out, void *ws,
                           const Shape &s, bool fused, int layout, bool bf16, cudaStream_t st);

}  // namespace im2win
