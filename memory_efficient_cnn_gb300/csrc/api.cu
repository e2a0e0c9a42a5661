// C ABI of the im2win library: argument validation, workspace sizing and
// dispatch to the kernels. No allocation, no synchronisation (except
// im2win_device_status), no CPU fallback: every result is computed on the GPU.
#include <cstdint>
#include <cstring>
#include <initializer_list>

#include "im2win_internal.cuh"

using namespace im2win;

namespace {

// Every element count a call can touch (input, window tensor, output, filter)
// stays at or below 2^50, so that byte counts and the kernels' 64-bit offsets
// derived from them cannot overflow. Products are formed in 128 bits.
constexpr int64_t kMaxElems = int64_t(1) << 50;

bool product_within(std::initializer_list<int64_t> factors, int64_t lim) {
    __int128 p = 1;
    for (const int64_t f : factors) {
        p *= (__int128)f;
        if (p > (__int128)lim) return false;
    }
    return true;
}

// The shape's tensors: x (padded extent), the window tensor, the output and the
// filter, each within kMaxElems elements.
im2win_status bound_tensors(const Shape &s) {
    const int64_t Hp = s.H_i + 2 * s.p_h, Wp = s.W_i + 2 * s.p_w;
    if (!product_within({s.N, s.C_i, Hp, Wp}, kMaxElems) ||
        !product_within({s.N, s.C_i, s.H_o, Wp, s.H_f}, kMaxElems) ||
        !product_within({s.N, s.C_o, s.H_o, s.W_o}, kMaxElems) ||
        !product_within({s.C_o, s.C_i, s.H_f, s.W_f}, kMaxElems))
        return IM2WIN_ERR_UNSUPPORTED;
    return IM2WIN_OK;
}

im2win_status make_shape(Shape &s, int64_t N, int64_t C_i, int64_t H_i, int64_t W_i, int64_t C_o,
                         int64_t H_f, int64_t W_f, int64_t s_h, int64_t s_w) {
    if (N < 0 || C_i <= 0 || H_i <= 0 || W_i <= 0 || C_o <= 0 || H_f <= 0 || W_f <= 0 ||
        s_h <= 0 || s_w <= 0 || H_f > H_i || W_f > W_i)
        return IM2WIN_ERR_INVALID_ARG;
    // keep every element count far from int64 overflow
    const int64_t lim = int64_t(1) << 40;
    if (N > lim || C_i > lim || H_i > lim || W_i > lim || C_o > lim ||
        N * C_i > lim || H_i * W_i > lim || C_o * C_i > lim || H_f * W_f > lim)
        return IM2WIN_ERR_UNSUPPORTED;
    s.N = N; s.C_i = C_i; s.H_i = H_i; s.W_i = W_i; s.C_o = C_o;
    s.H_f = H_f; s.W_f = W_f; s.s_h = s_h; s.s_w = s_w;
    s.H_o = (H_i - H_f) / s_h + 1;
    s.W_o = (W_i - W_f) / s_w + 1;
    return bound_tensors(s);
}

// make_shape with zero padding p_h, p_w >= 0 and dilation d_h, d_w >= 1; the
// dilated filter must fit the padded input.
im2win_status make_shape_pd(Shape &s, int64_t N, int64_t C_i, int64_t H_i, int64_t W_i, int64_t C_o,
                            int64_t H_f, int64_t W_f, int64_t s_h, int64_t s_w, int64_t p_h, int64_t p_w,
                            int64_t d_h, int64_t d_w) {
    const int64_t lim = int64_t(1) << 40;
    if (N < 0 || C_i <= 0 || H_i <= 0 || W_i <= 0 || C_o <= 0 || H_f <= 0 || W_f <= 0 || s_h <= 0 ||
        s_w <= 0 || p_h < 0 || p_w < 0 || d_h <= 0 || d_w <= 0)
        return IM2WIN_ERR_INVALID_ARG;
    if (p_h > lim || p_w > lim || d_h > lim || d_w > lim || H_f > lim || W_f > lim || H_i > lim || W_i > lim)
        return IM2WIN_ERR_UNSUPPORTED;
    if (d_h * (H_f - 1) + 1 > H_i + 2 * p_h || d_w * (W_f - 1) + 1 > W_i + 2 * p_w) return IM2WIN_ERR_INVALID_ARG;
    if (N > lim || C_i > lim || C_o > lim || N * C_i > lim || (H_i + 2 * p_h) * (W_i + 2 * p_w) > lim ||
        C_o * C_i > lim || H_f * W_f > lim)
        return IM2WIN_ERR_UNSUPPORTED;
    s.N = N; s.C_i = C_i; s.H_i = H_i; s.W_i = W_i; s.C_o = C_o;
    s.H_f = H_f; s.W_f = W_f; s.s_h = s_h; s.s_w = s_w;
    s.p_h = p_h; s.p_w = p_w; s.d_h = d_h; s.d_w = d_w; s.g_w = 1;
    s.H_o = (H_i + 2 * p_h - d_h * (H_f - 1) - 1) / s_h + 1;
    s.W_o = (W_i + 2 * p_w - d_w * (W_f - 1) - 1) / s_w + 1;
    return bound_tensors(s);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t window_bytes(const Shape &s, int esz) {
    return (size_t)(s.N * s.C_i * s.H_o * padded_w(s) * s.H_f) * (size_t)esz;
}

size_t conv_ws_bytes(const Shape &s, int dtype, bool fused, int layout) {
    const size_t f = dtype == IM2WIN_F32 ? conv_f32_filter_bytes(s, fused, layout)
                                         : conv_tc_filter_bytes(s, fused, layout);
    return kStatusBytes + round_up(f, 256);
}

im2win_status conv_shape(const Shape &s, const void *src, const void *filt, void *out, void *ws,
                         size_t ws_bytes, int dtype, void *stream, bool fused, int layout);

im2win_status conv_common(const void *src, const void *filt, void *out, void *ws, size_t ws_bytes,
                          int64_t N, int64_t C_i, int64_t H_i, int64_t W_i, int64_t C_o,
                          int64_t H_f, int64_t W_f, int64_t s_h, int64_t s_w, int dtype,
                          void *stream, bool fused, int layout) {
    Shape s;
    im2win_status st = make_shape(s, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w);
    if (st != IM2WIN_OK) return st;
    return conv_shape(s, src, filt, out, ws, ws_bytes, dtype, stream, fused, layout);
}

im2win_status conv_shape(const Shape &s, const void *src, const void *filt, void *out, void *ws,
                         size_t ws_bytes, int dtype, void *stream, bool fused, int layout) {
    if (elem_size(dtype) == 0) return IM2WIN_ERR_INVALID_ARG;
    if (s.N == 0) return IM2WIN_OK;  // empty batch: nothing to read or write
    if (!src || !filt || !out) return IM2WIN_ERR_INVALID_ARG;
    if (!aligned16(src) || !aligned16(filt) || !aligned16(out)) return IM2WIN_ERR_MISALIGNED;
    if (!ws || ws_bytes < conv_ws_bytes(s, dtype, fused, layout)) return IM2WIN_ERR_WORKSPACE;
    if (!aligned16(ws)) return IM2WIN_ERR_MISALIGNED;
    const bool ok = dtype == IM2WIN_F32 ? conv_f32_supported(s, fused, layout)
                                        : conv_tc_supported(s, fused, layout);
    if (!ok) return IM2WIN_ERR_UNSUPPORTED;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const cudaError_t e = dtype == IM2WIN_F32
                              ? launch_conv_f32(src, filt, out, ws, s, fused, layout, cs)
                              : launch_conv_tc(src, filt, out, ws, s, fused, layout, dtype == IM2WIN_BF16, cs);
    return e == cudaSuccess ? IM2WIN_OK : IM2WIN_ERR_CUDA;
}

im2win_status transform_shape(const Shape &s, const void *x, void *win, int dtype, void *stream, int layout);

im2win_status transform_common(const void *x, void *win, int64_t N, int64_t C_i, int64_t H_i,
                               int64_t W_i, int64_t C_o, int64_t H_f, int64_t W_f, int64_t s_h,
                               int64_t s_w, int dtype, void *stream, int layout) {
    Shape s;
    im2win_status st = make_shape(s, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w);
    if (st != IM2WIN_OK) return st;
    return transform_shape(s, x, win, dtype, stream, layout);
}

im2win_status transform_shape(const Shape &s, const void *x, void *win, int dtype, void *stream, int layout) {
    const int esz = elem_size(dtype);
    if (esz == 0) return IM2WIN_ERR_INVALID_ARG;
    if (s.N == 0) return IM2WIN_OK;  // empty batch: nothing to read or write
    if (!x || !win) return IM2WIN_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(win)) return IM2WIN_ERR_MISALIGNED;
    const bool cl = layout == LAYOUT_NHWC;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (!plain(s)) {
        if (!transform_pd_supported(s, esz)) return IM2WIN_ERR_UNSUPPORTED;
        e = launch_transform_pd(x, win, s, esz, layout, cs);
    } else {
        if (!(cl ? transform_nhwc_supported(s, esz) : transform_supported(s, esz))) return IM2WIN_ERR_UNSUPPORTED;
        e = cl ? launch_transform_nhwc(x, win, s, esz, cs) : launch_transform(x, win, s, esz, cs);
    }
    return e == cudaSuccess ? IM2WIN_OK : IM2WIN_ERR_CUDA;
}

}  // namespace

extern "C" {

im2win_status im2win_workspace_size(int op, int64_t N, int64_t C_i, int64_t H_i, int64_t W_i,
                                    int64_t C_o, int64_t H_f, int64_t W_f, int64_t s_h,
                                    int64_t s_w, int dtype, size_t *bytes) {
    if (!bytes) return IM2WIN_ERR_INVALID_ARG;
    Shape s;
    im2win_status st = make_shape(s, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w);
    if (st != IM2WIN_OK) return st;
    const int esz = elem_size(dtype);
    if (esz == 0) return IM2WIN_ERR_INVALID_ARG;
    switch (op) {
        case IM2WIN_OP_TRANSFORM: *bytes = window_bytes(s, esz); return IM2WIN_OK;
        case IM2WIN_OP_CONV: *bytes = conv_ws_bytes(s, dtype, false, LAYOUT_NCHW); return IM2WIN_OK;
        case IM2WIN_OP_CONV_FUSED: *bytes = conv_ws_bytes(s, dtype, true, LAYOUT_NCHW); return IM2WIN_OK;
        case IM2WIN_OP_CONV_NHWC: *bytes = conv_ws_bytes(s, dtype, false, LAYOUT_NHWC); return IM2WIN_OK;
        case IM2WIN_OP_CONV_FUSED_NHWC: *bytes = conv_ws_bytes(s, dtype, true, LAYOUT_NHWC); return IM2WIN_OK;
        default: return IM2WIN_ERR_INVALID_ARG;
    }
}

im2win_status im2win_transform(const void *x, void *win, int64_t N, int64_t C_i, int64_t H_i,
                               int64_t W_i, int64_t C_o, int64_t H_f, int64_t W_f,
                               int64_t s_h, int64_t s_w, int dtype, void *stream) {
    return transform_common(x, win, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, dtype, stream, LAYOUT_NCHW);
}

im2win_status im2win_transform_nhwc(const void *x, void *win, int64_t N, int64_t C_i, int64_t H_i,
                                    int64_t W_i, int64_t C_o, int64_t H_f, int64_t W_f,
                                    int64_t s_h, int64_t s_w, int dtype, void *stream) {
    return transform_common(x, win, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, dtype, stream, LAYOUT_NHWC);
}

im2win_status im2win_conv(const void *win, const void *filt, void *out, void *ws,
                          size_t ws_bytes, int64_t N, int64_t C_i, int64_t H_i, int64_t W_i,
                          int64_t C_o, int64_t H_f, int64_t W_f, int64_t s_h, int64_t s_w,
                          int dtype, void *stream) {
    return conv_common(win, filt, out, ws, ws_bytes, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w,
                       dtype, stream, false, LAYOUT_NCHW);
}

im2win_status im2win_conv_fused(const void *x, const void *filt, void *out, void *ws,
                                size_t ws_bytes, int64_t N, int64_t C_i, int64_t H_i,
                                int64_t W_i, int64_t C_o, int64_t H_f, int64_t W_f,
                                int64_t s_h, int64_t s_w, int dtype, void *stream) {
    return conv_common(x, filt, out, ws, ws_bytes, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w,
                       dtype, stream, true, LAYOUT_NCHW);
}

im2win_status im2win_conv_nhwc(const void *win, const void *filt, void *out, void *ws,
                               size_t ws_bytes, int64_t N, int64_t C_i, int64_t H_i, int64_t W_i,
                               int64_t C_o, int64_t H_f, int64_t W_f, int64_t s_h, int64_t s_w,
                               int dtype, void *stream) {
    return conv_common(win, filt, out, ws, ws_bytes, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w,
                       dtype, stream, false, LAYOUT_NHWC);
}

im2win_status im2win_conv_fused_nhwc(const void *x, const void *filt, void *out, void *ws,
                                     size_t ws_bytes, int64_t N, int64_t C_i, int64_t H_i,
                                     int64_t W_i, int64_t C_o, int64_t H_f, int64_t W_f,
                                     int64_t s_h, int64_t s_w, int dtype, void *stream) {
    return conv_common(x, filt, out, ws, ws_bytes, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w,
                       dtype, stream, true, LAYOUT_NHWC);
}

// ---- padding, dilation and layout as arguments

im2win_status im2win_workspace_size_ex(int op, int64_t N, int64_t C_i, int64_t H_i, int64_t W_i,
                                       int64_t C_o, int64_t H_f, int64_t W_f, int64_t s_h, int64_t s_w,
                                       int64_t p_h, int64_t p_w, int64_t d_h, int64_t d_w, int layout,
                                       int dtype, size_t *bytes) {
    if (!bytes || (layout != IM2WIN_LAYOUT_NCHW && layout != IM2WIN_LAYOUT_NHWC)) return IM2WIN_ERR_INVALID_ARG;
    Shape s;
    im2win_status st = make_shape_pd(s, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, p_h, p_w, d_h, d_w);
    if (st != IM2WIN_OK) return st;
    const int esz = elem_size(dtype);
    if (esz == 0) return IM2WIN_ERR_INVALID_ARG;
    switch (op) {
        case IM2WIN_OP_TRANSFORM: *bytes = window_bytes(s, esz); return IM2WIN_OK;
        case IM2WIN_OP_CONV: *bytes = conv_ws_bytes(s, dtype, false, layout); return IM2WIN_OK;
        case IM2WIN_OP_CONV_FUSED: *bytes = conv_ws_bytes(s, dtype, true, layout); return IM2WIN_OK;
        default: return IM2WIN_ERR_INVALID_ARG;
    }
}

im2win_status im2win_transform_ex(const void *x, void *win, int64_t N, int64_t C_i, int64_t H_i, int64_t W_i,
                                  int64_t C_o, int64_t H_f, int64_t W_f, int64_t s_h, int64_t s_w,
                                  int64_t p_h, int64_t p_w, int64_t d_h, int64_t d_w, int layout, int dtype,
                                  void *stream) {
    if (layout != IM2WIN_LAYOUT_NCHW && layout != IM2WIN_LAYOUT_NHWC) return IM2WIN_ERR_INVALID_ARG;
    Shape s;
    im2win_status st = make_shape_pd(s, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, p_h, p_w, d_h, d_w);
    if (st != IM2WIN_OK) return st;
    return transform_shape(s, x, win, dtype, stream, layout);
}

im2win_status im2win_conv_ex(const void *win, const void *filt, void *out, void *ws, size_t ws_bytes,
                             int64_t N, int64_t C_i, int64_t H_i, int64_t W_i, int64_t C_o, int64_t H_f,
                             int64_t W_f, int64_t s_h, int64_t s_w, int64_t p_h, int64_t p_w, int64_t d_h,
                             int64_t d_w, int layout, int dtype, void *stream) {
    if (layout != IM2WIN_LAYOUT_NCHW && layout != IM2WIN_LAYOUT_NHWC) return IM2WIN_ERR_INVALID_ARG;
    Shape s;
    im2win_status st = make_shape_pd(s, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, p_h, p_w, d_h, d_w);
    if (st != IM2WIN_OK) return st;
    return conv_shape(s, win, filt, out, ws, ws_bytes, dtype, stream, false, layout);
}

im2win_status im2win_conv_fused_ex(const void *x, const void *filt, void *out, void *ws, size_t ws_bytes,
                                   int64_t N, int64_t C_i, int64_t H_i, int64_t W_i, int64_t C_o, int64_t H_f,
                                   int64_t W_f, int64_t s_h, int64_t s_w, int64_t p_h, int64_t p_w, int64_t d_h,
                                   int64_t d_w, int layout, int dtype, void *stream) {
    if (layout != IM2WIN_LAYOUT_NCHW && layout != IM2WIN_LAYOUT_NHWC) return IM2WIN_ERR_INVALID_ARG;
    Shape s;
    im2win_status st = make_shape_pd(s, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, p_h, p_w, d_h, d_w);
    if (st != IM2WIN_OK) return st;
    return conv_shape(s, x, filt, out, ws, ws_bytes, dtype, stream, true, layout);
}

im2win_status im2win_plan(int op, int64_t N, int64_t C_i, int64_t H_i, int64_t W_i, int64_t C_o,
                          int64_t H_f, int64_t W_f, int64_t s_h, int64_t s_w, int64_t p_h, int64_t p_w,
                          int64_t d_h, int64_t d_w, int layout, int dtype, int sms, im2win_plan_info *info) {
    if (!info || (layout != IM2WIN_LAYOUT_NCHW && layout != IM2WIN_LAYOUT_NHWC) ||
        (op != IM2WIN_OP_CONV && op != IM2WIN_OP_CONV_FUSED) || elem_size(dtype) == 0)
        return IM2WIN_ERR_INVALID_ARG;
    Shape s;
    im2win_status st = make_shape_pd(s, N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, p_h, p_w, d_h, d_w);
    if (st != IM2WIN_OK) return st;
    const bool fused = op == IM2WIN_OP_CONV_FUSED;
    std::memset(info, 0, sizeof(*info));
    info->tap_mode = -1;
    if (dtype == IM2WIN_F32) {
        if (!conv_f32_supported(s, fused, layout)) return IM2WIN_ERR_UNSUPPORTED;
        info->kernel = IM2WIN_KERNEL_F32;
        return IM2WIN_OK;
    }
    TcPlanInfo t;
    if (!conv_tc_plan_info(s, fused, layout, sms, t)) return IM2WIN_ERR_UNSUPPORTED;
    info->kernel = t.kernel == 1 ? IM2WIN_KERNEL_TAP : IM2WIN_KERNEL_EXPAND;
    info->tap_mode = t.tap_mode;
    info->stacked = t.stacked;
    info->rows_per_tile = t.rows_per_tile;
    info->pitch = t.pitch;
    info->tmem_columns = t.tmem_columns;
    info->tmem_read_end = t.tmem_read_end;
    info->smem_bytes = t.smem_bytes;
    info->filter_stage_taps = t.filter_stage_taps;
    info->filter_stages = t.filter_stages;
    info->slab_stages = t.slab_stages;
    info->tiles = t.tiles;
    info->grid = t.grid;
    return IM2WIN_OK;
}

const char *im2win_status_string(int status) {
    switch (status) {
        case IM2WIN_OK: return "ok";
        case IM2WIN_ERR_INVALID_ARG: return "invalid argument";
        case IM2WIN_ERR_UNSUPPORTED: return "unsupported shape";
        case IM2WIN_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case IM2WIN_ERR_WORKSPACE: return "workspace missing or too small";
        case IM2WIN_ERR_CUDA: return "CUDA error";
        case IM2WIN_ERR_TIMEOUT: return "in-kernel wait timed out";
        default: return "unknown status";
    }
}

im2win_status im2win_device_status(const void *ws, size_t ws_bytes, void *stream) {
    if (!ws || ws_bytes < kStatusBytes) return IM2WIN_ERR_WORKSPACE;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(cs) != cudaSuccess) return IM2WIN_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return IM2WIN_ERR_CUDA;
    return word == 0 ? IM2WIN_OK : static_cast<im2win_status>(word);
}

}  // extern "C"
