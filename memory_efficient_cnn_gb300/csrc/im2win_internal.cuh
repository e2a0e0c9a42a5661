// Internal declarations shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "im2win.h"

namespace im2win {

// Problem shape with the valid-convolution output extents derived
// (Table I of the GPU im2win paper: no padding, floor division).
struct Shape {
    int64_t N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w, H_o, W_o;
};

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

// ---- launchers (each returns cudaSuccess or the launch error) ----

// Window transform of esz-byte elements.
cudaError_t launch_transform(const void *x, void *win, const Shape &s, int esz, cudaStream_t st);
bool transform_supported(const Shape &s, int esz);

// fp32 CUDA-core convolution; from_x selects the fused variant that gathers
// from the NCHW input instead of the window tensor. ws holds the status block
// followed by the re-laid filter.
size_t conv_f32_filter_bytes(const Shape &s);
bool conv_f32_supported(const Shape &s, bool from_x);
cudaError_t launch_conv_f32(const void *src, const void *filt, void *out, void *ws,
                            const Shape &s, bool from_x, cudaStream_t st);

// fp16/bf16 tensor-core convolution (tcgen05). mode: 0 = from window tensor,
// 1 = fused from NCHW input.
size_t conv_tc_filter_bytes(const Shape &s, bool fused);
bool conv_tc_supported(const Shape &s, bool fused);
cudaError_t launch_conv_tc(const void *src, const void *filt, void *out, void *ws,
                           const Shape &s, bool fused, bool bf16, cudaStream_t st);

}  // namespace im2win
