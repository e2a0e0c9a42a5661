"""im2win convolution for GB300 (sm_103a): a C-ABI CUDA library and its binding.

The library (libim2win.so, built from csrc/ by build.build()) implements the
im2win transformation and convolution of "Im2win: Memory Efficient Convolution
On SIMD Architectures" and "Enabling Memory-efficient Im2win Convolution with
Multi-precision Support on GPU CUDA and Tensor Cores": a window transform, an
fp32 CUDA-core convolution, an fp16/bf16 tensor-core (tcgen05) convolution and
a fused variant that never writes the window tensor, for NCHW and for
channels-last (NHWC) tensors. This package is the thin Python binding over it.
"""
from ._binding import (  # noqa: F401
    BF16, EXPORTS, F16, F32, NOALLOC_SCRATCH_BYTES, OP_CONV, OP_CONV_FUSED, OP_CONV_FUSED_NHWC, OP_CONV_NHWC,
    OP_TRANSFORM, Im2winError,
    conv, conv_fused, conv_fused_nhwc, conv_nhwc, im2win_conv, im2win_conv_fused, im2win_conv_fused_nhwc,
    im2win_conv_fused_noalloc, im2win_conv_nhwc, im2win_device_status, im2win_status_string,
    im2win_transform, im2win_transform_nhwc,
    im2win_workspace_size, lib, library_path, out_hw, status_string, transform, transform_nhwc, workspace,
    NCHW, NHWC, conv_ex, conv_fused_ex, im2win_conv_ex, im2win_conv_fused_ex, im2win_transform_ex,
    im2win_workspace_size_ex, out_hw_pd, transform_ex,
    KERNEL_EXPAND, KERNEL_F32, KERNEL_TAP, PlanInfo, im2win_plan)
