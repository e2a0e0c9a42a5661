// Fused convolution for callers that cannot allocate a workspace.
//
// Some callers only ever hold the input and output buffers: a plugin slot in
// a host framework that hands over tensor pointers and nothing else, or code
// running where a cudaMalloc is not acceptable because it may synchronise the
// device and stall other work. This entry point gives them the fused
// convolution without a workspace argument: the scratch the kernels need (a
// 256-byte status block and the re-laid filter) lives in one fixed array
// compiled into the library, in device memory of every GPU that loads it,
// for as long as the process runs.
//
// Properties a caller must know:
//  * the array holds IM2WIN_NOALLOC_SCRATCH_BYTES; problems whose fused
//    workspace is larger are rejected with IM2WIN_ERR_WORKSPACE before any
//    work is queued;
//  * every call looks up the array's device address on the current device
//    (cudaGetSymbolAddress), so a device reset, which may move the array, is
//    harmless; the first call on a device loads the library's module there:
//    make one call before capturing the stream into a graph;
//  * all calls share the array, which keeps whatever the last call left in
//    it: every call re-lays the filter and clears the status word itself, and
//    two calls whose kernels overlap on the GPU (different streams, no
//    ordering) race on it and may produce wrong results;
//  * nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include "im2win_internal.cuh"

namespace {

constexpr size_t kScratchBytes = IM2WIN_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of the scratch array on the current device.
im2win_status scratch_on_current_device(void **addr) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return IM2WIN_ERR_CUDA;
    *addr = p;
    return IM2WIN_OK;
}

}  // namespace

extern "C" im2win_status im2win_conv_fused_noalloc(const void *x, const void *filt, void *out,
                                                   int64_t N, int64_t C_i, int64_t H_i, int64_t W_i,
                                                   int64_t C_o, int64_t H_f, int64_t W_f,
                                                   int64_t s_h, int64_t s_w, int dtype, void *stream) {
    size_t need = 0;
    im2win_status st = im2win_workspace_size(IM2WIN_OP_CONV_FUSED, N, C_i, H_i, W_i, C_o, H_f, W_f,
                                             s_h, s_w, dtype, &need);
    if (st != IM2WIN_OK) return st;
    if (need > kScratchBytes) return IM2WIN_ERR_WORKSPACE;
    if (N == 0) return IM2WIN_OK;
    void *scratch = nullptr;
    st = scratch_on_current_device(&scratch);
    if (st != IM2WIN_OK) return st;
    return im2win_conv_fused(x, filt, out, scratch, kScratchBytes, N, C_i, H_i, W_i, C_o, H_f, W_f,
                             s_h, s_w, dtype, stream);
}
