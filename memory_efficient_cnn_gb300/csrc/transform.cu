// im2win transformation kernel (sm_103a).
//
// win[n][ci][ho][w*H_f + r] = x[n][ci][ho*s_h + r][w]: for each channel and
// output row the H_f input rows under it are flattened column by column into
// one contiguous window row ("Im2win: Memory Efficient Convolution On SIMD
// Architectures", Abstract; "Enabling Memory-efficient Im2win Convolution with
// Multi-precision Support on GPU CUDA and Tensor Cores", Fig. 1).
//
// The transform is pure data movement and HBM-bound: the window is
// H_f/s_h times the input. Design:
//  * one CTA per (plane = n*C_i + ci, band of T output rows); the input rows
//    of the band form one contiguous range of x, staged once into shared
//    memory with 16-byte loads (rows shared by neighbouring output rows are
//    read from HBM once per band);
//  * the band's window rows are assembled in shared memory: a thread takes one
//    input column w of one output row and copies its H_f elements (one per
//    staged row) to window positions w*H_f .. w*H_f + H_f - 1, so consecutive
//    lanes read consecutive shared-memory elements;
//  * the band's output is one contiguous range of win; it leaves shared
//    memory as whole 16-byte vectors (coalesced 128-bit stores), the buffer
//    being offset so that its vectors line up with the global ones; the
//    unaligned head and tail are written element by element, so neighbouring
//    CTAs never overlap.
// The element type is the raw bit pattern (uint16_t / uint32_t), so the copy
// is bit-exact for every dtype.
#include "im2win_internal.cuh"

namespace im2win {
namespace {

constexpr int kThreads = 256;
constexpr int kSmemBudget = 56 * 1024;  // per CTA (input + output band), 4 CTAs/SM

struct TParams {
    const void *x;
    void *win;
    int64_t x_elems;      // total elements of x
    int64_t H_i, W_i, H_f, s_h, H_o;
    int64_t tiles_per_plane;
    int T;                // output rows per band
    int in_cap;           // elements reserved for the staged input band (multiple of 8)
    uint32_t L;           // W_i * H_f
};

template <typename E>
__global__ void __launch_bounds__(kThreads) transform_kernel(TParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    constexpr int V = 16 / sizeof(E);
    E *s_in = reinterpret_cast<E *>(smem_raw);
    E *s_out = s_in + p.in_cap;

    const E *__restrict__ x = static_cast<const E *>(p.x);
    E *__restrict__ win = static_cast<E *>(p.win);

    const int64_t plane = blockIdx.x / p.tiles_per_plane;
    const int64_t tile = blockIdx.x - plane * p.tiles_per_plane;
    const int64_t ho0 = tile * p.T;
    const int64_t ho1 = min(ho0 + (int64_t)p.T, p.H_o);
    const int rows_out = (int)(ho1 - ho0);
    const int rows_in = (int)((rows_out - 1) * p.s_h + p.H_f);
    const int W_i = (int)p.W_i, H_f = (int)p.H_f, s_h = (int)p.s_h;
    const int L = (int)p.L;

    // ---- stage the band's input rows: x[in0, in0 + cnt) -> s_in[lead, lead + cnt)
    const int64_t in0 = (plane * p.H_i + ho0 * p.s_h) * p.W_i;
    const int cnt = rows_in * W_i;
    const int64_t base = in0 - (in0 % V);
    const int lead = (int)(in0 - base);
    const int nvec = (lead + cnt + V - 1) / V;
    for (int v = threadIdx.x; v < nvec; v += kThreads) {
        const int64_t g = base + (int64_t)v * V;
        if (g + V <= p.x_elems) {
            *reinterpret_cast<uint4 *>(s_in + v * V) = __ldg(reinterpret_cast<const uint4 *>(x + g));
        } else {
#pragma unroll
            for (int i = 0; i < V; ++i)
                if (g + i < p.x_elems) s_in[v * V + i] = x[g + i];
        }
    }
    __syncthreads();

    // ---- assemble the window rows: s_out[olead + hl*L + w*H_f + r] = s_in[lead + (hl*s_h + r)*W_i + w]
    const int64_t o0 = (plane * p.H_o + ho0) * (int64_t)L;
    const int64_t o1 = o0 + (int64_t)rows_out * L;
    const int olead = (int)(o0 % V);
    const E *sl = s_in + lead;
    E *so = s_out + olead;
    const int items = rows_out * W_i;
    for (int it = threadIdx.x; it < items; it += kThreads) {
        const int hl = it / W_i;
        const int w = it - hl * W_i;
        const E *src = sl + hl * s_h * W_i + w;
        E *dst = so + hl * L + w * H_f;
        for (int r = 0; r < H_f; ++r) dst[r] = src[r * W_i];
    }
    __syncthreads();

    // ---- write win[o0, o1): aligned 16-byte vectors, ragged head and tail by element
    int64_t a0 = (o0 + V - 1) / V * V;
    int64_t a1 = o1 / V * V;
    if (a0 > o1) a0 = o1;
    if (a1 < a0) a1 = a0;
    const int head = (int)(a0 - o0), tail = (int)(o1 - a1);
    if ((int)threadIdx.x < head) win[o0 + threadIdx.x] = so[threadIdx.x];
    if ((int)threadIdx.x < tail) win[a1 + threadIdx.x] = so[(int)(a1 - o0) + threadIdx.x];
    const int nbody = (int)((a1 - a0) / V);
    const uint4 *sv = reinterpret_cast<const uint4 *>(so + (a0 - o0));  // 16-byte aligned by olead
    uint4 *gv = reinterpret_cast<uint4 *>(win + a0);
    for (int v = threadIdx.x; v < nbody; v += kThreads) gv[v] = sv[v];
}

}  // namespace

cudaError_t launch_transform(const void *x, void *win, const Shape &s, int esz, cudaStream_t st) {
    if (s.N == 0) return cudaSuccess;
    const int64_t L = s.W_i * s.H_f;
    // bytes of a band of T output rows: staged input rows + assembled window rows
    auto band_bytes = [&](int64_t T) {
        const int64_t in_elems = ((T - 1) * s.s_h + s.H_f) * s.W_i + 16;
        return (in_elems + 8) / 8 * 8 * esz + (T * L + 16) * esz;
    };
    int64_t T = 1;
    while (T < s.H_o && band_bytes(T + 1) <= kSmemBudget) ++T;
    // balance the bands of a plane
    const int64_t tiles = (s.H_o + T - 1) / T;
    T = (s.H_o + tiles - 1) / tiles;
    const int64_t in_elems = ((T - 1) * s.s_h + s.H_f) * s.W_i + 16;

    TParams p;
    p.x = x;
    p.win = win;
    p.x_elems = s.N * s.C_i * s.H_i * s.W_i;
    p.H_i = s.H_i;
    p.W_i = s.W_i;
    p.H_f = s.H_f;
    p.s_h = s.s_h;
    p.H_o = s.H_o;
    p.tiles_per_plane = tiles;
    p.T = (int)T;
    p.in_cap = (int)((in_elems + 8) / 8 * 8);
    p.L = (uint32_t)L;
    const size_t smem = (size_t)band_bytes(T);

    const int64_t blocks = s.N * s.C_i * tiles;
    cudaError_t e;
    if (esz == 2) {
        e = cudaFuncSetAttribute(transform_kernel<uint16_t>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        transform_kernel<uint16_t><<<(unsigned)blocks, kThreads, smem, st>>>(p);
    } else {
        e = cudaFuncSetAttribute(transform_kernel<uint32_t>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        transform_kernel<uint32_t><<<(unsigned)blocks, kThreads, smem, st>>>(p);
    }
    return cudaGetLastError();
}

// The transform stages at least one output row (its H_f input rows and its
// window row) and indexes a band with 32-bit arithmetic.
bool transform_supported(const Shape &s, int esz) {
    // one output row: H_f staged rows plus one window row
    const int64_t one_row = (s.H_f * s.W_i + 32) * esz + (s.W_i * s.H_f + 16) * esz;
    return one_row <= 200 * 1024 && s.W_i * s.H_f * s.H_o < (1ll << 31) &&
           s.N * s.C_i * s.H_o < (1ll << 31);
}

}  // namespace im2win
