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
//  * the band's output is one contiguous range of win; every thread writes
//    whole 16-byte vectors of it (coalesced, 128-bit stores), assembling each
//    vector from shared memory; the unaligned head and tail of the range are
//    written element by element, so neighbouring CTAs never overlap;
//  * index arithmetic inside a band is 32-bit with multiply-high division.
// The element type is the raw bit pattern (uint16_t / uint32_t), so the copy
// is bit-exact for every dtype.
#include "im2win_internal.cuh"

namespace im2win {
namespace {

constexpr int kThreads = 256;
constexpr int kSmemBudget = 40 * 1024;  // per CTA, leaves room for 5 CTAs/SM

struct TParams {
    const void *x;
    void *win;
    int64_t x_elems;      // total elements of x
    int64_t H_i, W_i, H_f, s_h, H_o;
    int64_t tiles_per_plane;
    int T;                // output rows per band
    uint32_t L;           // W_i * H_f
    FastDiv div_L, div_Hf;
};

template <typename E>
__global__ void __launch_bounds__(kThreads) transform_kernel(TParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    E *s = reinterpret_cast<E *>(smem_raw);
    constexpr int V = 16 / sizeof(E);

    const E *__restrict__ x = static_cast<const E *>(p.x);
    E *__restrict__ win = static_cast<E *>(p.win);

    const int64_t plane = blockIdx.x / p.tiles_per_plane;
    const int64_t tile = blockIdx.x - plane * p.tiles_per_plane;
    const int64_t ho0 = tile * p.T;
    const int64_t ho1 = min(ho0 + (int64_t)p.T, p.H_o);
    const int rows_out = (int)(ho1 - ho0);
    const int rows_in = (int)((rows_out - 1) * p.s_h + p.H_f);
    const int W_i = (int)p.W_i, H_f = (int)p.H_f, s_h = (int)p.s_h;

    // ---- stage the band's input rows: x[in0, in0 + cnt) -> s[lead, lead + cnt)
    const int64_t in0 = (plane * p.H_i + ho0 * p.s_h) * p.W_i;
    const int cnt = rows_in * W_i;
    const int64_t base = in0 - (in0 % V);
    const int lead = (int)(in0 - base);
    const int nvec = (lead + cnt + V - 1) / V;
    for (int v = threadIdx.x; v < nvec; v += kThreads) {
        const int64_t g = base + (int64_t)v * V;
        if (g + V <= p.x_elems) {
            *reinterpret_cast<uint4 *>(s + v * V) = __ldg(reinterpret_cast<const uint4 *>(x + g));
        } else {
#pragma unroll
            for (int i = 0; i < V; ++i)
                if (g + i < p.x_elems) s[v * V + i] = x[g + i];
        }
    }
    __syncthreads();

    // ---- write the band's window rows: win[o0, o0 + rows_out*L)
    const uint32_t L = p.L;
    const int64_t o0 = (plane * p.H_o + ho0) * (int64_t)L;
    const int64_t o1 = o0 + (int64_t)rows_out * L;
    int64_t a0 = (o0 + V - 1) / V * V;
    int64_t a1 = o1 / V * V;
    if (a0 > o1) a0 = o1;
    if (a1 < a0) a1 = a0;
    const E *sl = s + lead;

    // element at local window index q (0 <= q < rows_out*L)
    auto fetch = [&](uint32_t q) -> E {
        uint32_t hl = fdiv(q, p.div_L);
        uint32_t rem = q - hl * L;
        uint32_t w = fdiv(rem, p.div_Hf);
        uint32_t r = rem - w * (uint32_t)H_f;
        return sl[((int)hl * s_h + (int)r) * W_i + (int)w];
    };

    // head and tail (fewer than V elements each)
    const int head = (int)(a0 - o0), tail = (int)(o1 - a1);
    if ((int)threadIdx.x < head) win[o0 + threadIdx.x] = fetch(threadIdx.x);
    if ((int)threadIdx.x < tail) {
        uint32_t q = (uint32_t)(a1 - o0) + threadIdx.x;
        win[a1 + threadIdx.x] = fetch(q);
    }

    // aligned body: whole 16-byte vectors
    const uint32_t nbody = (uint32_t)((a1 - a0) / V);
    for (uint32_t v = threadIdx.x; v < nbody; v += kThreads) {
        uint32_t q = (uint32_t)(a0 - o0) + v * V;
        uint32_t hl = fdiv(q, p.div_L);
        uint32_t rem = q - hl * L;
        uint32_t w = fdiv(rem, p.div_Hf);
        uint32_t r = rem - w * (uint32_t)H_f;
        int row = (int)hl * s_h + (int)r;
        int col = (int)w;
        union { uint4 u; E e[V]; } pack;
#pragma unroll
        for (int i = 0; i < V; ++i) {
            pack.e[i] = sl[row * W_i + col];
            // advance (r, w, hl) by one window element
            ++r;
            ++row;
            if ((int)r == H_f) {
                r = 0;
                row -= H_f;
                ++col;
                if (col == W_i) {
                    col = 0;
                    row += s_h;
                }
            }
        }
        *reinterpret_cast<uint4 *>(win + a0 + (int64_t)v * V) = pack.u;
    }
}

}  // namespace

cudaError_t launch_transform(const void *x, void *win, const Shape &s, int esz, cudaStream_t st) {
    if (s.N == 0) return cudaSuccess;
    const int64_t row_bytes = s.W_i * esz;
    // largest band whose staged input fits the budget (at least one output row)
    int64_t T = (kSmemBudget / row_bytes - s.H_f) / s.s_h + 1;
    if (T < 1) T = 1;
    if (T > s.H_o) T = s.H_o;
    // balance the bands of a plane
    const int64_t tiles = (s.H_o + T - 1) / T;
    T = (s.H_o + tiles - 1) / tiles;
    const int64_t rows_in = (T - 1) * s.s_h + s.H_f;
    const size_t smem = (size_t)(rows_in * row_bytes + 16);

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
    p.L = (uint32_t)(s.W_i * s.H_f);
    p.div_L = make_fastdiv(p.L);
    p.div_Hf = make_fastdiv((uint32_t)s.H_f);

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

// The transform stages at least one output row's input rows (H_f rows of
// W_i elements) and indexes a band with 32-bit arithmetic.
bool transform_supported(const Shape &s, int esz) {
    const int64_t one_row = s.H_f * s.W_i * esz + 16;
    return one_row <= 200 * 1024 && s.W_i * s.H_f * s.H_o < (1ll << 31) &&
           s.N * s.C_i * s.H_o < (1ll << 31);
}

}  // namespace im2win
