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
constexpr int kSmemBudget = 40 * 1024;  // per CTA (input + output band), 5 CTAs/SM

struct TParams {
    const void *x;
    void *win;
    int64_t x_elems;      // total elements of x
    int64_t H_i, W_i, H_f, s_h, H_o;
    int64_t tiles_per_plane;
    int T;                // output rows per band
    int Wt, ctiles;       // columns per tile and column tiles per band (1 unless a row is too wide)
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

    const int64_t tile_id = blockIdx.x / p.ctiles;
    const int ct = (int)(blockIdx.x - tile_id * p.ctiles);
    const int64_t plane = tile_id / p.tiles_per_plane;
    const int64_t tile = tile_id - plane * p.tiles_per_plane;
    const int64_t ho0 = tile * p.T;
    const int64_t ho1 = min(ho0 + (int64_t)p.T, p.H_o);
    const int rows_out = (int)(ho1 - ho0);
    const int rows_in = (int)((rows_out - 1) * p.s_h + p.H_f);
    const int W_i = (int)p.W_i, H_f = (int)p.H_f, s_h = (int)p.s_h;
    const int L = (int)p.L;
    const int w0 = ct * p.Wt;
    const int Wc = min(p.Wt, W_i - w0);  // columns of this tile

    // ---- stage the band's input rows (columns [w0, w0 + Wc)) in s_in, row pitch Wc
    int lead = 0;
    if (p.ctiles == 1) {
        // whole rows: one contiguous range of x, x[in0, in0 + cnt) -> s_in[lead, lead + cnt)
        const int64_t in0 = (plane * p.H_i + ho0 * p.s_h) * p.W_i;
        const int cnt = rows_in * W_i;
        const int64_t base = in0 - (in0 % V);
        lead = (int)(in0 - base);
        const int nvec = (lead + cnt + V - 1) / V;
        // vectors that lie wholly inside x: four loads in flight per thread
        const int64_t inside = (p.x_elems - base) / V;
        const int nfull = inside < (int64_t)nvec ? (int)inside : nvec;
        const uint4 *gx = reinterpret_cast<const uint4 *>(x + base);
        uint4 *sx = reinterpret_cast<uint4 *>(s_in);
        int v = threadIdx.x;
        for (; v + 3 * kThreads < nfull; v += 4 * kThreads) {
            const uint4 r0 = __ldg(gx + v), r1 = __ldg(gx + v + kThreads);
            const uint4 r2 = __ldg(gx + v + 2 * kThreads), r3 = __ldg(gx + v + 3 * kThreads);
            sx[v] = r0;
            sx[v + kThreads] = r1;
            sx[v + 2 * kThreads] = r2;
            sx[v + 3 * kThreads] = r3;
        }
        for (; v < nfull; v += kThreads) sx[v] = __ldg(gx + v);
        // the last, partial vector of x (if any)
        for (int e = nfull * V + (int)threadIdx.x; e < nvec * V; e += kThreads)
            if (base + e < p.x_elems) s_in[e] = x[base + e];
    } else {
        // a column segment of each input row (rows too wide for one band)
        const int64_t row0 = (plane * p.H_i + ho0 * p.s_h) * p.W_i + w0;
        for (int e = threadIdx.x; e < rows_in * Wc; e += kThreads) {
            const int lr = e / Wc, c = e - lr * Wc;
            s_in[e] = x[row0 + (int64_t)lr * p.W_i + c];
        }
    }
    __syncthreads();

    // ---- assemble the window rows: s_out[olead + hl*L + (w-w0)*H_f + r] = s_in[lead + (hl*s_h + r)*Wc + w - w0]
    // (a band of whole rows is one contiguous output range; a column tile is one output row)
    const int64_t o0 = (plane * p.H_o + ho0) * (int64_t)L + (int64_t)w0 * H_f;
    const int64_t o1 = o0 + (p.ctiles == 1 ? (int64_t)rows_out * L : (int64_t)Wc * H_f);
    const int olead = (int)(o0 % V);
    const E *sl = s_in + lead;
    E *so = s_out + olead;
    const int items = rows_out * Wc;
    for (int it = threadIdx.x; it < items; it += kThreads) {
        const int hl = it / Wc;
        const int w = it - hl * Wc;
        const E *src = sl + hl * s_h * Wc + w;
        E *dst = so + hl * L + w * H_f;
        for (int r = 0; r < H_f; ++r) dst[r] = src[r * Wc];
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
    // bytes of a band of T output rows of Wt columns: staged input rows + assembled window rows
    auto band_bytes = [&](int64_t T, int64_t Wt) {
        const int64_t in_elems = ((T - 1) * s.s_h + s.H_f) * Wt + 16;
        return (in_elems + 8) / 8 * 8 * esz + (T * Wt * s.H_f + 16) * esz;
    };
    int64_t T = 1, Wt = s.W_i;
    if (band_bytes(1, Wt) > kSmemBudget) {
        // rows too wide: one output row per band, split into column tiles
        while (Wt > 8 && band_bytes(1, Wt) > kSmemBudget) Wt = (Wt + 1) / 2;
    } else {
        while (T < s.H_o && band_bytes(T + 1, Wt) <= kSmemBudget) ++T;
    }
    const int64_t ctiles = (s.W_i + Wt - 1) / Wt;
    // balance the bands of a plane
    const int64_t tiles = (s.H_o + T - 1) / T;
    T = (s.H_o + tiles - 1) / tiles;
    const int64_t in_elems = ((T - 1) * s.s_h + s.H_f) * Wt + 16;

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
    p.Wt = (int)Wt;
    p.ctiles = (int)ctiles;
    p.in_cap = (int)((in_elems + 8) / 8 * 8);
    p.L = (uint32_t)L;
    const size_t smem = (size_t)band_bytes(T, Wt);

    const int64_t blocks = s.N * s.C_i * tiles * ctiles;
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

// The transform indexes a band with 32-bit arithmetic and launches one CTA per
// (plane, band, column tile).
bool transform_supported(const Shape &s, int esz) {
    // the narrowest tile (8 columns of one output row) must fit in shared memory
    const int64_t narrow = ((s.H_f * 8 + 24) + (8 * s.H_f + 16)) * esz;
    return narrow <= 200 * 1024 && s.W_i * s.H_f * s.H_o < (1ll << 31) &&
           s.N * s.C_i * s.H_o * ((s.W_i + 7) / 8) < (1ll << 31);
}

}  // namespace im2win
