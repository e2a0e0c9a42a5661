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
//  * a CTA owns a contiguous piece of the work: several whole planes
//    (plane = n*C_i + ci) when a plane is small, else a band of T output rows
//    of one plane, else (rows too wide) a column segment of one output row.
//    The input rows under that piece form one contiguous range of x, staged
//    once into shared memory with 16-byte loads (rows shared by neighbouring
//    output rows are read from HBM once per piece);
//  * the piece's output is one contiguous range of win. Each thread builds
//    whole 16-byte output vectors, aligned to the global ones, in registers:
//    it walks the window positions of its vector (window row, column w, row
//    offset r), gathers each element from the staged rows and stores the
//    vector straight to win (coalesced 128-bit stores across the warp). The
//    unaligned head and tail of the range are written element by element, so
//    neighbouring CTAs never overlap.
//  * 16-bit elements in rows of whole 16-byte vectors (W_i a multiple of 8)
//    skip the staging: a thread loads the H_f vectors under 8 columns of a
//    window row and interleaves them in registers (transform_rows16), which
//    replaces 8 gathered 2-byte shared-memory loads per output vector by two
//    byte permutes per output word.
// The element type is the raw bit pattern (uint16_t / uint32_t), so the copy
// is bit-exact for every dtype.
#include <algorithm>
#include <map>
#include <mutex>
#include <utility>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "im2win_internal.cuh"
#include "tc_ptx.cuh"

namespace im2win {
namespace {

constexpr int kThreads = 256;
constexpr int kSmemBudget = 32 * 1024;  // staged input band per CTA (up to 7 CTAs/SM)

struct TParams {
    const void *x;
    void *win;
    int64_t x_elems;      // total elements of x
    int64_t n_planes;     // N * C_i
    int64_t H_i, W_i, H_f, s_h, H_o;
    int64_t tiles_per_plane;
    int PPC;              // planes per CTA (> 1 only when whole planes fit)
    int T;                // output rows per band (H_o for whole planes)
    int RP;               // output rows per staged plane (H_o for whole planes, else T)
    int Wt, ctiles;       // columns per tile and column tiles per band (1 unless a row is too wide)
    uint32_t L;           // W_i * H_f
    int in_cap;           // elements reserved for the staged input (the offset table follows)
    int flip_bit;         // 16-bit gathers: lanes with this bit of their lane index set gather
                          // their vector's elements in the order i ^ 2 (-1: none)
    FastDiv div_L, div_Hf, div_RP;
};

constexpr int kMaxTableHf = 32;

template <typename E, bool TABLE>
__global__ void __launch_bounds__(kThreads) transform_kernel(TParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    constexpr int V = 16 / sizeof(E);
    E *s_in = reinterpret_cast<E *>(smem_raw);
    // offT[r0][i]: staged offset of element i of a vector whose first element is at
    // row offset r0 of column w, from column w's top: ((r0 + i) % H_f) * Wc + (r0 + i) / H_f
    int *offT = reinterpret_cast<int *>(smem_raw + (size_t)p.in_cap * sizeof(E));

    const E *__restrict__ x = static_cast<const E *>(p.x);
    E *__restrict__ win = static_cast<E *>(p.win);

    const int64_t tile_id = blockIdx.x / p.ctiles;
    const int ct = (int)(blockIdx.x - tile_id * p.ctiles);
    const int64_t group = tile_id / p.tiles_per_plane;
    const int64_t tile = tile_id - group * p.tiles_per_plane;
    const int64_t plane0 = group * p.PPC;
    const int nplanes = (int)min((int64_t)p.PPC, p.n_planes - plane0);
    const int64_t ho0 = tile * p.T;
    const int64_t ho1 = min(ho0 + (int64_t)p.T, p.H_o);
    const int rows_out = (int)(ho1 - ho0);               // output rows per plane of the piece
    const int rows_in = (int)((rows_out - 1) * p.s_h + p.H_f);
    const int W_i = (int)p.W_i, H_f = (int)p.H_f, s_h = (int)p.s_h;
    const int L = (int)p.L;
    const int w0 = ct * p.Wt;
    const int Wc = min(p.Wt, W_i - w0);  // columns of this tile
    const int plane_in = (int)p.H_i * Wc;  // staged elements between planes (whole planes only)

    // ---- stage the piece's input rows (columns [w0, w0 + Wc)) in s_in, row pitch Wc
    int lead = 0;
    if (p.ctiles == 1) {
        // whole rows: one contiguous range of x, x[in0, in0 + cnt) -> s_in[lead, lead + cnt)
        const int64_t in0 = (plane0 * p.H_i + ho0 * p.s_h) * p.W_i;
        const int cnt = (nplanes - 1) * plane_in + rows_in * W_i;
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
        const int64_t row0 = (plane0 * p.H_i + ho0 * p.s_h) * p.W_i + w0;
        for (int e = threadIdx.x; e < rows_in * Wc; e += kThreads) {
            const int lr = e / Wc, c = e - lr * Wc;
            s_in[e] = x[row0 + (int64_t)lr * p.W_i + c];
        }
    }
    if (TABLE) {
        for (int e = threadIdx.x; e < H_f * V; e += kThreads) {
            const int r0 = e / V, i = e - r0 * V;
            offT[e] = ((r0 + i) % H_f) * Wc + (r0 + i) / H_f;
        }
    }
    __syncthreads();

    // ---- write win[o0, o1): the piece's window rows (a column tile: one row segment)
    const int64_t o0 = (plane0 * p.H_o + ho0) * (int64_t)L + (int64_t)w0 * H_f;
    const int64_t o1 = o0 + (p.ctiles == 1 ? (int64_t)nplanes * rows_out * L : (int64_t)Wc * H_f);
    const E *sl = s_in + lead;
    const int rstep = s_h * Wc;  // staged elements between consecutive window rows of a plane
    // staged index of the first element of window row gh of the piece
    auto row_base = [&](int gh) -> int {
        const int pl = (int)fdiv((uint32_t)gh, p.div_RP);
        return pl * plane_in + (gh - pl * p.RP) * rstep;
    };
    // position q of the range -> (window row gh, column w, row offset r) and staged index
    int gh, w, r;
    auto locate = [&](int q) -> int {
        gh = p.ctiles == 1 ? (int)fdiv((uint32_t)q, p.div_L) : 0;
        const int rem = q - gh * L;
        w = (int)fdiv((uint32_t)rem, p.div_Hf);
        r = rem - w * H_f;
        return row_base(gh) + r * Wc + w;
    };
    int64_t a0 = (o0 + V - 1) / V * V;
    int64_t a1 = o1 / V * V;
    if (a0 > o1) a0 = o1;
    if (a1 < a0) a1 = a0;
    const int head = (int)(a0 - o0), tail = (int)(o1 - a1);
    if ((int)threadIdx.x < head + tail) {
        const int q = (int)threadIdx.x < head ? (int)threadIdx.x : (int)(a1 - o0) + (int)threadIdx.x - head;
        win[o0 + q] = sl[locate(q)];
    }
    const int nbody = (int)((a1 - a0) / V);
    uint4 *gv = reinterpret_cast<uint4 *>(win + a0);
    const int q_body = (int)(a0 - o0);
    const int Lw = p.ctiles == 1 ? L : Wc * H_f;  // window row length within the piece
    // 16-bit elements: the lanes whose flip bit is set gather element i ^ 2 at step i,
    // so that at each step the warp's 2-byte shared loads fall in fewer banks twice
    // over; the word pairs of their vector are swapped back before the store
    const bool flip = V == 8 && p.flip_bit >= 0 && ((threadIdx.x >> p.flip_bit) & 1) != 0;
    const int fx = flip ? 2 : 0;
    for (int v = threadIdx.x; v < nbody; v += kThreads) {
        int idx = locate(q_body + v * V);
        uint32_t e[V];
        bool swapped = false;  // e[] holds the elements in the flipped order
        if (TABLE && w * H_f + r + V <= Lw) {
            // the vector stays in one window row: element i is at a fixed offset from
            // the top of column w, given by the table row of r
            const int top = idx - r * Wc;
            int o[V];
#pragma unroll
            for (int j = 0; j < V / 4; ++j) {
                const int4 t = reinterpret_cast<const int4 *>(offT + r * V)[j];
                o[4 * j] = t.x;
                o[4 * j + 1] = t.y;
                o[4 * j + 2] = t.z;
                o[4 * j + 3] = t.w;
            }
            if (V == 8) {
                // element i ^ fx at step i (the offsets' order only)
#pragma unroll
                for (int i = 0; i < V; ++i) e[i] = (uint32_t)sl[top + (fx ? o[i ^ 2] : o[i])];
                swapped = fx != 0;
            } else {
#pragma unroll
                for (int i = 0; i < V; ++i) e[i] = (uint32_t)sl[top + o[i]];
            }
        } else if (!TABLE && H_f >= V && w * H_f + r + V <= Lw) {
            // H_f >= V and one window row: the vector is the rest of column w and at
            // most the start of column w + 1, so its elements' staged indices are
            // independent of one another
            // element i: idx + i*Wc in column w, or that minus (H_f*Wc - 1) once
            // r + i reaches the next column
            const int wrap = H_f * Wc - 1;
            const int th = H_f - r;
            const E *s0 = sl + idx;
#pragma unroll
            for (int i = 0; i < V; ++i) {
                const int j = i ^ fx;  // the element gathered at step i
                e[i] = (uint32_t)s0[j * Wc - (j >= th ? wrap : 0)];
            }
            swapped = fx != 0;
        } else {
#pragma unroll
            for (int i = 0; i < V; ++i) {
                e[i] = (uint32_t)sl[idx];
                // next window position: r + 1, else the next column, else the next window row
                if (++r < H_f) {
                    idx += Wc;
                } else if (++w < Wc) {
                    r = 0;
                    idx += 1 - (H_f - 1) * Wc;
                } else if (i + 1 < V) {
                    r = 0;
                    w = 0;
                    idx = row_base(++gh);
                }
            }
        }
        uint4 out;
        if (V == 8) {
            out = make_uint4(__byte_perm(e[0], e[1], 0x5410), __byte_perm(e[2], e[3], 0x5410),
                             __byte_perm(e[4], e[5], 0x5410), __byte_perm(e[6], e[7], 0x5410));
            // flipped order: e[i] is element i ^ 2, i.e. the vector's words 0,1 and 2,3 swapped
            if (swapped) out = make_uint4(out.y, out.x, out.w, out.z);
        } else {
            out = make_uint4(e[0], e[1], e[2], e[3]);
        }
        gv[v] = out;
    }
}

// 16-bit elements, W_i a multiple of 8 (every input row and window row starts
// on a 16-byte boundary) and H_f at most kMaxRowsHf: an item is one 8-column
// group g of one window row (plane, ho). Its window positions are the 8*H_f
// consecutive elements win[plane][ho][8g*H_f + e], e = c*H_f + r, holding
// x[plane][ho*s_h + r][8g + c]: the H_f input vectors under the group, read
// with one 16-byte load each, interleaved in registers (two elements per byte
// permute, all indices fixed at compile time) into H_f output vectors.
// Consecutive items are consecutive in win, so a warp's 32 items are one
// contiguous range of 32*H_f vectors: each thread puts its vectors in the
// warp's staging area, and the warp stores the range with 16-byte stores that
// are contiguous across its lanes. For s_h = 1 the lanes' loads of one r are
// contiguous too (the rows of a plane follow one another in x). (For 32-bit
// elements the staged kernel below is as fast: its vectors need no gathers.)
constexpr int kMaxRowsHf = 12;

struct TRParams {
    const uint4 *x;
    uint4 *win;
    int items;            // N * C_i * H_o * (W_i / 8)
    int H_i, s_h;
    int rvec;             // 16-byte vectors per input row (W_i / 8)
    FastDiv div_G, div_Ho;  // column groups per window row, output rows per plane
};

template <int HF>
__global__ void __launch_bounds__(kThreads) transform_rows16(TRParams p) {
    extern __shared__ uint4 tr_stage[];  // [warp][32 * HF]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint4 *stage = tr_stage + warp * 32 * HF;
    const int item0 = (blockIdx.x * (kThreads / 32) + warp) * 32;  // the warp's first item
    if (item0 >= p.items) return;
    const int item = item0 + lane;
    uint32_t in[HF][4];
    if (item < p.items) {
        const int wr = (int)fdiv((uint32_t)item, p.div_G);  // window row = plane*H_o + ho
        const int g = item - wr * (int)p.div_G.d;
        const int plane = (int)fdiv((uint32_t)wr, p.div_Ho);
        const int ho = wr - plane * (int)p.div_Ho.d;
        const uint4 *src = p.x + ((int64_t)plane * p.H_i + (int64_t)ho * p.s_h) * p.rvec + g;
#pragma unroll
        for (int r = 0; r < HF; ++r) {
            const uint4 v = __ldg(src + (int64_t)r * p.rvec);
            in[r][0] = v.x;
            in[r][1] = v.y;
            in[r][2] = v.z;
            in[r][3] = v.w;
        }
    } else {
#pragma unroll
        for (int r = 0; r < HF; ++r) in[r][0] = in[r][1] = in[r][2] = in[r][3] = 0u;
    }
#pragma unroll
    for (int i = 0; i < HF; ++i) {
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            // elements e = 8i + 2k and e + 1, element (c, r) being half c % 2 of word
            // c / 2 of input vector r
            const int e0 = 8 * i + 2 * k, e1 = e0 + 1;
            const int c0 = e0 / HF, r0 = e0 % HF, c1 = e1 / HF, r1 = e1 % HF;
            const uint32_t sel = (uint32_t)((2 * (c0 & 1)) | ((2 * (c0 & 1) + 1) << 4) |
                                            ((4 + 2 * (c1 & 1)) << 8) | ((5 + 2 * (c1 & 1)) << 12));
            o[k] = __byte_perm(in[r0][c0 >> 1], in[r1][c1 >> 1], sel);
        }
        stage[lane * HF + i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    __syncwarp();
    const int nvec = min(32, p.items - item0) * HF;
    uint4 *dst = p.win + (int64_t)item0 * HF;
    for (int j = lane; j < nvec; j += 32) dst[j] = stage[j];
}

// The lane bit whose lanes gather in the flipped order (-1: none) for 16-bit
// vectors over rows of pitch Wc and H_f rows: a model of the gather's
// shared-memory wavefronts (most distinct 4-byte words one bank serves, per
// warp and step) over 128 warps' worth of consecutive vectors, for no flip and
// for a flip on each of the lane bits 0..4; the fewest wins (ties: no flip).
static int flip_bit_for(int64_t Wc, int64_t H_f) {
    static std::mutex mu;
    static std::map<std::pair<int64_t, int64_t>, int> cache;
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_pair(Wc, H_f);
    const auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    auto cost = [&](int bit) {
        int64_t total = 0;
        for (int64_t v0 = 0; v0 < 128 * 32; v0 += 32) {
            for (int t = 0; t < 8; ++t) {
                int64_t words[32];
                int per_bank[32] = {0};
                for (int l = 0; l < 32; ++l) {
                    const int i = (bit >= 0 && ((l >> bit) & 1)) ? (t ^ 2) : t;
                    const int64_t q = 8 * (v0 + l) + i;
                    const int64_t w = q / H_f, r = q - w * H_f;
                    words[l] = (r * Wc + w) / 2;
                }
                for (int l = 0; l < 32; ++l) {
                    bool seen = false;
                    for (int l2 = 0; l2 < l; ++l2) seen = seen || words[l2] == words[l];
                    if (!seen) ++per_bank[words[l] % 32];
                }
                int mx = 0;
                for (int b = 0; b < 32; ++b) mx = std::max(mx, per_bank[b]);
                total += mx;
            }
        }
        return total;
    };
    int best = -1;
    int64_t best_cost = cost(-1);
    for (int bit = 0; bit < 5; ++bit) {
        const int64_t c = cost(bit);
        if (c < best_cost) { best_cost = c; best = bit; }
    }
    cache[key] = best;
    return best;
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    return n;
}

}  // namespace

// Whether the register-interleave kernel covers the shape (and the buffers'
// alignment).
static bool rows16_covers(const void *x, const void *win, const Shape &s, int esz) {
    if (esz != 2 || s.W_i % 8 != 0 || s.H_f < 1 || s.H_f > kMaxRowsHf) return false;
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(win)) & 15) return false;
    const int64_t items = s.N * s.C_i * s.H_o * (s.W_i / 8);
    return items + 256 < (1ll << 31) && s.N * s.C_i * s.H_o < (1ll << 31);
}

template <int HF>
static cudaError_t launch_rows16_hf(const TRParams &p, cudaStream_t st) {
    const size_t smem = (size_t)(kThreads / 32) * 32 * HF * 16;
    const cudaError_t e = cudaFuncSetAttribute(transform_rows16<HF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)smem);
    if (e != cudaSuccess) return e;
    const unsigned blocks = (unsigned)((p.items + kThreads - 1) / kThreads);
    transform_rows16<HF><<<blocks, kThreads, smem, st>>>(p);
    return cudaGetLastError();
}

static cudaError_t launch_rows16(const void *x, void *win, const Shape &s, cudaStream_t st) {
    TRParams p;
    p.x = static_cast<const uint4 *>(x);
    p.win = static_cast<uint4 *>(win);
    p.items = (int)(s.N * s.C_i * s.H_o * (s.W_i / 8));
    p.H_i = (int)s.H_i;
    p.s_h = (int)s.s_h;
    p.rvec = (int)(s.W_i / 8);
    p.div_G = make_fastdiv((uint32_t)(s.W_i / 8));
    p.div_Ho = make_fastdiv((uint32_t)s.H_o);
    switch (s.H_f) {
        case 1: return launch_rows16_hf<1>(p, st);
        case 2: return launch_rows16_hf<2>(p, st);
        case 3: return launch_rows16_hf<3>(p, st);
        case 4: return launch_rows16_hf<4>(p, st);
        case 5: return launch_rows16_hf<5>(p, st);
        case 6: return launch_rows16_hf<6>(p, st);
        case 7: return launch_rows16_hf<7>(p, st);
        case 8: return launch_rows16_hf<8>(p, st);
        case 9: return launch_rows16_hf<9>(p, st);
        case 10: return launch_rows16_hf<10>(p, st);
        case 11: return launch_rows16_hf<11>(p, st);
        default: return launch_rows16_hf<12>(p, st);
    }
}

cudaError_t launch_transform(const void *x, void *win, const Shape &s, int esz, cudaStream_t st) {
    if (s.N == 0) return cudaSuccess;
    if (rows16_covers(x, win, s, esz)) return launch_rows16(x, win, s, st);
    const int64_t L = s.W_i * s.H_f;
    const int64_t NP = s.N * s.C_i;
    const int64_t full_rows = (s.H_o - 1) * s.s_h + s.H_f;  // input rows a plane's windows use
    // bytes staged for `planes` whole planes, or for a band of T output rows of Wt columns
    auto stage_bytes = [&](int64_t elems) { return (elems + 16 + 8) / 8 * 8 * esz; };
    auto band_bytes = [&](int64_t T, int64_t Wt) { return stage_bytes(((T - 1) * s.s_h + s.H_f) * Wt); };
    auto planes_bytes = [&](int64_t P) { return stage_bytes((P - 1) * s.H_i * s.W_i + full_rows * s.W_i); };
    int64_t PPC = 1, T = 1, Wt = s.W_i;
    const bool whole = planes_bytes(1) <= kSmemBudget;
    if (whole) {
        // whole planes per CTA: as many as fit, but no more than ~16 output vectors a thread
        // and enough CTAs to fill every SM several times
        T = s.H_o;
        const int64_t plane_out_vecs = std::max<int64_t>(1, s.H_o * L * esz / 16);
        const int64_t by_work = std::max<int64_t>(1, 16 * kThreads / plane_out_vecs);
        const int64_t by_grid = std::max<int64_t>(1, NP / (sm_count() * 8));
        const int64_t cap = std::min(by_work, by_grid);
        while (PPC < cap && planes_bytes(PPC + 1) <= kSmemBudget) ++PPC;
    } else if (band_bytes(1, Wt) > kSmemBudget) {
        // rows too wide: one output row per band, split into column tiles
        while (Wt > 8 && band_bytes(1, Wt) > kSmemBudget) Wt = (Wt + 1) / 2;
    } else {
        while (T < s.H_o && band_bytes(T + 1, Wt) <= kSmemBudget) ++T;
        // balance the bands of a plane
        const int64_t tiles = (s.H_o + T - 1) / T;
        T = (s.H_o + tiles - 1) / tiles;
    }
    const int64_t ctiles = (s.W_i + Wt - 1) / Wt;
    const int64_t tiles = (s.H_o + T - 1) / T;
    const size_t staged = (size_t)(whole ? planes_bytes(PPC) : band_bytes(T, Wt));
    const int V = 16 / esz;
    // the table pays off when a vector spans several columns (H_f < V): there the
    // stepping would wrap more than once per vector; otherwise its extra shared-memory
    // loads cost more than the one wrap they save
    const bool use_table = s.H_f < V && s.H_f <= kMaxTableHf;
    const size_t smem = staged + (use_table ? (size_t)s.H_f * V * sizeof(int) : 0);

    TParams p;
    p.x = x;
    p.win = win;
    p.x_elems = s.N * s.C_i * s.H_i * s.W_i;
    p.n_planes = NP;
    p.H_i = s.H_i;
    p.W_i = s.W_i;
    p.H_f = s.H_f;
    p.s_h = s.s_h;
    p.H_o = s.H_o;
    p.tiles_per_plane = tiles;
    p.PPC = (int)PPC;
    p.T = (int)T;
    p.RP = (int)T;
    p.Wt = (int)Wt;
    p.ctiles = (int)ctiles;
    p.L = (uint32_t)L;
    p.in_cap = (int)(staged / esz);
    p.flip_bit = esz == 2 ? flip_bit_for(Wt, s.H_f) : -1;
    p.div_L = make_fastdiv((uint32_t)L);
    p.div_Hf = make_fastdiv((uint32_t)s.H_f);
    p.div_RP = make_fastdiv((uint32_t)T);

    const int64_t blocks = (NP + PPC - 1) / PPC * tiles * ctiles;
    auto go = [&](auto kernel) -> cudaError_t {
        const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kernel<<<(unsigned)blocks, kThreads, smem, st>>>(p);
        return cudaSuccess;
    };
    cudaError_t e;
    if (esz == 2)
        e = use_table ? go(transform_kernel<uint16_t, true>) : go(transform_kernel<uint16_t, false>);
    else
        e = use_table ? go(transform_kernel<uint32_t, true>) : go(transform_kernel<uint32_t, false>);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// ---- channels-last window transform
// win[n][ho][w*H_f + r][c] = x[n][ho*s_h + r][w][c]: the window row of (n, ho)
// is W_i*H_f runs of C_i contiguous elements, run (w, r) being the C_i
// channels of input position (ho*s_h + r, w). The output is written as whole
// 16-byte vectors in order (coalesced stores).
//  * C_i*esz a multiple of 16: every run is whole 16-byte vectors, copied one
//    to one by a grid-stride loop that keeps four in flight per thread;
//    consecutive output rows, which share input rows, are written at about the
//    same time, so shared rows are re-read from L2.
//  * otherwise, a CTA owns a band of output rows of one image: the input rows
//    under it are one contiguous range of x (rows of W_i*C_i elements), staged
//    once into shared memory with 16-byte loads; each thread builds 16-byte
//    output vectors from it, stepping (c, r, w, row) element by element, and
//    the band's unaligned head and tail are written element by element.
namespace {

struct TNParams {
    const void *x;
    void *win;
    int64_t elems;        // window elements
    int64_t vecs;         // 16-byte output vectors (the last may be partial)
    int64_t Lp;           // window row length W_i*H_f*C_i
    int C_i, H_i, W_i, H_f, s_h, H_o;
    int VPR;              // vectors per run (vector path: C_i*esz / 16)
    FastDiv div_vpr, div_wh, div_hf, div_ho;
    FastDiv div_lp, div_c;  // staged path: window row length, channels
    int T, tiles;         // staged path: output rows per band, bands per image
    int64_t x_elems;      // staged path: elements of x
};

// C_i*esz a multiple of 16: every run is whole, aligned 16-byte vectors.
__global__ void __launch_bounds__(256) transform_nhwc_vec(TNParams p) {
    const uint4 *__restrict__ x = static_cast<const uint4 *>(p.x);
    uint4 *__restrict__ win = static_cast<uint4 *>(p.win);
    const int WH = p.W_i * p.H_f;
    const int G = gridDim.x * blockDim.x;
    auto src_of = [&](int v) -> int64_t {
        const int R = (int)fdiv((uint32_t)v, p.div_vpr);  // run: (n, ho, w, r)
        const int k = v - R * p.VPR;
        const int row = (int)fdiv((uint32_t)R, p.div_wh);  // n*H_o + ho
        const int pp = R - row * WH;                      // w*H_f + r
        const int w = (int)fdiv((uint32_t)pp, p.div_hf);
        const int r = pp - w * p.H_f;
        const int n = (int)fdiv((uint32_t)row, p.div_ho);
        const int ho = row - n * p.H_o;
        return (((int64_t)n * p.H_i + (int64_t)ho * p.s_h + r) * p.W_i + w) * p.VPR + k;
    };
    for (int v0 = blockIdx.x * blockDim.x + threadIdx.x; v0 < p.vecs; v0 += 4 * G) {
        uint4 val[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int v = v0 + u * G;
            if (v < p.vecs) val[u] = __ldg(x + src_of(v));
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int v = v0 + u * G;
            if (v < p.vecs) win[v] = val[u];
        }
    }
}

// Any C_i: each thread builds one 16-byte output vector element by element,
// stepping (c, r, w, ho, n) from the vector's first element; a partial last
// vector is stored element by element.
template <typename E>
__global__ void __launch_bounds__(256) transform_nhwc_elem(TNParams p) {
    constexpr int V = 16 / sizeof(E);
    const E *__restrict__ x = static_cast<const E *>(p.x);
    E *__restrict__ win = static_cast<E *>(p.win);
    for (int64_t v = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; v < p.vecs;
         v += (int64_t)gridDim.x * blockDim.x) {
        const int64_t f0 = v * V;
        const int64_t row = f0 / p.Lp;
        const int64_t off = f0 - row * p.Lp;
        int n = (int)(row / p.H_o), ho = (int)(row - (int64_t)n * p.H_o);
        const int64_t pos = off / p.C_i;
        int c = (int)(off - pos * p.C_i);
        int w = (int)(pos / p.H_f), r = (int)(pos - (int64_t)w * p.H_f);
        union {
            uint4 u;
            E e[V];
        } out;
#pragma unroll
        for (int e = 0; e < V; ++e) {
            out.e[e] = f0 + e < p.elems
                           ? x[(((int64_t)n * p.H_i + (int64_t)ho * p.s_h + r) * p.W_i + w) * p.C_i + c]
                           : E(0);
            if (++c == p.C_i) {
                c = 0;
                if (++r == p.H_f) {
                    r = 0;
                    if (++w == p.W_i) {
                        w = 0;
                        if (++ho == p.H_o) { ho = 0; ++n; }
                    }
                }
            }
        }
        if (f0 + V <= p.elems) {
            *reinterpret_cast<uint4 *>(win + f0) = out.u;
        } else {
            for (int e = 0; f0 + e < p.elems; ++e) win[f0 + e] = out.e[e];
        }
    }
}

template <typename E>
__global__ void __launch_bounds__(256) transform_nhwc_staged(TNParams p) {
    extern __shared__ __align__(16) unsigned char smem_nhwc[];
    constexpr int V = 16 / sizeof(E);
    E *s_in = reinterpret_cast<E *>(smem_nhwc);
    const E *__restrict__ x = static_cast<const E *>(p.x);
    E *__restrict__ win = static_cast<E *>(p.win);
    const int n = blockIdx.x / p.tiles;
    const int tile = blockIdx.x - n * p.tiles;
    const int ho0 = tile * p.T;
    const int rows_out = min(p.T, p.H_o - ho0);
    const int rows_in = (rows_out - 1) * p.s_h + p.H_f;
    const int C = p.C_i, H_f = p.H_f, W_i = p.W_i;
    const int RL = W_i * C;  // elements of an input row

    // ---- stage x[in0, in0 + cnt) at s_in[lead, lead + cnt)
    const int64_t in0 = ((int64_t)n * p.H_i + (int64_t)ho0 * p.s_h) * RL;
    const int cnt = rows_in * RL;
    const int64_t base = in0 - (in0 % V);
    const int lead = (int)(in0 - base);
    const int nvec = (lead + cnt + V - 1) / V;
    const int64_t inside = (p.x_elems - base) / V;  // vectors wholly inside x
    const int nfull = inside < (int64_t)nvec ? (int)inside : nvec;
    const uint4 *gx = reinterpret_cast<const uint4 *>(x + base);
    uint4 *sx = reinterpret_cast<uint4 *>(s_in);
    int v = threadIdx.x;
    for (; v + 3 * 256 < nfull; v += 4 * 256) {
        const uint4 r0 = __ldg(gx + v), r1 = __ldg(gx + v + 256);
        const uint4 r2 = __ldg(gx + v + 512), r3 = __ldg(gx + v + 768);
        sx[v] = r0;
        sx[v + 256] = r1;
        sx[v + 512] = r2;
        sx[v + 768] = r3;
    }
    for (; v < nfull; v += 256) sx[v] = __ldg(gx + v);
    for (int e = nfull * V + (int)threadIdx.x; e < nvec * V; e += 256)
        if (base + e < p.x_elems) s_in[e] = x[base + e];
    __syncthreads();

    // staged index of band element g (g = t*Lp + (w*H_f + r)*C + c)
    const int Lp = (int)p.Lp;
    auto staged = [&](int g) -> int {
        const int t = (int)fdiv((uint32_t)g, p.div_lp), o = g - t * Lp;
        const int pos = (int)fdiv((uint32_t)o, p.div_c), c = o - pos * C;
        const int w = (int)fdiv((uint32_t)pos, p.div_hf), r = pos - w * H_f;
        return (t * p.s_h + r) * RL + w * C + c + lead;
    };
    const int64_t f0 = ((int64_t)n * p.H_o + ho0) * Lp;
    const int64_t f1 = f0 + (int64_t)rows_out * Lp;
    const int64_t head = min(f1, (f0 + V - 1) / V * V);  // first aligned element
    const int64_t vend = max(head, f1 / V * V);           // end of the whole vectors
    for (int64_t e = f0 + threadIdx.x; e < head; e += 256) win[e] = s_in[staged((int)(e - f0))];
    for (int64_t e = vend + threadIdx.x; e < f1; e += 256) win[e] = s_in[staged((int)(e - f0))];
    for (int64_t vv = head / V + threadIdx.x; vv < vend / V; vv += 256) {
        // (the vector's first element, by multiply-shift divisions)
        const int g = (int)(vv * V - f0);
        int t = (int)fdiv((uint32_t)g, p.div_lp);
        const int o = g - t * Lp;
        const int pos = (int)fdiv((uint32_t)o, p.div_c);
        int c = o - pos * C;
        int w = (int)fdiv((uint32_t)pos, p.div_hf), r = pos - w * H_f;
        int src = (t * p.s_h + r) * RL + w * C + c + lead;
        union {
            uint4 u;
            E e[V];
        } out;
#pragma unroll
        for (int e = 0; e < V; ++e) {
            out.e[e] = s_in[src];
            if (++c == C) {  // next row offset r of column w
                c = 0;
                src += RL - C + 1;
                if (++r == H_f) {  // next column w, back to the first row
                    r = 0;
                    src += C - H_f * RL;
                    if (++w == W_i) {  // next output row of the band
                        w = 0;
                        src += (p.s_h - 1) * RL;
                        ++t;
                    }
                }
            } else {
                ++src;
            }
        }
        *reinterpret_cast<uint4 *>(win + vv * V) = out.u;
    }
}

constexpr int kNhwcStageBudget = 48 * 1024;  // staged input rows per CTA

// Channels-last with C_i*esz a multiple of 16: window row (n, ho) is, for w in
// [0, W_i), the H_f input positions (ho*s_h + r, w) of C_i contiguous elements.
// Seen as a 4-D tensor of dimensions (C_i, rows, columns, N) — strides 1,
// W_i*C_i, C_i and H_i*W_i*C_i elements — the box (C_i, H_f, Wc, 1) at
// (0, ho*s_h, w0, n) lands in shared memory as [column][row][channel]: exactly
// the window row's elements [w0*H_f*C_i, (w0 + Wc)*H_f*C_i). So a unit (n, ho,
// column chunk) is one TMA tensor load and one bulk store of the same bytes;
// columns past W_i (a short last chunk) read as zero and are not stored. Each
// CTA is persistent: one thread cycles its units through a ring of kNhwcRing
// shared-memory buffers, the loads of the next units in flight while a unit is
// stored. The waits for the loads give up after 2 s (the CTA then stops; the
// copy engine completes every load it accepted, so none is expected).
constexpr int kNhwcRing = 3;
constexpr int kNhwcBoxBytes = 32 * 1024;

struct TTParams {
    CUtensorMap tmap;  // (the type is 128-byte aligned)
    uint8_t *win;
    int64_t units;        // N * H_o * chunks
    int chunks, Wc;       // column chunks per window row, columns per chunk
    int H_o, W_i, s_h;
    uint32_t box_bytes;   // C_i * H_f * Wc * esz
    uint32_t buf_bytes;   // box_bytes rounded up to 128 (each buffer 128-byte aligned)
    uint32_t col_bytes;   // H_f * C_i * esz: one column of a window row
};

__global__ void __launch_bounds__(32, 1) transform_nhwc_tma(const __grid_constant__ TTParams p) {
    extern __shared__ __align__(128) uint8_t tt_smem[];
    __shared__ uint64_t full[kNhwcRing];
    if (threadIdx.x != 0) return;
    using namespace tc;
    for (int b = 0; b < kNhwcRing; ++b) mbar_init(smem_u32(&full[b]), 1);
    fence_mbar_init();
    const int64_t first = blockIdx.x, step = gridDim.x;
    const int64_t mine = first < p.units ? (p.units - first + step - 1) / step : 0;
    auto load = [&](int64_t k) {  // the k-th unit of this CTA into buffer k % kNhwcRing
        const int64_t u = first + k * step;
        const int ch = (int)(u % p.chunks);
        const int64_t r = u / p.chunks;
        const int ho = (int)(r % p.H_o), n = (int)(r / p.H_o);
        const int b = (int)(k % kNhwcRing);
        const uint32_t bar = smem_u32(&full[b]);
        mbar_arrive_expect_tx(bar, p.box_bytes);
        tma_load_4d(smem_u32(tt_smem + (size_t)b * p.buf_bytes), &p.tmap, 0, ho * p.s_h, ch * p.Wc, n, bar);
    };
    for (int64_t k = 0; k < kNhwcRing - 1 && k < mine; ++k) load(k);
    for (int64_t k = 0; k < mine; ++k) {
        const int b = (int)(k % kNhwcRing);
        // wait (bounded) for the unit's load
        const uint32_t bar = smem_u32(&full[b]), par = (uint32_t)((k / kNhwcRing) & 1);
        bool ok = mbar_try_wait(bar, par);
        const uint64_t t0 = globaltimer();
        while (!ok && globaltimer() - t0 < kTimeoutNs) ok = mbar_try_wait(bar, par);
        if (!ok) break;
        const int64_t u = first + k * step;
        const int ch = (int)(u % p.chunks);
        const int64_t r = u / p.chunks;
        const int w0 = ch * p.Wc;
        const int ncols = min(p.Wc, p.W_i - w0);
        uint8_t *dst = p.win + ((r * p.W_i) + w0) * (int64_t)p.col_bytes;  // r = n*H_o + ho
        fence_async_smem();
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                     "r"(smem_u32(tt_smem + (size_t)b * p.buf_bytes)), "r"((uint32_t)ncols * p.col_bytes)
                     : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        // the next load reuses the buffer of the previous unit's store: wait until that
        // store has read it (this unit's store may still be in flight)
        if (k + kNhwcRing - 1 < mine) {
            asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
            load(k + kNhwcRing - 1);
        }
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// The channels-last TMA transform's tensor map, or false when it does not cover
// the shape (box limits: at most 256 per dimension).
static PFN_cuTensorMapEncodeTiled_v12000 transform_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

static bool nhwc_tma_params(TTParams &p, const void *x, void *win, const Shape &s, int esz) {
    if ((s.C_i * esz) % 16 != 0 || s.C_i > 256 || s.H_f > 256) return false;
    if (((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(win)) & 15) != 0) return false;
    const int64_t col_bytes = s.H_f * s.C_i * esz;
    if (col_bytes > kNhwcBoxBytes) return false;
    const int64_t wmax = std::min<int64_t>(256, kNhwcBoxBytes / col_bytes);
    const int64_t chunks = (s.W_i + wmax - 1) / wmax;
    const int64_t Wc = (s.W_i + chunks - 1) / chunks;
    const PFN_cuTensorMapEncodeTiled_v12000 enc = transform_map_encoder();
    if (!enc) return false;
    const cuuint64_t C = (cuuint64_t)s.C_i, W = (cuuint64_t)s.W_i, H = (cuuint64_t)s.H_i;
    const cuuint64_t e = (cuuint64_t)esz;
    const cuuint64_t dims[4] = {C, H, W, (cuuint64_t)s.N};
    const cuuint64_t strides[3] = {W * C * e, C * e, H * W * C * e};
    const cuuint32_t box[4] = {(cuuint32_t)C, (cuuint32_t)s.H_f, (cuuint32_t)Wc, 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    const CUresult r = enc(&p.tmap, esz == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT32, 4,
                           const_cast<void *>(x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    p.win = static_cast<uint8_t *>(win);
    p.chunks = (int)chunks;
    p.Wc = (int)Wc;
    p.units = s.N * s.H_o * chunks;
    p.H_o = (int)s.H_o;
    p.W_i = (int)s.W_i;
    p.s_h = (int)s.s_h;
    p.col_bytes = (uint32_t)col_bytes;
    p.box_bytes = (uint32_t)(col_bytes * Wc);
    p.buf_bytes = (p.box_bytes + 127u) / 128u * 128u;
    return true;
}

}  // namespace

cudaError_t launch_transform_nhwc(const void *x, void *win, const Shape &s, int esz, cudaStream_t st) {
    if (s.N > 0 && s.H_o > 0) {
        TTParams tp;
        if (nhwc_tma_params(tp, x, win, s, esz)) {
            int dev = 0, sms = 148;
            if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            const size_t smem = (size_t)kNhwcRing * tp.buf_bytes;
            const cudaError_t e =
                cudaFuncSetAttribute(transform_nhwc_tma, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            const int per_sm = (int)std::max<size_t>(1, std::min<size_t>(8, (200 * 1024) / smem));
            const unsigned blocks = (unsigned)std::min<int64_t>(tp.units, (int64_t)sms * per_sm);
            transform_nhwc_tma<<<blocks, 32, smem, st>>>(tp);
            return cudaGetLastError();
        }
    }
    TNParams p;
    p.x = x;
    p.win = win;
    p.Lp = s.W_i * s.H_f * s.C_i;
    p.elems = s.N * s.H_o * p.Lp;
    p.vecs = (p.elems * esz + 15) / 16;
    p.C_i = (int)s.C_i;
    p.H_i = (int)s.H_i;
    p.W_i = (int)s.W_i;
    p.H_f = (int)s.H_f;
    p.s_h = (int)s.s_h;
    p.H_o = (int)s.H_o;
    const bool vec = (s.C_i * esz) % 16 == 0;
    p.VPR = vec ? (int)(s.C_i * esz / 16) : 1;
    p.x_elems = s.N * s.H_i * s.W_i * s.C_i;
    // staged path: as many output rows per band as the budget holds, balanced
    const int64_t RLb = s.W_i * s.C_i * esz;  // bytes of an input row
    int64_t T = 0;
    while (T < s.H_o && (T * s.s_h + s.H_f) * RLb + 16 <= kNhwcStageBudget) ++T;
    const bool staged = !vec && T >= 1;
    if (staged) {
        const int64_t tiles = (s.H_o + T - 1) / T;
        T = (s.H_o + tiles - 1) / tiles;
        p.T = (int)T;
        p.tiles = (int)tiles;
    }
    p.div_vpr = make_fastdiv((uint32_t)p.VPR);
    p.div_wh = make_fastdiv((uint32_t)(s.W_i * s.H_f));
    p.div_hf = make_fastdiv((uint32_t)s.H_f);
    p.div_ho = make_fastdiv((uint32_t)s.H_o);
    p.div_lp = make_fastdiv((uint32_t)p.Lp);
    p.div_c = make_fastdiv((uint32_t)s.C_i);
    if (p.vecs == 0) return cudaSuccess;
    if (staged) {
        const size_t smem = (size_t)(((T - 1) * s.s_h + s.H_f) * RLb + 16 + 15) / 16 * 16;
        const unsigned blocks = (unsigned)(s.N * p.tiles);
        if (esz == 2) {
            cudaFuncSetAttribute(transform_nhwc_staged<uint16_t>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
            transform_nhwc_staged<uint16_t><<<blocks, 256, smem, st>>>(p);
        } else {
            cudaFuncSetAttribute(transform_nhwc_staged<uint32_t>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
            transform_nhwc_staged<uint32_t><<<blocks, 256, smem, st>>>(p);
        }
        return cudaGetLastError();
    }
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t per_pass = vec ? 4 : 1;  // vectors per thread and grid pass
    const int64_t need = (p.vecs + 256 * per_pass - 1) / (256 * per_pass);
    const unsigned blocks = (unsigned)std::max<int64_t>(1, std::min<int64_t>(need, (int64_t)sms * 8));
    if (vec)
        transform_nhwc_vec<<<blocks, 256, 0, st>>>(p);
    else if (esz == 2)
        transform_nhwc_elem<uint16_t><<<blocks, 256, 0, st>>>(p);
    else
        transform_nhwc_elem<uint32_t><<<blocks, 256, 0, st>>>(p);
    return cudaGetLastError();
}

// The vector path indexes output vectors and runs with 32-bit arithmetic.
bool transform_nhwc_supported(const Shape &s, int esz) {
    const int64_t runs = s.N * s.H_o * s.W_i * s.H_f;
    const int64_t bytes = runs * s.C_i * esz;
    return bytes / 16 < (1ll << 30) && runs < (1ll << 31) && s.W_i * s.H_f * s.C_i < (1ll << 40);
}

// ---- padded / dilated window transform (either layout)
// A plane is one (image, channel) of NCHW (C = 1 element per position) or one
// image of NHWC (C = C_i channels per position, innermost). Its window row ho
// holds, for the W_p = W_i + 2 p_w padded columns w and the H_f rows r,
//   win[plane][ho][(w*H_f + r)*C + c] = x[plane][ho*s_h + r*d_h - p_h][w - p_w][c]
// (zero outside x). A CTA owns a band of output rows of one plane; the input
// rows under it that exist are one contiguous range of x, staged in shared
// memory when they fit (else read from global memory); each thread builds
// 16-byte output vectors by stepping (c, r, w, row), the band's unaligned ends
// element by element.
namespace {

struct TPParams {
    const void *x;
    void *win;
    int64_t x_elems;
    int H_i, W_i, C, H_f, s_h, p_h, p_w, d_h, H_o, Wp;
    int Lp;              // window row length W_p*H_f*C
    int T, tiles;        // output rows per band, bands per plane
    int staged;          // 1: input rows staged in shared memory
};

template <typename E>
__global__ void __launch_bounds__(256) transform_pd_kernel(TPParams p) {
    extern __shared__ __align__(16) unsigned char smem_pd[];
    constexpr int V = 16 / sizeof(E);
    E *s_in = reinterpret_cast<E *>(smem_pd);
    const E *__restrict__ x = static_cast<const E *>(p.x);
    E *__restrict__ win = static_cast<E *>(p.win);
    const int64_t plane = blockIdx.x / p.tiles;
    const int tile = (int)(blockIdx.x - plane * p.tiles);
    const int ho0 = tile * p.T;
    const int rows_out = min(p.T, p.H_o - ho0);
    const int RL = p.W_i * p.C;
    // input rows [hs, he) of the plane under the band (clipped to x)
    const int hs = max(0, ho0 * p.s_h - p.p_h);
    const int he = min(p.H_i, (ho0 + rows_out - 1) * p.s_h + (p.H_f - 1) * p.d_h - p.p_h + 1);
    const int64_t in0 = (plane * p.H_i + hs) * (int64_t)RL;
    const E *src = x + in0;  // element (h, w, c) of the plane at src[(h - hs)*RL + w*C + c]
    if (p.staged) {
        const int cnt = max(0, he - hs) * RL;
        const int64_t base = in0 - (in0 % V);
        const int lead = (int)(in0 - base);
        const int nvec = (lead + cnt + V - 1) / V;
        const int64_t inside = (p.x_elems - base) / V;
        const int nfull = inside < (int64_t)nvec ? (int)inside : nvec;
        const uint4 *gx = reinterpret_cast<const uint4 *>(x + base);
        uint4 *sx = reinterpret_cast<uint4 *>(s_in);
        int v = threadIdx.x;
        for (; v + 3 * 256 < nfull; v += 4 * 256) {
            const uint4 r0 = __ldg(gx + v), r1 = __ldg(gx + v + 256);
            const uint4 r2 = __ldg(gx + v + 512), r3 = __ldg(gx + v + 768);
            sx[v] = r0;
            sx[v + 256] = r1;
            sx[v + 512] = r2;
            sx[v + 768] = r3;
        }
        for (; v < nfull; v += 256) sx[v] = __ldg(gx + v);
        for (int e = nfull * V + (int)threadIdx.x; e < nvec * V; e += 256)
            if (base + e < p.x_elems) s_in[e] = x[base + e];
        __syncthreads();
        src = s_in + lead;
    }
    const int C = p.C, H_f = p.H_f, Lp = p.Lp;
    // element g of the band: t = g / Lp, (w*H_f + r)*C + c = g % Lp
    auto value = [&](int t, int w, int r, int c) -> E {
        const int h = (ho0 + t) * p.s_h + r * p.d_h - p.p_h;
        const int wx = w - p.p_w;
        return ((unsigned)h < (unsigned)p.H_i && (unsigned)wx < (unsigned)p.W_i) ? src[(h - hs) * RL + wx * C + c]
                                                                                   : E(0);
    };
    auto value_at = [&](int g) -> E {
        const int t = g / Lp, o = g - t * Lp;
        const int pos = o / C, c = o - pos * C;
        const int w = pos / H_f, r = pos - w * H_f;
        return value(t, w, r, c);
    };
    const int64_t f0 = (plane * p.H_o + ho0) * (int64_t)Lp;
    const int64_t f1 = f0 + (int64_t)rows_out * Lp;
    const int64_t head = min(f1, (f0 + V - 1) / V * V);
    const int64_t vend = max(head, f1 / V * V);
    for (int64_t e = f0 + threadIdx.x; e < head; e += 256) win[e] = value_at((int)(e - f0));
    for (int64_t e = vend + threadIdx.x; e < f1; e += 256) win[e] = value_at((int)(e - f0));
    for (int64_t vv = head / V + threadIdx.x; vv < vend / V; vv += 256) {
        const int g = (int)(vv * V - f0);
        int t = g / Lp;
        const int o = g - t * Lp;
        const int pos = o / C;
        int c = o - pos * C;
        int w = pos / H_f, r = pos - w * H_f;
        union {
            uint4 u;
            E e[V];
        } out;
#pragma unroll
        for (int e = 0; e < V; ++e) {
            out.e[e] = value(t, w, r, c);
            if (++c == C) {
                c = 0;
                if (++r == H_f) {
                    r = 0;
                    if (++w == p.Wp) { w = 0; ++t; }
                }
            }
        }
        *reinterpret_cast<uint4 *>(win + vv * V) = out.u;
    }
}

constexpr int kPdStageBudget = 48 * 1024;

}  // namespace

cudaError_t launch_transform_pd(const void *x, void *win, const Shape &s, int esz, int layout,
                                cudaStream_t st) {
    const bool cl = layout == LAYOUT_NHWC;
    TPParams p;
    p.x = x;
    p.win = win;
    p.x_elems = s.N * s.C_i * s.H_i * s.W_i;
    p.H_i = (int)s.H_i;
    p.W_i = (int)s.W_i;
    p.C = cl ? (int)s.C_i : 1;
    p.H_f = (int)s.H_f;
    p.s_h = (int)s.s_h;
    p.p_h = (int)s.p_h;
    p.p_w = (int)s.p_w;
    p.d_h = (int)s.d_h;
    p.H_o = (int)s.H_o;
    p.Wp = (int)padded_w(s);
    p.Lp = (int)(padded_w(s) * s.H_f * p.C);
    const int64_t planes = cl ? s.N : s.N * s.C_i;
    const int64_t RLb = s.W_i * p.C * esz;
    // output rows per band: as many as the staging budget holds (at least one band
    // row per CTA; rows too long to stage are read from global memory)
    int64_t T = 0;
    while (T < s.H_o && (T * s.s_h + (s.H_f - 1) * s.d_h + 1) * RLb + 16 <= kPdStageBudget) ++T;
    p.staged = T >= 1 ? 1 : 0;
    if (T < 1) T = std::min<int64_t>(s.H_o, 4);
    const int64_t tiles = (s.H_o + T - 1) / T;
    T = (s.H_o + tiles - 1) / tiles;
    p.T = (int)T;
    p.tiles = (int)tiles;
    if (planes == 0 || s.H_o == 0) return cudaSuccess;
    const size_t smem =
        p.staged ? (size_t)((((T - 1) * s.s_h + (s.H_f - 1) * s.d_h + 1) * RLb + 16 + 15) / 16 * 16) : 0;
    const unsigned blocks = (unsigned)(planes * tiles);
    if (esz == 2) {
        if (smem) cudaFuncSetAttribute(transform_pd_kernel<uint16_t>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        transform_pd_kernel<uint16_t><<<blocks, 256, smem, st>>>(p);
    } else {
        if (smem) cudaFuncSetAttribute(transform_pd_kernel<uint32_t>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        transform_pd_kernel<uint32_t><<<blocks, 256, smem, st>>>(p);
    }
    return cudaGetLastError();
}

// 32-bit indexing within a band and a plane; one CTA per (plane, band).
bool transform_pd_supported(const Shape &s, int esz) {
    const int64_t Lp = padded_w(s) * s.H_f * s.C_i;  // the longest window row (NHWC)
    return s.H_o * Lp < (1ll << 31) && s.H_i * s.W_i * s.C_i < (1ll << 31) &&
           s.N * s.C_i * ((s.H_o + 3) / 4 + 1) < (1ll << 31) && esz > 0;
}

// The transform indexes a band with 32-bit arithmetic and launches one CTA per
// (plane, band, column tile).
bool transform_supported(const Shape &s, int esz) {
    // the narrowest tile (8 columns of one output row) must fit in shared memory
    const int64_t narrow = (s.H_f * 8 + 24) * esz;
    return narrow <= 200 * 1024 && s.W_i * s.H_f * s.H_o < (1ll << 31) &&
           s.N * s.C_i * s.H_o * ((s.W_i + 7) / 8) < (1ll << 31);
}

}  // namespace im2win
