// fp16/bf16 im2win convolution on the 5th-generation tensor cores (tcgen05,
// sm_103a), fp32 accumulation in tensor memory (TMEM).
//
// "Enabling Memory-efficient Im2win Convolution with Multi-precision Support
// on GPU CUDA and Tensor Cores", Abstract (half precision on tensor cores):
//   out[n][co][ho][wo] = sum_ci sum_{k < W_f*H_f} win[n][ci][ho][wo*s_w*H_f + k] * filt'[co][ci][k]
// with filt'[co][ci][j*H_f + r] = filt[co][ci][r][j]. As a GEMM:
//   D[co][p] = sum_K A[co][K] * B[p][K],  K = (ci, k),  p = output pixel,
// A = filt' (M = 128 output channels per tile), B[p][(ci, k)] = the pixel's
// contiguous window segment of channel ci (N = 256 pixels per tile).
//
// This file holds the "expand" kernel: every pipeline stage covers 64 values
// of K; producer warps gather, for each of the tile's 256 pixels, its 64
// window values of the stage (im2win order) into the canonical K-major
// operand layout in shared memory, reading either the window tensor (the
// two-step path) or the NCHW input directly (the fused path, which then never
// materialises the window tensor). The filter tile of the stage arrives by
// one bulk (TMA) copy from the workspace, where a small kernel has re-laid it
// into the same canonical layout. One thread issues tcgen05.mma (M=128,
// N=256, K=16) into a TMEM accumulator; a 4-stage mbarrier pipeline
// overlaps gathering, copying and MMA; the producer warps then drain TMEM
// (tcgen05.ld), round to the input dtype and store through shared memory so
// that global stores are coalesced along the output row.
//
// Operand layout (both A and B, no swizzle, K-major): core matrices of
// 8 rows x 16 bytes; the 8 core matrices of one 8-row group that cover the
// stage's 64 K values are adjacent (leading-dimension offset 128 B), and
// consecutive 8-row groups are 1024 B apart (stride-dimension offset).
//
// Every mbarrier wait is bounded (wall clock, 2 s): on expiry the CTA records
// IM2WIN_ERR_TIMEOUT in the workspace status word, drains its in-flight
// copies and MMAs, frees TMEM and exits.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "im2win_internal.cuh"
#include "tc_ptx.cuh"

namespace im2win {
namespace {

using namespace tc;

// ------------------------------------------------------------------ config
constexpr int BM = 128;               // output channels per tile (MMA M)
constexpr int KS = 64;                // K values per pipeline stage (4 MMAs of K = 16)
constexpr int NT = 256;               // pixels per tile (MMA N)
constexpr int STAGES = 4;
constexpr int PROD_WARPS = 8;         // one pixel per producer thread
constexpr int NTHREADS = (2 + PROD_WARPS) * 32;
constexpr uint32_t A_BYTES = BM * KS * 2;   // 16 KB
constexpr uint32_t B_BYTES = NT * KS * 2;   // 32 KB
constexpr uint32_t TMEM_COLS = NT;          // fp32 accumulator columns
constexpr size_t SMEM_BYTES = STAGES * (A_BYTES + B_BYTES) + 256;
static_assert(PROD_WARPS * 32 == NT, "one producer thread per pixel");

struct TcParams {
    const uint16_t *src;   // window tensor (two-step) or NCHW input (fused)
    const uint16_t *fa;    // filter tiles in the canonical operand layout
    uint16_t *out;
    uint32_t *status;
    int C_i, C_o, H_i, W_i, H_o, W_o, H_f, W_f, s_h, s_w;
    int KK, KKP;           // taps per channel, padded to a multiple of 8
    int P;                 // pixels per image
    int L, S;              // window row length W_i*H_f, window step s_w*H_f
    int kstages;           // K stages per tile
    int pos_tiles;         // pixel tiles per image
    int64_t img_src;       // elements of src per image
    int64_t fa_tile;       // elements of fa per channel tile
    FastDiv div_KKP, div_Hf, div_Wo;
    uint32_t idesc;
    int bf16;
};

template <bool FROM_X>
__global__ void __launch_bounds__(NTHREADS, 1) conv_tc_expand_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * A_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sB + STAGES * B_BYTES);
    // bars: full_a[S] | full_b[S] | empty[S] | done | drain
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 3 * STAGES + 2);
    int *abort_word = reinterpret_cast<int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = blockIdx.x / p.pos_tiles;
    const int tile = blockIdx.x - n * p.pos_tiles;
    const int mt = blockIdx.y;
    const int pos0 = tile * NT;

    auto full_a = [&](int s) { return smem_u32(bars + s); };
    auto full_b = [&](int s) { return smem_u32(bars + STAGES + s); };
    auto empty = [&](int s) { return smem_u32(bars + 2 * STAGES + s); };
    const uint32_t done = smem_u32(bars + 3 * STAGES);
    const uint32_t drain = smem_u32(bars + 3 * STAGES + 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_a(s), 1);
            mbar_init(full_b(s), PROD_WARPS * 32);
            mbar_init(empty(s), 1);
        }
        mbar_init(done, 1);
        mbar_init(drain, 1);
        *abort_word = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(tmem_slot);
    const Ctl ctl{reinterpret_cast<volatile int *>(abort_word), p.status};

    if (warp == 0) {
        // ---------------- MMA issuer
        if (lane == 0) {
            bool ok = true;
            for (int it = 0; it < p.kstages && ok; ++it) {
                const int s = it % STAGES;
                const uint32_t ph = (it / STAGES) & 1;
                ok = bar_wait(full_a(s), ph, ctl, SITE_FULL_A) && bar_wait(full_b(s), ph, ctl, SITE_FULL_B);
                if (!ok) break;
                tc_fence_after();
                const uint32_t a0 = smem_u32(sA + s * A_BYTES), b0 = smem_u32(sB + s * B_BYTES);
#pragma unroll
                for (int u = 0; u < KS / 16; ++u) {
                    const uint64_t ad = smem_desc(a0 + u * 256, 128, 1024);
                    const uint64_t bd = smem_desc(b0 + u * 256, 128, 1024);
                    mma_f16(tmem, ad, bd, p.idesc, (it | u) != 0);
                }
                mma_commit(empty(s));
            }
            mma_commit(done);
            if (!ok) bar_wait(done, 0, ctl, SITE_DRAIN, false);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- filter tiles: one bulk copy per stage
        if (lane == 0) {
            const uint16_t *fa = p.fa + (int64_t)mt * p.fa_tile;
            int issued = 0;
            for (int it = 0; it < p.kstages; ++it) {
                const int s = it % STAGES;
                const uint32_t ph = (it / STAGES) & 1;
                if (!bar_wait(empty(s), ph ^ 1, ctl, SITE_EMPTY_LOAD)) break;
                mbar_arrive_expect_tx(full_a(s), A_BYTES);
                bulk_g2s(smem_u32(sA + s * A_BYTES), fa + (int64_t)it * (BM * KS), A_BYTES, full_a(s));
                ++issued;
            }
            if (*ctl.abort_flag) {
                // let every copy still in flight land before the CTA exits
                for (int it = (issued > STAGES ? issued - STAGES : 0); it < issued; ++it)
                    bar_wait(full_a(it % STAGES), (it / STAGES) & 1, ctl, SITE_DRAIN, false);
            }
        }
        __syncwarp();
    } else {
        // ---------------- producers: one pixel each, 64 window values per stage
        const int pt = threadIdx.x - 64;
        const int pg = pos0 + pt;
        const bool valid = pg < p.P;
        int pos_off = 0;
        if (valid) {
            const int ho = (int)fdiv((uint32_t)pg, p.div_Wo);
            const int wo = pg - ho * p.W_o;
            pos_off = FROM_X ? ho * p.s_h * p.W_i + wo * p.s_w : ho * p.L + wo * p.S;
        }
        const uint16_t *__restrict__ src = p.src + (int64_t)n * p.img_src;
        const uint32_t row_off = (uint32_t)((pt >> 3) * 1024 + (pt & 7) * 16);
        const int HiWi = p.H_i * p.W_i, HoL = p.H_o * p.L;
        for (int it = 0; it < p.kstages; ++it) {
            const int s = it % STAGES;
            const uint32_t ph = (it / STAGES) & 1;
            if (!bar_wait(empty(s), ph ^ 1, ctl, SITE_EMPTY_PROD)) break;
            uint8_t *dstB = sB + s * B_BYTES + row_off;
#pragma unroll 2
            for (int c = 0; c < KS / 8; ++c) {
                const int kg0 = it * KS + c * 8;
                const int ci = (int)fdiv((uint32_t)kg0, p.div_KKP);
                const int kk0 = kg0 - ci * p.KKP;
                uint32_t v[8];
                if (valid && ci < p.C_i) {
                    if (FROM_X) {
                        int j = (int)fdiv((uint32_t)kk0, p.div_Hf);
                        int r = kk0 - j * p.H_f;
                        const uint16_t *b = src + ci * HiWi + pos_off;
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            v[e] = (kk0 + e < p.KK) ? (uint32_t)__ldg(b + r * p.W_i + j) : 0u;
                            if (++r == p.H_f) { r = 0; ++j; }
                        }
                    } else {
                        const uint16_t *b = src + ci * HoL + pos_off + kk0;
#pragma unroll
                        for (int e = 0; e < 8; ++e) v[e] = (kk0 + e < p.KK) ? (uint32_t)__ldg(b + e) : 0u;
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = 0u;
                }
                uint4 q;
                q.x = v[0] | (v[1] << 16);
                q.y = v[2] | (v[3] << 16);
                q.z = v[4] | (v[5] << 16);
                q.w = v[6] | (v[7] << 16);
                *reinterpret_cast<uint4 *>(dstB + c * 128) = q;
            }
            fence_async_smem();
            mbar_arrive(full_b(s));
        }

        // ---------------- epilogue: TMEM -> registers -> smem -> coalesced stores
        const bool ok = bar_wait(done, 0, ctl, SITE_DONE);
        tc_fence_after();
        if (ok) {
            const int q = warp & 3;              // TMEM lane quarter this warp may read
            const int hh = (warp - 2) >> 2;      // which half of the columns
            uint32_t *stage = reinterpret_cast<uint32_t *>(sB) + (warp - 2) * (32 * 17);
            const int co_base = mt * BM + q * 32;
            for (int blk = 0; blk < NT / 64; ++blk) {
                const int col = hh * (NT / 2) + blk * 32;
                uint32_t r[32];
                tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)col, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    stage[lane * 17 + i] = pack2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]), p.bf16);
                __syncwarp();
                const int pidx = pos0 + col + lane;
                const uint16_t *st16 = reinterpret_cast<const uint16_t *>(stage);
                for (int row = 0; row < 32; ++row) {
                    const int co = co_base + row;
                    if (co < p.C_o && pidx < p.P)
                        p.out[((int64_t)n * p.C_o + co) * p.P + pidx] = st16[row * 34 + lane];
                }
                __syncwarp();
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// Filter tiles for the expand kernel: for channel tile mt and stage ks, a
// 128 x 64 block in the canonical layout described above, holding
// filt'[co][ci][kk] at K index ci*KKP + kk (kk = j*H_f + r), zero-padded.
// Block 0 also clears the workspace status word for this call.
__global__ void relayout_filter_expand(const uint16_t *__restrict__ filt, uint16_t *__restrict__ fa,
                                       uint32_t *status, int64_t total, int C_i, int C_o, int H_f,
                                       int W_f, int KK, int KKP, int kstages) {
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        status[0] = 0;
        status[1] = 0;
        status[2] = 0;
    }
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int e = (int)(idx & 7), rw = (int)((idx >> 3) & 7), c = (int)((idx >> 6) & 7),
                  g = (int)((idx >> 9) & 15);
        const int64_t rest = idx >> 13;
        const int ks = (int)(rest % kstages);
        const int mt = (int)(rest / kstages);
        const int co = mt * BM + g * 8 + rw;
        const int kg = ks * KS + c * 8 + e;
        const int ci = kg / KKP, kk = kg - ci * KKP;
        uint16_t v = 0;
        if (co < C_o && ci < C_i && kk < KK) {
            const int j = kk / H_f, r = kk - j * H_f;
            v = filt[(((int64_t)co * C_i + ci) * H_f + r) * W_f + j];
        }
        fa[idx] = v;
    }
}

// =========================================================================
// Tap kernel (fused path, many input channels).
//
// The CTA owns Q whole output rows of one image and 128 output channels.
// Shared memory holds, per 16-channel chunk, the unique input elements under
// those rows (the (Q-1)*s_h + H_f input rows, every column) with the 16
// channels innermost, split into s_h x s_w polyphase blocks:
//   slab[c8][row % s_h][col % s_w][row / s_h][col / s_w][8 channels]  (16 B per entry)
// Output pixel (q, w') of the tile is "position" p = q*Wh + w' (Wh = ceil(W_i/s_w)),
// and for filter tap (r, j) the 16 B entries of consecutive positions are
// consecutive in the slab. So the B operand of tap (r, j) is the slab seen
// from a constant offset -- a plain K-major descriptor (8-row groups 128 B
// apart, the two 8-channel halves one plane apart) -- and no element is ever
// duplicated: each tap is one tcgen05.mma (M=128 channels, N<=256 positions,
// K=16 input channels) per half of the tile. Positions with w' >= W_o are
// computed and discarded. The filter arrives per (chunk, group of taps) by
// bulk copy, pre-laid by a re-layout kernel as [tap][co-group][8-ch half][8 co][8 ch].
// =========================================================================
constexpr int TAP_PROD_WARPS = 8;
constexpr int TAP_THREADS = (2 + TAP_PROD_WARPS) * 32;
constexpr uint32_t TAP_A_BYTES = BM * 16 * 2;  // one tap of one 16-channel chunk: 4 KB
constexpr int TAP_MAX_NT = 512;

struct TapParams {
    const uint16_t *x;
    const uint16_t *fa;
    uint16_t *out;
    uint32_t *status;
    int C_i, C_o, H_i, W_i, H_o, W_o, H_f, W_f, s_h, s_w;
    int C16;               // 16-channel chunks
    int T;                 // taps H_f*W_f
    int TG, ntg;           // taps per filter stage, filter stages per chunk
    int Q, tiles_h;        // output rows per tile, tiles per image
    int Wh, HH, RR;        // positions per row, phase rows, input rows per tile
    int NT, NTp, N0, N1;   // positions, padded, MMA N of the two halves
    uint32_t PB, CH;       // bytes of a phase block, of an 8-channel plane
    uint32_t stage_b;      // bytes of one slab stage
    int BST, AST;          // slab stages, filter stages
    uint32_t tmem_cols;
    int vec;               // 1: rows are 16 B aligned and W_i % 8 == 0 (vector loads)
    uint32_t idesc0, idesc1;
    int bf16;
};

__device__ __forceinline__ uint32_t tap_off(const TapParams &p, int r, int j) {
    return (uint32_t)((((r % p.s_h) * p.s_w + (j % p.s_w)) * p.PB) +
                      (((r / p.s_h) * p.Wh + (j / p.s_w)) * 16));
}

__global__ void __launch_bounds__(TAP_THREADS, 1) conv_tc_tap_kernel(const __grid_constant__ TapParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t a_stage = (uint32_t)p.TG * TAP_A_BYTES;
    uint8_t *sA = smem;
    uint8_t *sB = smem + (size_t)p.AST * a_stage;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sB + (size_t)p.BST * p.stage_b);
    // bars: full_a[AST] | empty_a[AST] | full_b[BST] | empty_b[BST] | done | drain
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * p.AST + 2 * p.BST + 2);
    int *abort_word = reinterpret_cast<int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = blockIdx.x / p.tiles_h;
    const int th = blockIdx.x - n * p.tiles_h;
    const int mt = blockIdx.y;
    const int ho0 = th * p.Q;

    auto full_a = [&](int s) { return smem_u32(bars + s); };
    auto empty_a = [&](int s) { return smem_u32(bars + p.AST + s); };
    auto full_b = [&](int s) { return smem_u32(bars + 2 * p.AST + s); };
    auto empty_b = [&](int s) { return smem_u32(bars + 2 * p.AST + p.BST + s); };
    const uint32_t done = smem_u32(bars + 2 * p.AST + 2 * p.BST);
    const uint32_t drain = smem_u32(bars + 2 * p.AST + 2 * p.BST + 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.AST; ++s) {
            mbar_init(full_a(s), 1);
            mbar_init(empty_a(s), 1);
        }
        for (int s = 0; s < p.BST; ++s) {
            mbar_init(full_b(s), TAP_PROD_WARPS * 32);
            mbar_init(empty_b(s), 1);
        }
        mbar_init(done, 1);
        mbar_init(drain, 1);
        *abort_word = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(tmem_slot);
    const Ctl ctl{reinterpret_cast<volatile int *>(abort_word), p.status};

    if (warp == 0) {
        // ---------------- MMA issuer
        if (lane == 0) {
            bool ok = true;
            int a_it = 0;
            for (int cc = 0; cc < p.C16 && ok; ++cc) {
                const int sb = cc % p.BST;
                if (!(ok = bar_wait(full_b(sb), (cc / p.BST) & 1, ctl, SITE_FULL_B))) break;
                const uint32_t slab = smem_u32(sB + (size_t)sb * p.stage_b);
                for (int tg = 0; tg < p.ntg && ok; ++tg, ++a_it) {
                    const int sa = a_it % p.AST;
                    if (!(ok = bar_wait(full_a(sa), (a_it / p.AST) & 1, ctl, SITE_FULL_A))) break;
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sA + (size_t)sa * a_stage);
                    const int t_end = min(p.T, (tg + 1) * p.TG);
                    for (int t = tg * p.TG; t < t_end; ++t) {
                        const int r = t / p.W_f, j = t - r * p.W_f;
                        const uint64_t ad = smem_desc(a0 + (uint32_t)(t - tg * p.TG) * TAP_A_BYTES, 128, 256);
                        const uint32_t bo = slab + tap_off(p, r, j);
                        const uint32_t acc = (cc | t) != 0;
                        mma_f16(tmem, ad, smem_desc(bo, p.CH, 128), p.idesc0, acc);
                        if (p.N1 > 0)
                            mma_f16(tmem + 256, ad, smem_desc(bo + 256 * 16, p.CH, 128), p.idesc1, acc);
                    }
                    mma_commit(empty_a(sa));
                }
                if (ok) mma_commit(empty_b(sb));
            }
            mma_commit(done);
            if (!ok) bar_wait(done, 0, ctl, SITE_DRAIN, false);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- filter loader
        if (lane == 0) {
            int issued = 0;
            bool ok = true;
            for (int cc = 0; cc < p.C16 && ok; ++cc) {
                for (int tg = 0; tg < p.ntg; ++tg) {
                    const int sa = issued % p.AST;
                    if (!(ok = bar_wait(empty_a(sa), ((issued / p.AST) & 1) ^ 1, ctl, SITE_EMPTY_LOAD)))
                        break;
                    const int t0 = tg * p.TG;
                    const uint32_t bytes = (uint32_t)(min(p.T, t0 + p.TG) - t0) * TAP_A_BYTES;
                    const uint16_t *src =
                        p.fa + (((int64_t)mt * p.C16 + cc) * p.T + t0) * (TAP_A_BYTES / 2);
                    mbar_arrive_expect_tx(full_a(sa), bytes);
                    bulk_g2s(smem_u32(sA + (size_t)sa * a_stage), src, bytes, full_a(sa));
                    ++issued;
                }
            }
            if (!ok) {
                for (int it = (issued > p.AST ? issued - p.AST : 0); it < issued; ++it)
                    bar_wait(full_a(it % p.AST), (it / p.AST) & 1, ctl, SITE_DRAIN, false);
            }
        }
        __syncwarp();
    } else {
        // ---------------- slab producers: NCHW -> [c8][phase][row][col][8 ch]
        const int pt = threadIdx.x - 64;
        const int R0 = ho0 * p.s_h;
        const int rows = min(p.RR, p.H_i - R0);
        const uint16_t *__restrict__ xn = p.x + (int64_t)n * p.C_i * p.H_i * p.W_i;
        const int64_t plane = (int64_t)p.H_i * p.W_i;
        for (int cc = 0; cc < p.C16; ++cc) {
            const int sb = cc % p.BST;
            if (!bar_wait(empty_b(sb), ((cc / p.BST) & 1) ^ 1, ctl, SITE_EMPTY_PROD)) break;
            uint8_t *slab = sB + (size_t)sb * p.stage_b;
            if (p.vec) {
                // 8 channels x 8 columns per item: 8 16-byte loads, 8x8 transpose, 8 16-byte stores
                const int cgs = p.W_i / 8;
                const int items = 2 * rows * cgs;
                for (int it = pt; it < items; it += TAP_PROD_WARPS * 32) {
                    const int cg = it % cgs;
                    const int t2 = it / cgs;
                    const int lr = t2 % rows;
                    const int c8 = t2 / rows;
                    const int ci0 = cc * 16 + c8 * 8;
                    uint4 v[8];
                    const uint16_t *src = xn + (int64_t)ci0 * plane + (int64_t)(R0 + lr) * p.W_i + cg * 8;
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        v[e] = (ci0 + e < p.C_i) ? __ldg(reinterpret_cast<const uint4 *>(src + e * plane))
                                                 : make_uint4(0, 0, 0, 0);
                    uint8_t *rowp = slab + (size_t)c8 * p.CH + (size_t)((lr % p.s_h) * p.s_w) * p.PB +
                                    (size_t)((lr / p.s_h) * p.Wh) * 16;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int col = cg * 8 + k;
                        const uint32_t sel = (k & 1) ? 0x7632u : 0x5410u;
                        uint32_t w0, w1, w2, w3;
                        const int wd = k >> 1;
#define IM2WIN_WORD(vv, i) ((i) == 0 ? (vv).x : (i) == 1 ? (vv).y : (i) == 2 ? (vv).z : (vv).w)
                        w0 = __byte_perm(IM2WIN_WORD(v[0], wd), IM2WIN_WORD(v[1], wd), sel);
                        w1 = __byte_perm(IM2WIN_WORD(v[2], wd), IM2WIN_WORD(v[3], wd), sel);
                        w2 = __byte_perm(IM2WIN_WORD(v[4], wd), IM2WIN_WORD(v[5], wd), sel);
                        w3 = __byte_perm(IM2WIN_WORD(v[6], wd), IM2WIN_WORD(v[7], wd), sel);
#undef IM2WIN_WORD
                        uint8_t *dst = rowp + (size_t)(col % p.s_w) * p.PB + (size_t)(col / p.s_w) * 16;
                        *reinterpret_cast<uint4 *>(dst) = make_uint4(w0, w1, w2, w3);
                    }
                }
            } else {
                // one column of 8 channels per item
                const int items = 2 * rows * p.W_i;
                for (int it = pt; it < items; it += TAP_PROD_WARPS * 32) {
                    const int col = it % p.W_i;
                    const int t2 = it / p.W_i;
                    const int lr = t2 % rows;
                    const int c8 = t2 / rows;
                    const int ci0 = cc * 16 + c8 * 8;
                    const uint16_t *src = xn + (int64_t)ci0 * plane + (int64_t)(R0 + lr) * p.W_i + col;
                    uint32_t e16[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) e16[e] = (ci0 + e < p.C_i) ? (uint32_t)__ldg(src + e * plane) : 0u;
                    uint8_t *dst = slab + (size_t)c8 * p.CH +
                                   (size_t)((lr % p.s_h) * p.s_w + col % p.s_w) * p.PB +
                                   (size_t)((lr / p.s_h) * p.Wh + col / p.s_w) * 16;
                    *reinterpret_cast<uint4 *>(dst) = make_uint4(e16[0] | (e16[1] << 16), e16[2] | (e16[3] << 16),
                                                                 e16[4] | (e16[5] << 16), e16[6] | (e16[7] << 16));
                }
            }
            fence_async_smem();
            mbar_arrive(full_b(sb));
        }

        // ---------------- epilogue
        const bool ok = bar_wait(done, 0, ctl, SITE_DONE);
        tc_fence_after();
        if (ok) {
            const int q = warp & 3;
            const int hh = (warp - 2) >> 2;
            uint32_t *stage = reinterpret_cast<uint32_t *>(sB) + (warp - 2) * (32 * 17);
            const int co_base = mt * BM + q * 32;
            const int nblk = (p.NTp + 31) / 32;
            for (int blk = hh; blk < nblk; blk += 2) {
                const int col = blk * 32;
                uint32_t r[32];
                tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)col, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    stage[lane * 17 + i] = pack2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]), p.bf16);
                __syncwarp();
                const int pp = col + lane;
                const int qrow = pp / p.Wh;
                const int wo = pp - qrow * p.Wh;
                const int ho = ho0 + qrow;
                const bool pv = pp < p.NT && wo < p.W_o && ho < p.H_o;
                const uint16_t *st16 = reinterpret_cast<const uint16_t *>(stage);
                for (int row = 0; row < 32; ++row) {
                    const int co = co_base + row;
                    if (pv && co < p.C_o)
                        p.out[(((int64_t)n * p.C_o + co) * p.H_o + ho) * p.W_o + wo] = st16[row * 34 + lane];
                }
                __syncwarp();
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, p.tmem_cols);
    }
}

// Filter tiles for the tap kernel: fa[mt][cc][t][g][c][row][e] holds
// filt[mt*128 + g*8 + row][cc*16 + c*8 + e][r][j] for tap t = r*W_f + j
// (zero outside the filter). Block 0 also clears the status word.
__global__ void relayout_filter_tap(const uint16_t *__restrict__ filt, uint16_t *__restrict__ fa,
                                    uint32_t *status, int64_t total, int C_i, int C_o, int T, int C16) {
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        status[0] = 0;
        status[1] = 0;
        status[2] = 0;
    }
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int e = (int)(idx & 7), rw = (int)((idx >> 3) & 7), c = (int)((idx >> 6) & 1),
                  g = (int)((idx >> 7) & 15);
        const int64_t rest = idx >> 11;
        const int t = (int)(rest % T);
        const int64_t rest2 = rest / T;
        const int cc = (int)(rest2 % C16);
        const int mt = (int)(rest2 / C16);
        const int co = mt * BM + g * 8 + rw;
        const int ci = cc * 16 + c * 8 + e;
        uint16_t v = 0;
        if (co < C_o && ci < C_i) v = filt[((int64_t)co * C_i + ci) * T + t];
        fa[idx] = v;
    }
}

struct TapPlan {
    bool ok;
    TapParams p;
    size_t smem;
    int mtiles;
};

// Choose the tap kernel's tiling for a shape, or report that it does not fit.
TapPlan plan_tap(const Shape &s) {
    TapPlan pl{};
    pl.ok = false;
    if (s.C_i < 16) return pl;
    const int64_t Wh = (s.W_i + s.s_w - 1) / s.s_w;
    if (Wh > TAP_MAX_NT || s.C_i * s.H_i * s.W_i >= (1ll << 31)) return pl;
    const int T = (int)(s.H_f * s.W_f);
    const int64_t smem_max = 227 * 1024 - 1024;
    for (int64_t Qmax = std::min<int64_t>(s.H_o, TAP_MAX_NT / Wh); Qmax >= 1; --Qmax) {
        const int64_t tiles = (s.H_o + Qmax - 1) / Qmax;
        const int64_t Q = (s.H_o + tiles - 1) / tiles;
        const int64_t NT = Q * Wh;
        const int64_t NTp = (NT + 15) / 16 * 16;
        const int64_t RR = (Q - 1) * s.s_h + s.H_f;
        const int64_t HH = (RR + s.s_h - 1) / s.s_h;
        const int64_t PB = HH * Wh * 16;
        const int64_t CH = s.s_h * s.s_w * PB;
        int64_t max_tap = 0;
        for (int64_t r = 0; r < s.H_f; ++r)
            for (int64_t j = 0; j < s.W_f; ++j)
                max_tap = std::max(max_tap, ((r % s.s_h) * s.s_w + j % s.s_w) * PB +
                                                ((r / s.s_h) * Wh + j / s.s_w) * 16);
        // plane 1 is written up to 2*CH and read up to CH + max_tap + NTp*16
        const int64_t stage_b = (std::max(2 * CH, CH + max_tap + NTp * 16) + 127) / 128 * 128;
        if (stage_b < 8 * 32 * 17 * 4) continue;  // too small to stage the epilogue (never at these sizes)
        for (int BST : {3, 2}) {
            for (int TG : {8, 5, 4, 3, 2, 1}) {
                if (TG > T && TG != 1) continue;
                const int tg = std::min(TG, T);
                for (int AST : {4, 3, 2}) {
                    int64_t total = (int64_t)AST * tg * TAP_A_BYTES + BST * stage_b + 256;
                    if (total > smem_max) continue;
                    // a 512-column TMEM accumulator needs the SM to itself
                    if (NTp > 256) total = std::max<int64_t>(total, 120 * 1024);
                    TapParams &p = pl.p;
                    p.C_i = (int)s.C_i; p.C_o = (int)s.C_o; p.H_i = (int)s.H_i; p.W_i = (int)s.W_i;
                    p.H_o = (int)s.H_o; p.W_o = (int)s.W_o; p.H_f = (int)s.H_f; p.W_f = (int)s.W_f;
                    p.s_h = (int)s.s_h; p.s_w = (int)s.s_w;
                    p.C16 = (int)((s.C_i + 15) / 16);
                    p.T = T;
                    p.TG = tg;
                    p.ntg = (T + tg - 1) / tg;
                    p.Q = (int)Q;
                    p.tiles_h = (int)tiles;
                    p.Wh = (int)Wh;
                    p.HH = (int)HH;
                    p.RR = (int)RR;
                    p.NT = (int)NT;
                    p.NTp = (int)NTp;
                    p.N0 = (int)std::min<int64_t>(256, NTp);
                    p.N1 = (int)(NTp - p.N0);
                    p.PB = (uint32_t)PB;
                    p.CH = (uint32_t)CH;
                    p.stage_b = (uint32_t)stage_b;
                    p.BST = BST;
                    p.AST = AST;
                    p.tmem_cols = NTp > 256 ? 512 : 256;
                    pl.smem = (size_t)total;
                    pl.mtiles = (int)((s.C_o + BM - 1) / BM);
                    pl.ok = tiles * s.N < (1ll << 31) && pl.mtiles < 65536;
                    return pl;
                }
            }
        }
    }
    return pl;
}

struct ExpandGeom {
    int KK, KKP, kstages, mtiles, pos_tiles;
    int64_t K_pad;
};

ExpandGeom expand_geom(const Shape &s) {
    ExpandGeom g;
    g.KK = (int)(s.H_f * s.W_f);
    g.KKP = (g.KK + 7) / 8 * 8;
    g.K_pad = (s.C_i * g.KKP + KS - 1) / KS * KS;
    g.kstages = (int)(g.K_pad / KS);
    g.mtiles = (int)((s.C_o + BM - 1) / BM);
    g.pos_tiles = (int)((s.H_o * s.W_o + NT - 1) / NT);
    return g;
}

}  // namespace

// The fused path takes the tap kernel when its tiling fits, else the expand
// kernel (which also serves the two-step path).
static bool use_tap(const Shape &s, bool fused) { return fused && plan_tap(s).ok; }

size_t conv_tc_filter_bytes(const Shape &s, bool fused) {
    if (use_tap(s, fused)) {
        const TapPlan pl = plan_tap(s);
        return round_up((size_t)pl.mtiles * pl.p.C16 * pl.p.T * TAP_A_BYTES, 256);
    }
    const ExpandGeom g = expand_geom(s);
    return round_up((size_t)g.mtiles * BM * (size_t)g.K_pad * 2, 256);
}

bool conv_tc_supported(const Shape &s, bool fused) {
    if (use_tap(s, fused)) return true;
    const int64_t img = fused ? s.C_i * s.H_i * s.W_i : s.C_i * s.H_o * s.W_i * s.H_f;
    const int64_t KKP = (s.H_f * s.W_f + 7) / 8 * 8;
    const int64_t P = s.H_o * s.W_o;
    const int64_t pos_tiles = (P + NT - 1) / NT;
    return img < (1ll << 31) && s.C_i * KKP < (1ll << 30) && P < (1ll << 31) &&
           pos_tiles * s.N < (1ll << 31) && (s.C_o + BM - 1) / BM < 65536;
}

static cudaError_t launch_tap(const void *x, const void *filt, void *out, void *ws, const Shape &s,
                              bool bf16, cudaStream_t st) {
    TapPlan pl = plan_tap(s);
    TapParams p = pl.p;
    uint32_t *status = static_cast<uint32_t *>(ws);
    uint16_t *fa = reinterpret_cast<uint16_t *>(static_cast<unsigned char *>(ws) + kStatusBytes);
    const int64_t total = (int64_t)pl.mtiles * p.C16 * p.T * (TAP_A_BYTES / 2);
    relayout_filter_tap<<<(unsigned)std::min<int64_t>((total + 255) / 256, 8192), 256, 0, st>>>(
        static_cast<const uint16_t *>(filt), fa, status, total, p.C_i, p.C_o, p.T, p.C16);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    p.x = static_cast<const uint16_t *>(x);
    p.fa = fa;
    p.out = static_cast<uint16_t *>(out);
    p.status = status;
    p.vec = (s.W_i % 8 == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0) ? 1 : 0;
    p.idesc0 = make_idesc(bf16, BM, p.N0);
    p.idesc1 = make_idesc(bf16, BM, p.N1 > 0 ? p.N1 : 16);
    p.bf16 = bf16 ? 1 : 0;
    e = cudaFuncSetAttribute(conv_tc_tap_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(p.tiles_h * s.N), (unsigned)pl.mtiles);
    conv_tc_tap_kernel<<<grid, TAP_THREADS, pl.smem, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_conv_tc(const void *src, const void *filt, void *out, void *ws, const Shape &s,
                           bool fused, bool bf16, cudaStream_t st) {
    if (use_tap(s, fused)) return launch_tap(src, filt, out, ws, s, bf16, st);
    const ExpandGeom g = expand_geom(s);
    uint32_t *status = static_cast<uint32_t *>(ws);
    uint16_t *fa = reinterpret_cast<uint16_t *>(static_cast<unsigned char *>(ws) + kStatusBytes);
    const int64_t total = (int64_t)g.mtiles * BM * g.K_pad;
    relayout_filter_expand<<<(unsigned)std::min<int64_t>((total + 255) / 256, 8192), 256, 0, st>>>(
        static_cast<const uint16_t *>(filt), fa, status, total, (int)s.C_i, (int)s.C_o, (int)s.H_f,
        (int)s.W_f, g.KK, g.KKP, g.kstages);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || s.N == 0) return e;

    TcParams p;
    p.src = static_cast<const uint16_t *>(src);
    p.fa = fa;
    p.out = static_cast<uint16_t *>(out);
    p.status = status;
    p.C_i = (int)s.C_i;
    p.C_o = (int)s.C_o;
    p.H_i = (int)s.H_i;
    p.W_i = (int)s.W_i;
    p.H_o = (int)s.H_o;
    p.W_o = (int)s.W_o;
    p.H_f = (int)s.H_f;
    p.W_f = (int)s.W_f;
    p.s_h = (int)s.s_h;
    p.s_w = (int)s.s_w;
    p.KK = g.KK;
    p.KKP = g.KKP;
    p.P = (int)(s.H_o * s.W_o);
    p.L = (int)(s.W_i * s.H_f);
    p.S = (int)(s.s_w * s.H_f);
    p.kstages = g.kstages;
    p.pos_tiles = g.pos_tiles;
    p.img_src = fused ? s.C_i * s.H_i * s.W_i : s.C_i * s.H_o * s.W_i * s.H_f;
    p.fa_tile = (int64_t)BM * g.K_pad;
    p.div_KKP = make_fastdiv((uint32_t)g.KKP);
    p.div_Hf = make_fastdiv((uint32_t)s.H_f);
    p.div_Wo = make_fastdiv((uint32_t)s.W_o);
    p.idesc = make_idesc(bf16, BM, NT);
    p.bf16 = bf16 ? 1 : 0;

    dim3 grid((unsigned)(g.pos_tiles * s.N), (unsigned)g.mtiles);
    if (fused) {
        e = cudaFuncSetAttribute(conv_tc_expand_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)SMEM_BYTES);
        if (e != cudaSuccess) return e;
        conv_tc_expand_kernel<true><<<grid, NTHREADS, SMEM_BYTES, st>>>(p);
    } else {
        e = cudaFuncSetAttribute(conv_tc_expand_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)SMEM_BYTES);
        if (e != cudaSuccess) return e;
        conv_tc_expand_kernel<false><<<grid, NTHREADS, SMEM_BYTES, st>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace im2win
