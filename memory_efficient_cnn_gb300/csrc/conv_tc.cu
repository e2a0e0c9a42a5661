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
// This file holds two kernel families. The tap kernels (second half of the
// file) run every shape a tiling exists for, in both layouts and with padding
// and dilation. The "expand" kernel is the NCHW fallback for the rest: every
// pipeline stage covers 64 values of K; producer warps gather, for each of the
// tile's 256 pixels, its 64
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

#include <cuda.h>
#include <cudaTypedefs.h>
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
                    // pixels 0..127 and 128..255 in two accumulators: independent MMAs
                    mma_f16(tmem, ad, bd, p.idesc, (it | u) != 0);
                    mma_f16(tmem + NT / 2, ad, bd + ((NT / 2 / 8 * 1024) >> 4), p.idesc, (it | u) != 0);
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
            if (!warp_bar_wait(empty(s), ph ^ 1, ctl, SITE_EMPTY_PROD)) break;
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

        // ---------------- epilogue: TMEM -> registers -> smem transpose -> coalesced stores
        const bool ok = warp_bar_wait(done, 0, ctl, SITE_DONE);
        tc_fence_after();
        if (ok) {
            const int q = warp & 3;              // TMEM lane quarter this warp may read
            const int hh = (warp - 2) >> 2;      // which half of the column blocks
            const int co0 = mt * BM + q * 32;
            uint16_t *out_c = p.out + ((int64_t)n * p.C_o + co0) * p.P;
            drain_accumulator(tmem + ((uint32_t)(q * 32) << 16), hh, NT / 32, 2,
                              reinterpret_cast<uint32_t *>(sB) + (warp - 2) * (32 * 17),
                              min(32, p.C_o - co0), (int64_t)p.P, p.bf16, [&](int col) -> uint16_t * {
                                  const int pidx = pos0 + col;
                                  return pidx < p.P ? out_c + pidx : nullptr;
                              });
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
// Tap kernels: every K step is a plain descriptor offset into a staged slab,
// so shared memory holds each staged element once (no im2col expansion).
//
// TAP_CH (fused, many input channels). The CTA owns Q whole output rows of one
// image and 128 output channels. Per 16-channel chunk the slab holds the
// unique input elements under those rows with the channels innermost, split
// into s_h x s_w polyphase blocks:
//   slab[c8][row % s_h][col % s_w][row / s_h][col / s_w][8 channels]   (16 B entries)
// Output pixel (q, w') is position p = q*pitch + w' (pitch = ceil(W_i/s_w));
// for filter tap (r, j) consecutive positions are consecutive slab entries, so
// the tap's B operand is the slab seen from a constant offset (K = the 16
// channels, the two 8-channel halves one plane apart).
//
// TAP_WX / TAP_WW (few input channels; fused from x / from the window tensor).
// The slab holds the im2win window rows of one channel under the tile's
// output rows, re-laid so that K runs along the window: with S = s_w*H_f the
// window row win[m*S + b] (b < S, m = column group) is stored as
//   slab[b / 8][q][m][b % 8]                                             (16 B entries)
// Output pixel (q, wo) uses window elements (wo + a)*S + b for a < ceil(W_f/s_w),
// so tap a, K group u is again a constant offset (a entries along m, 2u chunks
// along b): the contiguous-window property of im2win becomes a descriptor stride.
//
// In every mode one tcgen05.mma (M = 128 output channels, N <= 256 positions,
// K = 16) is issued per tap and half tile; positions whose column is >= W_o are
// computed and discarded. Filter tiles arrive per (chunk, group of taps) by
// bulk copy, pre-laid by a re-layout kernel as [tap][co group][K half][8 co][8 K].
// Raw source rows, where a staging ring exists, arrive by bulk copies too.
// The channel modes also take zero padding (the slab spans the padded width;
// producers zero-fill outside the input) and dilation (tap (r, j) reads slab
// row r*d_h, column j*d_w); TAP_CL is the channel mode on channels-last input.
// =========================================================================
// TAP_CL (channels-last input, C_i a multiple of 8): the slab of TAP_CH, whose
// 16-byte entries (8 channels of one input position) are 16 contiguous bytes of
// an NHWC input. Producers copy each entry straight from global memory with
// cp.async and never touch it; the copies' completion is tracked by the slab
// barrier (cp.async.mbarrier.arrive.noinc), and the MMA issuers order the
// copies before their reads with a proxy fence after the barrier wait.
enum TapMode { TAP_CH = 0, TAP_WX = 1, TAP_WW = 2, TAP_CL = 3 };

// Tap stacking (TAP_CH with C_o <= 64, so half of M = 128 would be idle).
// Taps (r, j) and (r, j + s_w) lie in the same polyphase block, one slab entry
// apart. One MMA at the B offset of (r, j) with A rows 0..63 = filter of (r, j)
// and rows 64..127 = filter of (r, j + s_w) leaves in accumulator rows 64..127
// the contribution of (r, j + s_w) to the position one column to the left; the
// epilogue adds D[co + 64][p + 1] to D[co][p]. Group k of a filter row has its
// top tap at j = (k / s_w) * 2 s_w + k % s_w (every column whose j / s_w is
// even) and its bottom tap at j + s_w when that is < W_f.
__host__ __device__ inline int stacked_top_j(int k, int s_w) { return (k / s_w) * 2 * s_w + k % s_w; }
__host__ __device__ inline int stacked_groups_per_row(int W_f, int s_w) {
    return (W_f / (2 * s_w)) * s_w + (W_f % (2 * s_w) < s_w ? W_f % (2 * s_w) : s_w);
}

constexpr int TAP_PROD_WARPS = 8;
constexpr int kMaxSlabStages = 6;
constexpr int kMnK = 2;  // 16-channel K steps per chunk of an MN-major 1x1 slab
constexpr int TAP_EPI_WARPS = 8;
constexpr int TAP_ISSUER1_WARP = 2 + TAP_PROD_WARPS + TAP_EPI_WARPS;  // the second MMA issuer
constexpr int TAP_THREADS = (3 + TAP_PROD_WARPS + TAP_EPI_WARPS) * 32;
constexpr uint32_t TAP_A_BYTES = BM * 16 * 2;  // one K=16 tap of 128 channels: 4 KB
constexpr int TAP_MAX_NT = 512;
// Epilogue staging per warp: 64-column blocks of 32 x 33 words. Without tap
// stacking a warp stages its whole share of an accumulator (two blocks) before
// releasing it; the stacked drain goes one block at a time.
constexpr int TAP_EPI_BLOCK_WORDS = 32 * 33;
__host__ __device__ constexpr uint32_t tap_epi_bytes(int blocks) {
    return (uint32_t)(TAP_EPI_WARPS * blocks * TAP_EPI_BLOCK_WORDS * 4);
}
// Transposed stacking (positions along M): the epilogue stages no outputs; its
// only shared memory is the hand-over of each lane quarter's first row,
// [tile parity][M block][lane quarter][channel half][32] fp32 values.
constexpr uint32_t TAP_XB_BYTES = 2 * 2 * 4 * 2 * 32 * 4;
__host__ __device__ constexpr uint32_t tap_epi_region(int blocks, int xpose) {
    return xpose ? TAP_XB_BYTES : tap_epi_bytes(blocks);
}

struct TapParams {
    // CH with a raw ring: the input as a 4-D tensor (W_i, H_i, C_i, N) whose box
    // (W_i, raw rows, 16 channels, 1) is one chunk's raw rows (tma_raw). CL with
    // whole 16-byte entries: the input as (C_i, W_i, H_i, N), box (8, pitch*s_w,
    // rows per phase*s_h, 1) traversed with element strides (1, s_w, s_h, 1): one
    // polyphase block of one 8-channel half of a chunk's slab (tma_slab).
    CUtensorMap tmap_x;    // (the type is 128-byte aligned)
    int tma_raw, tma_slab;
    int slab_hh;           // CL with tma_slab: rows of a polyphase block
    // CH, 1x1 filter at stride 1 without padding (the input is its own window): a
    // chunk is 16*mn_k channels, its slab the tile's input positions x those channels
    // held MN-major, one tensor copy per chunk; the MMAs read it with the B
    // transpose bit set, and its T = mn_k "taps" are the 16-channel K steps.
    //  mnb = 1: no swizzle (8 positions x 8 channels per 128-byte core matrix,
    //    [position group][channel][position]): the input seen as (8, C_i, H_i*W_i/8,
    //    N), box (8, 16*mn_k, mn_box/8, 1); K steps 256 bytes apart.
    //  mnb = 2: 128-byte swizzle, where planes and tiles are whole 64-position
    //    blocks: the input seen as (64, C_i, H_i*W_i/64, N), box (64, 16*mn_k,
    //    mn_box/64, 1) with the copy's 128-byte swizzle, so that [block][channel]
    //    rows of 64 positions (128 bytes) land with their 16-byte pieces permuted by
    //    the row index mod 8 -- the MMA's 128-byte-swizzled MN-major layout (8
    //    channels x 64 positions per 1024-byte atom; blocks lbo = 2048*mn_k bytes
    //    apart, 8-channel groups 1024); K steps 2048 bytes apart. The copy then
    //    moves 128-byte rows instead of 16-byte ones.
    // CL, the same filter with channels in whole 64s (mnb = 3): a chunk is 64
    // channels (mn_k = 4 K steps) of the tile's mn_box positions, held K-major with
    // the 128-byte swizzle: one tensor copy of the input seen as (C_i, W_i, H_i, N),
    // box (64, W_i, rows per tile, 1), writes each position's 64 channels as one
    // 128-byte row, 16-byte pieces permuted by the row index mod 8 (the MMA's
    // 128-byte-swizzled K-major layout: 8-position groups 1024 bytes apart); K steps
    // 32 bytes apart within the rows.
    int mnb, mn_box, mn_k;
    const uint16_t *src;   // NCHW input (CH, WX), window tensor (WW), NHWC input (CL)
    const uint16_t *fa;
    uint16_t *out;
    uint32_t *status;
    int C_i, C_o, H_i, W_i, H_o, W_o, H_f, W_f, s_h, s_w;
    int MT;                // 128-channel output tiles
    int NCH;               // chunks: 16-channel groups (CH) or channels (WX, WW)
    int T;                 // K=16 taps per chunk
    int TG, ntg;           // taps per filter stage, filter stages per chunk
    int Qmax;              // output rows per tile at most
    int tps;               // tiles per (image, channel tile)
    int64_t tiles_total;   // N * MT * tps
    int pitch;             // positions per output row of a tile
    uint32_t lbo;          // CH: bytes of an 8-channel plane; W*: bytes of a K chunk
    uint32_t PB;           // CH: bytes of a phase block
    int U, S, A;           // W*: K=16 groups per window step, window step s_w*H_f, taps along m
    int64_t L;             // WW: window row length W_i*H_f
    int64_t win_elems;     // WW: elements of the window tensor
    int N_img;             // images (bound of the staged reads)
    int raw_elems;         // elements of the raw staging area (all slots)
    int ring;              // 1: raw chunks staged two deep (next chunk's bulk copy in flight)
    int raw_slot;          // elements of one raw slot (a multiple of 64)
    int raw_ch;            // CH with ring: elements per channel plane of a slot (raw_rows x raw_w, padded)
    int raw_rows, raw_w;   // CH with ring: rows of a plane, elements per raw row (the tensor copy's
                           // box; W_i when per-channel bulk copies stage the rows)
    uint32_t stage_b;      // bytes of one slab stage
    int BST, AST;          // slab stages, filter stages
    int merge;             // one filter stage per chunk and AST == BST: a chunk's filter copy
                           // completes on its slab stage's full barrier and the stage's release
                           // is the slab's (one wait and one commit per chunk for the issuers)
    int vec;               // CH: 16-byte row loads possible
    int bf16;
    FastDiv div_pitch;     // W*: positions -> (output row, column group)
    FastDiv div_cgs, div_sh, div_sw;  // CH: 8-column groups per row, strides
    int stack;             // CH, C_o <= 64: two taps per MMA, stacked along M (see below)
    int xpose;             // stacked, transposed: positions along M, the two taps along N
    int Gr;                // stacked: tap groups per filter row
    int nhwc;              // output out[n][ho][wo][co] (else out[n][co][ho][wo])
    FastDiv div_wi;        // CL: positions of a slab row (W_i, or Wp when padded)
    // zero padding and dilation (CH / CL). Filter tap (r, j) reads slab row
    // r*dil_h and column (j / g_w)*dil_w*g_w + j % g_w relative to the output's
    // origin; the slab covers the Wp = W_i + 2 p_w padded columns, and with
    // padding its entry (row lr, column col) is input (ho0*s_h + lr - p_h, col - p_w),
    // zero outside the input.
    int p_h, p_w, dil_h, dil_w, g_w;
    int Hfe;               // slab rows a filter spans: (H_f - 1)*dil_h + 1
    int Wp;                // slab columns
    int padded;            // p_h or p_w > 0: the producers zero-fill outside the input
    int epi_blocks;        // staging blocks per epilogue warp (2, or 1 when stacked)
};

// A tile: output rows [ho0, ho0 + Q) of image n, output channels [mt*128, mt*128 + 128).
struct TapTile {
    int n, mt, ho0, Q;
};

// Tiles: each (image, channel tile) segment of H_o output rows is cut into
// tps tiles of at most Qmax rows; tile id = (n*MT + mt)*tps + th. CTA b takes
// tiles b, b + gridDim.x, ... Every role of the CTA walks the same sequence.
__device__ __forceinline__ void tile_at(const TapParams &p, int64_t id, TapTile &t) {
    const int64_t nm = id / p.tps;
    const int th = (int)(id - nm * p.tps);
    t.n = (int)(nm / p.MT);
    t.mt = (int)(nm - (int64_t)t.n * p.MT);
    t.ho0 = th * p.Qmax;
    t.Q = min(p.Qmax, p.H_o - t.ho0);
}

// MMA split of a tile's NTp positions into two accumulators [0, N0) and
// [N0, NTp) so that consecutive MMAs never wait on each other; N0 is a multiple
// of 32 so that each accumulator's columns start on a 32-column TMEM load (of
// 64 with a 128-byte-swizzled MN-major slab: the second accumulator's operand
// then starts on a swizzle atom). The
// boundary is the same for every tile of a launch (that of the widest tile):
// an accumulator is released as soon as it is drained, so the next tile's MMAs
// into it must not reach columns of the other, possibly still draining, one.
// A narrower tile may leave the second accumulator empty.
__host__ __device__ __forceinline__ int split_n0(int NTp, int step = 32) {
    return NTp >= step ? min(NTp, (NTp / 2 + step - 1) / step * step) : NTp;
}
// Accumulator columns of a tile of NT positions: whole 16-column MMA widths
// (with stacking one column more), whole 64-position blocks of a swizzled
// MN-major slab (a short last tile reads the zeros or rows past its own, which
// the epilogue does not store).
__device__ __forceinline__ int tile_ntp(const TapParams &p, int NT) {
    return p.mnb == 2 ? (NT + 63) / 64 * 64 : (NT + p.stack + 15) / 16 * 16;
}
__device__ __forceinline__ int tile_n0(const TapParams &p, int NTp) {
    return min(NTp, split_n0((p.Qmax * p.pitch + p.stack + 15) / 16 * 16, p.mnb == 2 ? 64 : 32));
}

// Slab row and column offsets of filter tap (r, j) (dilation; see TapParams).
__host__ __device__ inline int tap_dr(int r, int dil_h) { return r * dil_h; }
__host__ __device__ inline int tap_dc(int j, int dil_w, int g_w) { return (j / g_w) * dil_w * g_w + j % g_w; }

template <int MODE>
__device__ __forceinline__ uint32_t tap_offset(const TapParams &p, int t) {
    if (MODE == TAP_CH && p.mnb) return (uint32_t)t * (p.mnb == 2 ? 2048u : 256u);  // K step t, MN-major slab
    if (MODE == TAP_CL && p.mnb == 3) return (uint32_t)t * 32u;  // K step t, swizzled K-major 1x1 slab
    if (MODE == TAP_CH || MODE == TAP_CL) {
        const int r = t / p.W_f, j = t - r * p.W_f;
        const int dr = tap_dr(r, p.dil_h), dc = tap_dc(j, p.dil_w, p.g_w);
        return (uint32_t)((((dr % p.s_h) * p.s_w + (dc % p.s_w)) * p.PB) +
                          (((dr / p.s_h) * p.pitch + (dc / p.s_w)) * 16));
    } else {
        const int a = t / p.U, u = t - a * p.U;
        return (uint32_t)(2 * u) * p.lbo + (uint32_t)a * 16u;
    }
}

// 16-byte asynchronous copy global -> shared; bytes past src_bytes (0..16) are zero.
__device__ __forceinline__ void cp_async16z(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit_group() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// word i of v for a run-time i, by selects (no indexed registers)
__device__ __forceinline__ uint32_t word_sel(const uint4 &v, int i) {
    const uint32_t lo = (i & 1) ? v.y : v.x, hi = (i & 1) ? v.w : v.z;
    return (i & 2) ? hi : lo;
}

// Persistent: one CTA per SM, each owning an equal share of the output rows.
// Warp 0 issues the MMAs, warp 1 streams filter tiles, warps 2..9 fill the
// slabs and warps 10..17 drain the accumulators, so the epilogue of one tile
// and the slab fill of the next overlap the MMAs.
template <int MODE>
__global__ void __launch_bounds__(TAP_THREADS, 1) conv_tc_tap_kernel(const __grid_constant__ TapParams p) {
    constexpr bool CHAN = MODE == TAP_CH || MODE == TAP_CL;  // slab over channels
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t a_stage = (uint32_t)p.TG * TAP_A_BYTES;
    uint8_t *sA = smem;
    uint8_t *sB = smem + (size_t)p.AST * a_stage;
    uint16_t *sRaw = reinterpret_cast<uint16_t *>(sB + (size_t)p.BST * p.stage_b);
    uint32_t *sE = reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(sRaw) +
                                                ((size_t)p.raw_elems * 2 + 127) / 128 * 128);
    uint64_t *bars =
        reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(sE) + tap_epi_region(p.epi_blocks, p.xpose));
    // [A stages][slab stages][raw rows (W modes)][epilogue staging] then
    // bars: full_a[AST] | empty_a[AST] | full_b[BST] | empty_b[BST] | tmem_full[4] | tmem_empty[4]
    //       | drain | stacked hand-over: full[4] | empty[4] | raw slot full[2]
    const int nb = 2 * p.AST + 2 * p.BST + 9 + 8 + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + nb);
    int *abort_word = reinterpret_cast<int *>(tmem_slot + 1);
    uint32_t *toff = reinterpret_cast<uint32_t *>(bars + nb + 1);  // [T] tap offsets (16-byte units)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // W modes: per K chunk row c and element e of a slab entry, the raw offset
    // from the entry's base and the limit on m*mstride below which it exists
    int *wtab = reinterpret_cast<int *>((reinterpret_cast<uintptr_t>(toff + p.T) + 15) & ~(uintptr_t)15);
    if (!CHAN) {
        for (int b = threadIdx.x; b < 16 * p.U; b += blockDim.x) {
            if (MODE == TAP_WX) {
                const int jl = b / p.H_f, r = b - jl * p.H_f;
                wtab[b] = r * p.W_i + jl;
                wtab[16 * p.U + b] = b < p.S ? p.W_i - jl : 0;  // column m*s_w + jl < W_i
            } else {
                wtab[b] = b;
                wtab[16 * p.U + b] = b < p.S ? (int)p.L - b : 0;  // window index m*S + b < L
            }
        }
    }
    for (int t = threadIdx.x; t < p.T; t += blockDim.x) {
        // a stacked group is issued at its top tap
        const int tap = p.stack ? (t / p.Gr) * p.W_f + stacked_top_j(t % p.Gr, p.s_w) : t;
        toff[t] = tap_offset<MODE>(p, tap) >> 4;  // 16-byte units
    }

    auto full_a = [&](int s) { return smem_u32(bars + s); };
    auto empty_a = [&](int s) { return smem_u32(bars + p.AST + s); };
    auto full_b = [&](int s) { return smem_u32(bars + 2 * p.AST + s); };
    auto empty_b = [&](int s) { return smem_u32(bars + 2 * p.AST + p.BST + s); };
    // one full / empty pair per accumulator: the epilogue drains accumulator 0 and
    // then 1, so each issuer restarts as soon as its own accumulator is drained.
    // Accumulator 2*buf + which: transposed stacking double-buffers (buf = tile
    // parity), the other layouts use buf 0 only.
    auto tmem_full = [&](int a) { return smem_u32(bars + 2 * p.AST + 2 * p.BST + a); };
    auto tmem_empty = [&](int a) { return smem_u32(bars + 2 * p.AST + 2 * p.BST + 4 + a); };
    const uint32_t drain = smem_u32(bars + 2 * p.AST + 2 * p.BST + 8);
    auto xfull = [&](int i) { return smem_u32(bars + 2 * p.AST + 2 * p.BST + 9 + i); };
    auto xempty = [&](int i) { return smem_u32(bars + 2 * p.AST + 2 * p.BST + 13 + i); };
    // raw staging slots (TAP_CH ring, TAP_WX, TAP_WW): their bulk copies complete here
    auto raw_full = [&](int i) { return smem_u32(bars + 2 * p.AST + 2 * p.BST + 17 + i); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.AST; ++s) {
            mbar_init(full_a(s), 1);
            mbar_init(empty_a(s), 2);  // both MMA issuers commit
        }
        // a slab stage is filled by one producer group (all producers when there is one)
        // (with tma_slab one thread completes a stage: its arrival and the copies' bytes)
        const bool one_group = !(MODE == TAP_CH && p.ring);
        for (int s = 0; s < p.BST; ++s) {
            mbar_init(full_b(s), (((MODE == TAP_CL && p.tma_slab) || (MODE == TAP_CH && p.mnb)) ? 1
                                  : one_group                     ? TAP_PROD_WARPS * 32
                                                                  : TAP_PROD_WARPS * 16) +
                                     (p.merge ? 1 : 0));
            mbar_init(empty_b(s), 2);
        }
        for (int a = 0; a < 4; ++a) {
            mbar_init(tmem_full(a), 1);
            mbar_init(tmem_empty(a), TAP_EPI_WARPS);
        }
        mbar_init(drain, 2);
        for (int i = 0; i < 4; ++i) {
            mbar_init(xfull(i), 1);  // lane 0 of the writing / reading warp
            mbar_init(xempty(i), 1);
        }
        for (int i = 0; i < 2; ++i) mbar_init(raw_full(i), 1);
        *abort_word = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(tmem_slot);
    const Ctl ctl{reinterpret_cast<volatile int *>(abort_word), p.status};
    // Only the filter loader reads what the re-layout kernel writes (the filter
    // tiles); it alone waits for that kernel, so the prologue and the first slab
    // fills overlap it. (The re-layout kernel also clears the status word, in
    // microseconds; a wait gives up only after seconds.) Everything earlier in
    // the stream is complete: the re-layout kernel started after it.

    if (warp == 0 || warp == TAP_ISSUER1_WARP) {
        // ---------------- MMA issuers
        // A tile's positions are split over two accumulators, TMEM columns [0, N0)
        // and [N0, NTp); warp 0 issues the MMAs of the first, the last warp those of
        // the second, in parallel. One thread issues each stream, so its own
        // instruction latency bounds the rate: stage indices and phases are ring
        // counters, descriptors are built in 32-bit halves from tap offsets
        // pre-shifted to 16-byte units, and the next tap's offset is loaded while
        // the current one issues. Both issuers wait on every stage and both commit
        // (the stage, accumulator and teardown barriers count two arrivals); an
        // issuer with no columns (a tile of one accumulator) commits without MMAs.
        if (lane == 0) {
            const int which = warp == 0 ? 0 : 1;
            bool ok = true;
            int k = 0;
            int sb = 0, sa = 0;
            uint32_t phb = 0, pha = 0;
            // (an MN-major slab: K halves lbo = 128 bytes apart, position groups 256*mn_k;
            // swizzled: 64-position blocks lbo apart, 8-channel groups 1024 bytes,
            // layout type 2 = 128-byte swizzle; the swizzled K-major 1x1 slab:
            // 8-position groups 1024 bytes apart, the leading offset unused)
            const uint64_t adesc0 = smem_desc(0, 128, 256),
                           bdesc0 = p.mnb >= 2 ? (smem_desc(0, p.lbo, 1024u) | (2ull << 61))
                                               : smem_desc(0, p.lbo, p.mnb ? 256u * (uint32_t)p.mn_k : 128u);
            const uint32_t a_hi = (uint32_t)(adesc0 >> 32), b_hi = (uint32_t)(bdesc0 >> 32);
            const uint32_t a_lo_base = (uint32_t)adesc0 + (smem_u32(sA) >> 4);
            const uint32_t b_lo_base = (uint32_t)bdesc0 + (smem_u32(sB) >> 4);
            const uint32_t a_stage16 = a_stage >> 4, b_stage16 = p.stage_b >> 4;
            TapTile tl;
            for (int64_t id = blockIdx.x; ok && id < p.tiles_total; id += gridDim.x) {
                tile_at(p, id, tl);
                // transposed stacking: tile k uses TMEM buffer k & 1, last used by tile k - 2
                const int buf = p.xpose ? (k & 1) : 0;
                const int acc = 2 * buf + which;
                if (p.xpose ? k >= 2 : k > 0) {
                    // the accumulator's previous tile must be drained
                    const uint32_t par = (uint32_t)(p.xpose ? (k >> 1) - 1 : k - 1) & 1u;
                    if (!(ok = bar_wait(tmem_empty(acc), par, ctl, SITE_EMPTY_MMA))) break;
                    tc_fence_after();
                }
                int NW;          // this issuer's accumulator columns (0: none this tile)
                uint32_t col0;   // first slab position its MMAs read, relative to the tile
                uint32_t idesc, d_tmem;
                if (p.xpose) {
                    // M block `which` (positions which*128 ..) of the tile's Q*pitch + 1
                    // positions; D = slab rows x filter rows, 128 x 128
                    const int nmb = (tl.Q * p.pitch + 1 + 127) / 128;
                    NW = which < nmb ? 128 : 0;
                    col0 = (uint32_t)which * 128u;
                    idesc = make_idesc(p.bf16 != 0, 128, 128);
                    d_tmem = tmem + (uint32_t)(buf * 256 + which * 128);
                } else {
                    // stacked: one more column, read by the epilogue for the shifted rows
                    const int NTp = tile_ntp(p, tl.Q * p.pitch);
                    const int N0 = tile_n0(p, NTp);
                    NW = which == 0 ? N0 : NTp - N0;
                    // slab offset of the issuer's first position, in 16-byte units (MN-major:
                    // 32*mn_k bytes per position, in 8- or 64-position blocks; the swizzled
                    // K-major 1x1 slab: a 128-byte row per position)
                    col0 = which == 0 ? 0u
                                      : (uint32_t)N0 * (p.mnb == 3 ? 8u : p.mnb ? 2u * (uint32_t)p.mn_k : 1u);
                    idesc = make_idesc(p.bf16 != 0, BM, NW > 0 ? NW : 16) |
                            ((p.mnb == 1 || p.mnb == 2) ? 1u << 16 : 0u);
                    d_tmem = tmem + (which == 0 ? 0u : (uint32_t)N0);
                }
                for (int cc = 0; cc < p.NCH && ok; ++cc) {
                    if (!(ok = bar_wait(full_b(sb), phb, ctl, SITE_FULL_B))) break;
                    // CL: the slab was written by cp.async (generic proxy), the MMAs read
                    // it through the async proxy
                    if (MODE == TAP_CL) fence_async_smem();
                    const uint32_t b_lo_slab = b_lo_base + (uint32_t)sb * b_stage16 + col0;
                    for (int t0 = 0; t0 < p.T && ok; t0 += p.TG) {
                        // (the filter tile arrived by a bulk copy completing on the barrier:
                        // no tcgen05 fence is needed for the MMAs to read it, and one per
                        // stage costs the issuer ~12% of the MMA rate)
                        if (!p.merge && !(ok = bar_wait(full_a(sa), pha, ctl, SITE_FULL_A))) break;
                        if (NW > 0) {
                            const int t_end = min(p.T, t0 + p.TG);
                            uint32_t a_lo = a_lo_base + (uint32_t)sa * a_stage16;
                            uint32_t off = toff[t0];
                            if (p.xpose) {
                                // the slab is the M operand, the filter tile the N one
                                for (int t = t0; t < t_end; ++t, a_lo += TAP_A_BYTES >> 4) {
                                    const uint32_t off_next = toff[t + 1 < t_end ? t + 1 : t];
                                    const uint64_t ad = ((uint64_t)a_hi << 32) | a_lo;
                                    const uint64_t bd = ((uint64_t)b_hi << 32) | (b_lo_slab + off);
                                    mma_f16(d_tmem, bd, ad, idesc, (cc | t) != 0);
                                    off = off_next;
                                }
                            } else {
                                for (int t = t0; t < t_end; ++t, a_lo += TAP_A_BYTES >> 4) {
                                    const uint32_t off_next = toff[t + 1 < t_end ? t + 1 : t];
                                    const uint64_t ad = ((uint64_t)a_hi << 32) | a_lo;
                                    const uint64_t bd = ((uint64_t)b_hi << 32) | (b_lo_slab + off);
                                    mma_f16(d_tmem, ad, bd, idesc, (cc | t) != 0);
                                    off = off_next;
                                }
                            }
                        }
                        if (!p.merge) mma_commit(empty_a(sa));
                        if (++sa == p.AST) { sa = 0; pha ^= 1; }
                    }
                    if (ok) mma_commit(empty_b(sb));
                    if (++sb == p.BST) { sb = 0; phb ^= 1; }
                }
                if (ok) mma_commit(tmem_full(acc));
                ++k;
            }
            // let every MMA in flight finish before the CTA tears down
            mma_commit(drain);
            bar_wait(drain, 0, ctl, SITE_DRAIN, false);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- filter loader
        if (lane == 0) {
            grid_dependency_wait();
            int issued = 0;
            bool ok = true;
            TapTile tl;
            for (int64_t id = blockIdx.x; ok && id < p.tiles_total; id += gridDim.x) {
                tile_at(p, id, tl);
                for (int cc = 0; cc < p.NCH && ok; ++cc) {
                    for (int tg = 0; tg < p.ntg; ++tg) {
                        const int sa = issued % p.AST;
                        // merged: filter stage sa is the chunk's slab stage
                        const uint32_t ebar = p.merge ? empty_b(sa) : empty_a(sa);
                        const uint32_t fbar = p.merge ? full_b(sa) : full_a(sa);
                        if (!(ok = bar_wait(ebar, ((issued / p.AST) & 1) ^ 1, ctl, SITE_EMPTY_LOAD))) break;
                        const int t0 = tg * p.TG;
                        const uint32_t bytes = (uint32_t)(min(p.T, t0 + p.TG) - t0) * TAP_A_BYTES;
                        const uint16_t *src =
                            p.fa + (((int64_t)tl.mt * p.NCH + cc) * p.T + t0) * (TAP_A_BYTES / 2);
                        mbar_arrive_expect_tx(fbar, bytes);
                        bulk_g2s(smem_u32(sA + (size_t)sa * a_stage), src, bytes, fbar);
                        ++issued;
                    }
                }
            }
            if (!ok) {
                for (int it = (issued > p.AST ? issued - p.AST : 0); it < issued; ++it)
                    bar_wait(p.merge ? full_b(it % p.AST) : full_a(it % p.AST), (it / p.AST) & 1, ctl, SITE_DRAIN,
                             false);
            }
        }
        __syncwarp();
    } else if (warp < 2 + TAP_PROD_WARPS) {
        // ---------------- slab producers
        // Chunks are walked in order (tile by tile, NCH per tile). Their source rows
        // are contiguous in global memory; where a raw staging area exists they are
        // copied there by bulk copies (completing on the slot's barrier) and the slab
        // is built from shared memory. Without one (TAP_CH whose rows are not 16-byte
        // aligned, or whose staging does not fit) the slab is gathered straight from
        // global memory; TAP_CL copies its entries by TMA (or cp.async). For TAP_CH
        // with a raw ring a chunk's fill is mostly latency (copy, barriers,
        // shared-memory round trips), so the producers form two groups of four warps
        // that fill alternate chunks at the same time, each with its own raw slot and
        // named barrier. Otherwise all eight warps fill every chunk (with two slab
        // stages only one chunk can be filled at a time: the other stage is being
        // read by the MMAs, so eight warps halve the fill's latency — cv4 fused 810
        // → 717 µs against two groups), and with two raw slots the next chunk's copy
        // is in flight while this one is re-laid.
        const bool staged = !CHAN || (MODE == TAP_CH && p.ring);
        const int ngroups = (MODE == TAP_CH && p.ring) ? 2 : 1;
        const bool prefetch = ngroups == 1 && staged && p.ring;
        const int grp = ngroups == 2 ? (warp - 2) / (TAP_PROD_WARPS / 2) : 0;
        const int NPT = TAP_PROD_WARPS * 32 / ngroups;  // threads of the group
        const int pt = (threadIdx.x - 64) % NPT;         // thread within the group
        const int bar_id = 1 + grp;
        typedef uint16_t E16;
        bool pok = true;
        int sb = 0;
        uint32_t phb = 0;
        // source range of chunk (tile, cc) and its 16-byte aligned copy into raw slot `slot`
        auto raw_lead_of = [&](const TapTile &t, int cc) -> int {
            if (CHAN) return 0;
            const int64_t g0 = MODE == TAP_WX ? (((int64_t)t.n * p.C_i + cc) * p.H_i + t.ho0 * p.s_h) * p.W_i
                                              : (((int64_t)t.n * p.C_i + cc) * p.H_o + t.ho0) * p.L;
            return (int)(g0 & 7);
        };
        auto issue_raw = [&](const TapTile &t, int cc, int slot) {
            const uint32_t dst0 = smem_u32(sRaw + (size_t)slot * p.raw_slot);
            if (MODE == TAP_CH && p.tma_raw) {
                // Raw row lr of channel k is input row ho0*s_h - p_h + lr of channel
                // cc*16 + k: one tensor copy of the box at (0, ho0*s_h - p_h, cc*16, n),
                // rows outside the input and channels past C_i read as zero. (One copy:
                // the copy engine takes bulk copies one at a time, at a fixed cost each.)
                if (pt == 0) {
                    const uint32_t bar = raw_full(slot);
                    mbar_arrive_expect_tx(bar, (uint32_t)(16 * p.raw_ch) * 2u);
                    tma_load_4d(dst0, &p.tmap_x, 0, t.ho0 * p.s_h - p.p_h, cc * 16, t.n, bar);
                }
            } else if (MODE == TAP_CH) {
                // Raw row lr of channel k is input row ho0*s_h - p_h + lr of channel
                // cc*16 + k. The rows that exist are one contiguous, 16-byte aligned range
                // of each channel plane: one bulk copy per channel, completing on the
                // slot's barrier. Rows outside the input and channels past C_i are
                // zeroed by the group's threads (the group's barrier orders them).
                const int rows = (t.Q - 1) * p.s_h + p.Hfe;
                const int64_t plane = (int64_t)p.H_i * p.W_i;
                const int hb = t.ho0 * p.s_h - p.p_h;
                const int r0 = max(0, -hb), r1 = min(rows, p.H_i - hb);
                const int nch = min(16, p.C_i - cc * 16);
                const uint32_t row_bytes = (uint32_t)p.W_i * 2;
                const uint32_t ch_bytes = r1 > r0 ? (uint32_t)(r1 - r0) * row_bytes : 0u;
                if (pt == 0) {
                    const uint32_t bar = raw_full(slot);
                    if (ch_bytes > 0 && nch > 0) {
                        mbar_arrive_expect_tx(bar, ch_bytes * (uint32_t)nch);
                        const uint16_t *x0 = p.src + ((int64_t)t.n * p.C_i + cc * 16) * plane +
                                             (int64_t)(hb + r0) * p.W_i;
                        for (int k = 0; k < nch; ++k)
                            bulk_g2s(dst0 + (uint32_t)(k * p.raw_ch + r0 * p.W_i) * 2, x0 + (int64_t)k * plane,
                                     ch_bytes, bar);
                    } else {
                        mbar_arrive(bar);
                    }
                }
                if (r0 > 0 || r1 < rows || nch < 16) {
                    // zero rows [0, r0) and [r1, rows) of the channels that exist, every row of
                    // the channels that do not (16-byte stores)
                    const int vpr = p.W_i / 8;  // vectors per row
                    const int nv = 16 * rows * vpr;
                    uint4 *raw16 = reinterpret_cast<uint4 *>(sRaw + (size_t)slot * p.raw_slot);
                    for (int v = pt; v < nv; v += NPT) {
                        const int k = v / (rows * vpr);
                        const int lr = (v - k * rows * vpr) / vpr;
                        if (k >= nch || lr < r0 || lr >= r1)
                            raw16[(k * p.raw_ch + lr * p.W_i) / 8 + (v % vpr)] = make_uint4(0, 0, 0, 0);
                    }
                }
            } else {
                int64_t g0, cnt, total;
                if (MODE == TAP_WX) {
                    g0 = (((int64_t)t.n * p.C_i + cc) * p.H_i + t.ho0 * p.s_h) * p.W_i;
                    cnt = (int64_t)((t.Q - 1) * p.s_h + p.H_f) * p.W_i;
                    total = (int64_t)p.N_img * p.C_i * p.H_i * p.W_i;
                } else {
                    g0 = (((int64_t)t.n * p.C_i + cc) * p.H_o + t.ho0) * p.L;
                    cnt = (int64_t)t.Q * p.L;
                    total = p.win_elems;
                }
                // the rows are one contiguous range of the source: one bulk copy of the
                // 16-byte vectors that lie wholly inside it, completing on the slot's
                // barrier; a partial last vector (the source's end) is copied by hand
                const int lead = (int)(g0 & 7);
                const int64_t base = g0 - lead;
                const int nvec = (int)((lead + cnt + 7) / 8);
                const int64_t inside = (total - base) / 8;
                const int nfull = inside < (int64_t)nvec ? (int)inside : nvec;
                if (pt == 0) {
                    const uint32_t bar = raw_full(slot);
                    if (nfull > 0) {
                        mbar_arrive_expect_tx(bar, (uint32_t)nfull * 16u);
                        bulk_g2s(dst0, p.src + base, (uint32_t)nfull * 16u, bar);
                    } else {
                        mbar_arrive(bar);
                    }
                }
                if (nfull < nvec && pt == NPT - 1) {
                    uint16_t *d = sRaw + (size_t)slot * p.raw_slot + (size_t)nfull * 8;
                    for (int e = 0; e < 8; ++e) {
                        const int64_t gg = base + (int64_t)nfull * 8 + e;
                        d[e] = gg < total ? p.src[gg] : (uint16_t)0;
                    }
                }
            }
        };
        auto next_chunk = [&](int64_t &id, int &cc, TapTile &t) {
            if (++cc == p.NCH) {
                cc = 0;
                id += gridDim.x;
                if (id < p.tiles_total) tile_at(p, id, t);
            }
        };
        if (CHAN && (p.stack || (MODE == TAP_CH && p.vec && p.p_w > 0))) {
            // Entries that no fill writes must read as zero: with padding, the 16-byte
            // fills skip the padding columns; with tap stacking, a group whose second tap
            // is missing multiplies zero filter rows by the entries one column past the
            // input's last (for the column after the last output), and whatever bytes an
            // earlier kernel left there may decode as Inf or NaN. Every stage is cleared
            // once; all producers fence their clears and meet before any chunk is filled.
            const int ptid = threadIdx.x - 64;
            const int n16 = (int)(p.BST * p.stage_b / 16);
            for (int i = ptid; i < n16; i += TAP_PROD_WARPS * 32)
                reinterpret_cast<uint4 *>(sB)[i] = make_uint4(0, 0, 0, 0);
            fence_async_smem();
            asm volatile("bar.sync %0, %1;" ::"r"(3), "r"(TAP_PROD_WARPS * 32) : "memory");
        }
        const bool copy_slab = (MODE == TAP_CL && p.tma_slab) || (MODE == TAP_CH && p.mnb);
        if (copy_slab && warp == 2) {
            // Channels-last input in whole 16-byte entries: each polyphase block (ph_r,
            // ph_c) of each 8-channel half of a chunk's slab is one tensor copy, entry
            // (q, m) being input (row R0 + ph_r + q*s_h, column ph_c + m*s_w - p_w),
            // zero outside the input. An MN-major 1x1 slab (mnb) is one tensor copy of
            // the chunk's 16 channels at the tile's positions (zero past the plane's
            // end or channel C_i), a channels-last one (mnb = 3) one copy of the chunk's
            // 64 channels at the tile's rows (zero past the last input row). One thread
            // issues them all on the stage's barrier;
            // the other producer warps have nothing to do.
            int sbt = 0;
            uint32_t pht = 0;
            bool ok2 = true;
            int pend[kMaxSlabStages];  // per stage: parity of a copy not yet seen landed
            for (int s2 = 0; s2 < kMaxSlabStages; ++s2) pend[s2] = -1;
            const uint32_t bytes = MODE == TAP_CH ? (uint32_t)p.mn_box * 32u * (uint32_t)p.mn_k
                                   : p.mnb == 3   ? (uint32_t)p.mn_box * 128u
                                                  : 2u * (uint32_t)(p.s_h * p.s_w * p.slab_hh * p.pitch) * 16u;
            TapTile t2;
            for (int64_t id2 = blockIdx.x; ok2 && id2 < p.tiles_total; id2 += gridDim.x) {
                tile_at(p, id2, t2);
                const int R0 = t2.ho0 * p.s_h - p.p_h;
                for (int c2 = 0; c2 < p.NCH; ++c2) {
                    if (!(ok2 = warp_bar_wait(empty_b(sbt), pht ^ 1, ctl, SITE_EMPTY_PROD))) break;
                    if (lane == 0 && MODE == TAP_CH) {
                        const uint32_t slab = smem_u32(sB + (size_t)sbt * p.stage_b);
                        mbar_arrive_expect_tx(full_b(sbt), bytes);
                        tma_load_4d(slab, &p.tmap_x, 0, c2 * 16 * p.mn_k, (t2.ho0 * p.W_o) >> (p.mnb == 2 ? 6 : 3),
                                    t2.n, full_b(sbt));
                    } else if (lane == 0 && p.mnb == 3) {
                        // channels-last 1x1: 64 channels of every position of the tile's rows
                        const uint32_t slab = smem_u32(sB + (size_t)sbt * p.stage_b);
                        mbar_arrive_expect_tx(full_b(sbt), bytes);
                        tma_load_4d(slab, &p.tmap_x, c2 * 64, 0, t2.ho0, t2.n, full_b(sbt));
                    } else if (lane == 0) {
                        const uint32_t slab = smem_u32(sB + (size_t)sbt * p.stage_b);
                        mbar_arrive_expect_tx(full_b(sbt), bytes);
                        for (int c8 = 0; c8 < 2; ++c8)
                            for (int pr = 0; pr < p.s_h; ++pr)
                                for (int pc = 0; pc < p.s_w; ++pc)
                                    tma_load_4d(slab + (uint32_t)c8 * p.lbo + (uint32_t)(pr * p.s_w + pc) * p.PB,
                                                &p.tmap_x, c2 * 16 + c8 * 8, pc - p.p_w, R0 + pr, t2.n, full_b(sbt));
                    }
                    __syncwarp();
                    pend[sbt] = (int)pht;
                    if (++sbt == p.BST) { sbt = 0; pht ^= 1; }
                }
            }
            // after a wait gave up, copies still in flight land before the CTA exits
            if (!ok2 && lane == 0)
                for (int s2 = 0; s2 < p.BST; ++s2)
                    if (pend[s2] >= 0) bar_wait(full_b(s2), (uint32_t)pend[s2], ctl, SITE_DRAIN, false);
            __syncwarp();
        }
        // (with tensor-copied slabs the loop below has nothing to do)
        int64_t id = copy_slab ? p.tiles_total : (int64_t)blockIdx.x;
        int cc = 0;
        TapTile tl;
        // raw staging (TAP_CH ring, TAP_WX, TAP_WW): parity of each slot's next
        // completion, and whether a bulk copy into it is outstanding
        uint32_t raw_ph[2] = {0u, 0u};
        bool raw_issued[2] = {false, false};
        if (id < p.tiles_total) tile_at(p, id, tl);
        if (prefetch && id < p.tiles_total) {
            issue_raw(tl, cc, 0);
            raw_issued[0] = true;
        }
        for (int g = 0; id < p.tiles_total; ++g, next_chunk(id, cc, tl)) {
            // slab stage of chunk g, advanced for every chunk
            const int sb_g = sb;
            const uint32_t ph_g = phb;
            if (++sb == p.BST) { sb = 0; phb ^= 1; }
            if (ngroups == 2 && (g & 1) != grp) continue;  // the other group's chunk
            const int slot = prefetch ? (g & 1) : grp;
            if (prefetch) {
                // the next chunk's copy into the other slot, then wait for this one
                int64_t id2 = id;
                int cc2 = cc;
                TapTile t2 = tl;
                next_chunk(id2, cc2, t2);
                if (pok && id2 < p.tiles_total) {
                    issue_raw(t2, cc2, slot ^ 1);
                    raw_issued[slot ^ 1] = true;
                }
                if (raw_issued[slot] && pok) {
                    pok = warp_bar_wait(raw_full(slot), raw_ph[slot], ctl, SITE_RAW);
                    if (pok) {
                        raw_ph[slot] ^= 1u;
                        raw_issued[slot] = false;
                    }
                }
                asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(NPT) : "memory");
            } else if (staged) {
                if (pok) {
                    issue_raw(tl, cc, slot);
                    raw_issued[slot] = true;
                }
                if (pok) {
                    pok = warp_bar_wait(raw_full(slot), raw_ph[slot], ctl, SITE_RAW);
                    if (pok) {
                        raw_ph[slot] ^= 1u;
                        raw_issued[slot] = false;
                    }
                }
                asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(NPT) : "memory");
            }
            const int n = tl.n, ho0 = tl.ho0, Q = tl.Q;
            if (pok) pok = warp_bar_wait(empty_b(sb_g), ph_g ^ 1, ctl, SITE_EMPTY_PROD);
            uint8_t *slab = sB + (size_t)sb_g * p.stage_b;
            const E16 *raw_slot = sRaw + (size_t)slot * p.raw_slot;
            if (!pok) {
                // aborted: keep meeting the producers' barrier, do no work
            } else if (MODE == TAP_CL) {
                // entry (8-channel half c8, tile row lr, column col) is x[n][R0 + lr][col][cc*16 + c8*8 ..
                // + 8]: one 16-byte copy. Lane pairs take the two halves of a position (32
                // contiguous bytes); halves past C_i (a multiple of 8) are zero-filled.
                // With padding the slab spans Wp columns and the entries outside the input
                // are zero-filled copies. C_i not a multiple of 8 (vec == 0): each entry is
                // built from element loads and stored, then the usual fence and arrival.
                const int rows = (Q - 1) * p.s_h + p.Hfe;
                const int items = 2 * rows * p.Wp;
                const int R0 = ho0 * p.s_h - p.p_h;  // input row of slab row 0
                const uint16_t *xn = p.src + (int64_t)n * p.H_i * p.W_i * p.C_i + cc * 16;
                for (int it = pt; it < items; it += NPT) {
                    const int c8 = it & 1;
                    const int pos = it >> 1;
                    const int lr = (int)fdiv((uint32_t)pos, p.div_wi);
                    const int col = pos - lr * p.Wp;
                    const int lq = (int)fdiv((uint32_t)lr, p.div_sh);
                    const int cq = (int)fdiv((uint32_t)col, p.div_sw);
                    uint8_t *dstp = slab + (size_t)c8 * p.lbo +
                                    (size_t)((lr - lq * p.s_h) * p.s_w + (col - cq * p.s_w)) * p.PB +
                                    (size_t)(lq * p.pitch + cq) * 16;
                    const int h = R0 + lr, w = col - p.p_w;
                    const bool inside = (unsigned)h < (unsigned)p.H_i && (unsigned)w < (unsigned)p.W_i;
                    const int c0 = cc * 16 + c8 * 8;  // first channel of the entry
                    const uint16_t *src = xn + ((int64_t)h * p.W_i + w) * p.C_i + c8 * 8;
                    if (p.vec) {
                        const bool ok = inside && c0 < p.C_i;
                        cp_async16z(smem_u32(dstp), ok ? (const void *)src : (const void *)p.src, ok ? 16u : 0u);
                    } else {
                        uint32_t e16[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            e16[e] = (inside && c0 + e < p.C_i) ? (uint32_t)__ldg(src + e) : 0u;
                        *reinterpret_cast<uint4 *>(dstp) =
                            make_uint4(e16[0] | (e16[1] << 16), e16[2] | (e16[3] << 16),
                                       e16[4] | (e16[5] << 16), e16[6] | (e16[7] << 16));
                    }
                }
            } else if (MODE == TAP_CH) {
                const int rows = (Q - 1) * p.s_h + p.Hfe;
                const int64_t plane = (int64_t)p.H_i * p.W_i;
                const uint16_t *__restrict__ xn = p.src + (int64_t)n * p.C_i * plane;
                const int R0 = ho0 * p.s_h;
                if (p.padded && !p.vec) {
                    // one slab column of 8 channels per item over the Wp padded columns;
                    // input (R0 + lr - p_h, col - p_w), zero outside the input
                    const int items = 2 * rows * p.Wp;
                    for (int it = pt; it < items; it += NPT) {
                        const int t2 = it / p.Wp;
                        const int col = it - t2 * p.Wp;
                        const int c8 = t2 >= rows ? 1 : 0;
                        const int lr = t2 - c8 * rows;
                        const int ci0 = cc * 16 + c8 * 8;
                        const int h = R0 + lr - p.p_h, w = col - p.p_w;
                        const bool inside = (unsigned)h < (unsigned)p.H_i && (unsigned)w < (unsigned)p.W_i;
                        const uint16_t *src = xn + (int64_t)ci0 * plane + (int64_t)h * p.W_i + w;
                        uint32_t e16[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            e16[e] = (inside && ci0 + e < p.C_i) ? (uint32_t)__ldg(src + e * plane) : 0u;
                        uint8_t *dst = slab + (size_t)c8 * p.lbo +
                                       (size_t)((lr % p.s_h) * p.s_w + col % p.s_w) * p.PB +
                                       (size_t)((lr / p.s_h) * p.pitch + col / p.s_w) * 16;
                        *reinterpret_cast<uint4 *>(dst) =
                            make_uint4(e16[0] | (e16[1] << 16), e16[2] | (e16[3] << 16),
                                       e16[4] | (e16[5] << 16), e16[6] | (e16[7] << 16));
                    }
                } else if (p.vec && p.ring) {
                    // A block is 8 channels x 8 columns of one raw row. A warp moves four
                    // blocks per step: one matrix load (lane 8q + i gives channel row i of
                    // block q) and one transposing matrix store (lane 8q + i gives the slab
                    // entry of column i of block q: that column's 8 channels, 16 bytes).
                    // Raw planes lie an odd number of 16-byte units apart, so a load's eight
                    // rows hit eight bank groups; a store's eight entries are consecutive.
                    // A step's blocks past the last repeat the last one (the same values to
                    // the same addresses).
                    const int cgs = p.W_i / 8;
                    const int nblk = 2 * rows * cgs;
                    const int wq = lane >> 3, wi = lane & 7;
                    for (int b0 = (pt >> 5) * 4; b0 < nblk; b0 += NPT / 8) {
                        const int blk = min(b0 + wq, nblk - 1);
                        const int t2 = (int)fdiv((uint32_t)blk, p.div_cgs);
                        const int cg = blk - t2 * cgs;
                        const int c8 = t2 >= rows ? 1 : 0;
                        const int lr = t2 - c8 * rows;
                        uint32_t r0, r1, r2, r3;
                        ldsm_x4(smem_u32(raw_slot + (size_t)(c8 * 8 + wi) * p.raw_ch + lr * p.raw_w + cg * 8), r0, r1,
                                r2, r3);
                        const int lq = (int)fdiv((uint32_t)lr, p.div_sh);
                        const int col = p.p_w + cg * 8 + wi;
                        const int cq = (int)fdiv((uint32_t)col, p.div_sw);
                        uint8_t *dst = slab + (size_t)c8 * p.lbo +
                                       (size_t)((lr - lq * p.s_h) * p.s_w + (col - cq * p.s_w)) * p.PB +
                                       (size_t)(lq * p.pitch + cq) * 16;
                        stsm_x4_trans(smem_u32(dst), r0, r1, r2, r3);
                    }
                } else if (p.vec) {
                    // 8 channels x 8 columns per item: 8 16-byte loads from global memory,
                    // 8x8 transpose, 8 16-byte stores
                    const int cgs = p.W_i / 8;
                    const int items = 2 * rows * cgs;
                    for (int it = pt; it < items; it += NPT) {
                        const int t2 = (int)fdiv((uint32_t)it, p.div_cgs);
                        const int cg = it - t2 * cgs;
                        const int c8 = t2 >= rows ? 1 : 0;
                        const int lr = t2 - c8 * rows;
                        const int ci0 = cc * 16 + c8 * 8;
                        uint4 v[8];
                        {
                            // input row R0 - p_h + lr (zero outside the input)
                            const int h = R0 - p.p_h + lr;
                            const bool rok = (unsigned)h < (unsigned)p.H_i;
                            const uint16_t *src = xn + (int64_t)ci0 * plane + (int64_t)h * p.W_i + cg * 8;
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                v[e] = (rok && ci0 + e < p.C_i)
                                           ? __ldg(reinterpret_cast<const uint4 *>(src + e * plane))
                                           : make_uint4(0, 0, 0, 0);
                        }
                        const int lq = (int)fdiv((uint32_t)lr, p.div_sh);
                        uint8_t *rowp = slab + (size_t)c8 * p.lbo + (size_t)((lr - lq * p.s_h) * p.s_w) * p.PB +
                                        (size_t)(lq * p.pitch) * 16;
                        // input column cg*8 + kk is slab column col = p_w + cg*8 + kk, in phase
                        // block (col % s_w) at entry col / s_w. The lanes of a warp hold
                        // column groups 8 entries (128 bytes) apart, so lane l writes its
                        // entries starting at kk = l % 8: the 8 lanes of a group then store to
                        // 8 different bank groups instead of one.
                        const int rot = threadIdx.x & 7;
                        const int col0 = cg * 8 + p.p_w;
#pragma unroll
                        for (int st = 0; st < 8; ++st) {
                            const int kk = (st + rot) & 7;
                            const uint32_t sel = (kk & 1) ? 0x7632u : 0x5410u;
                            const int wd = kk >> 1;
                            const uint32_t w0 = __byte_perm(word_sel(v[0], wd), word_sel(v[1], wd), sel);
                            const uint32_t w1 = __byte_perm(word_sel(v[2], wd), word_sel(v[3], wd), sel);
                            const uint32_t w2 = __byte_perm(word_sel(v[4], wd), word_sel(v[5], wd), sel);
                            const uint32_t w3 = __byte_perm(word_sel(v[6], wd), word_sel(v[7], wd), sel);
                            const int col = col0 + kk;
                            const int cq = (int)fdiv((uint32_t)col, p.div_sw);
                            const int cph = col - cq * p.s_w;
                            uint8_t *dst = rowp + (size_t)cph * p.PB + (size_t)cq * 16;
                            *reinterpret_cast<uint4 *>(dst) = make_uint4(w0, w1, w2, w3);
                        }
                    }
                } else {
                    // one column of 8 channels per item
                    const int items = 2 * rows * p.W_i;
                    for (int it = pt; it < items; it += NPT) {
                        const int col = it % p.W_i;
                        const int t2 = it / p.W_i;
                        const int c8 = t2 >= rows ? 1 : 0;
                        const int lr = t2 - c8 * rows;
                        const int ci0 = cc * 16 + c8 * 8;
                        const uint16_t *src = xn + (int64_t)ci0 * plane + (int64_t)(R0 + lr) * p.W_i + col;
                        uint32_t e16[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            e16[e] = (ci0 + e < p.C_i) ? (uint32_t)__ldg(src + e * plane) : 0u;
                        uint8_t *dst = slab + (size_t)c8 * p.lbo +
                                       (size_t)((lr % p.s_h) * p.s_w + col % p.s_w) * p.PB +
                                       (size_t)((lr / p.s_h) * p.pitch + col / p.s_w) * 16;
                        *reinterpret_cast<uint4 *>(dst) =
                            make_uint4(e16[0] | (e16[1] << 16), e16[2] | (e16[3] << 16),
                                       e16[4] | (e16[5] << 16), e16[6] | (e16[7] << 16));
                    }
                }
            } else if (MODE == TAP_WW) {
                // window rows staged contiguously: entry (c, q, m) is the 8 consecutive
                // staged elements at q*L + m*S + 8c of window row q (zero past the row's
                // end, and past b = S: the K padding). Position by position (one division),
                // K chunk by K chunk, each element at a fixed offset from the chunk's start:
                // the fill is bound by instruction issue, and this takes about a third of
                // the instructions of gathering through the offset table.
                const int SC = 2 * p.U;
                const int per_c = Q * p.pitch;
                const E16 *raw = raw_slot + raw_lead_of(tl, cc);
                const int L = (int)p.L, S = p.S;
                for (int i = pt; i < per_c; i += NPT) {
                    const int q = (int)fdiv((uint32_t)i, p.div_pitch);
                    const int m = i - q * p.pitch;
                    const int mm = m * S;
                    const int lim = min(S, L - mm);  // elements of the position that exist
                    const E16 *rb = raw + q * L + mm;
                    uint8_t *dst = slab + (size_t)i * 16;
                    for (int c = 0; c < SC; ++c, rb += 8, dst += p.lbo) {
                        const int rem = lim - 8 * c;
                        uint32_t e16[8];
                        if (rem >= 8) {
#pragma unroll
                            for (int e = 0; e < 8; ++e) e16[e] = (uint32_t)rb[e];
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e) e16[e] = e < rem ? (uint32_t)rb[e] : 0u;
                        }
                        *reinterpret_cast<uint4 *>(dst) =
                            make_uint4(__byte_perm(e16[0], e16[1], 0x5410), __byte_perm(e16[2], e16[3], 0x5410),
                                       __byte_perm(e16[4], e16[5], 0x5410), __byte_perm(e16[6], e16[7], 0x5410));
                    }
                }
            } else {
                // TAP_WX: window rows of channel cc, re-laid from the staged input rows:
                //   entry (c, q, m)[e] = window row q of the tile at m*S + 8c + e
                //   = x[cc][(ho0+q)*s_h + r][m*s_w + jl] with 8c + e = jl*H_f + r
                // One K chunk c at a time, so that the 8 source offsets of an entry
                // (and which of them exist) stay in registers; per entry one division.
                const int SC = 2 * p.U;
                const int per_c = Q * p.pitch;
                const E16 *raw = raw_slot + raw_lead_of(tl, cc);
                const int qstride = MODE == TAP_WX ? p.s_h * p.W_i : (int)p.L;
                const int mstride = MODE == TAP_WX ? p.s_w : p.S;
                for (int c = 0; c < SC; ++c) {
                    // element e of an entry: raw offset boff[e] from the entry's base, present
                    // if m*mstride < lim[e] (the per-CTA table of the prologue)
                    int boff[8], lim[8];
                    {
                        const int4 *tb = reinterpret_cast<const int4 *>(wtab + 8 * c);
                        const int4 *tl4 = reinterpret_cast<const int4 *>(wtab + 16 * p.U + 8 * c);
                        const int4 b0 = tb[0], b1 = tb[1], l0 = tl4[0], l1 = tl4[1];
                        boff[0] = b0.x; boff[1] = b0.y; boff[2] = b0.z; boff[3] = b0.w;
                        boff[4] = b1.x; boff[5] = b1.y; boff[6] = b1.z; boff[7] = b1.w;
                        lim[0] = l0.x; lim[1] = l0.y; lim[2] = l0.z; lim[3] = l0.w;
                        lim[4] = l1.x; lim[5] = l1.y; lim[6] = l1.z; lim[7] = l1.w;
                    }
                    uint8_t *slab_c = slab + (size_t)c * p.lbo;
                    for (int i = pt; i < per_c; i += NPT) {
                        const int q = (int)fdiv((uint32_t)i, p.div_pitch);
                        const int m = i - q * p.pitch;
                        const int base = q * qstride + m * mstride;
                        const int mm = m * mstride;
                        uint32_t e16[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) e16[e] = mm < lim[e] ? (uint32_t)raw[base + boff[e]] : 0u;
                        *reinterpret_cast<uint4 *>(slab_c + (size_t)i * 16) =
                            make_uint4(e16[0] | (e16[1] << 16), e16[2] | (e16[3] << 16),
                                       e16[4] | (e16[5] << 16), e16[6] | (e16[7] << 16));
                    }
                }
            }
            if (pok) {
                if (MODE == TAP_CL && p.vec) {
                    cp_async_mbar_arrive_noinc(full_b(sb_g));  // once this thread's copies land
                } else {
                    fence_async_smem();
                    mbar_arrive(full_b(sb_g));
                }
            }
            if (staged) {
                // the raw slot is consumed: the group's next copy may overwrite it
                asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(NPT) : "memory");
            }
            if (CHAN && !staged && !pok) break;
        }
        cp_async_commit_group();
        cp_async_wait_group<0>();
        // bulk copies still in flight (an aborted wait) land before the CTA exits
        if (MODE != TAP_CL) {
            for (int s2 = 0; s2 < 2; ++s2)
                if (raw_issued[s2]) bar_wait(raw_full(s2), raw_ph[s2], ctl, SITE_DRAIN, false);
        }
    } else {
        // ---------------- epilogue: TMEM -> registers -> smem transpose -> coalesced stores
        const int ew = warp - 2 - TAP_PROD_WARPS;  // 0..7
        const int q4 = warp & 3;                  // TMEM lane quarter this warp may read
        const int hh = ew >> 2;                   // which half of the columns
        const int warp_words = p.epi_blocks * TAP_EPI_BLOCK_WORDS;
        uint32_t *stage = sE + ew * warp_words;
        const int64_t plane = (int64_t)p.H_o * p.W_o;
        int k = 0;
        uint32_t xk = 0;  // stacked hand-overs so far (the same count in both warps of a pair)
        TapTile tl;
        for (int64_t id = blockIdx.x; id < p.tiles_total; id += gridDim.x) {
            tile_at(p, id, tl);
            const int NT = tl.Q * p.pitch;
            const int NTp = tile_ntp(p, NT);  // the MMAs' columns
            const int N0 = tile_n0(p, NTp);
            const int pitch = p.pitch, W_o = p.W_o;
            auto off_of = [&](int pp) -> int {
                const int qrow = pp / pitch;
                const int wo = pp - qrow * pitch;
                return (pp < NT && wo < W_o) ? qrow * W_o + wo : -1;
            };
            const uint32_t taddr = tmem + ((uint32_t)(q4 * 32) << 16);
            // the two warps of a quarter split a column range in 64-column blocks
            auto half_range = [&](int a0, int a1, int &cb, int &ce) {
                const int nb = (a1 - a0 + 63) / 64;
                const int mid = a0 + ((nb + 1) / 2) * 64;
                cb = hh == 0 ? a0 : mid;
                ce = hh == 0 ? min(a1, mid) : a1;
            };
            bool ok = true;
            // channels-last: a position's channels are contiguous, positions C_o apart
            auto out_at = [&](int co0) -> uint16_t * {
                return p.nhwc ? p.out + (((int64_t)tl.n * p.H_o + tl.ho0) * p.W_o) * p.C_o + co0
                              : p.out + ((int64_t)tl.n * p.C_o + co0) * plane + (int64_t)tl.ho0 * p.W_o;
            };
            const int64_t ostride = p.nhwc ? (int64_t)p.C_o : plane;
            if (p.xpose) {
                // Transposed stacking: accumulator 2*buf + mb holds, in TMEM lane i,
                // position mb*128 + i of the tile; columns 0..63 the first taps' sums
                // for channel n, 64..127 the second taps' sums for channel n - 64,
                // which belong to the position one to the left. So output (position
                // pp, channel co) = D[pp][co] + D[pp + 1][64 + co]: the next lane of
                // the same warp, except for a lane quarter's last row, whose partner
                // is the next quarter's (or next M block's) first row. Each warp
                // (lane quarter q4, channel half hh) first hands its first row's
                // second-tap values over through shared memory; after the epilogue
                // warps meet, it adds the next lane's values by a shuffle.
                const int buf = k & 1;
                const uint32_t par = (uint32_t)(k >> 1) & 1u;
                const int NT = tl.Q * p.pitch;
                const int nmb = (NT + 1 + 127) / 128;
                float *xk = reinterpret_cast<float *>(sE) + (k & 1) * 512;  // [mb][q4][hh][32]
                const uint32_t tq = tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)(buf * 256);
                const bool okw = warp_bar_wait(tmem_full(2 * buf), par, ctl, SITE_DONE) &&
                                 warp_bar_wait(tmem_full(2 * buf + 1), par, ctl, SITE_DONE);
                if (okw) {
                    tc_fence_after();
#pragma unroll 1
                    for (int mb = 0; mb < nmb; ++mb) {
                        uint32_t u[32];
                        tmem_ld32(tq + (uint32_t)(mb * 128 + 64 + hh * 32), u);
                        tmem_wait_ld();
                        if (lane == 0) {
                            float4 *d = reinterpret_cast<float4 *>(xk + ((mb * 4 + q4) * 2 + hh) * 32);
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                d[i] = make_float4(__uint_as_float(u[4 * i]), __uint_as_float(u[4 * i + 1]),
                                                   __uint_as_float(u[4 * i + 2]), __uint_as_float(u[4 * i + 3]));
                        }
                    }
                }
                // every epilogue warp meets here once per tile; a failed wait in any
                // of them ends all of them. The hand-over area alternates with the
                // tile's parity: a warp writes the next tile's values only after
                // every warp has passed this tile's meeting, so nobody still reads them.
                ok = bar_red_and(5, TAP_EPI_WARPS * 32, okw);
                if (ok) {
                    const int pitch = p.pitch, W_o = p.W_o;
                    const int c_base = hh * 32;
                    const int nco = min(32, p.C_o - c_base);  // this warp's channels
#pragma unroll 1
                    for (int mb = 0; mb < nmb && nco > 0; ++mb) {
                        // the row after the quarter's last: the next quarter's first, or the
                        // next M block's (none after the last: that row is no output's)
                        const float *nx = q4 < 3 ? xk + ((mb * 4 + q4 + 1) * 2 + hh) * 32
                                                 : (mb + 1 < nmb ? xk + (((mb + 1) * 4) * 2 + hh) * 32 : nullptr);
                        const int pp = mb * 128 + q4 * 32 + lane;
                        const int qrow = pp / pitch;
                        const int wo = pp - qrow * pitch;
                        const bool valid = pp < NT && wo < W_o;
                        uint16_t *o = p.nhwc ? p.out + (((int64_t)tl.n * p.H_o + tl.ho0 + qrow) * W_o + wo) * p.C_o +
                                                   c_base
                                             : p.out + ((int64_t)tl.n * p.C_o + c_base) * plane +
                                                   (int64_t)(tl.ho0 + qrow) * W_o + wo;
                        // two halves of 16 channels (registers)
#pragma unroll 1
                        for (int h2 = 0; h2 < 2 && 16 * h2 < nco; ++h2) {
                            uint32_t t[16], u[16];
                            const uint32_t col = (uint32_t)(mb * 128 + c_base + 16 * h2);
                            tmem_ld16(tq + col, t);
                            tmem_ld16(tq + col + 64, u);
                            tmem_wait_ld();
                            // the sums, in place
#pragma unroll
                            for (int c = 0; c < 16; ++c) {
                                float nxt = __shfl_down_sync(0xffffffffu, __uint_as_float(u[c]), 1);
                                if (lane == 31) nxt = nx ? nx[16 * h2 + c] : 0.f;
                                t[c] = __float_as_uint(__uint_as_float(t[c]) + nxt);
                            }
                            if (!valid) continue;
                            const int nc = min(16, nco - 16 * h2);
                            auto f = [&](int c) { return __uint_as_float(t[c]); };
                            if (p.nhwc) {
                                uint16_t *oh = o + 16 * h2;
                                if (nc == 16 && (p.C_o & 7) == 0) {
#pragma unroll
                                    for (int i = 0; i < 2; ++i)
                                        reinterpret_cast<uint4 *>(oh)[i] =
                                            make_uint4(pack2(f(8 * i), f(8 * i + 1), p.bf16),
                                                       pack2(f(8 * i + 2), f(8 * i + 3), p.bf16),
                                                       pack2(f(8 * i + 4), f(8 * i + 5), p.bf16),
                                                       pack2(f(8 * i + 6), f(8 * i + 7), p.bf16));
                                } else {
#pragma unroll
                                    for (int c = 0; c < 16; ++c)
                                        if (c < nc) oh[c] = cvt16(f(c), p.bf16);
                                }
                            } else {
                                uint16_t *oh = o + (int64_t)(16 * h2) * plane;
#pragma unroll
                                for (int c = 0; c < 16; ++c)
                                    if (c < nc) oh[(int64_t)c * plane] = cvt16(f(c), p.bf16);
                            }
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(tmem_empty(2 * buf));
                        mbar_arrive(tmem_empty(2 * buf + 1));
                    }
                }
            } else if (!p.stack) {
                const int co0 = tl.mt * BM + q4 * 32;
                uint16_t *out_c = out_at(co0);
                for (int a = 0; a < 2 && ok; ++a) {
                    if (!(ok = warp_bar_wait(tmem_full(a), k & 1, ctl, SITE_DONE))) break;
                    if (co0 >= p.C_o) {
                        // the warp's 32 channels lie past C_o (zero filter rows): nothing
                        // to store, the accumulator is released at once
                        if (lane == 0) mbar_arrive(tmem_empty(a));
                        continue;
                    }
                    tc_fence_after();
                    int cb, ce;
                    half_range(a == 0 ? 0 : N0, a == 0 ? N0 : NTp, cb, ce);
                    // a block may reach past the range (into the other accumulator, which
                    // may still be accumulating): only columns of the range are stored
                    auto off_in = [&](int pp) -> int { return pp < ce ? off_of(pp) : -1; };
                    const int rows = min(32, p.C_o - co0);
                    if (p.epi_blocks == 2) {
                        // the warp's share (at most two 64-column blocks) goes to its staging
                        // area, the accumulator is released, then the stores run while the
                        // next tile's MMAs use it
                        if (p.nhwc)
                            stage_columns<true>(taddr, cb, ce, stage, TAP_EPI_BLOCK_WORDS, p.bf16);
                        else
                            stage_columns<false>(taddr, cb, ce, stage, TAP_EPI_BLOCK_WORDS, p.bf16);
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(tmem_empty(a));
                        for (int c0 = cb, bi = 0; c0 < ce; c0 += 64, ++bi) {
                            const uint32_t *blk = stage + bi * TAP_EPI_BLOCK_WORDS;
                            if (p.nhwc)
                                store_block_cl(blk, c0, rows, ostride, out_c, off_in);
                            else
                                store_block(blk, c0, rows, ostride, out_c, off_in);
                        }
                        __syncwarp();
                    } else {
                        if (p.nhwc)
                            drain_columns<true>(taddr, cb, ce, stage, rows, ostride, p.bf16, out_c, off_in);
                        else
                            drain_columns<false>(taddr, cb, ce, stage, rows, ostride, p.bf16, out_c, off_in);
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(tmem_empty(a));
                    }
                }
            } else {
                // the shifted add reads one column across the accumulators' boundary:
                // both accumulators are drained together.
                // Warps of quarters 2, 3 (rows 64..127) feed the warps of quarters 0, 1
                // (same channels, rows 0..63) of the same column half through the
                // lower warp's staging area and the pair's two mbarriers
                ok = warp_bar_wait(tmem_full(0), k & 1, ctl, SITE_DONE) &&
                     warp_bar_wait(tmem_full(1), k & 1, ctl, SITE_DONE);
                if (ok) {
                    tc_fence_after();
                    int cb, ce;
                    half_range(0, (NT + 15) / 16 * 16, cb, ce);
                    const int pair = (q4 & 1) + 2 * hh;
                    if (q4 >= 2) {
                        ok = drain_stacked_lower(taddr, cb, ce, reinterpret_cast<float *>(stage), xfull(pair),
                                                 xempty(pair), &xk, ctl, SITE_STACK);
                    } else {
                        const int co0 = q4 * 32;
                        uint16_t *out_c = out_at(co0);
                        const float *xbuf = reinterpret_cast<const float *>(sE + (ew - 2) * warp_words);
                        const int rows = max(0, min(32, p.C_o - co0));
                        if (p.nhwc)
                            ok = drain_stacked_upper<true>(taddr, cb, ce, stage, xbuf, xfull(pair), xempty(pair),
                                                           &xk, ctl, SITE_STACK, rows, ostride, p.bf16, out_c,
                                                           off_of);
                        else
                            ok = drain_stacked_upper<false>(taddr, cb, ce, stage, xbuf, xfull(pair), xempty(pair),
                                                            &xk, ctl, SITE_STACK, rows, ostride, p.bf16, out_c,
                                                            off_of);
                    }
                }
                if (ok) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(tmem_empty(0));
                        mbar_arrive(tmem_empty(1));
                    }
                }
            }
            if (!ok) break;
            ++k;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Filter tiles of the tap kernels: fa[mt][cc][t][g][h][row][e] (h = K half)
// holds, for output channel mt*128 + g*8 + row and K index k = h*8 + e of tap t,
// the element (ci, r, j) of the kernel's (virtual) filter C_v x H_fv x W_fv:
//   TAP_CH, TAP_CL: ci = cc*16 + k, (r, j) = (t / W_fv, t % W_fv);
//   TAP_W*: ci = cc, r = b % H_fv, j = a*s_wv + b / H_fv with t = a*U + u, b = 16u + k (b < S);
// zero outside the filter. `view` maps that element to the caller's filter
// C x H_f x W_f (filter_src_offset). Block 0 also clears the status word.
struct TapRelayout {
    int mode;
    int C_v, H_fv, W_fv, s_wv;  // the kernel's shape
    int view, C, H_f, W_f;      // the caller's filter and the view onto it
    int C_o, T, NCH, U, S, n_chunks, stack, Gr;
};

__global__ void relayout_filter_tap(const uint16_t *__restrict__ filt, uint16_t *__restrict__ fa,
                                    uint32_t *status, const TapRelayout a) {
    allow_dependents();  // the tap kernel may start its prologue meanwhile
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
        status[0] = 0;
        status[1] = 0;
        status[2] = 0;
    }
    const int per_chunk = a.T * (TAP_A_BYTES / 2);  // elements of one (mt, cc) chunk: T taps x 2048
    const int64_t frow = (int64_t)a.C * a.H_f * a.W_f;
    for (int chunk = blockIdx.y; chunk < a.n_chunks; chunk += gridDim.y) {
        const int cc = chunk % a.NCH, mt = chunk / a.NCH;
        uint16_t *dst = fa + (int64_t)chunk * per_chunk;
        for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < per_chunk; idx += gridDim.x * blockDim.x) {
            const int e = idx & 7, rw = (idx >> 3) & 7, h = (idx >> 6) & 1, g = (idx >> 7) & 15;
            const int t = idx >> 11;
            const int co = mt * BM + (a.stack ? (g & 7) : g) * 8 + rw;
            const int k = h * 8 + e;
            int ci = -1, r = 0, j = 0;
            if (a.mode == TAP_CH || a.mode == TAP_CL) {
                // tap of the filter: t itself, or for a stacked group the top tap (rows
                // 0..63) or the bottom tap (rows 64..127, absent past W_fv)
                if (a.stack) {
                    r = t / a.Gr;
                    const int jt = stacked_top_j(t % a.Gr, a.s_wv);
                    j = g < 8 ? jt : jt + a.s_wv;
                } else {
                    r = t / a.W_fv;
                    j = t - r * a.W_fv;
                }
                ci = cc * 16 + k;
                if (ci >= a.C_v || j >= a.W_fv) ci = -1;
            } else {
                const int ta = t / a.U, u = t - ta * a.U;
                const int b = 16 * u + k;
                if (b < a.S) {
                    const int jl = b / a.H_fv;
                    r = b - jl * a.H_fv;
                    j = ta * a.s_wv + jl;
                    if (j < a.W_fv) ci = cc;
                }
            }
            uint16_t v = 0;
            if (co < a.C_o && ci >= 0)
                v = filt[(int64_t)co * frow + filter_src_offset(a.view, ci, r, j, a.C, a.H_f, a.W_f)];
            dst[idx] = v;
        }
    }
}

struct TapPlan {
    bool ok;
    int mode;
    TapParams p;
    size_t smem;
    int mtiles;
    int64_t kslots;        // MMA K values per output pixel (cost model)
    int view;              // how the kernel's filter maps to the caller's (FilterView)
};

static int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    return n;
}

// Modelled time of one tile of NT positions: two MMAs of N = NTp/2 per K step,
// at rates measured for tcgen05.mma M=128 with two accumulators (MAC/clk/SM:
// N=64 1962, 128 2880, 224 3347, 256 3542), plus a fixed drain/restart cost.
static double tile_cost(int64_t NT) {
    const double n = (double)((NT + 15) / 16 * 16) / 2.0;
    const double pts[5][2] = {{16, 600}, {64, 1962}, {128, 2880}, {224, 3347}, {256, 3542}};
    double rate = pts[4][1];
    for (int i = 0; i < 4; ++i)
        if (n <= pts[i + 1][0]) {
            const double f = (n - pts[i][0]) / (pts[i + 1][0] - pts[i][0]);
            rate = pts[i][1] + (n < pts[i][0] ? 0.0 : f) * (pts[i + 1][1] - pts[i][1]);
            break;
        }
    return 2.0 * n / rate + 0.15;  // relative units
}

// The same for transposed stacking: one 128 x 128 MMA per M block and K step, the
// M blocks on their own issuers (MAC/clk/SM measured for M = N = 128 with A and
// B in shared memory: one issuer 2096, two 3210), in the units of tile_cost.
static double tile_cost_xpose(int64_t NT) {
    const int64_t nmb = (NT + 1 + 127) / 128;
    return (nmb == 1 ? 128.0 / 2096.0 : 256.0 / 3210.0) + 0.15;
}

// Tiling of a tap kernel for a shape (mode TAP_CH / TAP_WX / TAP_WW) on `sms`
// SMs, or !ok: the tiling with the least modelled time among those whose slab
// stages fit shared memory. Whether a plan exists, and its filter layout, do
// not depend on `sms`.
TapPlan plan_tap_epi(const Shape &s, int mode, int64_t sms, int epi_blocks, bool xpose = false) {
    TapPlan pl{};
    pl.ok = false;
    pl.mode = mode;
    const int64_t smem_max = 227 * 1024 - 1024;
    if (s.C_i * s.H_i * s.W_i >= (1ll << 31)) return pl;
    const bool chan = mode == TAP_CH || mode == TAP_CL;
    if (!chan && !plain(s)) return pl;  // padding / dilation: channel modes only
    const int64_t Wp = padded_w(s);
    const int64_t Hfe = (s.H_f - 1) * s.d_h + 1;  // slab rows a filter spans
    if (Wp * s.C_i * (s.H_i + 2 * s.p_h) >= (1ll << 31)) return pl;
    int64_t pitch, T, U = 0, S = 0, A = 0, NCH;
    // stacking (TAP_CH / TAP_CL, C_o <= 64, some tap has a partner, no dilation): T
    // counts tap groups
    const int stack = (chan && s.C_o <= 64 && s.W_f > s.s_w && s.d_h == 1 && s.d_w == 1) ? 1 : 0;
    const int Gr = stack ? stacked_groups_per_row((int)s.W_f, (int)s.s_w) : 0;
    if (xpose && !stack) return pl;
    // a 1x1 filter at stride 1 without padding on rows of whole 8-position groups: the
    // input is its own window, copied MN-major into the slab by one tensor copy per
    // chunk of 16*mn_k channels
    const bool mnb = mode == TAP_CH && s.H_f == 1 && s.W_f == 1 && s.s_h == 1 && s.s_w == 1 && plain(s) &&
                     s.W_o % 8 == 0;
    // the same filter channels-last, with channels in whole 64s: a chunk's slab is 64
    // channels of the tile's rows, copied K-major (one 128-byte row per position, the
    // copy's 128-byte swizzle) by one tensor copy per chunk
    const bool kmb = mode == TAP_CL && s.H_f == 1 && s.W_f == 1 && s.s_h == 1 && s.s_w == 1 && plain(s) &&
                     s.C_i % 64 == 0 && s.W_i % 8 == 0 && s.W_i <= 256;
    const bool copy1 = mnb || kmb;  // a 1x1 slab by one tensor copy per chunk
    const int64_t mn_k = mnb ? std::min<int64_t>(kMnK, (s.C_i + 15) / 16) : kmb ? 4 : 1;
    if (chan) {
        pitch = (Wp + s.s_w - 1) / s.s_w;
        T = copy1 ? mn_k : stack ? s.H_f * Gr : s.H_f * s.W_f;
        NCH = (s.C_i + 16 * mn_k - 1) / (16 * mn_k);
    } else {
        S = s.s_w * s.H_f;
        U = (S + 15) / 16;
        A = (s.W_f + s.s_w - 1) / s.s_w;
        pitch = std::max<int64_t>((s.W_i + s.s_w - 1) / s.s_w, s.W_o + A - 1);
        T = A * U;
        NCH = s.C_i;
        if (mode == TAP_WW && s.N * s.C_i * s.H_o * s.W_i * s.H_f >= (1ll << 40)) return pl;
        if (s.H_o * s.W_i * s.H_f >= (1ll << 31)) return pl;
    }
    // stacked tiles need one more accumulator column, and the epilogue reads one
    // column past a 64-column block: at most 448 columns; transposed stacking
    // double-buffers at most two M blocks of 128 positions
    const int64_t max_nt = xpose ? 2 * 128 - 1 : stack ? 448 - 1 : TAP_MAX_NT;
    if (pitch > max_nt || T > 4096) return pl;
    const int64_t Qcap = std::min<int64_t>(s.H_o, max_nt / pitch);
    const int64_t MT = (s.C_o + BM - 1) / BM;
    for (int64_t Qfit = Qcap; Qfit >= 1; --Qfit) {
        // rows per tile: among tilings with at most Qfit rows, the one with the least
        // modelled time = rounds of tiles over the SMs x time of one tile
        int64_t Q = Qfit;
        double best = 1e30;
        for (int64_t tps = (s.H_o + Qfit - 1) / Qfit; tps <= (s.H_o + Qfit - 1) / Qfit + 4 && tps <= s.H_o; ++tps) {
            const int64_t q = (s.H_o + tps - 1) / tps;
            const int64_t tiles = s.N * MT * tps;
            const int64_t rounds = (tiles + sms - 1) / sms;
            const double t = (double)rounds * (xpose ? tile_cost_xpose(q * pitch) : tile_cost(q * pitch));
            if (t < best * 0.99) { best = t; Q = q; }
        }
        // positions the MMAs read from the slab (transposed: whole M blocks)
        const int64_t NTp = xpose ? (Q * pitch + 1 + 127) / 128 * 128 : (Q * pitch + stack + 15) / 16 * 16;
        const int64_t RR = (Q - 1) * s.s_h + Hfe;  // slab rows under a tile of Q rows
        int64_t PB = 0, lbo, stage_b;
        // the 128-byte-swizzled MN-major slab where the plane and the tile are whole
        // 64-position blocks
        const bool mn_sw = mnb && (s.H_i * s.W_i) % 64 == 0 && (Q * s.W_o) % 64 == 0;
        if (mnb) {
            // the two 8-channel core matrices of a 16-channel K step; swizzled, the
            // stride of the 64-position blocks
            lbo = mn_sw ? 2048 * mn_k : 128;
            stage_b = NTp * 32 * mn_k;
        } else if (kmb) {
            lbo = 16;  // (unused: a K step lies within the 128-byte rows)
            stage_b = NTp * 128;
        } else if (chan) {
            const int64_t HH = (RR + s.s_h - 1) / s.s_h;
            // a multiple of 128 bytes, so that every polyphase block of a stage can be the
            // destination of a tensor copy (its tail past the block's rows is never written)
            PB = (HH * pitch * 16 + 127) / 128 * 128;
            lbo = s.s_h * s.s_w * PB;
            int64_t max_tap = 0;
            for (int64_t r = 0; r < s.H_f; ++r)
                for (int64_t j = 0; j < s.W_f; ++j) {
                    const int64_t dr = tap_dr((int)r, (int)s.d_h), dc = tap_dc((int)j, (int)s.d_w, (int)s.g_w);
                    max_tap = std::max(max_tap, ((dr % s.s_h) * s.s_w + dc % s.s_w) * PB +
                                                    ((dr / s.s_h) * pitch + dc / s.s_w) * 16);
                }
            // plane 1 is written up to 2*lbo and read up to lbo + max_tap + NTp*16
            stage_b = std::max(2 * lbo, lbo + max_tap + NTp * 16);
        } else {
            lbo = Q * pitch * 16;
            // chunks 0..2U-1 are written; tap (a, u) reads chunks 2u, 2u+1 from a*16
            stage_b = std::max(2 * U * lbo, (2 * U - 1) * lbo + (A - 1 + NTp) * 16);
        }
        stage_b = (stage_b + 127) / 128 * 128;
        // raw staging slot (elements, a multiple of 64): TAP_CH 16 channel planes of the
        // tile's input rows (only when rows are whole 16-byte vectors), TAP_WX one
        // channel's input rows, TAP_WW its window rows, each with room for the alignment
        // lead; TAP_CL copies straight into the slab. A TAP_CH plane is RR rows of W_i
        // elements or, where it fits (tried first at each pipeline depth), Rb rows of Wb
        // elements, Rb in {RR, RR + 1} and Wb in {W_i, W_i + 8} both odd in 8-element
        // units, so that planes lie an odd number of 16-byte units apart: the eight
        // channel rows of a matrix load then fall in eight different bank groups.
        const int64_t Wb = (s.W_i / 8) % 2 ? s.W_i : s.W_i + 8, Rb = RR % 2 ? RR : RR + 1;
        auto slot_elems = [&](bool pad) -> int64_t {
            const int64_t slot = (mode == TAP_CL || mnb) ? 0
                                 : mode == TAP_CH ? (s.W_i % 8 == 0 ? 16 * (pad ? Rb * Wb : RR * s.W_i) : 0)
                                 : mode == TAP_WX ? RR * s.W_i + 16
                                                  : Q * s.W_i * s.H_f + 16;
            return (slot + 63) / 64 * 64;
        };
        // search: filter stages of at least 8 taps (or all of them) first, since every
        // stage costs the MMA issuers a fixed overhead; within that a ring of two raw
        // slots (the next chunk's copy in flight) before one slot (TAP_W*) or none
        // (TAP_CH); then larger filter stages, then three slab stages, then three
        // filter stages
        // Transposed stacking issues 128 x 128 MMAs, for which the issuers' fixed cost
        // per filter stage is large: there the candidates are the fewest stages per
        // chunk that fit (the smallest stage for each count), two stages first.
        int tg_list[64], n_tg = 0;
        if (xpose) {
            for (int64_t ns = 1; ns <= T && n_tg < 64; ++ns) {
                const int tg = (int)((T + ns - 1) / ns);
                if (n_tg == 0 || tg_list[n_tg - 1] != tg) tg_list[n_tg++] = tg;
            }
        } else {
            for (int v : {9, 8, 6, 5, 4, 3, 2, 1}) tg_list[n_tg++] = v;
        }
        const int ast_list[5] = {xpose ? 2 : 3, xpose ? 3 : 2, 4, 6, 0};
        for (int pass = 0; pass < 2; ++pass)
        for (int ring : {1, 0}) {
          if (ring && slot_elems(false) == 0) continue;
          for (int ti = 0; ti < n_tg; ++ti) {
            const int TG = tg_list[ti];
            const int tg = (int)std::min<int64_t>(TG, T);
            if (TG > T && TG != 1) continue;
            if (pass == 0 && !xpose && tg < std::min<int64_t>(T, 8)) continue;
            // a 1x1 slab copied by tensor copies: each stage is one copy in flight; up
            // to six stages, as many filter stages (a chunk's K steps each)
            const int bst_list[4] = {copy1 ? 6 : 3, copy1 ? 4 : 2, copy1 ? 3 : 0, copy1 ? 2 : 0};
            for (int BST : bst_list) {
              if (BST == 0) continue;
              for (int AST : ast_list) {
                if (AST == 0 || (copy1 ? AST != BST : AST == 6)) continue;
                for (int pad : {1, 0}) {
                    if (pad && !(mode == TAP_CH && ring)) continue;
                    const int64_t slot_e = slot_elems(pad != 0);
                    const int64_t raw_e = chan ? (ring ? 2 * slot_e : 0) : (ring ? 2 : 1) * slot_e;
                    int64_t total = (int64_t)AST * tg * TAP_A_BYTES + BST * stage_b + raw_e * 2 +
                                    tap_epi_region(epi_blocks, xpose) + 512 + 4 * T + 16 + 128 * U;
                    if (total > smem_max) continue;
                    // the 512-column TMEM accumulator needs the SM to itself
                    total = std::max<int64_t>(total, 120 * 1024);
                    TapParams &p = pl.p;
                    p.C_i = (int)s.C_i; p.C_o = (int)s.C_o; p.H_i = (int)s.H_i; p.W_i = (int)s.W_i;
                    p.H_o = (int)s.H_o; p.W_o = (int)s.W_o; p.H_f = (int)s.H_f; p.W_f = (int)s.W_f;
                    p.s_h = (int)s.s_h; p.s_w = (int)s.s_w;
                    p.MT = (int)((s.C_o + BM - 1) / BM);
                    p.NCH = (int)NCH;
                    p.T = (int)T;
                    p.stack = stack;
                    p.xpose = xpose ? 1 : 0;
                    p.Gr = Gr;
                    p.p_h = (int)s.p_h; p.p_w = (int)s.p_w;
                    p.dil_h = (int)s.d_h; p.dil_w = (int)s.d_w; p.g_w = (int)s.g_w;
                    p.Hfe = (int)Hfe;
                    p.Wp = (int)Wp;
                    p.padded = (s.p_h > 0 || s.p_w > 0) ? 1 : 0;
                    p.epi_blocks = xpose ? 0 : epi_blocks;
                    p.TG = tg;
                    p.ntg = (int)((T + tg - 1) / tg);
                    p.Qmax = (int)Q;
                    p.tps = (int)((s.H_o + Q - 1) / Q);
                    p.tiles_total = s.N * p.MT * p.tps;
                    p.pitch = (int)pitch;
                    p.lbo = (uint32_t)lbo;
                    p.PB = (uint32_t)PB;
                    p.U = (int)U;
                    p.S = (int)S;
                    p.A = (int)A;
                    p.L = s.W_i * s.H_f;
                    p.win_elems = s.N * s.C_i * s.H_o * s.W_i * s.H_f;
                    p.N_img = (int)s.N;
                    p.raw_elems = (int)raw_e;
                    p.ring = ring;
                    p.raw_slot = (int)slot_e;
                    p.mnb = mnb ? (mn_sw ? 2 : 1) : kmb ? 3 : 0;
                    p.mn_box = (int)(kmb ? Q * s.W_i : NTp);  // positions of a tile's copy
                    p.mn_k = (int)mn_k;
                    p.raw_rows = (int)(pad ? Rb : RR);
                    p.raw_w = (int)(pad ? Wb : s.W_i);
                    p.raw_ch = p.raw_rows * p.raw_w;
                    p.stage_b = (uint32_t)stage_b;
                    p.BST = BST;
                    p.AST = AST;
                    p.merge = (p.ntg == 1 && AST == BST) ? 1 : 0;
                    pl.smem = (size_t)total;
                    pl.mtiles = p.MT;
                    pl.kslots = NCH * T * 16;
                    pl.ok = p.tiles_total < (1ll << 40) && s.N < (1ll << 31) && raw_e < (1ll << 30);
                    return pl;
                }
              }
            }
          }
        }
    }
    return pl;
}

// Epilogue staging of two blocks per warp (release the accumulator before the
// stores) when it costs the tiling nothing: the same rows per tile and filter
// stages of at least min(T, 8) taps as with one block; one block otherwise, and
// always with tap stacking (its drain goes block by block).
TapPlan plan_tap(const Shape &s, int mode, int64_t sms) {
    // tap stacking with rows of at most 255 positions: transposed, TMEM double-buffered
    const TapPlan x = plan_tap_epi(s, mode, sms, 0, true);
    if (x.ok) return x;
    const TapPlan one = plan_tap_epi(s, mode, sms, 1);
    if (!one.ok || one.p.stack) return one;
    const TapPlan two = plan_tap_epi(s, mode, sms, 2);
    const int need_tg = std::min(one.p.TG, 8);
    if (two.ok && two.p.Qmax == one.p.Qmax && two.p.TG >= need_tg) return two;
    return one;
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

// The convolution from the window tensor is itself a valid convolution: each
// window row win[n][ci][ho][:] (W_i*H_f elements) is an input row, the filter is
// the re-laid filter as one row of W_f*H_f taps, and output pixel wo starts at
// window offset wo*s_w*H_f (the dot product of the im2win convolution). So the
// window tensor is an input of H_o x W_i*H_f, filtered by 1 x W_f*H_f at stride
// (1, s_w*H_f); the output extents are unchanged. A padded window tensor has
// rows of W_p*H_f elements and needs no padding of its own; with column
// dilation d_w, filter column j (run j / H_f) starts (j / H_f)*d_w*H_f + j % H_f
// into the pixel's window (g_w = H_f).
static Shape window_as_input(const Shape &s) {
    Shape v = s;
    v.H_i = s.H_o;
    v.W_i = padded_w(s) * s.H_f;
    v.H_f = 1;
    v.W_f = s.W_f * s.H_f;
    v.s_h = 1;
    v.s_w = s.s_w * s.H_f;
    v.p_h = v.p_w = 0;
    v.d_h = 1;
    v.d_w = s.d_w;
    v.g_w = s.d_w > 1 ? s.H_f : 1;
    return v;
}

// A channels-last tensor x[n][h][w][c] is, row by row, one channel of H x W*C
// elements: the convolution with C_i channels is the one-channel convolution
// of that image by the H_f x W_f*C_i filter whose column j*C_i + c is channel c
// of filter column j, at stride (s_h, s_w*C_i). The output extents are unchanged.
static Shape channels_as_columns(const Shape &s) {
    Shape v = s;
    v.C_i = 1;
    v.W_i = s.W_i * s.C_i;
    v.W_f = s.W_f * s.C_i;
    v.s_w = s.s_w * s.C_i;
    return v;
}

// Kernel choice: among the tap kernels that apply, the one that needs the
// fewest MMA K values per pixel (ties: the first listed).
//   NCHW fused:   TAP_CH over channels; TAP_WX over window rows.
//   NCHW window:  TAP_CH over the channels of the window tensor seen as an input
//                 (window_as_input); TAP_WW over window rows.
//   NHWC fused:   TAP_CL over channels (C_i a multiple of 8); TAP_WX over the
//                 input seen as one channel (channels_as_columns).
//   NHWC window:  TAP_CL over the window tensor seen as an input; TAP_WW over it
//                 seen as one channel.
// NCHW falls back to the expand kernel when the choice's K padding costs more
// than half again the expand kernel's K; NHWC has no fallback. Padding and
// dilation run the channel modes only (TAP_CH / TAP_CL), without fallback.
static bool has_expand(const Shape &s, int layout) { return layout == LAYOUT_NCHW && plain(s); }

static TapPlan choose_tap(const Shape &s, bool fused, int layout, int64_t sms = 148) {
    struct Cand {
        int mode;
        Shape v;
        int view;
    };
    Cand cand[2];
    if (layout == LAYOUT_NHWC) {
        const Shape base = fused ? s : window_as_input(s);
        cand[0] = {TAP_CL, base, fused ? VIEW_IDENT : VIEW_WIN};
        cand[1] = {fused ? TAP_WX : TAP_WW, channels_as_columns(base), fused ? VIEW_CL_X : VIEW_CL_WIN};
    } else if (fused) {
        cand[0] = {TAP_CH, s, VIEW_IDENT};
        cand[1] = {TAP_WX, s, VIEW_IDENT};
    } else {
        cand[0] = {TAP_CH, window_as_input(s), VIEW_WIN};
        cand[1] = {TAP_WW, s, VIEW_IDENT};
    }
    TapPlan best{};
    best.ok = false;
    for (const Cand &c : cand) {
        TapPlan pl = plan_tap(c.v, c.mode, sms);
        pl.view = c.view;
        if (pl.ok && (!best.ok || pl.kslots < best.kslots)) best = pl;
    }
    const int64_t expand_k = s.C_i * ((s.H_f * s.W_f + 7) / 8 * 8);
    if (has_expand(s, layout) && best.ok && best.kslots * 2 > expand_k * 3) best.ok = false;
    return best;
}

size_t conv_tc_filter_bytes(const Shape &s, bool fused, int layout) {
    const TapPlan pl = choose_tap(s, fused, layout);
    if (pl.ok) return round_up((size_t)pl.mtiles * pl.p.NCH * pl.p.T * TAP_A_BYTES, 256);
    if (!has_expand(s, layout)) return 0;
    const ExpandGeom g = expand_geom(s);
    return round_up((size_t)g.mtiles * BM * (size_t)g.K_pad * 2, 256);
}

bool conv_tc_supported(const Shape &s, bool fused, int layout) {
    if (choose_tap(s, fused, layout).ok) return true;
    if (!has_expand(s, layout)) return false;
    const int64_t img = fused ? s.C_i * s.H_i * s.W_i : s.C_i * s.H_o * s.W_i * s.H_f;
    const int64_t KKP = (s.H_f * s.W_f + 7) / 8 * 8;
    const int64_t P = s.H_o * s.W_o;
    const int64_t pos_tiles = (P + NT - 1) / NT;
    return img < (1ll << 31) && s.C_i * KKP < (1ll << 30) && P < (1ll << 31) &&
           pos_tiles * s.N < (1ll << 31) && (s.C_o + BM - 1) / BM < 65536;
}

bool conv_tc_plan_info(const Shape &s, bool fused, int layout, int64_t sms, TcPlanInfo &info) {
    if (!conv_tc_supported(s, fused, layout)) return false;
    if (sms <= 0) sms = sm_count();
    info = TcPlanInfo{};
    const TapPlan pl = choose_tap(s, fused, layout, sms);
    if (!pl.ok) {
        info.kernel = 2;
        info.tap_mode = -1;
        return true;
    }
    const TapParams &p = pl.p;
    info.kernel = 1;
    info.tap_mode = pl.mode;
    info.stacked = p.stack ? (p.xpose ? 2 : 1) : 0;
    info.rows_per_tile = p.Qmax;
    info.pitch = p.pitch;
    const int NT = p.Qmax * p.pitch;  // the widest tile's positions
    if (p.xpose) {
        // two TMEM buffers of up to two 128-column M blocks; the MMAs write, and the
        // epilogue reads, buffer 1 up to its last M block's end
        const int nmb = (NT + 1 + 127) / 128;
        info.tmem_columns = 256 + nmb * 128;
        info.tmem_read_end = info.tmem_columns;
        info.smem_bytes = (int)pl.smem;
        info.filter_stage_taps = p.TG;
        info.filter_stages = p.AST;
        info.slab_stages = p.BST;
        info.tiles = p.tiles_total;
        info.grid = std::min<int64_t>(sms, p.tiles_total);
        return true;
    }
    const int NTp = (NT + p.stack + 15) / 16 * 16;
    info.tmem_columns = NTp;
    // The epilogue's column walk: the two warps of a lane quarter split a range in
    // 64-column blocks; without stacking a warp reads 32-column loads while they
    // start inside its share, with stacking every block whole plus (lower half)
    // the column after it.
    int end = 0;
    auto walk = [&](int a0, int a1) {
        const int nb = (a1 - a0 + 63) / 64;
        const int mid = a0 + ((nb + 1) / 2) * 64;
        for (int hh = 0; hh < 2; ++hh) {
            const int cb = hh == 0 ? a0 : mid, ce = hh == 0 ? std::min(a1, mid) : a1;
            if (cb >= ce) continue;
            end = std::max(end, p.stack ? cb + (ce - cb + 63) / 64 * 64 + 1 : cb + (ce - cb + 31) / 32 * 32);
        }
    };
    if (p.stack) {
        walk(0, (NT + 15) / 16 * 16);
    } else {
        const int N0 = split_n0(NTp, p.mnb == 2 ? 64 : 32);
        walk(0, N0);
        walk(N0, NTp);
    }
    info.tmem_read_end = end;
    info.smem_bytes = (int)pl.smem;
    info.filter_stage_taps = p.TG;
    info.filter_stages = p.AST;
    info.slab_stages = p.BST;
    info.tiles = p.tiles_total;
    info.grid = std::min<int64_t>(sms, p.tiles_total);
    return true;
}

// cuTensorMapEncodeTiled, from the driver through the runtime (no link to the
// driver library); null when the driver does not provide it.
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// The tensor map of TAP_CH's raw rows: the kernel's input (16-bit elements; the
// window tensor when it is read as one) as a 4-D tensor (W_i, H_i, C_i, N) of
// the kernel's shape, box (raw_w, raw_rows, 16, 1), zero fill outside (the
// padding columns and row of a raw plane). False when the box is out of the
// copy engine's limits (at most 256 per dimension) or the encoder refuses it;
// the per-channel bulk copies then stage the rows.
static bool encode_raw_map(TapParams &p, const void *src) {
    if (p.raw_w > 256 || p.raw_rows > 256 || (reinterpret_cast<uintptr_t>(src) & 15) != 0) return false;
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t W = (cuuint64_t)p.W_i, H = (cuuint64_t)p.H_i, C = (cuuint64_t)p.C_i;
    const cuuint64_t dims[4] = {W, H, C, (cuuint64_t)p.N_img};
    const cuuint64_t strides[3] = {W * 2, H * W * 2, C * H * W * 2};
    const cuuint32_t box[4] = {(cuuint32_t)p.raw_w, (cuuint32_t)p.raw_rows, 16u, 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    const CUresult r = enc(&p.tmap_x, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<void *>(src), dims, strides,
                           box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The tensor map of TAP_CL's slab: the kernel's channels-last input as a 4-D
// tensor (C_i, W_i, H_i, N), box (8 channels, pitch*s_w columns, rows per
// polyphase block * s_h, 1) traversed with element strides (1, s_w, s_h, 1), so
// that one copy writes one polyphase block of one 8-channel half as its dense
// [row][column][8 channels] entries; zero fill outside. False when out of the
// copy engine's limits (box at most 256 and element strides at most 8 per
// dimension) or the encoder refuses it; the producers' 16-byte copies fill the
// slab instead.
static bool encode_slab_map(TapParams &p, const void *src) {
    const int64_t HH = ((int64_t)(p.Qmax - 1) * p.s_h + p.Hfe + p.s_h - 1) / p.s_h;  // rows of a polyphase block
    // every block starts a multiple of PB into a 128-byte aligned stage: the copies'
    // shared-memory destinations are 128-byte aligned only when PB is
    if ((int64_t)p.pitch * p.s_w > 256 || HH * p.s_h > 256 || p.s_w > 8 || p.s_h > 8 || p.PB % 128 != 0 ||
        p.stage_b % 128 != 0 || (reinterpret_cast<uintptr_t>(src) & 15) != 0)
        return false;
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t W = (cuuint64_t)p.W_i, H = (cuuint64_t)p.H_i, C = (cuuint64_t)p.C_i;
    const cuuint64_t dims[4] = {C, W, H, (cuuint64_t)p.N_img};
    const cuuint64_t strides[3] = {C * 2, W * C * 2, H * W * C * 2};
    const cuuint32_t box[4] = {8u, (cuuint32_t)(p.pitch * p.s_w), (cuuint32_t)(HH * p.s_h), 1u};
    const cuuint32_t estr[4] = {1u, (cuuint32_t)p.s_w, (cuuint32_t)p.s_h, 1u};
    const CUresult r = enc(&p.tmap_x, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<void *>(src), dims, strides,
                           box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    p.slab_hh = (int)HH;
    return r == CUDA_SUCCESS;
}

// The tensor map of an MN-major 1x1 slab (mnb), zero fill outside (past the
// plane's last position group, channels past C_i); false when the encoder
// refuses it.
//  mnb = 1: the input as a 4-D tensor (8, C_i, H_i*W_i/8, N) -- eight consecutive
//    positions, channels, position groups, images -- box (8, 16*mn_k, mn_box/8, 1).
//  mnb = 2: the same with 64-position blocks, box (64, 16*mn_k, mn_box/64, 1), and
//    the copy's 128-byte swizzle (rows of 128 bytes). The planner chose it only
//    where the plane and every tile are whole blocks.
static bool encode_mn_map(TapParams &p, const void *src) {
    const int64_t P = (int64_t)p.H_i * p.W_i;
    const int64_t G = p.mnb == 2 ? 64 : 8;  // positions per row of the box
    if (P % G != 0 || p.mn_box % G != 0 || p.mn_box / G > 256 || (reinterpret_cast<uintptr_t>(src) & 15) != 0)
        return false;
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)G, (cuuint64_t)p.C_i, (cuuint64_t)(P / G), (cuuint64_t)p.N_img};
    const cuuint64_t strides[3] = {(cuuint64_t)P * 2, (cuuint64_t)G * 2, (cuuint64_t)p.C_i * P * 2};
    const cuuint32_t box[4] = {(cuuint32_t)G, 16u * (cuuint32_t)p.mn_k, (cuuint32_t)(p.mn_box / G), 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    const CUresult r = enc(&p.tmap_x, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<void *>(src), dims, strides,
                           box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           p.mnb == 2 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The tensor map of a channels-last K-major 1x1 slab (mnb = 3): the input as
// (C_i, W_i, H_i, N), box (64, W_i, Qmax, 1) -- 64 channels of every position of
// a tile's rows -- with the copy's 128-byte swizzle; rows past H_i read as zero.
// False when the shape or the encoder refuses it.
static bool encode_kmb_map(TapParams &p, const void *src) {
    if (p.C_i % 64 != 0 || p.W_i > 256 || p.Qmax > 256 || (reinterpret_cast<uintptr_t>(src) & 15) != 0)
        return false;
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t W = (cuuint64_t)p.W_i, H = (cuuint64_t)p.H_i, C = (cuuint64_t)p.C_i;
    const cuuint64_t dims[4] = {C, W, H, (cuuint64_t)p.N_img};
    const cuuint64_t strides[3] = {C * 2, W * C * 2, H * W * C * 2};
    const cuuint32_t box[4] = {64u, (cuuint32_t)p.W_i, (cuuint32_t)p.Qmax, 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    const CUresult r = enc(&p.tmap_x, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<void *>(src), dims, strides,
                           box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

static cudaError_t launch_tap(const TapPlan &pl, const void *src, const void *filt, void *out,
                              void *ws, const Shape &s, int layout, bool bf16, cudaStream_t st) {
    TapParams p = pl.p;
    uint32_t *status = static_cast<uint32_t *>(ws);
    uint16_t *fa = reinterpret_cast<uint16_t *>(static_cast<unsigned char *>(ws) + kStatusBytes);
    // (an MN-major 1x1 slab's chunk of mn_k K steps is mn_k 16-channel chunks of one tap)
    const int relay_nch = p.mnb ? p.NCH * p.mn_k : p.NCH, relay_t = p.mnb ? 1 : p.T;
    const int n_chunks = pl.mtiles * relay_nch;
    const int per_chunk = relay_t * (int)(TAP_A_BYTES / 2);
    const dim3 rgrid((unsigned)std::min(std::max(1, (per_chunk + 255) / 256), 64),
                     (unsigned)std::min(n_chunks, 65535));
    TapRelayout ra;
    ra.mode = pl.mode;
    ra.C_v = p.C_i; ra.H_fv = p.H_f; ra.W_fv = p.W_f; ra.s_wv = p.s_w;
    ra.view = pl.view; ra.C = (int)s.C_i; ra.H_f = (int)s.H_f; ra.W_f = (int)s.W_f;
    ra.C_o = p.C_o; ra.T = relay_t; ra.NCH = relay_nch; ra.U = p.U; ra.S = p.S;
    ra.n_chunks = n_chunks; ra.stack = p.stack; ra.Gr = p.Gr;
    relayout_filter_tap<<<rgrid, 256, 0, st>>>(static_cast<const uint16_t *>(filt), fa, status, ra);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    p.src = static_cast<const uint16_t *>(src);
    p.fa = fa;
    p.out = static_cast<uint16_t *>(out);
    p.status = status;
    p.vec = (p.W_i % 8 == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0) ? 1 : 0;
    if (pl.mode == TAP_CL)  // 16-byte entries: 8 channels of one position
        p.vec = (p.C_i % 8 == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0) ? 1 : 0;
    if (pl.mode == TAP_CH && !p.vec) p.ring = 0;  // 16-byte copies need 16-byte rows
    p.tma_raw = (pl.mode == TAP_CH && p.ring && !p.mnb && encode_raw_map(p, src)) ? 1 : 0;
    if (pl.mode == TAP_CH && p.mnb && !encode_mn_map(p, src)) return cudaErrorInvalidValue;
    if (!p.tma_raw) p.raw_w = p.W_i;  // per-channel bulk copies: contiguous rows
    if (pl.mode == TAP_CL && p.mnb == 3) {
        // the plan's slab layout is the swizzled copy's: no other fill writes it
        if (!p.vec || !encode_kmb_map(p, src)) return cudaErrorInvalidValue;
        p.tma_slab = 1;
    } else {
        p.tma_slab = (pl.mode == TAP_CL && p.vec && encode_slab_map(p, src)) ? 1 : 0;
    }
    p.div_pitch = make_fastdiv((uint32_t)p.pitch);
    p.div_cgs = make_fastdiv((uint32_t)std::max(1, p.W_i / 8));
    p.div_sh = make_fastdiv((uint32_t)p.s_h);
    p.div_sw = make_fastdiv((uint32_t)p.s_w);
    p.div_wi = make_fastdiv((uint32_t)p.Wp);
    p.nhwc = layout == LAYOUT_NHWC ? 1 : 0;
    p.bf16 = bf16 ? 1 : 0;
    const unsigned grid = (unsigned)std::min<int64_t>(sm_count(), p.tiles_total);
    auto go = [&](auto kernel) -> cudaError_t {
        cudaError_t e2 = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
        if (e2 != cudaSuccess) return e2;
        // launched as a programmatic dependent of the re-layout kernel: the prologue
        // overlaps it, the kernel waits for it before touching its output
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(TAP_THREADS);
        cfg.dynamicSmemBytes = pl.smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kernel, p);
    };
    if (pl.mode == TAP_CH) return go(conv_tc_tap_kernel<TAP_CH>);
    if (pl.mode == TAP_CL) return go(conv_tc_tap_kernel<TAP_CL>);
    if (pl.mode == TAP_WX) return go(conv_tc_tap_kernel<TAP_WX>);
    return go(conv_tc_tap_kernel<TAP_WW>);
}

cudaError_t launch_conv_tc(const void *src, const void *filt, void *out, void *ws, const Shape &s,
                           bool fused, int layout, bool bf16, cudaStream_t st) {
    const TapPlan pl = choose_tap(s, fused, layout, sm_count());
    if (pl.ok) return launch_tap(pl, src, filt, out, ws, s, layout, bf16, st);
    if (!has_expand(s, layout)) return cudaErrorNotSupported;
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
    p.idesc = make_idesc(bf16, BM, NT / 2);
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
