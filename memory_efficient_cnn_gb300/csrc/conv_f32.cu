// fp32 im2win convolution on the CUDA cores (sm_103a).
//
// "Enabling Memory-efficient Im2win Convolution with Multi-precision Support
// on GPU CUDA and Tensor Cores", Abstract (full precision on CUDA cores):
//   out[n][co][ho][wo] = sum_ci sum_{k < W_f*H_f} win[n][ci][ho][wo*s_w*H_f + k] * filt'[co][ci][k]
//   filt'[co][ci][j*H_f + r] = filt[co][ci][r][j]
// Seen as a product of the filter matrix filt' (C_o x K, K = C_i*W_f*H_f,
// row-major) with a matrix whose column for output pixel p = (ho, wo) is the
// concatenation over ci of that pixel's contiguous window segments.
//
// Kernel: a CTA computes TM output channels x 128 pixels of one image.
// The K dimension is walked in chunks of KC; each chunk's window segments
// (KC x 128) and filter slice (KC x TM) are staged in shared memory, double
// buffered through registers, and every thread accumulates an 8 x 8
// (channels x pixels) register tile with FFMA (4 operand reads of 16 bytes
// per 64 FFMA). Warps are 4 channel-groups x 8 pixel-groups so that every
// shared-memory operand read is one conflict-free wavefront.
// The fused variant (FROM_X) gathers the same matrix straight from the NCHW
// input (x[n][ci][ho*s_h + r][wo*s_w + j] for k = j*H_f + r) and never
// materialises the window tensor.
//
// Channels-last tensors (NHWC) run the window path over a virtual shape:
//  * from the channels-last window tensor, whose window row is one run of
//    W_i*H_f*C_i elements: one channel, K = W_f*H_f*C_i contiguous elements per
//    pixel starting at wo*s_w*H_f*C_i;
//  * fused from the NHWC input: the H_f filter rows play the channels, each a
//    contiguous run of W_f*C_i elements of input row ho*s_h + r starting at
//    column wo*s_w (channel stride W_i*C_i, pixel stride s_w*C_i).
// In both the filter is re-laid in the matching order and the epilogue writes
// out[n][ho][wo][co].
//
// Zero padding and dilation (GEN): the same kernel with the fused variant's
// lane mapping and a general gather: element (ci, r, j) of pixel (ho, wo) is
// x[ci][ho*s_h + r*d_h - p_h][wo*s_w + j*d_w - p_w] (zero outside x; either
// layout), or, from the padded window tensor, window column
// (wo*s_w + j*d_w)*H_f + r of window row (ci, ho).
#include <algorithm>

#include "im2win_internal.cuh"
#include "tc_ptx.cuh"

namespace im2win {
namespace {

constexpr int TP = 128;  // pixels per CTA

struct F32Params {
    const float *src;    // window tensor or NCHW input
    const float *filt;   // filt' transposed and zero padded: [K_pad][C_o_pad]
    float *out;
    uint32_t *status;
    int C_i, C_o, H_o, W_o, H_i, W_i, H_f, s_h, s_w;
    int P;               // H_o * W_o
    int K;               // C_i * W_f * H_f
    int KK;              // W_f * H_f
    int pos_tiles;       // ceil(P / TP)
    int L;               // W_i * H_f
    int S;               // s_w * H_f
    int64_t img_src;     // elements of src per image
    int cs;              // window path: element stride between channels (H_o*L for the NCHW window)
    // general gather (padding / dilation)
    int from_win;        // source is the padded window tensor (else the input)
    int p_h, p_w, d_h, d_w, W_f;
    int Lw;              // padded window row length W_p*H_f
    int C_o_pad;         // row length of the transposed filter (a multiple of the channel tile)
    FastDiv div_KK, div_Wo, div_Hf;
};

// The filter is padded along K to a multiple of every chunk length (16, 24, 48).
constexpr int K_ALIGN = 48;

// Kernel configurations per channel tile: TM, RI (channels per thread), KC (k
// per chunk), pipeline stages, CTAs per SM the registers are budgeted for. The
// 96-channel tile runs 6 x 8 register tiles in 256 threads: 16 warps per SM
// instead of the 12 of 8 x 8 tiles in 192 threads.
#ifndef F32_CFG_128
#define F32_CFG_128 128, 8, 16, 3, 2
#endif
#ifndef F32_CFG_96
#define F32_CFG_96 96, 6, 16, 3, 2
#endif
#ifndef F32_CFG_64
#define F32_CFG_64 64, 8, 16, 3, 3
#endif
#ifndef F32_CFG_32
#define F32_CFG_32 32, 8, 8, 3, 4
#endif

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// 4-byte asynchronous copy global -> shared; src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async4(uint32_t dst, const float *src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}
// 16-byte asynchronous copy global -> shared (L2 only).
__device__ __forceinline__ void cp_async16(uint32_t dst, const float *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// The RI filter values of a thread's channels at one k: two 16-byte loads (RI =
// 8) or three 8-byte loads (RI = 6: a 24-byte group, 8-byte aligned).
template <int RI>
__device__ __forceinline__ void load_b(const float *b, float (&bv)[RI]) {
    if (RI == 8) {
        const float4 b0 = *reinterpret_cast<const float4 *>(b);
        const float4 b1 = *reinterpret_cast<const float4 *>(b + 4);
        const float t[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int i = 0; i < RI; ++i) bv[i] = t[i];
    } else {
#pragma unroll
        for (int i = 0; i < RI; i += 2) {
            const float2 v = *reinterpret_cast<const float2 *>(b + i);
            bv[i] = v.x;
            bv[i + 1] = v.y;
        }
    }
}

// TM output channels x 128 pixels per CTA, RI x 8 register tile per thread
// (channels ty*RI..+RI-1, pixels tx*4..+3 and 64 + tx*4..+3). K is staged KC at a
// time through a STAGES-deep cp.async pipeline (gathers go straight to shared
// memory, so no registers hold prefetched data). The filter slice arrives as
// 16-byte vectors. The 4-byte gathers follow the contiguous direction of the
// source: from the window tensor consecutive k of a pixel are consecutive
// elements, so a warp's copy covers 8 consecutive k of 4 pixels (lane l: k
// offset l % 8, pixel offset l / 8) -- 32-byte runs in global memory and, with
// the 4-word padding of a shared row, 32 distinct banks; warp w keeps k group
// w % (KC/8) and walks every (NW/(KC/8))-th group of 4 pixels. From the NCHW
// input consecutive pixels of a row are (unit stride), so lane l of warp w
// gathers pixels l + 32i at the KPT values of k w*KPT ...
template <int TM, int RI, int KC, int STAGES, int MINB, bool FROM_X, bool CL, bool GEN>
__global__ void __launch_bounds__(TM / RI * 16, MINB) conv_f32_kernel(F32Params p) {
    constexpr int NT = TM / RI * 16;           // (TM/RI) x 16 threads
    constexpr int NW = NT / 32;                           // warps
    constexpr int KG = KC / 8;                            // window path: 8-k groups per chunk
    constexpr int PPT = FROM_X ? TP / 32 : TP * KG / (4 * NW);  // pixels each thread gathers
    constexpr int KPT = FROM_X ? KC * 32 / NT : 1;        // k values each thread gathers
    constexpr int B_N = KC * TM / 4;                      // 16-byte filter vectors of a chunk
    constexpr int B_VEC = (B_N + NT - 1) / NT;            // ... each thread stages at most
    static_assert((FROM_X ? KPT * NW == KC : (KC % 8 == 0 && NW % KG == 0 && PPT * 4 * NW == TP * KG)) &&
                      (RI == 8 || RI == 6) && TM % RI == 0 && (TP + 4) % 32 == 4,
                  "tile");
    static_assert(K_ALIGN % KC == 0, "filter padding");
    extern __shared__ __align__(16) float smem_f[];
    float (*As)[KC][TP + 4] = reinterpret_cast<float (*)[KC][TP + 4]>(smem_f);
    float (*Bs)[KC][TM + 4] = reinterpret_cast<float (*)[KC][TM + 4]>(smem_f + STAGES * KC * (TP + 4));

    const int tid = threadIdx.x;
    const int n = blockIdx.x / p.pos_tiles;
    const int p0 = (blockIdx.x - n * p.pos_tiles) * TP;
    const int co0 = blockIdx.y * TM;
    const float *__restrict__ src = p.src + (int64_t)n * p.img_src;
    const float *__restrict__ filt = p.filt;

    // ---- staging coordinates
    // thread's first pixel, pixel step, first k and shared-memory row/column
    const int px0 = FROM_X ? (tid & 31) : ((tid >> 5) / KG) * 4 + ((tid & 31) >> 3);
    constexpr int PXS = FROM_X ? 32 : 4 * (NW / KG);
    const int k0 = FROM_X ? (tid >> 5) * KPT : ((tid >> 5) % KG) * 8 + (tid & 7);
    int pos_off[PPT];     // offset of the pixel's window segment; pixels past P read offset 0, size 0
    uint32_t pos_ok = 0;  // bit i: pixel i exists
    int gh[GEN ? PPT : 1], gw[GEN ? PPT : 1];  // GEN: the pixel's first input row / column
#pragma unroll
    for (int i = 0; i < PPT; ++i) {
        const int pg = p0 + px0 + PXS * i;
        pos_off[i] = 0;
        if (GEN) gh[i] = gw[i] = 0;
        if (pg < p.P) {
            const int ho = (int)fdiv((uint32_t)pg, p.div_Wo);
            const int wo = pg - ho * p.W_o;
            pos_off[i] = FROM_X ? (ho * p.s_h * p.W_i + wo * p.s_w) : (ho * p.L + wo * p.S);
            if (GEN) {
                gh[i] = p.from_win ? ho : ho * p.s_h - p.p_h;
                gw[i] = p.from_win ? wo * p.s_w : wo * p.s_w - p.p_w;
            }
            pos_ok |= 1u << i;
        }
    }
    const uint32_t a_dst0 = smem_addr(&As[0][k0][px0]);
    const uint32_t b_dst0 = smem_addr(&Bs[0][0][0]);
    constexpr uint32_t A_BUF = KC * (TP + 4) * 4, B_BUF = KC * (TM + 4) * 4;
    const float *__restrict__ fcol = filt + co0;

    auto issue_chunk = [&](int c) {
        const int buf = c % STAGES;
        const uint32_t a_dst = a_dst0 + buf * A_BUF;
#pragma unroll
        for (int j = 0; j < (GEN ? KPT : 0); ++j) {
            // general gather: k = ci*KK + jj*H_f + r
            const int kg = c * KC + k0 + j;
            int ci = 0, jj = 0, r = 0;
            const bool kin = kg < p.K;
            if (kin) {
                ci = (int)fdiv((uint32_t)kg, p.div_KK);
                const int kk = kg - ci * p.KK;
                jj = (int)fdiv((uint32_t)kk, p.div_Hf);
                r = kk - jj * p.H_f;
            }
#pragma unroll
            for (int i = 0; i < PPT; ++i) {
                bool ok = kin && ((pos_ok >> i) & 1u);
                int off = 0;
                if (p.from_win) {
                    const int col = (gw[i] + jj * p.d_w) * p.H_f + r;
                    off = CL ? (gh[i] * p.Lw + col) * p.C_i + ci : (ci * p.H_o + gh[i]) * p.Lw + col;
                } else {
                    const int h = gh[i] + r * p.d_h, w = gw[i] + jj * p.d_w;
                    ok = ok && (unsigned)h < (unsigned)p.H_i && (unsigned)w < (unsigned)p.W_i;
                    off = CL ? (h * p.W_i + w) * p.C_i + ci : (ci * p.H_i + h) * p.W_i + w;
                }
                cp_async4(a_dst + (j * (TP + 4) + PXS * i) * 4, ok ? src + off : src, ok ? 4u : 0u);
            }
        }
#pragma unroll
        for (int j = 0; j < (GEN ? 0 : KPT); ++j) {
            const int kg = c * KC + k0 + j;
            int coff = 0;
            uint32_t ok = 0;
            if (kg < p.K) {
                const int ci = (int)fdiv((uint32_t)kg, p.div_KK);
                const int kk = kg - ci * p.KK;
                if (FROM_X) {
                    const int jj = (int)fdiv((uint32_t)kk, p.div_Hf);
                    const int r = kk - jj * p.H_f;
                    coff = (ci * p.H_i + r) * p.W_i + jj;
                } else {
                    coff = ci * p.cs + kk;
                }
                ok = pos_ok;
            }
#pragma unroll
            for (int i = 0; i < PPT; ++i)
                cp_async4(a_dst + (j * (TP + 4) + PXS * i) * 4, src + (pos_off[i] + coff), ((ok >> i) & 1u) * 4u);
        }
        // filter rows c*KC .. c*KC + KC - 1, channels co0 .. co0 + TM - 1 (zero padded in memory)
        const uint32_t b_dst = b_dst0 + buf * B_BUF;
#pragma unroll
        for (int v = 0; v < B_VEC; ++v) {
            const int q = tid + v * NT;            // vector index in the KC x TM/4 slice
            if (B_N % NT != 0 && q >= B_N) break;
            const int kr = q / (TM / 4), cv = q - kr * (TM / 4);
            cp_async16(b_dst + (kr * (TM + 4) + cv * 4) * 4, fcol + (int64_t)(c * KC + kr) * p.C_o_pad + cv * 4);
        }
    };

    // ---- compute coordinates: warps of 4 channel groups x 8 pixel groups
    const int warp = tid >> 5, lane = tid & 31;
    const int ty = (warp >> 1) * 4 + (lane >> 3);  // channel group (RI channels)
    const int tx = (warp & 1) * 8 + (lane & 7);     // pixel group (2 x 4 pixels)

    float acc[RI][8];
#pragma unroll
    for (int i = 0; i < RI; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    // Pacing of the pipeline. Channel tiles below 128 (24- and 16-k chunks): stage
    // s has mbarriers; full[s] completes when every thread's copies of its chunk
    // have landed (one cp.async.mbarrier.arrive.noinc per thread), empty[s] when
    // every warp has computed it. Chunk c - 1's stage is refilled (with chunk
    // c - 1 + STAGES) after this warp has computed chunk c, so a warp waits for
    // the others only when it is a whole chunk ahead of the slowest (cv1: 574
    // instead of 581 us). Waits are bounded: one that gives up records
    // IM2WIN_ERR_TIMEOUT in the status word. The 128-channel tile's chunks are
    // short (16 k); there a barrier per chunk, with two chunks in flight, measured
    // faster (990 instead of 1002 us on the 3x3 sweep layer).
    constexpr bool MBAR = TM < 128;
    __shared__ uint64_t bar_full[STAGES], bar_empty[STAGES];
    if (MBAR && tid == 0) {
        for (int st = 0; st < STAGES; ++st) {
            tc::mbar_init(tc::smem_u32(&bar_full[st]), NT);
            tc::mbar_init(tc::smem_u32(&bar_empty[st]), NW);
        }
        tc::fence_mbar_init();
    }
    __syncthreads();
    auto wait_bar = [&](uint64_t *bar, uint32_t parity) -> bool {
        const uint32_t a = tc::smem_u32(bar);
        if (tc::mbar_try_wait(a, parity)) return true;
        const uint64_t t0 = tc::globaltimer();
        for (uint32_t spin = 1;; ++spin) {
            if (tc::mbar_try_wait(a, parity)) return true;
            if ((spin & 255u) == 0 && tc::globaltimer() - t0 > tc::kTimeoutNs) {
                atomicCAS(p.status, 0u, (uint32_t)IM2WIN_ERR_TIMEOUT);
                return false;
            }
        }
    };

    const int nchunks = (p.K + KC - 1) / KC;
#pragma unroll
    for (int c = 0; c < (MBAR ? STAGES : STAGES - 1); ++c) {
        if (c < nchunks) issue_chunk(c);
        if (MBAR) {
            if (c < nchunks) tc::cp_async_mbar_arrive_noinc(tc::smem_u32(&bar_full[c]));
        } else {
            cp_async_commit();
        }
    }
    // k values of the last chunk (the rest of it is the filter's zero padding);
    // the 128-channel tile, whose registers are capped at 128, always runs whole
    // chunks (a separate short loop makes it spill)
    const int k_last = TM == 128 ? KC : p.K - (nchunks - 1) * KC;
    for (int c = 0; c < nchunks; ++c) {
        const int buf = c % STAGES;
        if (MBAR) {
            if (!wait_bar(&bar_full[buf], (uint32_t)(c / STAGES) & 1u)) break;
        } else {
            cp_async_wait<STAGES - 2>();  // chunk c has landed (this thread's copies)
            __syncthreads();              // ... and every thread's; chunk c-1's buffer is free
            if (c + STAGES - 1 < nchunks) issue_chunk(c + STAGES - 1);
            cp_async_commit();
        }
        if (TM == 128 || c + 1 < nchunks || k_last == KC) {
#pragma unroll
            for (int k = 0; k < KC; ++k) {
                const float4 a0 = *reinterpret_cast<const float4 *>(&As[buf][k][tx * 4]);
                const float4 a1 = *reinterpret_cast<const float4 *>(&As[buf][k][64 + tx * 4]);
                const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                float bv[RI];
                load_b<RI>(&Bs[buf][k][ty * RI], bv);
#pragma unroll
                for (int i = 0; i < RI; ++i)
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(bv[i], av[j], acc[i][j]);
            }
        } else {
            // the same k steps, only the k_last that are not padding
#pragma unroll 1
            for (int k = 0; k < k_last; ++k) {
                const float4 a0 = *reinterpret_cast<const float4 *>(&As[buf][k][tx * 4]);
                const float4 a1 = *reinterpret_cast<const float4 *>(&As[buf][k][64 + tx * 4]);
                const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                float bv[RI];
                load_b<RI>(&Bs[buf][k][ty * RI], bv);
#pragma unroll
                for (int i = 0; i < RI; ++i)
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(bv[i], av[j], acc[i][j]);
            }
        }
        if (!MBAR) continue;
        __syncwarp();
        if ((tid & 31) == 0) tc::mbar_arrive(tc::smem_u32(&bar_empty[buf]));
        // refill chunk c - 1's stage once every warp has computed it
        const int cr = c - 1 + STAGES;
        if (c >= 1 && cr < nchunks) {
            const int sr = (c - 1) % STAGES;
            if (!wait_bar(&bar_empty[sr], (uint32_t)((c - 1) / STAGES) & 1u)) break;
            issue_chunk(cr);
            tc::cp_async_mbar_arrive_noinc(tc::smem_u32(&bar_full[sr]));
        }
    }
    cp_async_commit();
    cp_async_wait<0>();

    // ---- epilogue: out[n][co][p], or (CL) out[n][p][co] (RI consecutive channels per pixel)
    if (CL) {
        const int cb = co0 + ty * RI;
        const bool vec = RI == 8 ? ((p.C_o & 3) == 0 && cb + 8 <= p.C_o) : ((p.C_o & 1) == 0 && cb + RI <= p.C_o);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int pg = p0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
            if (pg >= p.P) continue;
            float *d = p.out + ((int64_t)n * p.P + pg) * p.C_o + cb;
            if (vec && RI == 8) {
                reinterpret_cast<float4 *>(d)[0] = make_float4(acc[0][j], acc[1][j], acc[2][j], acc[3][j]);
                reinterpret_cast<float4 *>(d)[1] = make_float4(acc[4 % RI][j], acc[5 % RI][j], acc[6 % RI][j],
                                                               acc[7 % RI][j]);
            } else if (vec) {
#pragma unroll
                for (int i = 0; i < RI; i += 2) reinterpret_cast<float2 *>(d)[i / 2] = make_float2(acc[i][j], acc[i + 1][j]);
            } else {
#pragma unroll
                for (int i = 0; i < RI; ++i)
                    if (cb + i < p.C_o) d[i] = acc[i][j];
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < RI; ++i) {
            const int co = co0 + ty * RI + i;
            if (co >= p.C_o) continue;
            float *orow = p.out + ((int64_t)n * p.C_o + co) * p.P;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int pg = p0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
                if (pg < p.P) orow[pg] = acc[i][j];
            }
        }
    }
}

template <int TM, int KC, int STAGES>
constexpr size_t f32_smem_bytes() {
    return (size_t)STAGES * KC * ((TP + 4) + (TM + 4)) * sizeof(float);
}

// fT[k][co] = filt'[co][k] with filt'[co][ci*KK + j*H_f + r] = filt[co][ci][r][j]
// for the kernel's (virtual) shape, C_v x H_fv x W_fv; `view` maps that element
// to the caller's filter, C x H_f x W_f (filter_src_offset). Zero for k >= K or
// co >= C_o; block 0 also clears the workspace status word for this call.
__global__ void relayout_filter_f32(const float *__restrict__ filt, float *__restrict__ fT,
                                    uint32_t *status, int K, int K_pad, int C_o, int C_o_pad, int H_fv,
                                    int W_fv, int view, int C, int H_f, int W_f) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) status[0] = 0;
    const int KK = H_fv * W_fv;
    for (int k = blockIdx.y; k < K_pad; k += gridDim.y) {
        int src_k = -1;
        if (k < K) {
            const int ci = k / KK, kk = k - ci * KK;
            const int j = kk / H_fv, r = kk - j * H_fv;
            src_k = (int)filter_src_offset(view, ci, r, j, C, H_f, W_f);  // within filt[co]
        }
        for (int co = blockIdx.x * blockDim.x + threadIdx.x; co < C_o_pad; co += gridDim.x * blockDim.x)
            fT[(int64_t)k * C_o_pad + co] = (src_k >= 0 && co < C_o) ? filt[(int64_t)co * K + src_k] : 0.f;
    }
}

template <int TM, int RI, int KC, int STAGES, int MINB, bool FROM_X, bool CL = false, bool GEN = false>
cudaError_t launch_tm(const F32Params &p, int N, cudaStream_t st) {
    dim3 grid((unsigned)(p.pos_tiles * N), (unsigned)((p.C_o + TM - 1) / TM));
    constexpr size_t smem = f32_smem_bytes<TM, KC, STAGES>();
    cudaError_t e = cudaFuncSetAttribute(conv_f32_kernel<TM, RI, KC, STAGES, MINB, FROM_X, CL, GEN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    conv_f32_kernel<TM, RI, KC, STAGES, MINB, FROM_X, CL, GEN><<<grid, TM / RI * 16, smem, st>>>(p);
    return cudaGetLastError();
}

}  // namespace

// Channel tile with the least padding (ties: the larger tile).
static int choose_tm(const Shape &s) {
    int best = 128;
    int64_t best_pad = (s.C_o + 127) / 128 * 128 - s.C_o;
    for (int tm : {96, 64, 32}) {
        const int64_t pad = (s.C_o + tm - 1) / tm * tm - s.C_o;
        if (pad < best_pad) { best = tm; best_pad = pad; }
    }
    return best;
}

static int64_t k_pad(const Shape &s) {
    const int64_t K = s.C_i * s.H_f * s.W_f;
    return (K + K_ALIGN - 1) / K_ALIGN * K_ALIGN;
}

static int64_t c_o_pad(const Shape &s) {
    const int tm = choose_tm(s);
    return (s.C_o + tm - 1) / tm * tm;
}

// The filter's K (C_i*H_f*W_f) and channel padding do not depend on the layout.
size_t conv_f32_filter_bytes(const Shape &s, bool, int) {
    return round_up((size_t)(k_pad(s) * c_o_pad(s)) * 4, 256);
}

bool conv_f32_supported(const Shape &s, bool from_x, int) {
    // elements of one image of the source (the same count in either layout)
    const int64_t img = from_x ? s.C_i * s.H_i * s.W_i : s.C_i * s.H_o * padded_w(s) * s.H_f;
    const int64_t P = s.H_o * s.W_o;
    const int64_t tiles = (P + TP - 1) / TP;
    return img < (1ll << 31) && k_pad(s) < (1ll << 30) && tiles * s.N < (1ll << 31) &&
           (s.C_o + 31) / 32 < 65536 && k_pad(s) * c_o_pad(s) < (1ll << 40);
}

cudaError_t launch_conv_f32(const void *src, const void *filt, void *out, void *ws,
                            const Shape &s, bool from_x, int layout, cudaStream_t st) {
    uint32_t *status = static_cast<uint32_t *>(ws);
    float *fp = reinterpret_cast<float *>(static_cast<unsigned char *>(ws) + kStatusBytes);
    const int64_t Kp = k_pad(s), Cp = c_o_pad(s);
    const bool cl = layout == LAYOUT_NHWC;
    const bool gen = !plain(s);  // padding or dilation: the general gather, filter in NCHW window order
    // virtual filter extents and view (see the head of this file)
    const bool view_cl = cl && !gen;
    const int64_t H_fv = view_cl ? 1 : s.H_f;
    const int64_t W_fv = !view_cl ? s.W_f : from_x ? s.W_f * s.C_i : s.W_f * s.H_f * s.C_i;
    const int view = !view_cl ? VIEW_IDENT : from_x ? VIEW_CL_ROWS : VIEW_CL_WIN;
    const dim3 rgrid((unsigned)std::min<int64_t>((Cp + 127) / 128, 8), (unsigned)std::min<int64_t>(Kp, 65535));
    relayout_filter_f32<<<rgrid, 128, 0, st>>>(static_cast<const float *>(filt), fp, status,
                                               (int)(s.C_i * s.H_f * s.W_f), (int)Kp, (int)s.C_o, (int)Cp,
                                               (int)H_fv, (int)W_fv, view, (int)s.C_i, (int)s.H_f,
                                               (int)s.W_f);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || s.N == 0) return e;

    F32Params p;
    p.src = static_cast<const float *>(src);
    p.filt = fp;
    p.out = static_cast<float *>(out);
    p.status = status;
    p.C_i = (int)s.C_i;
    p.C_o = (int)s.C_o;
    p.H_o = (int)s.H_o;
    p.W_o = (int)s.W_o;
    p.H_i = (int)s.H_i;
    p.W_i = (int)s.W_i;
    p.H_f = (int)s.H_f;
    p.s_h = (int)s.s_h;
    p.s_w = (int)s.s_w;
    p.P = (int)(s.H_o * s.W_o);
    p.K = (int)(s.C_i * s.H_f * s.W_f);
    p.KK = (int)(s.H_f * s.W_f);
    p.pos_tiles = (p.P + TP - 1) / TP;
    p.L = (int)(s.W_i * s.H_f);
    p.S = (int)(s.s_w * s.H_f);
    p.img_src = from_x ? s.C_i * s.H_i * s.W_i : s.C_i * s.H_o * padded_w(s) * s.H_f;
    p.cs = (int)(s.H_o * s.W_i * s.H_f);
    p.from_win = from_x ? 0 : 1;
    p.p_h = (int)s.p_h;
    p.p_w = (int)s.p_w;
    p.d_h = (int)s.d_h;
    p.d_w = (int)s.d_w;
    p.W_f = (int)s.W_f;
    p.Lw = (int)(padded_w(s) * s.H_f);
    p.C_o_pad = (int)Cp;
    p.div_KK = make_fastdiv((uint32_t)(s.H_f * s.W_f));
    p.div_Wo = make_fastdiv((uint32_t)s.W_o);
    p.div_Hf = make_fastdiv((uint32_t)s.H_f);
    if (view_cl) {
        // the window path over the virtual shape: KK = H_fv*W_fv taps per channel
        p.KK = (int)(H_fv * W_fv);
        p.div_KK = make_fastdiv((uint32_t)p.KK);
        if (from_x) {
            p.L = (int)(s.s_h * s.W_i * s.C_i);  // output row step
            p.S = (int)(s.s_w * s.C_i);          // pixel step
            p.cs = (int)(s.W_i * s.C_i);         // filter row r = channel r
        } else {
            p.L = (int)(s.W_i * s.H_f * s.C_i);
            p.S = (int)(s.s_w * s.H_f * s.C_i);
            p.cs = (int)(s.H_o * p.L);           // one channel
        }
    }

    const int best = choose_tm(s);
    const int N = (int)s.N;
    if (gen) {  // padding or dilation: the general gather
        if (cl) {
            if (best == 128) return launch_tm<F32_CFG_128, true, true, true>(p, N, st);
            if (best == 96) return launch_tm<F32_CFG_96, true, true, true>(p, N, st);
            if (best == 64) return launch_tm<F32_CFG_64, true, true, true>(p, N, st);
            return launch_tm<F32_CFG_32, true, true, true>(p, N, st);
        }
        if (best == 128) return launch_tm<F32_CFG_128, true, false, true>(p, N, st);
        if (best == 96) return launch_tm<F32_CFG_96, true, false, true>(p, N, st);
        if (best == 64) return launch_tm<F32_CFG_64, true, false, true>(p, N, st);
        return launch_tm<F32_CFG_32, true, false, true>(p, N, st);
    }
    if (cl) {  // the window path with the channels-last epilogue
        if (best == 128) return launch_tm<F32_CFG_128, false, true>(p, N, st);
        if (best == 96) return launch_tm<F32_CFG_96, false, true>(p, N, st);
        if (best == 64) return launch_tm<F32_CFG_64, false, true>(p, N, st);
        return launch_tm<F32_CFG_32, false, true>(p, N, st);
    }
    if (from_x) {
        if (best == 128) return launch_tm<F32_CFG_128, true>(p, N, st);
        if (best == 96) return launch_tm<F32_CFG_96, true>(p, N, st);
        if (best == 64) return launch_tm<F32_CFG_64, true>(p, N, st);
        return launch_tm<F32_CFG_32, true>(p, N, st);
    }
    if (best == 128) return launch_tm<F32_CFG_128, false>(p, N, st);
    if (best == 96) return launch_tm<F32_CFG_96, false>(p, N, st);
    if (best == 64) return launch_tm<F32_CFG_64, false>(p, N, st);
    return launch_tm<F32_CFG_32, false>(p, N, st);
}

}  // namespace im2win
