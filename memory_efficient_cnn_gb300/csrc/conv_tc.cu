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

namespace im2win {
namespace {

// ------------------------------------------------------------------ PTX
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
        "r"(bytes)
        : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// bulk copy global -> shared::cta, completion counted in bytes on `bar`
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16, one CTA
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive on `bar` once every tcgen05 operation issued so far by this thread is done
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05): start address, leading- and
// stride-dimension byte offsets (all >> 4), fixed version bits 46..48 = 1,
// base offset 0, no swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) |
           ((uint64_t)(sbo >> 4) << 32) | (1ull << 46);
}

// Instruction descriptor, kind::f16: fp32 accumulator, A/B fp16 (0) or bf16
// (1), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
inline uint32_t make_idesc(bool bf16, int M, int N) {
    const uint32_t t = bf16 ? 1u : 0u;
    return (1u << 4) | (t << 7) | (t << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

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
constexpr uint64_t kTimeoutNs = 2000000000ull;
static_assert(PROD_WARPS * 32 == NT, "one producer thread per pixel");

enum WaitSite : uint32_t { SITE_FULL_A = 1, SITE_FULL_B, SITE_EMPTY_MMA, SITE_EMPTY_LOAD,
                           SITE_EMPTY_PROD, SITE_DONE, SITE_DRAIN };

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

struct Ctl {
    volatile int *abort_flag;
    uint32_t *status;
};

// Bounded wait: true when the phase of parity `parity` of `bar` completed;
// false when the CTA aborted or the wait gave up (which records the timeout).
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, const Ctl &c, uint32_t site,
                                         bool honour_abort = true) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t spin = 1;; ++spin) {
        if (mbar_try_wait(bar, parity)) return true;
        if (honour_abort && *c.abort_flag) return false;
        if ((spin & 63u) == 0) {
            if (honour_abort && *reinterpret_cast<volatile uint32_t *>(c.status) != 0) {
                *c.abort_flag = 1;
                return false;
            }
            if (globaltimer() - t0 > kTimeoutNs) {
                *c.abort_flag = 1;
                if (atomicCAS(c.status, 0u, (uint32_t)IM2WIN_ERR_TIMEOUT) == 0u) {
                    c.status[1] = site;
                    c.status[2] = blockIdx.x + blockIdx.y * gridDim.x;
                }
                return false;
            }
        }
    }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, int bf16) {
    uint16_t a, b;
    if (bf16) {
        a = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
        b = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    } else {
        a = __half_as_ushort(__float2half_rn(lo));
        b = __half_as_ushort(__float2half_rn(hi));
    }
    return (uint32_t)a | ((uint32_t)b << 16);
}

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

size_t conv_tc_filter_bytes(const Shape &s, bool /*fused*/) {
    const ExpandGeom g = expand_geom(s);
    return round_up((size_t)g.mtiles * BM * (size_t)g.K_pad * 2, 256);
}

bool conv_tc_supported(const Shape &s, bool fused) {
    const int64_t img = fused ? s.C_i * s.H_i * s.W_i : s.C_i * s.H_o * s.W_i * s.H_f;
    const int64_t KKP = (s.H_f * s.W_f + 7) / 8 * 8;
    const int64_t P = s.H_o * s.W_o;
    const int64_t pos_tiles = (P + NT - 1) / NT;
    return img < (1ll << 31) && s.C_i * KKP < (1ll << 30) && P < (1ll << 31) &&
           pos_tiles * s.N < (1ll << 31) && (s.C_o + BM - 1) / BM < 65536;
}

cudaError_t launch_conv_tc(const void *src, const void *filt, void *out, void *ws, const Shape &s,
                           bool fused, bool bf16, cudaStream_t st) {
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
