// PTX wrappers and small device helpers for the tcgen05 kernels (sm_103a):
// mbarriers, bulk (TMA) copies, tensor-memory allocation, tcgen05.mma /
// commit / ld, shared-memory matrix descriptors, and a bounded mbarrier wait.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "im2win_internal.cuh"

namespace im2win {
namespace tc {

constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait

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
// The same with a suspend-time hint: a thread whose phase is not complete sleeps
// in hardware until it completes or `ns` nanoseconds pass, instead of returning
// at once; polling warps then take no issue slots from the warps they share a
// scheduler with (the MMA issuers among them).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}
// TMA tensor copy of one 4-D box (tile mode) global -> shared::cta at box
// coordinates (x, y, z, w), completion counted in bytes on `bar`; elements
// outside the tensor read as zero. `tmap` is the generic address of a tensor
// map in kernel parameter space.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void *tmap, int x, int y, int z, int w,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
        : "memory");
}
// bulk copy global -> shared::cta, completion counted in bytes on `bar`
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
// cp.async 16-byte copies of this thread still in flight count towards one
// arrival on `bar` when they complete (the barrier's expected count covers it).
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Warp-wide loads and stores of four 8 x 8 matrices of 16-bit elements in
// shared memory. Lane 8q + i gives the 16-byte aligned address of row i of
// matrix q. In registers, lane t holds in r_q elements (t / 4, 2(t % 4)) (low
// half) and (t / 4, 2(t % 4) + 1) of matrix q. The transposing store writes
// matrix q's column i, as 8 consecutive elements, at the row address of lane
// 8q + i.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}
__device__ __forceinline__ void stsm_x4_trans(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(r0),
                 "r"(r1), "r"(r2), "r"(r3)
                 : "memory");
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
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld1(uint32_t taddr, uint32_t &r) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr) : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start before the previous kernel of the stream has
// finished; grid_dependency_wait() returns once that kernel has completed and
// its writes are visible (immediately when launched without the attribute).
// allow_dependents() lets the next such kernel start launching early.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void allow_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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
__host__ __device__ inline uint32_t make_idesc(bool bf16, int M, int N) {
    const uint32_t t = bf16 ? 1u : 0u;
    return (1u << 4) | (t << 7) | (t << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

enum WaitSite : uint32_t { SITE_FULL_A = 1, SITE_FULL_B, SITE_EMPTY_MMA, SITE_EMPTY_LOAD,
                           SITE_EMPTY_PROD, SITE_DONE, SITE_DRAIN, SITE_STACK, SITE_RAW };

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
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (honour_abort && *c.abort_flag) return false;
        if ((spin & 255u) == 0 && globaltimer() - t0 > kTimeoutNs) {
            *c.abort_flag = 1;
            if (atomicCAS(c.status, 0u, (uint32_t)IM2WIN_ERR_TIMEOUT) == 0u) {
                c.status[1] = site;
                c.status[2] = blockIdx.x + blockIdx.y * gridDim.x;
            }
            return false;
        }
    }
}

// The same wait for a whole warp: lane 0 polls, the others sleep in the
// warp barrier; every lane gets lane 0's result.
__device__ __forceinline__ bool warp_bar_wait(uint32_t bar, uint32_t parity, const Ctl &c, uint32_t site) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = bar_wait(bar, parity, c, site) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Named barrier `id` over `count` threads (a multiple of 32) that also returns
// whether `v` held in every one of them.
__device__ __forceinline__ bool bar_red_and(int id, int count, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.and.pred po, %2, %3, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// One fp32 value rounded to fp16 / bf16 (round to nearest even), as its bits.
__device__ __forceinline__ uint16_t cvt16(float v, int bf16) {
    return bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(v)) : __half_as_ushort(__float2half_rn(v));
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, int bf16) {
    if (bf16) {
        const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t *>(&v);
    }
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// Epilogue of one warp: drains TMEM column blocks first_blk, first_blk+step, ...
// (< nblk, 32 columns each) of the warp's 32 accumulator lanes (taddr = lane
// quarter base), rounds to fp16/bf16, transposes through the warp's shared
// staging area (32 x 17 words) and stores: lane l writes column blk*32 + l of
// rows 0..rows-1 at dst_of(blk*32 + l) + row*row_stride (dst_of returns
// nullptr for columns that are not outputs). The TMEM load of the next block
// is in flight while the current block is stored.
template <typename DstFn>
__device__ __forceinline__ void drain_accumulator(uint32_t taddr, int first_blk, int nblk, int step,
                                                  uint32_t *stage, int rows, int64_t row_stride,
                                                  int bf16, DstFn dst_of) {
    const int lane = threadIdx.x & 31;
    const uint16_t *st16 = reinterpret_cast<const uint16_t *>(stage);
    if (first_blk >= nblk) return;
    uint32_t r[32];
    int blk = first_blk;
    tmem_ld32(taddr + (uint32_t)(blk * 32), r);
    while (true) {
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i)
            stage[lane * 17 + i] = pack2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]), bf16);
        __syncwarp();
        const int next = blk + step;
        if (next < nblk) tmem_ld32(taddr + (uint32_t)(next * 32), r);
        uint16_t v[32];
#pragma unroll
        for (int row = 0; row < 32; ++row) v[row] = st16[row * 34 + lane];
        __syncwarp();
        uint16_t *d = dst_of(blk * 32 + lane);
        if (d != nullptr) {
#pragma unroll
            for (int row = 0; row < 32; ++row)
                if (row < rows) d[row * row_stride] = v[row];
        }
        if (next >= nblk) break;
        blk = next;
    }
}

// Stores one staged block of the tap kernels' drain: the warp's staging area
// holds 32 rows x 64 columns of rounded results (u16 pairs, row pitch 33
// words); lane l stores positions 2l and 2l+1 of every row. off_of(col) gives
// the output element offset of column col within a channel plane (or -1 if the
// column is not an output); row r lives at out_c + r*row_stride. When, for
// every lane, the two positions are adjacent outputs at a 4-byte aligned
// address in every row, the block is stored as 4-byte pairs; otherwise as
// 2-byte elements. Either way a lane's row loop is branch-free.
template <typename OffFn>
__device__ __forceinline__ void store_block(const uint32_t *stage, int c0, int rows, int64_t row_stride,
                                            uint16_t *out_c, OffFn off_of) {
    const int lane = threadIdx.x & 31;
    const int o0 = off_of(c0 + 2 * lane), o1 = off_of(c0 + 2 * lane + 1);
    const bool pair_ok = o0 < 0 || (o1 == o0 + 1 && (reinterpret_cast<uintptr_t>(out_c + o0) & 3) == 0);
    const bool pairs = (row_stride & 1) == 0 && __all_sync(0xffffffffu, pair_ok);
    const uint32_t *src = stage + lane;
    if (pairs) {
        if (o0 >= 0) {
            uint32_t *d = reinterpret_cast<uint32_t *>(out_c + o0);
            const int64_t st = row_stride >> 1;
            if (rows == 32) {
#pragma unroll 8
                for (int row = 0; row < 32; ++row, d += st) *d = src[row * 33];
            } else {
                for (int row = 0; row < rows; ++row, d += st) *d = src[row * 33];
            }
        }
    } else if (o0 >= 0 || o1 >= 0) {
        // a lane whose first position is not an output stores through its second
        // address for both (the store of the missing one is predicated off)
        uint16_t *d0 = out_c + (o0 >= 0 ? o0 : o1);
        uint16_t *d1 = out_c + (o1 >= 0 ? o1 : o0);
        const bool v0 = o0 >= 0, v1 = o1 >= 0;
        if (rows == 32) {
#pragma unroll 8
            for (int row = 0; row < 32; ++row, d0 += row_stride, d1 += row_stride) {
                const uint32_t w = src[row * 33];
                if (v0) *d0 = (uint16_t)(w & 0xFFFFu);
                if (v1) *d1 = (uint16_t)(w >> 16);
            }
        } else {
            for (int row = 0; row < rows; ++row, d0 += row_stride, d1 += row_stride) {
                const uint32_t w = src[row * 33];
                if (v0) *d0 = (uint16_t)(w & 0xFFFFu);
                if (v1) *d1 = (uint16_t)(w >> 16);
            }
        }
    }
}

// Channels-last staging of 32 columns (half `half` of a 64-column block): lane
// l holds channel l of columns half*32 + i in v[i]. Lane pairs swap values so
// that each lane packs two adjacent channels of one column:
//   stage[col*16 + l/2] = (channel 2(l/2), channel 2(l/2)+1) of column col,
// i.e. a column's 32 channels are 64 contiguous bytes. Every store is one
// conflict-free wavefront (32 consecutive words).
__device__ __forceinline__ void stage_half_cl(uint32_t *stage, int half, const float (&v)[32], int bf16) {
    const int lane = threadIdx.x & 31;
    const bool odd = (lane & 1) != 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float a = v[2 * i], b = v[2 * i + 1];
        const float recv = __shfl_xor_sync(0xffffffffu, odd ? a : b, 1);
        const float lo = odd ? recv : a, hi = odd ? b : recv;
        stage[(half * 32 + 2 * i + (odd ? 1 : 0)) * 16 + (lane >> 1)] = pack2(lo, hi, bf16);
    }
}

// Stores a channels-last staged block of 64 columns: column col of the block
// goes to out_c + off_of(c0 + col)*cstride (off_of < 0: not an output), its
// channels 0..rows-1 contiguous. Four lanes cover a column's 32 channels with
// 16-byte stores when cstride is a multiple of 8 (rows then is too), element
// stores otherwise.
template <typename OffFn>
__device__ __forceinline__ void store_block_cl(const uint32_t *stage, int c0, int rows, int64_t cstride,
                                               uint16_t *out_c, OffFn off_of) {
    const int lane = threadIdx.x & 31;
    const int oa = off_of(c0 + lane), ob = off_of(c0 + 32 + lane);
    const bool vec = (cstride & 7) == 0;
    const int q = lane & 3;
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int col = it * 8 + (lane >> 2);
        const int o = __shfl_sync(0xffffffffu, it < 4 ? oa : ob, col & 31);
        if (o < 0 || q * 8 >= rows) continue;
        const uint4 val = *reinterpret_cast<const uint4 *>(stage + col * 16 + q * 4);
        uint16_t *d = out_c + (int64_t)o * cstride + q * 8;
        if (vec) {
            *reinterpret_cast<uint4 *>(d) = val;
        } else {
            const uint32_t w[4] = {val.x, val.y, val.z, val.w};
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (q * 8 + e < rows) d[e] = (uint16_t)(w[e >> 1] >> (16 * (e & 1)));
        }
    }
}

// Stages TMEM columns [c_begin, c_end) of the warp's 32 accumulator lanes (at
// most two 64-column blocks) into consecutive staging blocks of block_words
// words each, rounded to fp16/bf16, in the layout store_block (NCHW) or
// store_block_cl (CL) reads. The caller releases the accumulator afterwards and
// stores the blocks from shared memory.
template <bool CL>
__device__ __forceinline__ void stage_columns(uint32_t taddr, int c_begin, int c_end, uint32_t *stage,
                                              int block_words, int bf16) {
    const int lane = threadIdx.x & 31;
    if (c_begin >= c_end) return;
    uint32_t r[32];
    tmem_ld32(taddr + (uint32_t)c_begin, r);
    for (int c0 = c_begin, bi = 0; c0 < c_end; c0 += 64, ++bi) {
        uint32_t *blk = stage + bi * block_words;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            tmem_wait_ld();
            if (CL) {
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
                stage_half_cl(blk, half, v, bf16);
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    blk[lane * 33 + half * 16 + i] =
                        pack2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]), bf16);
            }
            const int nxt = half == 0 ? c0 + 32 : c0 + 64;
            if (nxt < c_end) tmem_ld32(taddr + (uint32_t)nxt, r);
        }
    }
    __syncwarp();
}

// Channels-last store of 32 columns straight from registers: lane l holds
// channel l of columns c0 + i in v[i] (fp32 bit patterns). Lane pairs swap values with one shuffle
// per two columns, so that the even lane of a pair holds channels (l, l+1) of
// column c0 + 2i and the odd lane the same channels of column c0 + 2i + 1; each
// store instruction then writes the warp's 32 channels of two columns as two
// runs of 64 contiguous bytes. off_of(col) < 0: not an output; rows: channels
// of the warp that exist; cstride: elements between positions (C_o). 4-byte
// stores when cstride is even, else 2-byte.
template <typename OffFn>
__device__ __forceinline__ void store_half_cl(const uint32_t (&v)[32], int c0, int rows, int64_t cstride,
                                              uint16_t *out_c, OffFn off_of, int bf16) {
    const int lane = threadIdx.x & 31;
    const bool odd = (lane & 1) != 0;
    const int ch = lane & ~1;  // first channel of the lane's pair
    const int o_mine = off_of(c0 + lane);
    const bool pairs = (cstride & 1) == 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float a = __uint_as_float(v[2 * i]), b = __uint_as_float(v[2 * i + 1]);
        const float recv = __shfl_xor_sync(0xffffffffu, odd ? a : b, 1);
        const float lo = odd ? recv : a, hi = odd ? b : recv;
        const int o = __shfl_sync(0xffffffffu, o_mine, 2 * i + (odd ? 1 : 0));
        if (o < 0 || ch >= rows) continue;
        uint16_t *d = out_c + (int64_t)o * cstride + ch;
        const uint32_t w = pack2(lo, hi, bf16);
        if (pairs && ch + 1 < rows) {
            *reinterpret_cast<uint32_t *>(d) = w;
        } else {
            d[0] = (uint16_t)(w & 0xFFFFu);
            if (ch + 1 < rows) d[1] = (uint16_t)(w >> 16);
        }
    }
}

// Faster drain for the tap kernels. The warp owns TMEM columns [c_begin,
// c_end) of its 32 accumulator lanes (taddr = lane quarter base). Per block of
// 64 columns: two 32-column TMEM loads (the next block's first load is in
// flight while this block is stored), rounding to fp16/bf16, a transpose
// through the warp's staging area (32 rows x 33 words), then store_block.
// The last block may reach past c_end: off_of must return -1 for its columns
// that are not the warp's to store. CL: channels-last output (stage_half_cl,
// store_block_cl; row_stride is then the stride between positions).
template <bool CL, typename OffFn>
__device__ __forceinline__ void drain_columns(uint32_t taddr, int c_begin, int c_end, uint32_t *stage,
                                              int rows, int64_t row_stride, int bf16,
                                              uint16_t *out_c, OffFn off_of) {
    const int lane = threadIdx.x & 31;
    if (c_begin >= c_end) return;
    uint32_t r[32];
    tmem_ld32(taddr + (uint32_t)c_begin, r);
    for (int c0 = c_begin; c0 < c_end; c0 += 64) {
        // ---- columns c0..c0+31, then c0+32..c0+63 into the staging area (u16 [32][66])
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            tmem_wait_ld();
            if (CL) {
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
                stage_half_cl(stage, half, v, bf16);
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    stage[lane * 33 + half * 16 + i] =
                        pack2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]), bf16);
            }
            const int nxt = half == 0 ? c0 + 32 : c0 + 64;
            if (nxt < c_end) tmem_ld32(taddr + (uint32_t)nxt, r);
        }
        __syncwarp();
        if (CL)
            store_block_cl(stage, c0, rows, row_stride, out_c, off_of);
        else
            store_block(stage, c0, rows, row_stride, out_c, off_of);
        __syncwarp();
    }
}

// Stacked drain, lower half: the warp reads accumulator rows 64..95 or 96..127
// (the second tap of each stacked group) and hands, per 32-column half block
// starting at column c, the fp32 values of columns c+1 .. c+32 to its partner
// through xbuf (32 rows x 33 words). Hand-over number k (counted over the whole
// kernel in *k, identically by both warps) completes phase k of bar_full; xbuf
// is reused once phase k-1 of bar_empty has completed. Each side signals with
// one arrival by lane 0 after a warp barrier, which orders every lane's shared
// memory accesses before it (one arrival measured faster than 32). Waits are
// bounded; false means the CTA aborted.
__device__ __forceinline__ bool drain_stacked_lower(uint32_t taddr, int c_begin, int c_end, float *xbuf,
                                                    uint32_t bar_full, uint32_t bar_empty, uint32_t *k,
                                                    const Ctl &ctl, uint32_t site) {
    const int lane = threadIdx.x & 31;
    for (int c0 = c_begin; c0 < c_end; c0 += 64) {
        for (int half = 0; half < 2; ++half, ++*k) {
            const int cc = c0 + 32 * half;
            uint32_t r[32], extra;
            tmem_ld32(taddr + (uint32_t)cc, r);
            tmem_ld1(taddr + (uint32_t)(cc + 32), extra);
            tmem_wait_ld();
            if (*k > 0 && !warp_bar_wait(bar_empty, (*k - 1) & 1, ctl, site)) return false;
#pragma unroll
            for (int i = 0; i < 31; ++i) xbuf[lane * 33 + i] = __uint_as_float(r[i + 1]);
            xbuf[lane * 33 + 31] = __uint_as_float(extra);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_full);
        }
    }
    return true;
}

// Stacked drain, upper half: accumulator rows 0..63 plus the partner's shifted
// values give the outputs; rounding, transpose and store as in drain_columns,
// except that channels-last outputs are stored from registers (store_half_cl),
// which measured faster here than staging them.
template <bool CL, typename OffFn>
__device__ __forceinline__ bool drain_stacked_upper(uint32_t taddr, int c_begin, int c_end, uint32_t *stage,
                                                    const float *xbuf, uint32_t bar_full, uint32_t bar_empty,
                                                    uint32_t *k, const Ctl &ctl, uint32_t site, int rows,
                                                    int64_t row_stride, int bf16, uint16_t *out_c, OffFn off_of) {
    const int lane = threadIdx.x & 31;
    for (int c0 = c_begin; c0 < c_end; c0 += 64) {
#pragma unroll
        for (int half = 0; half < 2; ++half, ++*k) {
            uint32_t r[32];
            tmem_ld32(taddr + (uint32_t)(c0 + 32 * half), r);
            tmem_wait_ld();
            if (!warp_bar_wait(bar_full, *k & 1, ctl, site)) return false;
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) + xbuf[lane * 33 + i]);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty);  // the partner's buffer is read
            if (CL) {
                store_half_cl(r, c0 + 32 * half, rows, row_stride, out_c, off_of, bf16);
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    stage[lane * 33 + half * 16 + i] =
                        pack2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]), bf16);
            }
        }
        if (!CL) {
            __syncwarp();
            store_block(stage, c0, rows, row_stride, out_c, off_of);
            __syncwarp();
        }
    }
    return true;
}

}  // namespace tc
}  // namespace im2win
