// tc_util.cuh -- 5th-generation tensor core (tcgen05) helpers: tensor memory, shared-memory operand
// descriptors, MMA issue/commit, bounded mbarrier waits and tensor-memory loads.
//
// Operand tiles live in shared memory in the canonical no-swizzle "core matrix" layout: a tile of R rows
// and C columns (fp16) is split into 8 x 8 core matrices of 128 contiguous bytes, row-major inside
// (16 bytes per row); core matrix (r/8, c/8) sits at (r/8) * (C/8) * 128 + (c/8) * 128.  The same tile
// serves as an MMA operand in two ways:
//   K-major view : operand rows = tile rows, reduction = tile columns
//                  LBO = 128 (next core matrix along the reduction), SBO = (C/8) * 128
//   MN-major view: operand rows = tile columns, reduction = tile rows (the transposed matrix)
//                  LBO = (C/8) * 128, SBO = 128
// i.e. for both majors LBO is the byte stride between core matrices adjacent along the reduction
// dimension and SBO the stride along M/N.  One MMA consumes 16 reduction elements.
#pragma once

#include <stdint.h>

#include "gdr_common.cuh"

namespace gdr {
namespace tc {

__device__ __forceinline__ uint32_t tile_off(int r, int c, int C) {
    return (uint32_t)((r >> 3) * (C >> 3) * 128 + (c >> 3) * 128 + (r & 7) * 16 + (c & 7) * 2);
}

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;  // descriptor version for this architecture; no swizzle
    return d;
}

// Descriptor of reduction step kk (16 elements) of a tile used in K-major / MN-major view.
__device__ __forceinline__ uint64_t desc_k(uint32_t tile, int C, int kk) {
    return smem_desc(tile + kk * 256, 128, (C >> 3) * 128);
}
__device__ __forceinline__ uint64_t desc_mn(uint32_t tile, int C, int kk) {
    return smem_desc(tile + kk * 2 * (C >> 3) * 128, (C >> 3) * 128, 128);
}

// Instruction descriptor: fp16 A and B, fp32 accumulator, M x N, operand majors.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

// D[M x N] (+)= A[M x Kr] B[N x Kr]^T over Kr / 16 MMAs; a_mn / b_mn select the operand views.
__device__ __forceinline__ void gemm(uint32_t d_tmem, uint32_t a_tile, int a_C, bool a_mn, uint32_t b_tile, int b_C,
                                     bool b_mn, int M, int N, int Kr, bool accumulate) {
    const uint32_t id = idesc_f16(M, N, a_mn, b_mn);
    // only the start-address field changes between reduction steps (shared addresses stay below 2^18,
    // so adding the 16-byte-unit offset cannot carry out of the 14-bit field)
    const uint64_t a0 = a_mn ? desc_mn(a_tile, a_C, 0) : desc_k(a_tile, a_C, 0);
    const uint64_t b0 = b_mn ? desc_mn(b_tile, b_C, 0) : desc_k(b_tile, b_C, 0);
    const uint32_t a_step = a_mn ? 2 * (a_C >> 3) * 128 / 16 : 256 / 16;
    const uint32_t b_step = b_mn ? 2 * (b_C >> 3) * 128 / 16 : 256 / 16;
    for (int kk = 0; kk < Kr / 16; ++kk)
        mma(d_tmem, a0 + (uint64_t)(kk * a_step), b0 + (uint64_t)(kk * b_step), id,
            (accumulate || kk > 0) ? 1u : 0u);
}

// An MMA operand: its descriptor at reduction step 0, the descriptor advance per 16-element reduction step
// (in the 16-byte units of the start-address field) and whether it is read MN-major.
struct Operand {
    uint64_t desc;
    uint32_t step;
    bool mn;
};

// Operand of a row-block-major tile with C columns (core matrix (r/8, c/8) at ((r/8)(C/8) + c/8) * 128; the
// workspace tiles): as desc_k / desc_mn.
__device__ __forceinline__ Operand op_rows(uint32_t tile, int C, bool mn) {
    return mn ? Operand{desc_mn(tile, C, 0), (uint32_t)(2 * (C >> 3) * 128 / 16), true}
              : Operand{desc_k(tile, C, 0), 256u / 16u, false};
}
// Operand of a column-block-major tile with R rows (core matrix (r/8, c/8) at ((c/8)(R/8) + r/8) * 128: the
// layout a TMA box of 8-element rows lands in).  K-major view: the next core matrix along the reduction (the
// columns) is (R/8) * 128 bytes on, the next along the rows 128; MN-major view: the reduction runs along the
// rows (128 bytes per core matrix) and the operand rows along the columns ((R/8) * 128 bytes).
__device__ __forceinline__ Operand op_cols(uint32_t tile, int R, bool mn) {
    const uint32_t cb = (uint32_t)(R >> 3) * 128u;
    return mn ? Operand{smem_desc(tile, 128, cb), 256u / 16u, true} : Operand{smem_desc(tile, cb, 128), 2u * cb / 16u, false};
}

// D (+)= A B^T with A in tensor memory: M = 128 rows on the lanes, the 16-bit elements of a row packed two per
// 32-bit column (element 2m in the low half of column m), so a reduction step of 16 is 8 columns on.
__device__ __forceinline__ void mma_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void gemm_ta(uint32_t d_tmem, uint32_t a_tmem, Operand b, int N, int Kr, bool accumulate) {
    const uint32_t id = idesc_f16(128, N, false, b.mn);
    for (int kk = 0; kk < Kr / 16; ++kk)
        mma_ta(d_tmem, a_tmem + 8u * kk, b.desc + (uint64_t)(kk * b.step), id, (accumulate || kk > 0) ? 1u : 0u);
}

// D[M x N] (+)= A[M x Kr] B[N x Kr]^T for operands of either tile order.
__device__ __forceinline__ void gemm_ops(uint32_t d_tmem, Operand a, Operand b, int M, int N, int Kr, bool accumulate) {
    const uint32_t id = idesc_f16(M, N, a.mn, b.mn);
    for (int kk = 0; kk < Kr / 16; ++kk)
        mma(d_tmem, a.desc + (uint64_t)(kk * a.step), b.desc + (uint64_t)(kk * b.step), id,
            (accumulate || kk > 0) ? 1u : 0u);
}

// ---- tensor-map (TMA) loads: a 4-D box of the global tensor described by `map` (a kernel parameter) at
// the given coordinates (innermost first) into shared memory, completion counted on `bar`.
__device__ __forceinline__ void tma_load_4d(void *dst, const void *map, int x0, int x1, int x2, int x3, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
        "[%6];\n" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x0), "r"(x1), "r"(x2), "r"(x3), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void *dst, const void *map, int x0, int x1, int x2, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];\n" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x0), "r"(x1), "r"(x2), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
        smem_u32(bar)));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, int count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}

// Wait for the mbarrier phase with the given parity; gives up after `limit` polls and returns false.
// A poll is a try_wait, which the hardware may suspend for a while before it reports an incomplete phase.
// Limits below 2^16 (set only to make waits run out in tests) poll with the non-blocking test_wait
// instead, so that a short limit really is short.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t limit) {
    uint32_t done = 0;
    if (limit < (1u << 16)) {
        for (uint32_t it = 0; it < limit; ++it) {
            asm volatile(
                "{\n.reg .pred p;\nmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                : "=r"(done)
                : "r"(smem_u32(bar)), "r"(parity)
                : "memory");
            if (done) return true;
        }
        return false;
    }
    for (uint32_t it = 0; it < limit; ++it) {
        asm volatile(
            "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(smem_u32(bar)), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}

// ---- bulk (TMA engine) copies of contiguous tiles
// Arm an mbarrier phase for `bytes` of incoming bulk copies (one arrival by the calling thread).
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
// global -> shared, completion counted on `bar` (bytes and addresses multiples of 16).
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}
// shared -> global, tracked by bulk groups of the issuing thread.
__device__ __forceinline__ void bulk_s2g(void *dst, const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(dst), "r"(smem_u32(src)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
// Wait until this thread's bulk stores no longer read shared memory (sources may be overwritten).
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory"); }
// Wait until this thread's bulk stores are complete.
__device__ __forceinline__ void bulk_wait() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
// Make this thread's generic-proxy shared-memory writes visible to the tensor core (async proxy).
__device__ __forceinline__ void fence_smem_to_async() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

// Allocation by one full warp; the column base is written to *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(slot)),
                 "r"(ncols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(base), "r"(ncols));
}

// 32 consecutive columns of this warp's 32 lanes (lane quarter of the warp) -> 32 registers per thread.
__device__ __forceinline__ void ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive columns of this warp's 32 lanes -> 16 registers per thread.
__device__ __forceinline__ void ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Two 16-column loads (addresses a and b) and one wait, in one statement so that no use of the registers
// can be scheduled before the wait: the second load's latency overlaps the first's.
__device__ __forceinline__ void ld16x2(uint32_t a, float (&va)[16], uint32_t b, float (&vb)[16]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, "
        "[%33];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(a), "r"(b)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        va[i] = __uint_as_float(r[i]);
        vb[i] = __uint_as_float(r[16 + i]);
    }
}

// 32 registers per thread -> 32 consecutive columns of this warp's 32 lanes.
__device__ __forceinline__ void st32(uint32_t taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
        "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
        "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31])));
}
// 32 values of this thread's row -> 16 consecutive columns of fp16 pairs (an A operand in tensor memory).
__device__ __forceinline__ void st32_f16(uint32_t taddr, const float (&v)[32]) {
    uint32_t p[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const __half2 h = __floats2half2_rn(v[2 * m], v[2 * m + 1]);
        p[m] = *reinterpret_cast<const uint32_t *>(&h);
    }
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(
            taddr),
        "r"(p[0]), "r"(p[1]), "r"(p[2]), "r"(p[3]), "r"(p[4]), "r"(p[5]), "r"(p[6]), "r"(p[7]), "r"(p[8]), "r"(p[9]),
        "r"(p[10]), "r"(p[11]), "r"(p[12]), "r"(p[13]), "r"(p[14]), "r"(p[15]));
}
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

// Tensor-memory address of (lane quarter of this warp, column).
__device__ __forceinline__ uint32_t taddr(uint32_t base, int col) {
    return base + ((uint32_t)((threadIdx.x >> 5) & 3) * 32u << 16) + (uint32_t)col;
}

// Lane l of the warp returns the sum over the warp of v[l] (v is consumed).
__device__ __forceinline__ float warp_transpose_sum32(float (&v)[32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        const bool up = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < s; ++i) {
            float send = up ? v[i] : v[i + s];
            float keep = up ? v[i + s] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
    return v[0];
}

// Lanes l and l ^ 16 of the warp return the sum over the warp of v[l % 16] (v is consumed).
__device__ __forceinline__ float warp_transpose_sum16(float (&v)[16]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int s = 8; s >= 1; s >>= 1) {
        const bool up = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < s; ++i) {
            float send = up ? v[i] : v[i + s];
            float keep = up ? v[i + s] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 16);
}

// Lanes l and l ^ 8 return the sum over the 16 lanes of their half-warp of v[l % 8] (v is consumed).
__device__ __forceinline__ float half_transpose_sum8(float (&v)[8]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int s = 4; s >= 1; s >>= 1) {
        const bool up = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < s; ++i) {
            float send = up ? v[i] : v[i + s];
            float keep = up ? v[i + s] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 8);
}

// The rows of an M = 64 accumulator sit in lanes 0..15 of a lane quarter.  After a 16-column load, lane l
// gets in x the columns 8 (l / 16) .. +7 of row l % 16 (lanes 16..31 take the upper half from lane l - 16),
// so that all 32 lanes share the element-wise work.
__device__ __forceinline__ void split_rows16(const float (&v)[16], float (&x)[8]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const float hi = __shfl_sync(0xffffffffu, v[8 + t], lane & 15);
        x[t] = lane < 16 ? v[t] : hi;
    }
}

// Write 8 fp32 values as one 16-byte row segment of core matrix (r/8, c0/8) of a tile (c0 % 8 == 0).
__device__ __forceinline__ void st_tile8(unsigned char *tile, int r, int c0, int C, const float *x) {
    uint4 p;
    __half2 *h2 = reinterpret_cast<__half2 *>(&p);
#pragma unroll
    for (int i = 0; i < 4; ++i) h2[i] = __floats2half2_rn(x[2 * i], x[2 * i + 1]);
    *reinterpret_cast<uint4 *>(tile + tile_off(r, c0, C)) = p;
}

__device__ __forceinline__ float ld_tile(const unsigned char *tile, int r, int c, int C) {
    return __half2float(*reinterpret_cast<const __half *>(tile + tile_off(r, c, C)));
}

}  // namespace tc
}  // namespace gdr
