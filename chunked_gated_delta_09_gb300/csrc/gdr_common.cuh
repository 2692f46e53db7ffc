// gdr_common.cuh -- device-side building blocks shared by the backward kernels.
//
// Tile geometry: every chunk is handled as a CT x DT tile (CT = 64 tokens, DT = 128 features).  A chunk
// shorter than CT (the ragged tail of a sequence, or BT < 64) and K or V smaller than DT are zero-padded;
// the padding is exact for this recurrence (a zero key row adds nothing to any state, a zero feature
// column stays zero), so one tile shape serves every size the API accepts.
//
// Arithmetic: tensor-core operands are fp16 with fp32 accumulation; the states, gate math, cumulative
// sums and every reduction stay in fp32.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace gdr {

constexpr int CT = 64;        // tokens per chunk tile
constexpr int DT = 128;       // features per tile (K and V padded to this)
constexpr int PADH = 8;       // fp16 row padding in shared memory (keeps ldmatrix rows on distinct banks)
constexpr int LDD = DT + PADH;  // pitch (halves) of a [*][DT] shared tile
constexpr int LDC = CT + PADH;  // pitch (halves) of a [*][CT] shared tile

// Device status bits (OR-ed into the workspace status word).
constexpr int ST_BAD_SEQLENS = 1;
constexpr int ST_TIMEOUT = 2;
constexpr int ST_RANGE = 4;  // an input value does not fit the fp16 tensor-core operands (|x| > 65504, inf, nan)

// Bounded waits.  A wait that gives up after its plan's poll limit (Params::spin) flags ST_TIMEOUT; before
// the CTA moves on it waits once more, up to DRAIN_LIMIT polls, for every copy or tensor-core operation that
// is still tracked by an armed barrier phase, so that nothing lands in shared or tensor memory after the
// CTA has released it.
constexpr uint32_t WAIT_LIMIT_DEFAULT = 1u << 24;
constexpr uint32_t DRAIN_LIMIT = 1u << 24;
constexpr float F16_MAX = 65504.f;

enum DType { F32 = 0, BF16 = 1, F16 = 2 };

// Everything a kernel needs, passed by value.
struct Params {
    // sizes
    int B, T, Hk, Hv, K, V, BT, G, N, per_channel, dense, max_chunks, nts;  // nts: chunks per dense seq
    float scale;
    int qkv_dtype, beta_dtype, dqdk_dtype, dv_dtype;
    uint32_t spin;  // polls of a bounded mbarrier wait before it is declared lost
    // inputs
    const void *q, *k, *v, *beta, *dO;
    const float *g, *h0, *dht;
    const int32_t *cu;
    // outputs (backward)
    void *dq, *dk, *dv;
    float *dbeta, *dg, *dh0;
    // outputs (forward): o [T][Hv][V] in qkv dtype, final state ht [N][Hv][V][K] fp32 (may be null)
    void *o;
    float *ht;
    // output of the WY-gradient stage taken alone: dA [T][Hv][BT] fp32 (gradient with respect to A_kk)
    float *dA_out;
    // workspace
    int *status;
    int32_t *chunk_idx;  // [max_chunks][2]
    int32_t *chunk_off;  // [N + 1]
    // Per chunk x value head unit u = n Hv + hv.  fp16 matrices are stored as core-matrix tiles
    // ("tile [R][C]": see ctile_off), each moved whole by bulk copies.
    float *gam;          // [u][CT] or [u][CT][DT]  chunk-local cumulative gate (fp32)
    float *sc;           // [u][4][CT] scalar gate, backward: beta, exp(gamma), exp(gamma_C - gamma), gamma
    __half *Tm;          // tile [r][i]   64 x 64    (I + A_kk)^-1
    __half *Aqk;         // tile [r][j]   64 x 64    M (.) Q K^T (causal, decayed, unscaled)
    __half *Kd;          // tile [i][j]   64 x 64    per-channel gate: sum_k k_i k_j exp(gamma_i - gamma_j), j < i
    __half *W, *U;       // W tile [c][k] 64 x 128; U^T tile [v][c] 128 x 64
    __half *Kt;          // tile [c][k]   64 x 128   K (.) exp(gamma_C - gamma)
    __half *Qg;          // tile [r][k]   64 x 128   Q (.) exp(gamma)
    __half *Dt;          // tile [r][v]   64 x 128   scale * dO
    __half *h, *dh;      // tile [v][k]   128 x 128  state entering / adjoint leaving the chunk
    __half *Vn;          // tile [v][c]   128 x 64   V_new^T
    __half *dVn;         // tile [v][c]   128 x 64   -dV_new^T
    float *dgam;         // [u][CT] or [u][CT][DT]
    float *dq_h, *dk_h;  // [T][Hv][K] per value head (GQA with the mma.sync gradient kernel; else null), in
                         // gqa_part_dtype (workspace sized for fp32)
    // segment-parallel scans: NS segments of Lseg chunks per sequence; per (sequence, head, segment)
    // fp32 [DT][DT] summaries: local end state E, transition product Phi (and its transpose), local
    // start gradient F,
    // exact entry state Sin and exact exit gradient dS
    int NS, Lseg;
    float *segE, *segPhi, *segPhiT, *segF, *segSin, *segdS;
    // factored state-gradient local pass (null: unfactored): QR = Q~ - Aqk W per unit, tile [r][k], in the
    // U^T region (dead once the forward scan has run)
    __half *QR;
};

// Element type of the per-value-head dq / dk partials that the GQA reduction sums: the output's own type
// (fp32 outputs keep fp32 partials; 16-bit outputs take 16-bit partials, half the bytes to write and read).
__device__ __forceinline__ int gqa_part_dtype(const Params &P) { return P.dqdk_dtype; }
__device__ __forceinline__ char *gqa_part(float *base, size_t elem, const Params &P) {
    return reinterpret_cast<char *>(base) + elem * (P.dqdk_dtype == F32 ? 4 : 2);
}

// ---------------------------------------------------------------- sequence / chunk bookkeeping
struct ChunkInfo {
    int s, c, tok0, len;
};

__device__ __forceinline__ void seq_range(const Params &P, int s, int &bos, int &eos) {
    if (P.dense) {
        bos = s * P.T;
        eos = bos + P.T;
    } else {
        bos = P.cu[s];
        eos = P.cu[s + 1];
    }
}

// Chunk n of the global, sequence-major list.  Returns false for entries past the total.
__device__ __forceinline__ bool chunk_info(const Params &P, int n, ChunkInfo &ci) {
    int s, c;
    if (P.dense) {
        s = n / P.nts;
        c = n - s * P.nts;
        if (s >= P.N) return false;
    } else {
        s = P.chunk_idx[2 * n];
        c = P.chunk_idx[2 * n + 1];
        if (s < 0) return false;
    }
    int bos, eos;
    seq_range(P, s, bos, eos);
    ci.s = s;
    ci.c = c;
    ci.tok0 = bos + c * P.BT;
    int len = eos - ci.tok0;
    ci.len = len < P.BT ? len : P.BT;
    return ci.len > 0;
}

__device__ __forceinline__ int seq_chunk_base(const Params &P, int s) {
    return P.dense ? s * P.nts : P.chunk_off[s];
}

// ---------------------------------------------------------------- element conversion
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }

// Load 8 consecutive elements (16- or 32-byte aligned) as floats.
__device__ __forceinline__ void load8(const float *p, float (&o)[8]) {
    float4 a = *reinterpret_cast<const float4 *>(p);
    float4 b = *reinterpret_cast<const float4 *>(p + 4);
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
    o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&o)[8]) {
    uint4 r = *reinterpret_cast<const uint4 *>(p);
    const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __bfloat1622float2(h2[i]);
        o[2 * i] = f.x;
        o[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void load8(const __half *p, float (&o)[8]) {
    uint4 r = *reinterpret_cast<const uint4 *>(p);
    const __half2 *h2 = reinterpret_cast<const __half2 *>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __half22float2(h2[i]);
        o[2 * i] = f.x;
        o[2 * i + 1] = f.y;
    }
}

__device__ __forceinline__ uint4 pack8_half(const float (&x)[8]) {
    uint4 r;
    __half2 *h2 = reinterpret_cast<__half2 *>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) h2[i] = __floats2half2_rn(x[2 * i], x[2 * i + 1]);
    return r;
}

// Whether any of the 8 values cannot be an fp16 operand (|x| > 65504, inf or nan).
__device__ __forceinline__ bool out_of_f16(const float (&x)[8]) {
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 8; ++i) bad |= !(fabsf(x[i]) <= F16_MAX);
    return bad;
}

template <typename To> __device__ __forceinline__ To to_out_t(float x);
template <> __device__ __forceinline__ float to_out_t<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 to_out_t<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <> __device__ __forceinline__ __half to_out_t<__half>(float x) { return __float2half_rn(x); }

__device__ __forceinline__ float load_scalar(const void *p, size_t i, int dt) {
    if (dt == F32) return reinterpret_cast<const float *>(p)[i];
    if (dt == BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[i]);
    return __half2float(reinterpret_cast<const __half *>(p)[i]);
}

__device__ __forceinline__ void store_scalar(void *p, size_t i, float x, int dt) {
    if (dt == F32) reinterpret_cast<float *>(p)[i] = x;
    else if (dt == BF16) reinterpret_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(x);
    else reinterpret_cast<__half *>(p)[i] = __float2half_rn(x);
}

// Stage a [rows][ncols] block of a strided input (row r at src + r * stride) into a shared fp16 tile
// [CT][LDD], multiplying row r by rowmul (nullable).  Rows >= rows and columns >= ncols become zero.
// ncols must be a multiple of 8 or the full row is loaded element-wise.
template <typename Tin>
__device__ __forceinline__ void stage_rows_f16(__half *dst, const Tin *src, size_t stride, int rows, int ncols,
                                               const float *rowmul, float mul, int tid, int nthr) {
    for (int e = tid; e < CT * (DT / 8); e += nthr) {
        int r = e / (DT / 8), c8 = (e % (DT / 8)) * 8;
        float x[8];
        if (r < rows && c8 + 8 <= ncols) {
            load8(src + (size_t)r * stride + c8, x);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                x[j] = (r < rows && c8 + j < ncols) ? to_f32(src[(size_t)r * stride + c8 + j]) : 0.f;
        }
        float m = mul * (rowmul ? rowmul[r] : 1.f);
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] *= m;
        *reinterpret_cast<uint4 *>(dst + r * LDD + c8) = pack8_half(x);
    }
}

// ---------------------------------------------------------------- tensor-core fragments (mma.sync)
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n"
                 : "=r"(r[0]), "=r"(r[1])
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t (&r)[2], const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];\n"
                 : "=r"(r[0]), "=r"(r[1])
                 : "r"(smem_u32(p)));
}

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// m16n8k8: c (16 x 8, fp32) += A (16 x 8, fp16: a0 rows lane/4, a1 rows lane/4 + 8) B (8 x 8, fp16).
__device__ __forceinline__ void mma1688(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(b0));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// One warp accumulates a (16*MT) x (8*NT) tile: acc += A[m0.., 0:kdim] * B[0:kdim, n0..].
//   AT = false: A(m, k) = A[m * lda + k]  (row-major M x K)
//   AT = true : A(m, k) = A[k * lda + m]  (stored transposed, K x M)
//   BT = false: B(k, n) = B[k * ldb + n]  (row-major K x N)
//   BT = true : B(k, n) = B[n * ldb + k]  (stored transposed, N x K)
// kdim is a multiple of 16.
template <int MT, int NT, bool AT, bool BT>
__device__ __forceinline__ void warp_mma(float (&acc)[MT][NT][4], const __half *A, int lda, const __half *B, int ldb,
                                         int m0, int n0, int kdim) {
    const int lane = threadIdx.x & 31;
    const int r8 = lane & 7, mat = lane >> 3;
    for (int k0 = 0; k0 < kdim; k0 += 16) {
        uint32_t a[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            int mb = m0 + mt * 16;
            if (!AT) {
                const __half *p = A + (size_t)(mb + (lane & 15)) * lda + k0 + (lane >> 4) * 8;
                ldsm_x4(a[mt], p);
            } else {
                const __half *p = A + (size_t)(k0 + r8 + (mat >> 1) * 8) * lda + mb + (mat & 1) * 8;
                ldsm_x4_t(a[mt], p);
            }
        }
#pragma unroll
        for (int nt = 0; nt + 1 < NT; nt += 2) {
            int nb = n0 + nt * 8;
            uint32_t b[4];
            if (BT) {
                const __half *p = B + (size_t)(nb + r8 + (mat >> 1) * 8) * ldb + k0 + (mat & 1) * 8;
                ldsm_x4(b, p);
            } else {
                const __half *p = B + (size_t)(k0 + r8 + (mat & 1) * 8) * ldb + nb + (mat >> 1) * 8;
                ldsm_x4_t(b, p);
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                mma16816(acc[mt][nt], a[mt], b[0], b[1]);
                mma16816(acc[mt][nt + 1], a[mt], b[2], b[3]);
            }
        }
        if (NT & 1) {
            constexpr int nt = NT - 1;
            int nb = n0 + nt * 8;
            int m2 = (lane >> 3) & 1;
            uint32_t b[2];
            if (BT) {
                const __half *p = B + (size_t)(nb + r8) * ldb + k0 + m2 * 8;
                ldsm_x2(b, p);
            } else {
                const __half *p = B + (size_t)(k0 + r8 + m2 * 8) * ldb + nb;
                ldsm_x2_t(b, p);
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) mma16816(acc[mt][nt], a[mt], b[0], b[1]);
        }
    }
}

// Byte offset of element (r, c) in a core-matrix tile with C columns: 8 x 8 blocks of 128 contiguous
// bytes, block (r/8, c/8) at (r/8) (C/8) 128 + (c/8) 128 (the layout the tensor-core descriptors read).
__device__ __forceinline__ uint32_t ctile_off(int r, int c, int C) {
    return (uint32_t)((r >> 3) * (C >> 3) * 128 + (c >> 3) * 128 + (r & 7) * 16 + (c & 7) * 2);
}
// Byte offset of element (r, c) in a column-block-major core-matrix tile with R rows: block (r/8, c/8) at
// ((c/8) (R/8) + r/8) 128 (the layout a tensor-map box of 8-element rows lands in).
__device__ __forceinline__ uint32_t cbtile_off(int r, int c, int R) {
    return (uint32_t)((c >> 3) * (R >> 3) * 128 + (r >> 3) * 128 + (r & 7) * 16 + (c & 7) * 2);
}
// Byte offset of element (r, c) in a 64-row tile of 128-byte-swizzled halves (the layout of two 64-column
// tensor-map boxes with the 128-byte swizzle, on a 1024-byte-aligned base): columns 64 h .. 64 h + 63 in half h
// (64 rows of 128 bytes each), the 16-byte chunk j of row r at position j ^ (r % 8).
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
    return (uint32_t)((c >> 6) * (CT * 128) + r * 128 + ((((c >> 3) & 7) ^ (r & 7)) << 4) + (c & 7) * 2);
}
// Tile layouts: TL_ROWB row-block-major core-matrix tile (D its column count), TL_COLB column-block-major (D its
// row count), TL_SW128 the swizzled halves above (D unused).
constexpr int TL_ROWB = 0, TL_COLB = 1, TL_SW128 = 2;
template <int L> __device__ __forceinline__ uint32_t tile_at(int r, int c, int D) {
    return L == TL_SW128 ? sw128_off(r, c) : L == TL_COLB ? cbtile_off(r, c, D) : ctile_off(r, c, D);
}
__device__ __forceinline__ float ctile_get(const unsigned char *t, int r, int c, int C) {
    return __half2float(*reinterpret_cast<const __half *>(t + ctile_off(r, c, C)));
}
__device__ __forceinline__ void ctile_set(unsigned char *t, int r, int c, int C, float x) {
    *reinterpret_cast<__half *>(t + ctile_off(r, c, C)) = __float2half_rn(x);
}

// m16n8k16 with bf16 operands (BF) or fp16 operands, fp32 accumulators
template <bool BF>
__device__ __forceinline__ void mma16816t(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    if constexpr (BF)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};\n"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    else
        mma16816(c, a, b0, b1);
}

// warp_mma on core-matrix tiles (each 8 x 8 ldmatrix block is one contiguous core matrix):
//   A(m, k) = tile element (m, k) (AT = false) or (k, m) (AT = true);
//   B(k, n) = tile element (k, n) (BT = false) or (n, k) (BT = true);
// AL / BL: the tiles' layouts (TL_*; A_D / B_D as tile_at takes them); BF: both tiles hold bf16 rather than fp16.
template <int MT, int NT, bool AT, bool BT, int AL = TL_ROWB, int BL = TL_ROWB, bool BF = false>
__device__ __forceinline__ void warp_mma_ct(float (&acc)[MT][NT][4], const unsigned char *A, int A_D,
                                            const unsigned char *B, int B_D, int m0, int n0, int kdim) {
    const int lane = threadIdx.x & 31;
    const int r8 = lane & 7, mat = lane >> 3;
    for (int k0 = 0; k0 < kdim; k0 += 16) {
        uint32_t a[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            int mb = m0 + mt * 16;
            if (!AT) ldsm_x4(a[mt], A + tile_at<AL>(mb + (lane & 15), k0 + (lane >> 4) * 8, A_D));
            else ldsm_x4_t(a[mt], A + tile_at<AL>(k0 + r8 + (mat >> 1) * 8, mb + (mat & 1) * 8, A_D));
        }
#pragma unroll
        for (int nt = 0; nt + 1 < NT; nt += 2) {
            int nb = n0 + nt * 8;
            uint32_t b[4];
            if (BT) ldsm_x4(b, B + tile_at<BL>(nb + r8 + (mat >> 1) * 8, k0 + (mat & 1) * 8, B_D));
            else ldsm_x4_t(b, B + tile_at<BL>(k0 + r8 + (mat & 1) * 8, nb + (mat >> 1) * 8, B_D));
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                mma16816t<BF>(acc[mt][nt], a[mt], b[0], b[1]);
                mma16816t<BF>(acc[mt][nt + 1], a[mt], b[2], b[3]);
            }
        }
        if (NT & 1) {
            constexpr int nt = NT - 1;
            int nb = n0 + nt * 8;
            int m2 = (lane >> 3) & 1;
            uint32_t b[2];
            if (BT) ldsm_x2(b, B + tile_at<BL>(nb + r8, k0 + m2 * 8, B_D));
            else ldsm_x2_t(b, B + tile_at<BL>(k0 + r8 + m2 * 8, nb, B_D));
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) mma16816t<BF>(acc[mt][nt], a[mt], b[0], b[1]);
        }
    }
}

// Convert two strided [rows][cols] input blocks into fp16 [CT][DT] core-matrix tiles (rows >= nrows or
// columns >= ncols become zero), multiplying by m0 / m1, with every global load of the thread issued
// before the first conversion.  Work item `it` of warp w covers rows 8 (it / 4) .. +7 and 16-byte
// columns 4 (it % 4) .. +3: the 8 lanes of each 16-byte store phase write the 8 rows of one core matrix
// (distinct banks), and each row reads 64 contiguous bytes from global memory.
// Eight consecutive input elements as loaded (16 bytes for 16-bit types, 32 for fp32), converted later.
template <typename Tin> struct Raw8 { uint4 v; };
template <> struct Raw8<float> { float4 a, b; };
__device__ __forceinline__ void raw_load(Raw8<float> &x, const float *p) {
    x.a = *reinterpret_cast<const float4 *>(p);
    x.b = *reinterpret_cast<const float4 *>(p + 4);
}
template <typename Tin> __device__ __forceinline__ void raw_load(Raw8<Tin> &x, const Tin *p) {
    x.v = *reinterpret_cast<const uint4 *>(p);
}
__device__ __forceinline__ void raw_zero(Raw8<float> &x) { x.a = x.b = make_float4(0.f, 0.f, 0.f, 0.f); }
template <typename Tin> __device__ __forceinline__ void raw_zero(Raw8<Tin> &x) { x.v = make_uint4(0u, 0u, 0u, 0u); }
__device__ __forceinline__ void raw_get(const Raw8<float> &x, float (&o)[8]) {
    o[0] = x.a.x; o[1] = x.a.y; o[2] = x.a.z; o[3] = x.a.w;
    o[4] = x.b.x; o[5] = x.b.y; o[6] = x.b.z; o[7] = x.b.w;
}
__device__ __forceinline__ void raw_get(const Raw8<__nv_bfloat16> &x, float (&o)[8]) {
    const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&x.v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __bfloat1622float2(h2[i]);
        o[2 * i] = f.x;
        o[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void raw_get(const Raw8<__half> &x, float (&o)[8]) {
    const __half2 *h2 = reinterpret_cast<const __half2 *>(&x.v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __half22float2(h2[i]);
        o[2 * i] = f.x;
        o[2 * i + 1] = f.y;
    }
}

// Stage NW row-major [rows x cols] inputs, each times its multiplier, as fp16 core-matrix tiles (CT x DT,
// zero padded) in shared or global memory.  Every global load of all NW tiles is issued before the first
// conversion (one memory round trip, not NW).
// A non-null range_status gets ST_RANGE when a converted value does not fit fp16.
template <typename Tin, int NTHR, int NW>
__device__ __forceinline__ void stage_ct_n(unsigned char *const (&t)[NW], const Tin *const (&src)[NW],
                                           const size_t (&st)[NW], const int (&nc)[NW], const float (&mul)[NW],
                                           int nrows, int tid, int *range_status = nullptr) {
    constexpr int PER = CT * (DT / 8) / NTHR;
    static_assert(PER * NTHR == CT * (DT / 8), "thread count must divide the tile");
    const int wid = tid >> 5, lane = tid & 31;
    Raw8<Tin> x[NW][PER];
    bool bad = false;
#pragma unroll
    for (int w = 0; w < NW; ++w)
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            int it = wid + (NTHR / 32) * i;
            int r = 8 * (it >> 2) + (lane & 7), c8 = 8 * (4 * (it & 3) + (lane >> 3));
            if (r < nrows && c8 + 8 <= nc[w]) raw_load(x[w][i], src[w] + (size_t)r * st[w] + c8);
            else raw_zero(x[w][i]);
        }
#pragma unroll
    for (int w = 0; w < NW; ++w)
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            int it = wid + (NTHR / 32) * i;
            int r = 8 * (it >> 2) + (lane & 7), c8 = 8 * (4 * (it & 3) + (lane >> 3));
            float f[8];
            raw_get(x[w][i], f);
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] *= mul[w];
            bad |= out_of_f16(f);
            *reinterpret_cast<uint4 *>(t[w] + ctile_off(r, c8, DT)) = pack8_half(f);
        }
    if (bad && range_status) atomicOr(range_status, ST_RANGE);
}



// Store two adjacent values (columns c, c+1) of an output row in the output dtype.
__device__ __forceinline__ void store_pair(void *p, size_t i, float a, float b, int dt) {
    if (dt == F32) *reinterpret_cast<float2 *>(reinterpret_cast<float *>(p) + i) = make_float2(a, b);
    else if (dt == BF16)
        *reinterpret_cast<__nv_bfloat162 *>(reinterpret_cast<__nv_bfloat16 *>(p) + i) = __floats2bfloat162_rn(a, b);
    else *reinterpret_cast<__half2 *>(reinterpret_cast<__half *>(p) + i) = __floats2half2_rn(a, b);
}

template <int MT, int NT>
__device__ __forceinline__ void zero_acc(float (&acc)[MT][NT][4]) {
#pragma unroll
    for (int i = 0; i < MT; ++i)
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[i][j][e] = 0.f;
}

// Row / column of accumulator element e of tile (mt, nt) for the calling lane.
__device__ __forceinline__ int acc_row(int m0, int mt, int e) {
    return m0 + mt * 16 + ((threadIdx.x & 31) >> 2) + ((e >> 1) << 3);
}
__device__ __forceinline__ int acc_col(int n0, int nt, int e) {
    return n0 + nt * 8 + ((threadIdx.x & 3) << 1) + (e & 1);
}

// ---------------------------------------------------------------- async copies
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
// 16-byte copy that reads src_bytes (0 or 16) bytes and zero-fills the rest.
__device__ __forceinline__ void cp_async16_zfill(void *smem, const void *gmem, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem)), "l"(gmem), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(void *smem, const void *gmem) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Copy a dense [rows][cols] fp16 block (cols multiple of 8) from global into a padded shared tile.
__device__ __forceinline__ void cp_block_f16(__half *dst, int ldd, const __half *src, int rows, int cols, int tid,
                                             int nthr) {
    const int per_row = cols / 8;
    for (int e = tid; e < rows * per_row; e += nthr) {
        int r = e / per_row, c8 = (e % per_row) * 8;
        cp_async16(dst + r * ldd + c8, src + (size_t)r * cols + c8);
    }
}

__device__ __forceinline__ void flag_status(int *status, int bits) { atomicOr(status, bits); }

}  // namespace gdr
