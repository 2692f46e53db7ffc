// k1_wy_prep.cu -- chunk-local WY preparation (one CTA per chunk x value head).
//
// Per chunk of C tokens with chunk-local cumulative gate gamma_r = sum_{i<=r} g_i ("FlashQLA backward
// explained", section 1: the gate arrives as its chunk-local cumsum; here the raw gate is summed in
// place), this kernel forms the strictly-lower, beta-weighted, gate-decayed key Gram matrix
//     A_kk[i, j] = beta_i exp(gamma_i - gamma_j) (k_i . k_j),   j < i
// and its triangular inverse T = (I + A_kk)^{-1}, the "intra-chunk triangular matrix" A [B, T, H, BT] of
// MindSpeed-Ops chunk_kda_bwd.md (input table), by blocked forward substitution in shared memory.  It
// then writes the WY factors W = T diag(beta Gamma) K and U = T diag(beta) V, the decayed attention
// matrix Aqk = M (.) Q K^T (M[i, j] = exp(gamma_i - gamma_j), j <= i), the decayed copies
// K~ = K (.) exp(gamma_C - gamma) and Q~ = Q (.) exp(gamma) that the two scans use, and D = scale dO.
// Per-channel gate: each exp(gamma_a - gamma_b) is taken per key channel inside the K contraction.  For the
// scalar gate's backward it also writes each unit's per-token record (beta, exp(gamma), exp(gamma_C - gamma),
// gamma) that the per-chunk gradient kernel fetches whole.  16-bit input rows arrive by tensor-map loads (two
// 64-column boxes per input with the 128-byte swizzle, so that every row segment of 16 bytes can be read without
// bank conflicts) in their own type: the key Gram and Aqk products take them as they are (bf16 or fp16 operands),
// and the element-wise pass that forms the decayed copies reads them there.
//
// Every matrix output is written in the core-matrix tile layout that the tensor-core kernels read,
// straight from registers: 8 lanes of an element-wise pass write one contiguous 128-byte core matrix, and
// a warp's pair stores of an MMA accumulator cover whole core matrices (no store waits at the end of a
// CTA, so the next CTA on the SM starts at once).  The forward pass runs the same kernel without dO.
#include <string.h>

#include <type_traits>

#include "gdr_common.cuh"
#include "gdr_kernels.h"
#include "tc_util.cuh"

namespace gdr {

constexpr int K1_THREADS = 256;
// row strides (floats) of the fp32 A / T array and the doubling scratch: 4 mod 32, so that the 8 rows x 4 columns
// of a TF32 fragment read fall on 32 distinct banks
constexpr int ATLD = CT + 4, XLD = 32 + 4;
constexpr int GKLD = DT + 4;  // row stride of the per-channel cumulative gate in shared memory (rows 16 bytes
                              // apart in bank terms, so a quarter-warp's 16-byte row reads do not collide)

// 8 consecutive fp16 values of a core-matrix tile row segment / 8 fp32 values (16-byte aligned) as floats
template <typename TT> __device__ __forceinline__ void ld8t(const unsigned char *p, float (&x)[8]) {
    Raw8<TT> r;
    r.v = *reinterpret_cast<const uint4 *>(p);
    raw_get(r, x);
}
// two consecutive 16-bit values as floats
__device__ __forceinline__ float2 ld2t(const __half *p) { return __half22float2(*reinterpret_cast<const __half2 *>(p)); }
__device__ __forceinline__ float2 ld2t(const __nv_bfloat16 *p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(p));
}
__device__ __forceinline__ void ld8f(const float *p, float (&x)[8]) {
    const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
    x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w, x[4] = b.x, x[5] = b.y, x[6] = b.z, x[7] = b.w;
}

struct __align__(1024) K1Smem {
    // Ks, Qs, Vs: the chunk's K, Q, V rows as 128-byte-swizzled halves (sw128_off; bf16 for bf16 inputs, fp16
    // otherwise).  Ks later holds T as the fp16 operand of the W and U products (row-block-major) and the
    // scratch of the inverse's block products; Qs later holds beta Gamma K and Vs beta V (fp16, in place).  AT
    // holds the raw dO rows on their way to the D tile, then A_kk, then in place its inverse T (fp32).
    unsigned char Ks[CT * DT * 2], Qs[CT * DT * 2], Vs[CT * DT * 2];
    float AT[CT][ATLD];
    float gam[CT];
    float beta[CT];
    uint64_t rbar;  // 16-bit inputs: the raw rows' bulk copies
};

// TF32 rounding (round to nearest, ties away) of an fp32 value: the bit pattern the TF32 products take
__device__ __forceinline__ uint32_t tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(r) : "f"(x));
    return r;
}
// c (16 x 8, fp32) += A (16 x 8) B (8 x 8) with TF32 operands.  Fragments (g = lane / 4, t = lane % 4):
// a0 (g, t), a1 (g + 8, t), a2 (g, t + 4), a3 (g + 8, t + 4); b0 (t, g), b1 (t + 4, g); c as for m16n8k16.
__device__ __forceinline__ void mma1688_tf32(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// The same product at about fp32 accuracy by the three-pass TF32 split (Ootomo and Yokota, 2022): each
// operand x = x_hi + x_lo with x_hi its TF32 rounding and x_lo the TF32 rounding of the remainder, and
// A B ~ A_lo B_hi + A_hi B_lo + A_hi B_hi (the small terms first; A_lo B_lo is below fp32 rounding).
__device__ __forceinline__ void mma1688_3xtf32(float (&c)[4], const float (&a)[4], const float (&b)[2]) {
    uint32_t ah[4], al[4], bh[2], bl[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        ah[i] = tf32_rna(a[i]);
        al[i] = tf32_rna(a[i] - __uint_as_float(ah[i]));
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        bh[i] = tf32_rna(b[i]);
        bl[i] = tf32_rna(b[i] - __uint_as_float(bh[i]));
    }
    mma1688_tf32(c, al, bh);
    mma1688_tf32(c, ah, bl);
    mma1688_tf32(c, ah, bh);
}

// One doubling level of the unit-lower-triangular inverse T = (I + A)^-1, built in place over A in fp32 shared
// memory: for every diagonal pair of B x B blocks (lo, hi = lo + B), with the B x B diagonal blocks of T already
// final, X = A[hi][lo] T[lo][lo] and then T[hi][lo] = -T[hi][hi] X.  Each product is a set of 16 x 8 output
// tiles, one per warp, as three-pass TF32 warp MMAs over the reduction in steps of 8.  A level reads A only in
// the blocks it then overwrites, after the barrier between its two products.
template <int B>
__device__ __forceinline__ void inv_level_tc(float (&T)[CT][ATLD], float (&X)[32][XLD], int wid, int lane) {
    constexpr int NP = CT / (2 * B);         // block pairs
    constexpr int PT = (B / 16) * (B / 8);   // 16 x 8 output tiles of one pair's B x B product
    static_assert(NP * PT <= K1_THREADS / 32 && NP * B <= 32, "one output tile per warp; X holds every pair");
    const bool act = wid < NP * PT;
    const int p = wid / PT, tm = (wid % PT) / (B / 8), tn = wid % (B / 8);
    const int lo = 2 * B * p, hi = lo + B, r0 = 16 * tm, c0 = 8 * tn;
    const int g = lane >> 2, t = lane & 3;
    if (act) {  // X[p B + r][c] = sum_k A[hi + r][lo + k] T[lo + k][lo + c]
        float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k0 = 0; k0 < B; k0 += 8) {
            const float a[4] = {T[hi + r0 + g][lo + k0 + t], T[hi + r0 + g + 8][lo + k0 + t],
                                T[hi + r0 + g][lo + k0 + t + 4], T[hi + r0 + g + 8][lo + k0 + t + 4]};
            const float b[2] = {T[lo + k0 + t][lo + c0 + g], T[lo + k0 + t + 4][lo + c0 + g]};
            mma1688_3xtf32(c, a, b);
        }
        *reinterpret_cast<float2 *>(&X[p * B + r0 + g][c0 + 2 * t]) = make_float2(c[0], c[1]);
        *reinterpret_cast<float2 *>(&X[p * B + r0 + g + 8][c0 + 2 * t]) = make_float2(c[2], c[3]);
    }
    __syncthreads();
    if (act) {  // T[hi + r][lo + c] = -sum_k T[hi + r][hi + k] X[p B + k][c]
        float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k0 = 0; k0 < B; k0 += 8) {
            const float a[4] = {T[hi + r0 + g][hi + k0 + t], T[hi + r0 + g + 8][hi + k0 + t],
                                T[hi + r0 + g][hi + k0 + t + 4], T[hi + r0 + g + 8][hi + k0 + t + 4]};
            const float b[2] = {X[p * B + k0 + t][c0 + g], X[p * B + k0 + t + 4][c0 + g]};
            mma1688_3xtf32(c, a, b);
        }
        *reinterpret_cast<float2 *>(&T[hi + r0 + g][lo + c0 + 2 * t]) = make_float2(-c[0], -c[1]);
        *reinterpret_cast<float2 *>(&T[hi + r0 + g + 8][lo + c0 + 2 * t]) = make_float2(-c[2], -c[3]);
    }
    __syncthreads();
}

// The tensor maps (16-bit inputs only; unused for fp32) describe k, q (key heads) and v, dO (value heads) as
// encode_rows_map_sw128 does.
template <typename Tin, bool PC>
__global__ void __launch_bounds__(K1_THREADS, PC ? 2 : 3)
    k1_wy_prep(const Params P, const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmq,
               const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmo) {
    // element type of the staged input tiles and of the key Gram / Aqk products
    using TT = typename std::conditional<std::is_same<Tin, __nv_bfloat16>::value, __nv_bfloat16, __half>::type;
    constexpr bool kBF = std::is_same<Tin, __nv_bfloat16>::value;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // the swizzled tiles need a 1024-byte-aligned base (the launch asks for 1 KB more than the layout)
    unsigned char *const sbase = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    K1Smem &S = *reinterpret_cast<K1Smem *>(sbase);
    float *gamK = reinterpret_cast<float *>(sbase + sizeof(K1Smem));  // [CT][GKLD], per-channel only

    if (*P.status & ST_BAD_SEQLENS) return;
    // heads fastest: CTAs that run at the same time read the same tokens' rows of all heads (whole rows of the
    // [token][head][feature] inputs) rather than one head's rows of many tokens
    const int n = (int)(blockIdx.x / (unsigned)P.Hv), hv = (int)(blockIdx.x % (unsigned)P.Hv), hk = hv / P.G;
    ChunkInfo ci;
    if (!chunk_info(P, n, ci)) return;
    const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
    const size_t u = (size_t)n * P.Hv + hv;
    const int len = ci.len;

    // ---- stage q, k (key head) and v, scale * dO (value head) as fp16 tiles (all loads in flight first)
    const Tin *kp = reinterpret_cast<const Tin *>(P.k) + ((size_t)ci.tok0 * P.Hk + hk) * P.K;
    const Tin *qp = reinterpret_cast<const Tin *>(P.q) + ((size_t)ci.tok0 * P.Hk + hk) * P.K;
    const Tin *vp = reinterpret_cast<const Tin *>(P.v) + ((size_t)ci.tok0 * P.Hv + hv) * P.V;
    const Tin *dop = P.dO ? reinterpret_cast<const Tin *>(P.dO) + ((size_t)ci.tok0 * P.Hv + hv) * P.V : nullptr;
    // the per-token scalars are read first so that their loads overlap the tile loads
    float beta_r = 0.f, gx0 = 0.f, gx1 = 0.f;
    if (tid < len) beta_r = load_scalar(P.beta, (size_t)(ci.tok0 + tid) * P.Hv + hv, P.beta_dtype);
    if (!PC && wid == 0) {
        if (2 * lane < len) gx0 = P.g[(size_t)(ci.tok0 + 2 * lane) * P.Hv + hv];
        if (2 * lane + 1 < len) gx1 = P.g[(size_t)(ci.tok0 + 2 * lane + 1) * P.Hv + hv];
    }
    if constexpr (PC) {
        // the chunk's per-channel gate rows, raw, into the gate tile by asynchronous copies (every thread, all in
        // flight at once; 16 bytes each when the gate tensor is 16-byte aligned, else 4); the cumulative sum below
        // runs over shared memory
        if ((reinterpret_cast<uintptr_t>(P.g) & 15u) == 0) {
            const int c4n = P.K >> 2;
            for (int e = tid; e < len * c4n; e += K1_THREADS) {
                const int i = e / c4n, c4 = 4 * (e - i * c4n);
                cp_async16(gamK + i * GKLD + c4, P.g + ((size_t)(ci.tok0 + i) * P.Hv + hv) * P.K + c4);
            }
        } else {
            for (int e = tid; e < len * P.K; e += K1_THREADS) {
                const int i = e / P.K, c = e - i * P.K;
                cp_async4(gamK + i * GKLD + c, P.g + ((size_t)(ci.tok0 + i) * P.Hv + hv) * P.K + c);
            }
        }
        cp_async_commit();
    }
    const int nin = P.dO ? 4 : 3;
    unsigned char *const slot[4] = {S.Ks, S.Qs, S.Vs, reinterpret_cast<unsigned char *>(&S.AT[0][0])};
    const int nc[4] = {P.K, P.K, P.V, P.V};
    bool bad = false;  // an input value that the fp16 operand tiles cannot hold
    if constexpr (sizeof(Tin) == 2) {
        // one tensor-map load per input (k, q, v, and dO into the A / T buffer, not yet in use), on one mbarrier
        if (tid == 0) {
            tc::mbar_init(&S.rbar, 1);
            asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        }
        __syncthreads();
        if (tid == 0) {
            const int hK = (P.K + 63) >> 6, hV = (P.V + 63) >> 6;  // 64-column boxes per input
            tc::mbar_expect_tx(&S.rbar, (uint32_t)((2 * hK + (nin - 2) * hV) * CT * 128));
            for (int h = 0; h < hK; ++h) {
                tc::tma_load_3d(S.Ks + h * CT * 128, &tmk, 64 * h, hk, ci.tok0, &S.rbar);
                tc::tma_load_3d(S.Qs + h * CT * 128, &tmq, 64 * h, hk, ci.tok0, &S.rbar);
            }
            for (int h = 0; h < hV; ++h) {
                tc::tma_load_3d(S.Vs + h * CT * 128, &tmv, 64 * h, hv, ci.tok0, &S.rbar);
                if (P.dO) tc::tma_load_3d(slot[3] + h * CT * 128, &tmo, 64 * h, hv, ci.tok0, &S.rbar);
            }
        }
        const bool landed = tc::mbar_wait(&S.rbar, 0, P.spin);
        if (__syncthreads_or(!landed)) {
            if (tid == 0) {
                flag_status(P.status, ST_TIMEOUT);
                tc::mbar_wait(&S.rbar, 0, DRAIN_LIMIT);  // the tiles still in flight land before the CTA exits
            }
            if constexpr (PC) cp_async_wait<0>();  // (and this thread's gate-row copies)
            return;
        }
        // a ragged chunk or narrow features: zero the rows past the chunk (the boxes also cover the next
        // sequence's rows) and a half no box filled (columns past K or V inside a box arrive as zero)
        if (len < CT || P.K <= 64 || P.V <= 64) {
            for (int w = 0; w < nin; ++w)
                for (int e = tid; e < CT * DT / 8; e += K1_THREADS) {
                    const int r = e & (CT - 1), c8 = 8 * (e >> 6);
                    if (r >= len || (c8 >= 64 && nc[w] <= 64))
                        *reinterpret_cast<uint4 *>(slot[w] + sw128_off(r, c8)) = make_uint4(0u, 0u, 0u, 0u);
                }
            __syncthreads();
        }
        if (P.dO) {  // D = scale dO, straight from the landed tile to its (row-block-major) workspace tile
            unsigned char *dg = reinterpret_cast<unsigned char *>(P.Dt + u * CT * DT);
            for (int e = tid; e < CT * DT / 8; e += K1_THREADS) {
                const int r = e & (CT - 1), c8 = 8 * (e >> 6);
                float f[8];
                ld8t<TT>(slot[3] + sw128_off(r, c8), f);
                bad |= out_of_f16(f);
#pragma unroll
                for (int t = 0; t < 8; ++t) f[t] *= P.scale;
                *reinterpret_cast<uint4 *>(dg + ctile_off(r, c8, DT)) = pack8_half(f);
            }
        }
    } else {
        // fp32 inputs: each 16-byte fp16 chunk of the swizzled tiles from 8 input values (rows past the chunk
        // and columns past K / V zero); D goes straight to its workspace tile
        const float *const src[4] = {reinterpret_cast<const float *>(kp), reinterpret_cast<const float *>(qp),
                                     reinterpret_cast<const float *>(vp), reinterpret_cast<const float *>(dop)};
        const size_t st[4] = {(size_t)P.Hk * P.K, (size_t)P.Hk * P.K, (size_t)P.Hv * P.V, (size_t)P.Hv * P.V};
        for (int w = 0; w < nin; ++w)
            for (int e = tid; e < CT * DT / 8; e += K1_THREADS) {
                const int r = e & (CT - 1), c8 = 8 * (e >> 6);
                float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                if (r < len && c8 < nc[w]) load8(src[w] + (size_t)r * st[w] + c8, f);
                bad |= out_of_f16(f);
                if (w == 3) {
#pragma unroll
                    for (int t = 0; t < 8; ++t) f[t] *= P.scale;
                    *reinterpret_cast<uint4 *>(reinterpret_cast<unsigned char *>(P.Dt + u * CT * DT) +
                                               ctile_off(r, c8, DT)) = pack8_half(f);
                } else {
                    *reinterpret_cast<uint4 *>(slot[w] + sw128_off(r, c8)) = pack8_half(f);
                }
            }
    }

    // ---- beta, gate cumsum
    if (tid < CT) S.beta[tid] = beta_r;
    if (!PC) {
        if (wid == 0) {
            const float x0 = gx0, x1 = gx1;
            const int r0 = 2 * lane, r1 = 2 * lane + 1;
            float s = x0 + x1;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                float y = __shfl_up_sync(0xffffffffu, s, o);
                if (lane >= o) s += y;
            }
            float excl = s - (x0 + x1);
            S.gam[r0] = excl + x0;
            S.gam[r1] = excl + x0 + x1;
            P.gam[u * CT + r0] = excl + x0;
            P.gam[u * CT + r1] = excl + x0 + x1;
        }
    } else {
        cp_async_wait<0>();
        __syncthreads();  // the raw gate rows have landed
        if (tid < DT) {
            const int c = tid;
            float run = 0.f;
#pragma unroll 8
            for (int i = 0; i < CT; ++i) {
                if (i < len && c < P.K) run += gamK[i * GKLD + c];
                gamK[i * GKLD + c] = run;
                P.gam[(u * CT + i) * DT + c] = run;
            }
        }
    }
    __syncthreads();
    if (!PC && P.sc && P.dO && tid < CT) {  // backward: the per-token record the gradient kernel fetches whole
        float *rec = P.sc + u * 4 * CT;
        const float gt = S.gam[tid], gl = S.gam[len - 1];
        rec[tid] = S.beta[tid];
        rec[CT + tid] = expf(gt);
        rec[2 * CT + tid] = expf(gl - gt);
        rec[3 * CT + tid] = gt;
    }

    // ---- A_kk (fp32, shared) and Aqk (fp16 tile)
    if (!PC) {
        const int m0 = (wid & 3) * 16, n0 = (wid >> 2) * 32;
        float kk[1][4][4], qk[1][4][4];
        zero_acc(kk);
        zero_acc(qk);
        warp_mma_ct<1, 4, false, true, TL_SW128, TL_SW128, kBF>(kk, S.Ks, 0, S.Ks, 0, m0, n0, DT);
        warp_mma_ct<1, 4, false, true, TL_SW128, TL_SW128, kBF>(qk, S.Qs, 0, S.Ks, 0, m0, n0, DT);
        unsigned char *aqk_g = reinterpret_cast<unsigned char *>(P.Aqk + u * CT * CT);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
                const int i = acc_row(m0, 0, e), j = acc_col(n0, nt, e);
                float aq[2], ak[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float d = __expf(S.gam[i] - S.gam[j + h]);  // selected only where the argument is <= 0
                    ak[h] = j + h < i ? S.beta[i] * d * kk[0][nt][e + h] : 0.f;
                    aq[h] = j + h <= i ? d * qk[0][nt][e + h] : 0.f;
                }
                *reinterpret_cast<float2 *>(&S.AT[i][j]) = make_float2(ak[0], ak[1]);
                *reinterpret_cast<__half2 *>(aqk_g + ctile_off(i, j, CT)) = __floats2half2_rn(aq[0], aq[1]);
            }
    } else {
        // per-channel sums sum_c x_ic k_jc exp(gamma_i[c] - gamma_j[c]) (x = k: the decayed key Gram, x = q: Aqk)
        // over the causal part of the chunk, by 16-row blocks I >= J:
        //  * I > J: sub-chunk factorisation around the first row ref = 16 I of block I, exp(gamma_i - gamma_j) =
        //    exp(gamma_i - gamma_ref) exp(gamma_ref - gamma_j), both factors at most 1: one warp per block pair
        //    runs two MMAs over the rescaled rows (built straight into the fragments), K = 128 channels;
        //  * I = J: the block splits at its middle row mid = 16 I + 8: the cross 8 x 8 quarter (upper rows, lower
        //    columns) by the same factorisation around mid (warps 0 and 1, two blocks each), the two 8 x 8
        //    triangles term by term over their 2 x 2 blocks, the 128 channels split between the two lanes of a pair
        //    (their halves added by one shuffle).
        // The blocks above the diagonal are zero.
        unsigned char *aqk_g = reinterpret_cast<unsigned char *>(P.Aqk + u * CT * CT);
        // the decayed key Gram itself (before beta) for the gradient kernel's dbeta, when it is wanted
        unsigned char *kd_g = P.Kd ? reinterpret_cast<unsigned char *>(P.Kd + u * CT * CT) : nullptr;
        auto put2 = [&](int i, int j0, const float (&akk)[2], const float (&aqk)[2]) {  // row i, columns j0, j0 + 1
            float aq[2], kd[2];
#pragma unroll
            for (int bb = 0; bb < 2; ++bb) {
                const int j = j0 + bb;
                kd[bb] = (j < i && i < len) ? akk[bb] : 0.f;
                aq[bb] = (j <= i && i < len) ? aqk[bb] : 0.f;
            }
            *reinterpret_cast<float2 *>(&S.AT[i][j0]) = make_float2(S.beta[i] * kd[0], S.beta[i] * kd[1]);
            *reinterpret_cast<__half2 *>(aqk_g + ctile_off(i, j0, CT)) = __floats2half2_rn(aq[0], aq[1]);
            if (kd_g) *reinterpret_cast<__half2 *>(kd_g + ctile_off(i, j0, CT)) = __floats2half2_rn(kd[0], kd[1]);
        };
        // ---- diagonal triangles: 4 blocks x 2 halves x 10 lower 2 x 2 blocks x 2 channel halves (warps 0..4)
        constexpr int NDIAG = 4 * 2 * 10 * 2;
        for (int t = tid; t < NDIAG; t += K1_THREADS) {
            const int half = t & 1, b2 = t >> 1, blk = b2 / 20, sh = (b2 % 20) / 10, l = b2 % 10;
            const int li = l < 1 ? 0 : (l < 3 ? 1 : (l < 6 ? 2 : 3));  // row of l in a 4 x 4 lower triangle
            const int lj = l - li * (li + 1) / 2;
            const int i0 = 16 * blk + 8 * sh + 2 * li, j0 = 16 * blk + 8 * sh + 2 * lj;
            float akk[2][2] = {{0.f, 0.f}, {0.f, 0.f}}, aqk[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
            if (i0 < len) {
                for (int c8 = 64 * half; c8 < 64 * half + 64; c8 += 8) {
                    float ki[2][8], qi[2][8], kj[2][8], gi[2][8], gj[2][8];
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        ld8t<TT>(S.Ks + sw128_off(i0 + r, c8), ki[r]);
                        ld8t<TT>(S.Qs + sw128_off(i0 + r, c8), qi[r]);
                        ld8t<TT>(S.Ks + sw128_off(j0 + r, c8), kj[r]);
                        ld8f(gamK + (i0 + r) * GKLD + c8, gi[r]);
                        ld8f(gamK + (j0 + r) * GKLD + c8, gj[r]);
                    }
#pragma unroll
                    for (int a = 0; a < 2; ++a)
#pragma unroll
                        for (int bb = 0; bb < 2; ++bb)
#pragma unroll
                            for (int t8 = 0; t8 < 8; ++t8) {
                                // (exponent <= 0 on every element that is kept below)
                                const float kd = kj[bb][t8] * __expf(gi[a][t8] - gj[bb][t8]);
                                akk[a][bb] += ki[a][t8] * kd;
                                aqk[a][bb] += qi[a][t8] * kd;
                            }
                }
            }
            // the other channel half is in the partner lane (tasks 2m, 2m + 1 sit in lanes 2m', 2m' + 1)
#pragma unroll
            for (int a = 0; a < 2; ++a)
#pragma unroll
                for (int bb = 0; bb < 2; ++bb) {
                    akk[a][bb] += __shfl_xor_sync(0xffffffffu, akk[a][bb], 1);
                    aqk[a][bb] += __shfl_xor_sync(0xffffffffu, aqk[a][bb], 1);
                }
            if (!half) {
                put2(i0, j0, akk[0], aqk[0]);
                put2(i0 + 1, j0, akk[1], aqk[1]);
            }
        }
        // ---- cross quarters of the diagonal blocks, on the warps without triangle tasks: warp 5 blocks 0 and 1,
        // warp 6 block 2, warp 7 block 3; the upper 8 rows sit in the fragments' rows 8..15, rows 0..7 stay zero
        if (wid >= 5) {
            const int g4 = lane >> 2, kq = 2 * (lane & 3);
            for (int bi = 0; bi < (wid == 5 ? 2 : 1); ++bi) {
                const int blk = wid == 5 ? bi : wid - 4, mid = 16 * blk + 8;
                float kk[4] = {}, qk[4] = {};
                for (int k0 = 0; k0 < DT; k0 += 16) {
                    uint32_t ak[4] = {0u, 0u, 0u, 0u}, aq[4] = {0u, 0u, 0u, 0u}, bk[2];
#pragma unroll
                    for (int q = 1; q < 4; q += 2) {  // a[1], a[3]: row mid + g4, channels k0 + kq (+8)
                        const int row = mid + g4, c = k0 + kq + 8 * (q >> 1);
                        const float2 gr = *reinterpret_cast<const float2 *>(gamK + mid * GKLD + c);
                        const float2 gx = *reinterpret_cast<const float2 *>(gamK + row * GKLD + c);
                        const float e0 = __expf(gx.x - gr.x), e1 = __expf(gx.y - gr.y);
                        const float2 kv = ld2t(reinterpret_cast<const TT *>(S.Ks + sw128_off(row, c)));
                        const float2 qv = ld2t(reinterpret_cast<const TT *>(S.Qs + sw128_off(row, c)));
                        ak[q] = pack_half2(kv.x * e0, kv.y * e1);
                        aq[q] = pack_half2(qv.x * e0, qv.y * e1);
                    }
#pragma unroll
                    for (int q = 0; q < 2; ++q) {  // key rows 16 blk + g4 (the lower half)
                        const int row = 16 * blk + g4, c = k0 + kq + 8 * q;
                        const float2 gr = *reinterpret_cast<const float2 *>(gamK + mid * GKLD + c);
                        const float2 gx = *reinterpret_cast<const float2 *>(gamK + row * GKLD + c);
                        const float2 kv = ld2t(reinterpret_cast<const TT *>(S.Ks + sw128_off(row, c)));
                        bk[q] = pack_half2(kv.x * __expf(gr.x - gx.x), kv.y * __expf(gr.y - gx.y));
                    }
                    mma16816(kk, ak, bk[0], bk[1]);
                    mma16816(qk, aq, bk[0], bk[1]);
                }
                const float a2[2] = {kk[2], kk[3]}, q2[2] = {qk[2], qk[3]};
                put2(mid + g4, 16 * blk + kq, a2, q2);
            }
        }
        // ---- blocks below the diagonal: warp 2 + p takes the pair p: (I, J) = (1,0) (2,0) (2,1) (3,0) (3,1) (3,2)
        if (wid >= 2) {
            const int p = wid - 2;
            const int I = p < 1 ? 1 : (p < 3 ? 2 : 3), J = p < 1 ? 0 : (p < 3 ? p - 1 : p - 3);
            const int ref = 16 * I, g4 = lane >> 2, kq = 2 * (lane & 3);
            float kk[2][4] = {}, qk[2][4] = {};
            for (int k0 = 0; k0 < DT; k0 += 16) {
                // A fragments (rows 16 I + g4, + 8; channels k0 + kq, +1, +8, +9), rescaled by exp(g[row] - g[ref])
                uint32_t ak[4], aq[4], bk[2][2];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int row = ref + g4 + 8 * (q & 1), c = k0 + kq + 8 * (q >> 1);
                    const float2 gr = *reinterpret_cast<const float2 *>(gamK + ref * GKLD + c);
                    const float2 gx = *reinterpret_cast<const float2 *>(gamK + row * GKLD + c);
                    const float e0 = __expf(gx.x - gr.x), e1 = __expf(gx.y - gr.y);
                    const float2 kv = ld2t(reinterpret_cast<const TT *>(S.Ks + sw128_off(row, c)));
                    const float2 qv = ld2t(reinterpret_cast<const TT *>(S.Qs + sw128_off(row, c)));
                    const __half2 hk = __floats2half2_rn(kv.x * e0, kv.y * e1), hq = __floats2half2_rn(qv.x * e0, qv.y * e1);
                    ak[q] = *reinterpret_cast<const uint32_t *>(&hk);
                    aq[q] = *reinterpret_cast<const uint32_t *>(&hq);
                }
                // B fragments (key rows 16 J + 8 nt + g4; channels k0 + kq, +1 and +8, +9), rescaled by
                // exp(g[ref] - g[row])
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const int row = 16 * J + 8 * nt + g4, c = k0 + kq + 8 * q;
                        const float2 gr = *reinterpret_cast<const float2 *>(gamK + ref * GKLD + c);
                        const float2 gx = *reinterpret_cast<const float2 *>(gamK + row * GKLD + c);
                        const float2 kv = ld2t(reinterpret_cast<const TT *>(S.Ks + sw128_off(row, c)));
                        const __half2 hb = __floats2half2_rn(kv.x * __expf(gr.x - gx.x), kv.y * __expf(gr.y - gx.y));
                        bk[nt][q] = *reinterpret_cast<const uint32_t *>(&hb);
                    }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    mma16816(kk[nt], ak, bk[nt][0], bk[nt][1]);
                    mma16816(qk[nt], aq, bk[nt][0], bk[nt][1]);
                }
            }
            // accumulators: rows ref + g4 (+ 8), columns 16 J + 8 nt + kq (+1), each times exp(g[row] - g[ref])
            // already folded in; write out
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float a2[2] = {kk[nt][2 * h], kk[nt][2 * h + 1]}, q2[2] = {qk[nt][2 * h], qk[nt][2 * h + 1]};
                    put2(ref + g4 + 8 * h, 16 * J + 8 * nt + kq, a2, q2);
                }
        }
        for (int e = tid; e < CT * CT / 2; e += K1_THREADS) {  // pairs (i, j0 .. j0 + 1) above the diagonal blocks
            const int i = e / (CT / 2), j0 = 2 * (e % (CT / 2));
            if (j0 / 2 > i / 2) {
                S.AT[i][j0] = 0.f;
                S.AT[i][j0 + 1] = 0.f;
                *reinterpret_cast<__half2 *>(aqk_g + ctile_off(i, j0, CT)) = __floats2half2_rn(0.f, 0.f);
                if (kd_g) *reinterpret_cast<__half2 *>(kd_g + ctile_off(i, j0, CT)) = __floats2half2_rn(0.f, 0.f);
            }
        }
    }
    __syncthreads();

    // ---- decayed copies of K and Q (to global); W and U operands (beta Gamma K over Q's tile, beta V)
    {
        const float gC = PC ? 0.f : S.gam[len - 1];
        unsigned char *Ktg = reinterpret_cast<unsigned char *>(P.Kt + u * CT * DT);
        unsigned char *Qgg = reinterpret_cast<unsigned char *>(P.Qg + u * CT * DT);
        for (int e = tid; e < CT * DT / 8; e += K1_THREADS) {
            // one 16-byte row segment (row i, columns c8 .. c8 + 7); consecutive lanes walk 8 rows (distinct
            // banks in the swizzled tiles), which are one contiguous core matrix of the row-block-major
            // global tiles
            const int i = e & (CT - 1), c8 = 8 * (e >> 6);
            const uint32_t off = ctile_off(i, c8, DT), so = sw128_off(i, c8);
            float kx[8], qx[8], vx[8], o1[8], o2[8], o3[8], o4[8];
            ld8t<TT>(S.Ks + so, kx);
            ld8t<TT>(S.Qs + so, qx);
            ld8t<TT>(S.Vs + so, vx);
            if constexpr (sizeof(Tin) == 2) bad |= out_of_f16(kx) | out_of_f16(qx) | out_of_f16(vx);
            const float bi = S.beta[i];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                float gi = PC ? gamK[i * GKLD + c8 + t] : S.gam[i];
                float gc = PC ? gamK[(len - 1) * GKLD + c8 + t] : gC;
                float Gi = __expf(gi);
                o1[t] = kx[t] * __expf(gc - gi);  // K~
                o2[t] = qx[t] * Gi;             // Q~
                o3[t] = bi * Gi * kx[t];        // beta Gamma K
                o4[t] = bi * vx[t];             // beta V
            }
            *reinterpret_cast<uint4 *>(Ktg + off) = pack8_half(o1);
            *reinterpret_cast<uint4 *>(Qgg + off) = pack8_half(o2);
            *reinterpret_cast<uint4 *>(S.Qs + so) = pack8_half(o3);  // in place (fp16 from here on)
            *reinterpret_cast<uint4 *>(S.Vs + so) = pack8_half(o4);
        }
        if (bad) flag_status(P.status, ST_RANGE);
    }

    // ---- T = (I + A_kk)^-1: diagonal 16x16 blocks by per-column forward substitution, then doubling
    // (in place: every thread has read its diagonal block of A before any T column is written)
    {
        const bool dact = wid < 4 && lane < 16;
        const int b0 = wid * 16, m = lane;
        float x[16];
        if (dact) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float acc = (i == m) ? 1.f : 0.f;
#pragma unroll
                for (int j = 0; j < i; ++j) acc -= S.AT[b0 + i][b0 + j] * x[j];
                x[i] = acc;
            }
        }
        __syncthreads();
        if (dact) {
#pragma unroll
            for (int i = 0; i < 16; ++i) S.AT[b0 + i][b0 + m] = x[i];
        }
    }
    __syncthreads();
    unsigned char *const oT = S.Ks;  // K is no longer needed
    float (&X32)[32][XLD] = *reinterpret_cast<float (*)[32][XLD]>(S.Ks + CT * CT * 2);
    // off-diagonal blocks by recursive doubling: for a lower block split [[T_11, 0], [X, T_22]] of an inverse,
    // X = -T_22 A_21 T_11.  First the two 32 x 32 diagonal blocks from their 16 x 16 halves, then the whole.
    inv_level_tc<16>(S.AT, X32, wid, lane);
    inv_level_tc<32>(S.AT, X32, wid, lane);
    for (int e = tid; e < CT * CT / 8; e += K1_THREADS) {
        int i = e / (CT / 8), j8 = (e % (CT / 8)) * 8;
        float x[8];
#pragma unroll
        for (int t = 0; t < 8; t += 4) {
            const float4 v = *reinterpret_cast<const float4 *>(&S.AT[i][j8 + t]);
            x[t] = v.x, x[t + 1] = v.y, x[t + 2] = v.z, x[t + 3] = v.w;
        }
        tc::st_tile8(oT, i, j8, CT, x);
        // (the forward, which runs without dO, needs T only for W and U)
        if (P.dO) tc::st_tile8(reinterpret_cast<unsigned char *>(P.Tm + u * CT * CT), i, j8, CT, x);
    }
    __syncthreads();

    // ---- W = T (beta Gamma K) and U^T = (beta V)^T T^T (a [v][c] tile), stored from the accumulators
    {
        float acc[1][8][4];
        {
            const int m0 = (wid & 3) * 16, n0 = (wid >> 2) * 64;
            zero_acc(acc);
            warp_mma_ct<1, 8, false, false, TL_ROWB, TL_SW128>(acc, oT, CT, S.Qs, 0, m0, n0, CT);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    int i = acc_row(m0, 0, e), j = acc_col(n0, nt, e);
                    *reinterpret_cast<__half2 *>(reinterpret_cast<unsigned char *>(P.W + u * CT * DT) +
                                                 ctile_off(i, j, DT)) = __floats2half2_rn(acc[0][nt][e], acc[0][nt][e + 1]);
                }
        }
        {
            const int m0 = wid * 16;  // 8 warps x 16 value rows, all 64 chunk columns
            zero_acc(acc);
            warp_mma_ct<1, 8, true, true, TL_SW128, TL_ROWB>(acc, S.Vs, 0, oT, CT, m0, 0, CT);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    int v = acc_row(m0, 0, e), c = acc_col(0, nt, e);
                    *reinterpret_cast<__half2 *>(reinterpret_cast<unsigned char *>(P.U + u * CT * DT) +
                                                 ctile_off(v, c, CT)) = __floats2half2_rn(acc[0][nt][e], acc[0][nt][e + 1]);
                }
        }
    }
}

template <typename Tin, bool PC>
static cudaError_t launch_k1_t(const Params &P, cudaStream_t stream) {
    size_t smem = sizeof(K1Smem) + (PC ? sizeof(float) * CT * GKLD : 0) + 1024;  // (+ alignment slack)
    cudaError_t e = smem_opt_in((const void *)k1_wy_prep<Tin, PC>, smem);
    if (e != cudaSuccess) return e;
    CUtensorMap mk, mq, mv, mo;
    memset(&mk, 0, sizeof(mk));
    memset(&mq, 0, sizeof(mq));
    memset(&mv, 0, sizeof(mv));
    memset(&mo, 0, sizeof(mo));
    if (sizeof(Tin) == 2) {
        const long long tokens = (long long)P.B * P.T;
        if ((e = encode_rows_map_sw128(&mk, P.k, P.qkv_dtype, tokens, P.Hk, P.K)) != cudaSuccess) return e;
        if ((e = encode_rows_map_sw128(&mq, P.q, P.qkv_dtype, tokens, P.Hk, P.K)) != cudaSuccess) return e;
        if ((e = encode_rows_map_sw128(&mv, P.v, P.qkv_dtype, tokens, P.Hv, P.V)) != cudaSuccess) return e;
        if (P.dO && (e = encode_rows_map_sw128(&mo, P.dO, P.qkv_dtype, tokens, P.Hv, P.V)) != cudaSuccess) return e;
    }
    if ((long long)P.max_chunks * P.Hv > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    dim3 grid((unsigned)P.max_chunks * (unsigned)P.Hv);  // CTA n Hv + hv
    k1_wy_prep<Tin, PC><<<grid, K1_THREADS, smem, stream>>>(P, mk, mq, mv, mo);
    return cudaGetLastError();
}

cudaError_t launch_k1(const Params &P, cudaStream_t stream) {
    if (P.qkv_dtype == F32) return P.per_channel ? launch_k1_t<float, true>(P, stream) : launch_k1_t<float, false>(P, stream);
    if (P.qkv_dtype == BF16)
        return P.per_channel ? launch_k1_t<__nv_bfloat16, true>(P, stream) : launch_k1_t<__nv_bfloat16, false>(P, stream);
    return P.per_channel ? launch_k1_t<__half, true>(P, stream) : launch_k1_t<__half, false>(P, stream);
}

}  // namespace gdr
