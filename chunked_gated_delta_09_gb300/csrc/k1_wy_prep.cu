// k1_wy_prep.cu -- chunk-local WY preparation (one CTA per chunk x value head).
//
// Per chunk of C tokens with chunk-local cumulative gate gamma_r = sum_{i<=r} g_i ("FlashQLA backward
// explained", section 1: the gate arrives as its chunk-local cumsum; here the raw gate is summed in
// place), this kernel forms the strictly-lower, beta-weighted, gate-decayed key Gram matrix
//     A_kk[i, j] = beta_i exp(gamma_i - gamma_j) (k_i . k_j),   j < i
// and its triangular inverse T = (I + A_kk)^{-1}, the "intra-chunk triangular matrix" A [B, T, H, BT] of
// MindSpeed-Ops chunk_kda_bwd.md (input table), by blocked forward substitution in shared memory.  It
// then writes the WY factors W = T diag(beta Gamma) K and U = T diag(beta) V, the decayed attention
// matrix Aqk = M (.) Q K^T (M[i, j] = exp(gamma_i - gamma_j), j <= i), and the decayed copies
// K (.) exp(gamma_C - gamma) and Q (.) exp(gamma) that the two scans use.
// Per-channel gate: each exp(gamma_a - gamma_b) is taken per key channel inside the K contraction.
#include "gdr_common.cuh"
#include "gdr_kernels.h"

namespace gdr {

constexpr int K1_THREADS = 256;

struct K1Smem {
    __half Ks[CT * LDD], Qs[CT * LDD], Vs[CT * LDD], KB[CT * LDD], VB[CT * LDD];
    __half Th[CT * LDC];
    float A32[CT][CT + 1];
    float T32[CT][CT + 1];
    float X32[3][16][17];
    float gam[CT];
    float beta[CT];
};

template <typename Tin, bool PC>
__global__ void __launch_bounds__(K1_THREADS) k1_wy_prep(const Params P) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    K1Smem &S = *reinterpret_cast<K1Smem *>(smem_raw);
    float *gamK = reinterpret_cast<float *>(smem_raw + sizeof(K1Smem));  // [CT][DT], per-channel only

    if (*P.status & ST_BAD_SEQLENS) return;
    const int n = blockIdx.x, hv = blockIdx.y, hk = hv / P.G;
    ChunkInfo ci;
    if (!chunk_info(P, n, ci)) return;
    const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
    const size_t u = (size_t)n * P.Hv + hv;
    const int len = ci.len;

    // ---- beta, gate cumsum
    if (tid < CT) S.beta[tid] = tid < len ? load_scalar(P.beta, (size_t)(ci.tok0 + tid) * P.Hv + hv, P.beta_dtype) : 0.f;
    if (!PC) {
        if (wid == 0) {
            float x0 = 0.f, x1 = 0.f;
            int r0 = 2 * lane, r1 = 2 * lane + 1;
            if (r0 < len) x0 = P.g[(size_t)(ci.tok0 + r0) * P.Hv + hv];
            if (r1 < len) x1 = P.g[(size_t)(ci.tok0 + r1) * P.Hv + hv];
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
        if (tid < DT) {
            const int c = tid;
            float run = 0.f;
            for (int i = 0; i < CT; ++i) {
                if (i < len && c < P.K) run += P.g[((size_t)(ci.tok0 + i) * P.Hv + hv) * P.K + c];
                gamK[i * DT + c] = run;
                P.gam[(u * CT + i) * DT + c] = run;
            }
        }
    }
    // ---- stage q, k (key head) and v (value head) as fp16
    const Tin *kp = reinterpret_cast<const Tin *>(P.k) + ((size_t)ci.tok0 * P.Hk + hk) * P.K;
    const Tin *qp = reinterpret_cast<const Tin *>(P.q) + ((size_t)ci.tok0 * P.Hk + hk) * P.K;
    const Tin *vp = reinterpret_cast<const Tin *>(P.v) + ((size_t)ci.tok0 * P.Hv + hv) * P.V;
    stage_rows_f16(S.Ks, kp, (size_t)P.Hk * P.K, len, P.K, nullptr, 1.f, tid, K1_THREADS);
    stage_rows_f16(S.Qs, qp, (size_t)P.Hk * P.K, len, P.K, nullptr, 1.f, tid, K1_THREADS);
    stage_rows_f16(S.Vs, vp, (size_t)P.Hv * P.V, len, P.V, nullptr, 1.f, tid, K1_THREADS);
    for (int e = tid; e < CT * (CT + 1); e += K1_THREADS) (&S.T32[0][0])[e] = 0.f;
    __syncthreads();

    __half *Aqk_g = P.Aqk + u * CT * CT;
    // ---- A_kk (fp32, shared) and Aqk (fp16, global)
    if (!PC) {
        const int m0 = (wid & 3) * 16, n0 = (wid >> 2) * 32;
        float kk[1][4][4], qk[1][4][4];
        zero_acc(kk);
        zero_acc(qk);
        warp_mma<1, 4, false, true>(kk, S.Ks, LDD, S.Ks, LDD, m0, n0, DT);
        warp_mma<1, 4, false, true>(qk, S.Qs, LDD, S.Ks, LDD, m0, n0, DT);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                int i = acc_row(m0, 0, e), j = acc_col(n0, nt, e);
                float d = expf(S.gam[i] - S.gam[j]);
                S.A32[i][j] = j < i ? S.beta[i] * d * kk[0][nt][e] : 0.f;
                Aqk_g[i * CT + j] = __float2half_rn(j <= i ? d * qk[0][nt][e] : 0.f);
            }
    } else {
        for (int e = tid; e < CT * CT; e += K1_THREADS) {
            int i = e / CT, j = e % CT;
            float akk = 0.f, aqk = 0.f;
            if (j <= i && i < len) {
                for (int c = 0; c < DT; ++c) {
                    float d = expf(gamK[i * DT + c] - gamK[j * DT + c]);
                    float kj = __half2float(S.Ks[j * LDD + c]);
                    akk += __half2float(S.Ks[i * LDD + c]) * kj * d;
                    aqk += __half2float(S.Qs[i * LDD + c]) * kj * d;
                }
            }
            S.A32[i][j] = j < i ? S.beta[i] * akk : 0.f;
            Aqk_g[i * CT + j] = __float2half_rn(j <= i ? aqk : 0.f);
        }
    }
    __syncthreads();

    // ---- T = (I + A_kk)^-1: diagonal 16x16 blocks by per-column forward substitution
    if (wid < 4 && lane < 16) {
        const int b0 = wid * 16, m = lane;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float acc = (i == m) ? 1.f : 0.f;
#pragma unroll
            for (int j = 0; j < i; ++j) acc -= S.A32[b0 + i][b0 + j] * x[j];
            x[i] = acc;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) S.T32[b0 + i][b0 + m] = x[i];
    }
    __syncthreads();
    // off-diagonal blocks, one block row at a time: T_IJ = -T_II * sum_{J<=k<I} A_Ik T_kJ
    for (int I = 1; I < 4; ++I) {
        for (int e = tid; e < I * 256; e += K1_THREADS) {
            int J = e >> 8, a = (e >> 4) & 15, b = e & 15;
            float acc = 0.f;
            for (int col = 16 * J; col < 16 * I; ++col) acc += S.A32[16 * I + a][col] * S.T32[col][16 * J + b];
            S.X32[J][a][b] = acc;
        }
        __syncthreads();
        for (int e = tid; e < I * 256; e += K1_THREADS) {
            int J = e >> 8, a = (e >> 4) & 15, b = e & 15;
            float acc = 0.f;
            for (int c = 0; c <= a; ++c) acc += S.T32[16 * I + a][16 * I + c] * S.X32[J][c][b];
            S.T32[16 * I + a][16 * J + b] = -acc;
        }
        __syncthreads();
    }

    // ---- operands for W and U, decayed copies of K and Q, T in fp16
    __half *Kt_g = P.Kt + u * CT * DT, *Qg_g = P.Qg + u * CT * DT;
    const float gC = PC ? 0.f : S.gam[len - 1];
    for (int e = tid; e < CT * DT; e += K1_THREADS) {
        int i = e / DT, c = e % DT;
        float gi = PC ? gamK[i * DT + c] : S.gam[i];
        float gc = PC ? gamK[(len - 1) * DT + c] : gC;
        float kv = __half2float(S.Ks[i * LDD + c]);
        float qv = __half2float(S.Qs[i * LDD + c]);
        float Gi = expf(gi);
        S.KB[i * LDD + c] = __float2half_rn(S.beta[i] * Gi * kv);
        S.VB[i * LDD + c] = __float2half_rn(S.beta[i] * __half2float(S.Vs[i * LDD + c]));
        Kt_g[e] = __float2half_rn(kv * expf(gc - gi));
        Qg_g[e] = __float2half_rn(qv * Gi);
    }
    __half *T_g = P.Tm + u * CT * CT;
    for (int e = tid; e < CT * CT; e += K1_THREADS) {
        int i = e / CT, j = e % CT;
        __half t = __float2half_rn(S.T32[i][j]);
        S.Th[i * LDC + j] = t;
        T_g[e] = t;
    }
    __syncthreads();

    // ---- W = T (beta Gamma K), U = T (beta V)
    {
        const int m0 = (wid & 3) * 16, n0 = (wid >> 2) * 64;
        float acc[1][8][4];
        __half *W_g = P.W + u * CT * DT, *U_g = P.U + u * CT * DT;
        zero_acc(acc);
        warp_mma<1, 8, false, false>(acc, S.Th, LDC, S.KB, LDD, m0, n0, CT);
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
                int i = acc_row(m0, 0, e), j = acc_col(n0, nt, e);
                *reinterpret_cast<__half2 *>(W_g + i * DT + j) = __floats2half2_rn(acc[0][nt][e], acc[0][nt][e + 1]);
            }
        zero_acc(acc);
        warp_mma<1, 8, false, false>(acc, S.Th, LDC, S.VB, LDD, m0, n0, CT);
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
                int i = acc_row(m0, 0, e), j = acc_col(n0, nt, e);
                *reinterpret_cast<__half2 *>(U_g + i * DT + j) = __floats2half2_rn(acc[0][nt][e], acc[0][nt][e + 1]);
            }
    }
}

template <typename Tin, bool PC>
static cudaError_t launch_k1_t(const Params &P, cudaStream_t stream) {
    size_t smem = sizeof(K1Smem) + (PC ? sizeof(float) * CT * DT : 0);
    cudaError_t e = cudaFuncSetAttribute(k1_wy_prep<Tin, PC>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(P.max_chunks, P.Hv);
    k1_wy_prep<Tin, PC><<<grid, K1_THREADS, smem, stream>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_k1(const Params &P, cudaStream_t stream) {
    if (P.qkv_dtype == F32) return P.per_channel ? launch_k1_t<float, true>(P, stream) : launch_k1_t<float, false>(P, stream);
    if (P.qkv_dtype == BF16)
        return P.per_channel ? launch_k1_t<__nv_bfloat16, true>(P, stream) : launch_k1_t<__nv_bfloat16, false>(P, stream);
    return P.per_channel ? launch_k1_t<__half, true>(P, stream) : launch_k1_t<__half, false>(P, stream);
}

}  // namespace gdr
