// k4_intra_grad_tc.cu -- per-chunk gradients on the 5th-generation tensor cores (scalar gate).
//
// Same mathematics as k4_intra_grad.cu (the WY-gradient stage of MindSpeed-Ops chunk_kda_bwd.md,
// "implementation principle", with the scalar gate of "FlashQLA backward explained", section 2), with
// every matrix product issued as tcgen05.mma (fp16 operands from shared memory, fp32 accumulators in
// tensor memory) by one thread, completion tracked by an mbarrier with a bounded wait, and results
// read back with tcgen05.ld.  Products whose output is chunk x feature are computed transposed
// (feature x chunk, M = 128) so that each epilogue thread owns one feature row and writes coalesced;
// chunk x chunk products use M = 64.  Operands are staged once in the core-matrix layout and used in
// either K-major or MN-major view, so no transposed copies are made.
//
// Five MMA phases, each followed by an epilogue that produces the next phase's operands:
//   1: P0 = D V_new^T, dq_inter^T = S0^T D^T, dk_SC^T = dS^T V_new^T, dW^T = -S0^T dV^T,
//      dT2 = dV V^T, TdU^T = dV^T T, KK = K K^T
//   2: dq_intra^T = K^T P^T, dk_O^T = Q^T P, TdW^T = dW^T T, dT1 = dW K^T
//   3: X = dT T^T        4: dA' = T^T X        5: dk_Ar^T = K^T E^T, dk_Ac^T = K^T E
#include "gdr_common.cuh"
#include "gdr_kernels.h"
#include "tc_util.cuh"

namespace gdr {

constexpr int K4T_THREADS = 256;
constexpr uint32_t K4T_TMEM_COLS = 512;
constexpr uint32_t K4T_WAIT_LIMIT = 1u << 24;  // mbarrier polls before a wait is declared lost

// tensor-memory column map (64 columns each; C_* regions use the M = 64 lane layout)
constexpr int C_G1 = 0, R_DQI = 64, R_DKSC = 128, R_DWT = 192, C_DT2 = 256, R_TDU = 320, C_KK = 384;
constexpr int R_DQA = 0, R_DKO = 128, R_TDW = 192, C_DT1 = 320;
constexpr int C_X = 0, C_DA = 64, R_DKAR = 128, R_DKAC = 192;

struct __align__(1024) K4TSmem {
    unsigned char Q[CT * DT * 2], K[CT * DT * 2], V[CT * DT * 2], D[CT * DT * 2];
    unsigned char Vn[DT * CT * 2], dVn[DT * CT * 2];  // V_new^T and -dV_new^T, tiles [v][c]
    unsigned char H[DT * DT * 2], dH[DT * DT * 2];    // [v][k] tiles: S_0 and dS_next
    unsigned char T[CT * CT * 2];
    unsigned char Pm[CT * CT * 2];   // P, later X
    unsigned char dWT[DT * CT * 2];  // dW^T [k][r]
    unsigned char dT[CT * CT * 2];   // dT, later E
    float gam[CT], G[CT], GC[CT], beta[CT];
    // partial sums in fixed slots, added in a fixed order at the end (run-to-run reproducible):
    // dbeta: 4 lane quarters x (TdU, TdW) + 2 column halves x (A term); dgrow: 4 quarters; lastrow: 8 warps
    float db_tdu[4][CT], db_tdw[4][CT], db_a[2][CT], dg_q[4][CT], last_w[8];
    uint64_t bar, lbar;
    uint32_t tslot;
};

template <typename Tin>
__global__ void __launch_bounds__(K4T_THREADS, 1) k4_intra_grad_tc(const Params P) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    K4TSmem &S = *reinterpret_cast<K4TSmem *>(smem_raw);
    if (*P.status & ST_BAD_SEQLENS) return;
    const int n = blockIdx.x, hv = blockIdx.y, hk = hv / P.G;
    ChunkInfo ci;
    if (!chunk_info(P, n, ci)) return;
    const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
    const size_t u = (size_t)n * P.Hv + hv;
    const int len = ci.len, rl = len - 1;

    if (wid == 0) tc::tmem_alloc(&S.tslot, K4T_TMEM_COLS);
    if (tid == 0) {
        tc::mbar_init(&S.bar, 1);
        tc::mbar_init(&S.lbar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        // ---- workspace tiles by bulk copy
        tc::mbar_expect_tx(&S.lbar, 2 * DT * DT * 2 + 2 * DT * CT * 2 + CT * CT * 2 + CT * DT * 2);
        tc::bulk_g2s(S.H, P.h + u * DT * DT, DT * DT * 2, &S.lbar);
        tc::bulk_g2s(S.dH, P.dh + u * DT * DT, DT * DT * 2, &S.lbar);
        tc::bulk_g2s(S.Vn, P.Vn + u * DT * CT, DT * CT * 2, &S.lbar);
        tc::bulk_g2s(S.dVn, P.dVn + u * DT * CT, DT * CT * 2, &S.lbar);
        tc::bulk_g2s(S.T, P.Tm + u * CT * CT, CT * CT * 2, &S.lbar);
        tc::bulk_g2s(S.D, P.Dt + u * CT * DT, CT * DT * 2, &S.lbar);
    }
    if (tid < CT) {
        S.beta[tid] = tid < len ? load_scalar(P.beta, (size_t)(ci.tok0 + tid) * P.Hv + hv, P.beta_dtype) : 0.f;
        S.gam[tid] = P.gam[u * CT + tid];
        S.db_a[0][tid] = 0.f;
        S.db_a[1][tid] = 0.f;
    }
    tc::fence_before();
    __syncthreads();  // barrier initialisation and the tensor-memory address visible
    tc::fence_after();
    // thread 0 waits for the bulk loads and starts the tile-only MMAs; everyone else converts inputs
    // meanwhile (the barrier after the conversion orders their later reads after that wait)
    const bool loaded = tid == 0 ? tc::mbar_wait(&S.lbar, 0, K4T_WAIT_LIMIT) : true;
    const uint32_t tm = S.tslot;
    const uint32_t sQ = smem_u32(S.Q), sK = smem_u32(S.K), sV = smem_u32(S.V), sD = smem_u32(S.D);
    const uint32_t sVn = smem_u32(S.Vn), sdVn = smem_u32(S.dVn), sH = smem_u32(S.H), sdH = smem_u32(S.dH);
    const uint32_t sT = smem_u32(S.T), sPm = smem_u32(S.Pm), sdWT = smem_u32(S.dWT), sdT = smem_u32(S.dT);
    unsigned char *Xs = S.Pm, *Es = S.dT;
    const uint32_t sX = sPm, sE = sdT;
    // phase 1, part 1: products of workspace tiles only, overlapping the input conversion below
    if (tid == 0 && loaded) {
        tc::gemm(tm + R_DKSC, sdH, DT, true, sVn, CT, true, 128, 64, DT, false);
        tc::gemm(tm + R_DWT, sH, DT, true, sdVn, CT, true, 128, 64, DT, false);
        tc::gemm(tm + R_TDU, sdVn, CT, false, sT, CT, true, 128, 64, CT, false);
    }
    const Tin *kp = reinterpret_cast<const Tin *>(P.k) + ((size_t)ci.tok0 * P.Hk + hk) * P.K;
    const Tin *qp = reinterpret_cast<const Tin *>(P.q) + ((size_t)ci.tok0 * P.Hk + hk) * P.K;
    const Tin *vp = reinterpret_cast<const Tin *>(P.v) + ((size_t)ci.tok0 * P.Hv + hv) * P.V;
    {
        unsigned char *const dst[3] = {S.K, S.Q, S.V};
        const Tin *const src[3] = {kp, qp, vp};
        const size_t st[3] = {(size_t)P.Hk * P.K, (size_t)P.Hk * P.K, (size_t)P.Hv * P.V};
        const int nc[3] = {P.K, P.K, P.V};
        const float mul[3] = {1.f, 1.f, 1.f};
        stage_ct_n<Tin, K4T_THREADS, 3>(dst, src, st, nc, mul, len, tid);
    }
    if (tid < CT) {
        S.G[tid] = expf(S.gam[tid]);
        S.GC[tid] = expf(S.gam[rl] - S.gam[tid]);
    }
    tc::fence_smem_to_async();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    uint32_t parity = 0;
    bool lost = __syncthreads_or(!loaded) != 0;

    // Each phase: one thread issues, everyone waits (bounded) and agrees on the outcome.
    auto finish_phase = [&]() {
        if (tid == 0) tc::commit(&S.bar);
        bool ok = tc::mbar_wait(&S.bar, parity, K4T_WAIT_LIMIT);
        parity ^= 1u;
        lost = __syncthreads_or(!ok || lost) != 0;
        tc::fence_after();
    };
    auto publish_tiles = [&]() {  // make epilogue-written tiles visible to the next phase's MMAs
        tc::fence_smem_to_async();
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
    };

    // Epilogue ownership: warp w reads lane quarter q = w % 4 and the column half c0 = 32 (w / 4).
    const int q = wid & 3, c0 = 32 * (wid >> 2);
    const int k = 32 * q + lane;        // feature row in M = 128 regions
    const int r64 = 16 * q + lane;      // chunk row in M = 64 regions (lanes 0..15)
    const bool own64 = lane < 16;
    float dk[32], dg[32], kreg[32];
    float lastpart = 0.f;
#pragma unroll
    for (int t = 0; t < 32; ++t) kreg[t] = tc::ld_tile(S.K, c0 + t, k, DT);

    // ---------------- phase 1, part 2 (needs the converted inputs)
    if (tid == 0 && !lost) {
        tc::gemm(tm + C_G1, sD, DT, false, sVn, CT, true, 64, 64, DT, false);
        tc::gemm(tm + R_DQI, sH, DT, true, sD, DT, false, 128, 64, DT, false);
        tc::gemm(tm + C_DT2, sdVn, CT, true, sV, DT, false, 64, 64, DT, false);
        tc::gemm(tm + C_KK, sK, DT, false, sK, DT, false, 64, 64, DT, false);
    }
    finish_phase();
    if (!lost) {
        float g[32];
        // P = (D V_new^T) (.) M  -> Pm tile
        tc::ld32(tc::taddr(tm, C_G1 + c0), g);
        if (own64) {
            const float gr = S.gam[r64];
#pragma unroll
            for (int j8 = 0; j8 < 32; j8 += 8) {
                float x[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    int j = c0 + j8 + t;
                    x[t] = j <= r64 ? g[j8 + t] * expf(gr - S.gam[j]) : 0.f;
                }
                tc::st_tile8(S.Pm, r64, c0 + j8, CT, x);
            }
        }
        // dW^T -> dWT tile (the stored dV tile is negated, so the product already is dW^T)
        tc::ld32(tc::taddr(tm, R_DWT + c0), g);
#pragma unroll
        for (int j8 = 0; j8 < 32; j8 += 8) tc::st_tile8(S.dWT, k, c0 + j8, CT, g + j8);
        // dk_SC = exp(gamma_C - gamma_j) (V_new dS)_j
        tc::ld32(tc::taddr(tm, R_DKSC + c0), g);
#pragma unroll
        for (int t = 0; t < 32; ++t) {
            float x = g[t] * S.GC[c0 + t];
            float kx = kreg[t] * x;
            dk[t] = x;
            dg[t] = -kx;
            lastpart += kx;
        }
        // TdU^T -> dv (coalesced over the feature index), dbeta += rowsum(TdU (.) V)
        tc::ld32(tc::taddr(tm, R_TDU + c0), g);
#pragma unroll
        for (int t = 0; t < 32; ++t) g[t] = -g[t];  // negated dV tile
        {
            float db[32];
#pragma unroll
            for (int t = 0; t < 32; ++t) {
                int r = c0 + t;
                db[t] = g[t] * tc::ld_tile(S.V, r, k, DT);
                if (r < len && k < P.V)
                    store_scalar(P.dv, ((size_t)(ci.tok0 + r) * P.Hv + hv) * P.V + k, S.beta[r] * g[t], P.dv_dtype);
            }
            S.db_tdu[q][c0 + lane] = tc::warp_transpose_sum32(db);
        }
    }
    publish_tiles();

    // ---------------- phase 2
    if (tid == 0 && !lost) {
        tc::gemm(tm + R_DQA, sK, DT, true, sPm, CT, false, 128, 64, CT, false);
        tc::gemm(tm + R_DKO, sQ, DT, true, sPm, CT, true, 128, 64, CT, false);
        tc::gemm(tm + R_TDW, sdWT, CT, false, sT, CT, true, 128, 64, CT, false);
        tc::gemm(tm + C_DT1, sdWT, CT, true, sK, DT, false, 64, 64, DT, false);
    }
    if (!lost) finish_phase();
    if (!lost) {
        float a[32], b[32];
        // dq = Gamma (.) dq_inter + dq_intra
        tc::ld32(tc::taddr(tm, R_DQI + c0), a);
        tc::ld32(tc::taddr(tm, R_DQA + c0), b);
#pragma unroll
        for (int t = 0; t < 32; ++t) {
            int r = c0 + t;
            float x = S.G[r] * a[t] + b[t];
            dg[t] += tc::ld_tile(S.Q, r, k, DT) * x;
            if (r < len && k < P.K) {
                if (P.G == 1)
                    store_scalar(P.dq, ((size_t)(ci.tok0 + r) * P.Hk + hk) * P.K + k, x, P.dqdk_dtype);
                else
                    P.dq_h[((size_t)(ci.tok0 + r) * P.Hv + hv) * P.K + k] = x;
            }
        }
        // dk_O
        tc::ld32(tc::taddr(tm, R_DKO + c0), a);
#pragma unroll
        for (int t = 0; t < 32; ++t) {
            dk[t] += a[t];
            dg[t] -= kreg[t] * a[t];
        }
        // TdW^T -> dk_W, dbeta
        tc::ld32(tc::taddr(tm, R_TDW + c0), a);
        {
#pragma unroll
            for (int t = 0; t < 32; ++t) {
                int j = c0 + t;
                float x = S.beta[j] * S.G[j] * a[t];
                dk[t] += x;
                dg[t] += kreg[t] * x;
                b[t] = S.G[j] * kreg[t] * a[t];
            }
            S.db_tdw[q][c0 + lane] = tc::warp_transpose_sum32(b);
        }
        // dT = dT1 (.) beta Gamma + dT2 (.) beta   -> dT tile
        tc::ld32(tc::taddr(tm, C_DT1 + c0), a);
        tc::ld32(tc::taddr(tm, C_DT2 + c0), b);
        if (own64) {
#pragma unroll
            for (int j8 = 0; j8 < 32; j8 += 8) {
                float x[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    int j = c0 + j8 + t;
                    x[t] = S.beta[j] * (S.G[j] * a[j8 + t] - b[j8 + t]);  // dT2 came negated
                }
                tc::st_tile8(S.dT, r64, c0 + j8, CT, x);
            }
        }
    }
    publish_tiles();

    // ---------------- phase 3: X = dT T^T
    if (tid == 0 && !lost) tc::gemm(tm + C_X, sdT, CT, false, sT, CT, false, 64, 64, CT, false);
    if (!lost) finish_phase();
    if (!lost) {
        float a[32];
        tc::ld32(tc::taddr(tm, C_X + c0), a);
        if (own64) {
#pragma unroll
            for (int j8 = 0; j8 < 32; j8 += 8) tc::st_tile8(Xs, r64, c0 + j8, CT, a + j8);
        }
    }
    publish_tiles();

    // ---------------- phase 4: dA' = T^T X; dA = strict_lower(-dA'); E = beta L dA
    if (tid == 0 && !lost) tc::gemm(tm + C_DA, sT, CT, true, sX, CT, true, 64, 64, CT, false);
    if (!lost) finish_phase();
    if (!lost) {
        float a[32], kk[32];
        tc::ld32(tc::taddr(tm, C_DA + c0), a);
        tc::ld32(tc::taddr(tm, C_KK + c0), kk);
        if (own64) {
            const int i = r64;
            const float gi = S.gam[i], bi = S.beta[i];
            float rb = 0.f;
#pragma unroll
            for (int j8 = 0; j8 < 32; j8 += 8) {
                float x[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    int j = c0 + j8 + t;
                    float e = 0.f;
                    if (j < i) {
                        float L = expf(gi - S.gam[j]);
                        float dA = -a[j8 + t];
                        rb += dA * L * kk[j8 + t];
                        e = bi * L * dA;
                    }
                    x[t] = e;
                }
                tc::st_tile8(Es, i, c0 + j8, CT, x);
            }
            S.db_a[c0 >> 5][i] = rb;
        }
    }
    publish_tiles();

    // ---------------- phase 5: dk_Ar^T = K^T E^T (+), dk_Ac^T = K^T E (-)
    if (tid == 0 && !lost) {
        tc::gemm(tm + R_DKAR, sK, DT, true, sE, CT, false, 128, 64, CT, false);
        tc::gemm(tm + R_DKAC, sK, DT, true, sE, CT, true, 128, 64, CT, false);
    }
    if (!lost) finish_phase();
    if (!lost) {
        float a[32], b[32];
        tc::ld32(tc::taddr(tm, R_DKAR + c0), a);
        tc::ld32(tc::taddr(tm, R_DKAC + c0), b);
#pragma unroll
        for (int t = 0; t < 32; ++t) {
            dk[t] += a[t] + b[t];
            dg[t] += kreg[t] * (a[t] - b[t]);
        }
#pragma unroll
        for (int t = 0; t < 32; ++t) {
            int j = c0 + t;
            if (j < len && k < P.K) {
                if (P.G == 1)
                    store_scalar(P.dk, ((size_t)(ci.tok0 + j) * P.Hk + hk) * P.K + k, dk[t], P.dqdk_dtype);
                else
                    P.dk_h[((size_t)(ci.tok0 + j) * P.Hv + hv) * P.K + k] = dk[t];
            }
        }
        // gate gradient: column sums over the feature rows
        S.dg_q[q][c0 + lane] = tc::warp_transpose_sum32(dg);
        // last row: Gamma_C <S_0, dS_next> (this warp's half of the v range) + sum_j k_j (.) dk_SC_j
        float hd = 0.f;
        {
            // <S_0, dS_next> over the whole tile: warp w takes the 8-column chunk 4 (w % 4) + lane / 8 over
            // rows 64 (w / 4) .. +63; a quarter-warp reads the 8 rows of one core matrix (no bank conflicts)
            const int cc8 = 8 * (4 * (wid & 3) + (lane >> 3));
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t off = tc::tile_off(64 * (wid >> 2) + 8 * j + (lane & 7), cc8, DT);
                const __half2 *a2 = reinterpret_cast<const __half2 *>(S.H + off);
                const __half2 *b2 = reinterpret_cast<const __half2 *>(S.dH + off);
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    float2 a = __half22float2(a2[t]), b = __half22float2(b2[t]);
                    hd += a.x * b.x + a.y * b.y;
                }
            }
        }
        float tot = lastpart + S.G[rl] * hd;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
        if (lane == 0) S.last_w[wid] = tot;
    }
    tc::fence_before();
    __syncthreads();
    if (lost) {
        if (tid == 0) flag_status(P.status, ST_TIMEOUT);
    } else if (tid < CT) {
        float x = (S.dg_q[0][tid] + S.dg_q[1][tid]) + (S.dg_q[2][tid] + S.dg_q[3][tid]);
        if (tid == rl) {
            float l = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) l += S.last_w[w];
            x += l;
        }
        P.dgam[u * CT + tid] = tid < len ? x : 0.f;
        float b = (S.db_tdu[0][tid] + S.db_tdu[1][tid]) + (S.db_tdu[2][tid] + S.db_tdu[3][tid]);
        b += (S.db_tdw[0][tid] + S.db_tdw[1][tid]) + (S.db_tdw[2][tid] + S.db_tdw[3][tid]);
        b += S.db_a[0][tid] + S.db_a[1][tid];
        if (tid < len) P.dbeta[(size_t)(ci.tok0 + tid) * P.Hv + hv] = b;
    }
    if (wid == 0) {
        tc::fence_after();
        tc::tmem_dealloc(tm, K4T_TMEM_COLS);
    }
}

template <typename Tin>
static cudaError_t launch_k4_tc_t(const Params &P, cudaStream_t stream) {
    size_t smem = sizeof(K4TSmem);
    cudaError_t e = cudaFuncSetAttribute(k4_intra_grad_tc<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(P.max_chunks, P.Hv);
    k4_intra_grad_tc<Tin><<<grid, K4T_THREADS, smem, stream>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_k4_tc(const Params &P, cudaStream_t stream) {
    if (P.qkv_dtype == F32) return launch_k4_tc_t<float>(P, stream);
    if (P.qkv_dtype == BF16) return launch_k4_tc_t<__nv_bfloat16>(P, stream);
    return launch_k4_tc_t<__half>(P, stream);
}

}  // namespace gdr
