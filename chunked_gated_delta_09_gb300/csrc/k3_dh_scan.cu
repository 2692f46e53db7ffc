// k3_dh_scan.cu -- reverse scan of the state gradient, serial over the chunks of each sequence.
//
// The adjoint of the state walks the chunks from last to first ("FlashQLA backward explained",
// section 2: the state-gradient recursion dS <- g_last dS + Q^T (dO g) - K^T (dV g), accumulated into
// dh0; section 1: dh0 is accumulated in fp32, dht is optional and absent means zero).  With
// D = scale dO, Aqk = M (.) Q K^T and the WY factor W of the chunk:
//     dh_n   = dS                                      (adjoint of the state leaving chunk n)
//     dV_new = Aqk^T D + (K (.) exp(gamma_C - gamma)) dS^T          (C x V)
//     dS    <- Gamma_C dS + D^T (Q (.) Gamma) - dV_new^T W           (KDA: dS diag(Gamma_C) + ...)
// and dh0 is the dS left after the first chunk.  As in the forward scan, rows of dS (the V index)
// are independent, so a CTA owns a BV-wide slice of V and keeps dS^T (K x BV) in fp32 registers.
#include "gdr_common.cuh"
#include "gdr_kernels.h"

namespace gdr {

constexpr int K3_THREADS = 128;

template <int BV>
struct ScanLd3 {
    static constexpr int value = BV == 8 ? 24 : BV + 8;
};

template <typename Tin, int BV, bool PC>
__global__ void __launch_bounds__(K3_THREADS) k3_dh_scan(const Params P, int nvt) {
    constexpr int LDB = ScanLd3<BV>::value;
    constexpr int NT = BV / 8;
    constexpr int DV8 = CT * (BV / 8);                  // 8-element vectors in one D slice
    constexpr int DREG = (DV8 + K3_THREADS - 1) / K3_THREADS;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __half *Ws = reinterpret_cast<__half *>(smem_raw);  // [2][CT][LDD]
    __half *Kts = Ws + 2 * CT * LDD;                    // [2][CT][LDD]
    __half *Qgs = Kts + 2 * CT * LDD;                   // [2][CT][LDD]
    __half *Aqs = Qgs + 2 * CT * LDD;                   // [2][CT][LDC]
    __half *Ds = Aqs + 2 * CT * LDC;                    // [2][CT][LDB]  scale * dO slice
    __half *dSts = Ds + 2 * CT * LDB;                   // [DT][LDB]
    __half *dVs = dSts + DT * LDB;                      // [CT][LDB]   -dV_new slice
    float *gC = reinterpret_cast<float *>(dVs + CT * LDB);  // [2][DT]

    if (*P.status & ST_BAD_SEQLENS) return;
    const int vt = blockIdx.x % nvt, hv = (blockIdx.x / nvt) % P.Hv, s = blockIdx.x / (nvt * P.Hv);
    const int v0 = vt * BV;
    const int tid = threadIdx.x, wid = tid >> 5;
    int bos, eos;
    seq_range(P, s, bos, eos);
    const int nc = (eos - bos + P.BT - 1) / P.BT;
    const int base = seq_chunk_base(P, s);
    const Tin *dOp = reinterpret_cast<const Tin *>(P.dO);

    float acc[2][NT][4];
    const int m0 = wid * 32;
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                int kk = acc_row(m0, mt, e), vv = v0 + acc_col(0, nt, e);
                float x = 0.f;
                if (P.dht && kk < P.K && vv < P.V) x = P.dht[(((size_t)s * P.Hv + hv) * P.V + vv) * P.K + kk];
                acc[mt][nt][e] = x;
            }

    // D slice prefetch through registers (it needs a dtype conversion, so no cp.async)
    float dreg[DREG][8];
    auto load_d = [&](int c) {
        int tok0 = bos + c * P.BT;
        int len = eos - tok0;
        len = len < P.BT ? len : P.BT;
#pragma unroll
        for (int i = 0; i < DREG; ++i) {
            int e = tid + i * K3_THREADS;
            int r = e / (BV / 8), c8 = (e % (BV / 8)) * 8;
            bool ok = e < DV8 && r < len;
            if (ok && v0 + c8 + 8 <= P.V) {
                load8(dOp + ((size_t)(tok0 + r) * P.Hv + hv) * P.V + v0 + c8, dreg[i]);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    dreg[i][j] = (ok && v0 + c8 + j < P.V) ? to_f32(dOp[((size_t)(tok0 + r) * P.Hv + hv) * P.V + v0 + c8 + j]) : 0.f;
            }
        }
    };
    auto store_d = [&](int buf) {
#pragma unroll
        for (int i = 0; i < DREG; ++i) {
            int e = tid + i * K3_THREADS;
            if (e < DV8) {
                int r = e / (BV / 8), c8 = (e % (BV / 8)) * 8;
                float x[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) x[j] = dreg[i][j] * P.scale;
                *reinterpret_cast<uint4 *>(Ds + buf * CT * LDB + r * LDB + c8) = pack8_half(x);
            }
        }
    };
    auto issue = [&](int c, int buf) {
        const size_t u = (size_t)(base + c) * P.Hv + hv;
        cp_block_f16(Ws + buf * CT * LDD, LDD, P.W + u * CT * DT, CT, DT, tid, K3_THREADS);
        cp_block_f16(Kts + buf * CT * LDD, LDD, P.Kt + u * CT * DT, CT, DT, tid, K3_THREADS);
        cp_block_f16(Qgs + buf * CT * LDD, LDD, P.Qg + u * CT * DT, CT, DT, tid, K3_THREADS);
        cp_block_f16(Aqs + buf * CT * LDC, LDC, P.Aqk + u * CT * CT, CT, CT, tid, K3_THREADS);
        int len = eos - (bos + c * P.BT);
        len = len < P.BT ? len : P.BT;
        if (PC) {
            for (int e = tid; e < DT; e += K3_THREADS) gC[buf * DT + e] = P.gam[(u * CT + len - 1) * DT + e];
        } else if (tid == 0) {
            gC[buf * DT] = P.gam[u * CT + len - 1];
        }
        cp_async_commit();
    };

    if (nc > 0) {
        load_d(nc - 1);
        store_d((nc - 1) & 1);
        issue(nc - 1, (nc - 1) & 1);
    }
    for (int c = nc - 1; c >= 0; --c) {
        const int buf = c & 1;
        const size_t u = (size_t)(base + c) * P.Hv + hv;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    dSts[acc_row(m0, mt, e) * LDB + acc_col(0, nt, e)] = __float2half_rn(acc[mt][nt][e]);
        cp_async_wait<0>();
        __syncthreads();
        if (c > 0) {
            issue(c - 1, buf ^ 1);
            load_d(c - 1);
        }
        {
            __half *dhg = P.dh + u * DT * DT;
            for (int e = tid; e < BV * DT; e += K3_THREADS) {
                int vv = e / DT, kk = e % DT;
                dhg[(size_t)(v0 + vv) * DT + kk] = dSts[kk * LDB + vv];
            }
        }
        // dV_new = Aqk^T D + K~ dS^T
        {
            float dv[1][NT][4];
            zero_acc(dv);
            warp_mma<1, NT, true, false>(dv, Aqs + buf * CT * LDC, LDC, Ds + buf * CT * LDB, LDB, wid * 16, 0, CT);
            warp_mma<1, NT, false, false>(dv, Kts + buf * CT * LDD, LDD, dSts, LDB, wid * 16, 0, DT);
            __half *dvg = P.dVn + u * CT * DT;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    int r = acc_row(wid * 16, 0, e), cc = acc_col(0, nt, e);
                    *reinterpret_cast<__half2 *>(dvg + (size_t)r * DT + v0 + cc) =
                        __floats2half2_rn(dv[0][nt][e], dv[0][nt][e + 1]);
                    *reinterpret_cast<__half2 *>(dVs + r * LDB + cc) = __floats2half2_rn(-dv[0][nt][e], -dv[0][nt][e + 1]);
                }
        }
        __syncthreads();
        // dS^T <- Gamma_C dS^T + (Q Gamma)^T D - W^T dV_new
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float G = expf(PC ? gC[buf * DT + acc_row(m0, mt, e)] : gC[buf * DT]);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) acc[mt][nt][e] *= G;
            }
        warp_mma<2, NT, true, false>(acc, Qgs + buf * CT * LDD, LDD, Ds + buf * CT * LDB, LDB, m0, 0, CT);
        warp_mma<2, NT, true, false>(acc, Ws + buf * CT * LDD, LDD, dVs, LDB, m0, 0, CT);
        if (c > 0) store_d(buf ^ 1);
    }
    if (P.dh0) {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    int kk = acc_row(m0, mt, e), vv = v0 + acc_col(0, nt, e);
                    if (kk < P.K && vv < P.V) P.dh0[(((size_t)s * P.Hv + hv) * P.V + vv) * P.K + kk] = acc[mt][nt][e];
                }
    }
}

template <typename Tin, int BV, bool PC>
static cudaError_t launch_k3_t(const Params &P, cudaStream_t stream) {
    constexpr int LDB = ScanLd3<BV>::value;
    size_t smem = sizeof(__half) * (6 * CT * LDD + 2 * CT * LDC + 2 * CT * LDB + DT * LDB + CT * LDB) +
                  sizeof(float) * 2 * DT;
    cudaError_t e = cudaFuncSetAttribute(k3_dh_scan<Tin, BV, PC>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int nvt = DT / BV;
    k3_dh_scan<Tin, BV, PC><<<P.N * P.Hv * nvt, K3_THREADS, smem, stream>>>(P, nvt);
    return cudaGetLastError();
}

template <typename Tin>
static cudaError_t launch_k3_d(const Params &P, int bv, cudaStream_t stream) {
    switch (bv) {
        case 8: return P.per_channel ? launch_k3_t<Tin, 8, true>(P, stream) : launch_k3_t<Tin, 8, false>(P, stream);
        case 16: return P.per_channel ? launch_k3_t<Tin, 16, true>(P, stream) : launch_k3_t<Tin, 16, false>(P, stream);
        case 32: return P.per_channel ? launch_k3_t<Tin, 32, true>(P, stream) : launch_k3_t<Tin, 32, false>(P, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_k3(const Params &P, int bv, cudaStream_t stream) {
    if (P.qkv_dtype == F32) return launch_k3_d<float>(P, bv, stream);
    if (P.qkv_dtype == BF16) return launch_k3_d<__nv_bfloat16>(P, bv, stream);
    return launch_k3_d<__half>(P, bv, stream);
}

}  // namespace gdr
