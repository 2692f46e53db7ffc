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
    constexpr int EPC = 16 / sizeof(Tin);              // input elements per 16-byte copy
    constexpr int DCH = CT * (BV / EPC);                // 16-byte copies per raw dO slice
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __half *Ws = reinterpret_cast<__half *>(smem_raw);  // [2][CT][LDD]
    __half *Kts = Ws + 2 * CT * LDD;                    // [2][CT][LDD]
    __half *Qgs = Kts + 2 * CT * LDD;                   // [2][CT][LDD]
    __half *Aqs = Qgs + 2 * CT * LDD;                   // [2][CT][LDC]
    __half *Ds = Aqs + 2 * CT * LDC;                    // [2][CT][LDB]  scale * dO slice
    __half *dSts = Ds + 2 * CT * LDB;                   // [DT][LDB]
    __half *dVs = dSts + DT * LDB;                      // [CT][LDB]   -dV_new slice
    float *gC = reinterpret_cast<float *>(dVs + CT * LDB);  // [2][DT]
    Tin *Draw = reinterpret_cast<Tin *>(gC + 2 * DT);        // [2][CT][BV] raw dO slice

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

    // raw dO slice: one 16-byte copy per (row, EPC columns); rows past the chunk or columns past V zero-fill
    auto issue_d = [&](int c, int buf) {
        int tok0 = bos + c * P.BT;
        int len = eos - tok0;
        len = len < P.BT ? len : P.BT;
        for (int e = tid; e < DCH; e += K3_THREADS) {
            int r = e / (BV / EPC), cc = (e % (BV / EPC)) * EPC;
            bool ok = r < len && v0 + cc + EPC <= P.V;
            const Tin *src = ok ? dOp + ((size_t)(tok0 + r) * P.Hv + hv) * P.V + v0 + cc : dOp;
            cp_async16_zfill(Draw + (buf * CT + r) * BV + cc, src, ok ? 16 : 0);
        }
    };
    // scale and convert the copies this thread made (visible to it after its own wait)
    auto convert_d = [&](int buf) {
        for (int e = tid; e < DCH; e += K3_THREADS) {
            int r = e / (BV / EPC), cc = (e % (BV / EPC)) * EPC;
            const Tin *src = Draw + (buf * CT + r) * BV + cc;
            __half *dst = Ds + buf * CT * LDB + r * LDB + cc;
#pragma unroll
            for (int j = 0; j < EPC; j += 2)
                *reinterpret_cast<__half2 *>(dst + j) =
                    __floats2half2_rn(to_f32(src[j]) * P.scale, to_f32(src[j + 1]) * P.scale);
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
            for (int e = tid; e < DT / 4; e += K3_THREADS)
                cp_async16(gC + buf * DT + 4 * e, P.gam + (u * CT + len - 1) * DT + 4 * e);
        } else if (tid == 0) {
            cp_async4(gC + buf * DT, P.gam + u * CT + len - 1);
        }
        issue_d(c, buf);
        cp_async_commit();
    };

    if (nc > 0) {
        issue(nc - 1, (nc - 1) & 1);
        cp_async_wait<0>();
        convert_d((nc - 1) & 1);
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
        __syncthreads();  // chunk c's operands (waited for and converted at the end of the previous step)
        if (c > 0) issue(c - 1, buf ^ 1);
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
        if (c > 0) {
            cp_async_wait<0>();
            convert_d(buf ^ 1);
        }
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
                  sizeof(float) * 2 * DT + sizeof(Tin) * 2 * CT * BV;
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
