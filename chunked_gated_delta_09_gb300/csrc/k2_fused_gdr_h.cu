// k2_fused_gdr_h.cu -- forward state recompute, serial over the chunks of each sequence.
//
// The backward needs the state entering every chunk ("FlashQLA backward explained", section 1, step 2:
// fused_gdr_h rebuilds the forward's chunk states h, which MindSpeed-Ops chunk_kda_bwd.md lists as
// h [B, NT, H, K, V] fp32 "chunk state").  With the WY factors of the chunk,
//     h_n   = S_0
//     V_new = U - W S_0^T                                  (C x V)
//     S_C   = Gamma_C S_0 + V_new^T (K (.) exp(gamma_C - gamma))     (KDA: S_0 diag(Gamma_C) + ...)
// The rows of S (the V index) evolve independently, so a CTA owns a BV-wide slice of V and the grid
// is sequences x value heads x V / BV.  The CTA keeps S^T (K x BV) in fp32 registers as tensor-core
// accumulators and prefetches the next chunk's W, K~ and U slice with cp.async while it works.
#include "gdr_common.cuh"
#include "gdr_kernels.h"

namespace gdr {

constexpr int K2_THREADS = 128;

template <int BV>
struct ScanLd {
    static constexpr int value = BV == 8 ? 24 : BV + 8;  // bank-conflict-free pitch of a [*][BV] tile
};

template <int BV, bool PC>
__global__ void __launch_bounds__(K2_THREADS) k2_fused_gdr_h(const Params P, int nvt) {
    constexpr int LDB = ScanLd<BV>::value;
    constexpr int NT = BV / 8;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __half *Ws = reinterpret_cast<__half *>(smem_raw);   // [2][CT][LDD]
    __half *Kts = Ws + 2 * CT * LDD;                     // [2][CT][LDD]
    __half *Us = Kts + 2 * CT * LDD;                     // [2][CT][LDB]
    __half *Sts = Us + 2 * CT * LDB;                     // [DT][LDB]  S^T as fp16
    __half *Vns = Sts + DT * LDB;                        // [CT][LDB]  V_new slice
    float *gC = reinterpret_cast<float *>(Vns + CT * LDB);  // [2][DT] gate of the chunk's last row

    if (*P.status & ST_BAD_SEQLENS) return;
    const int vt = blockIdx.x % nvt, hv = (blockIdx.x / nvt) % P.Hv, s = blockIdx.x / (nvt * P.Hv);
    const int v0 = vt * BV;
    const int tid = threadIdx.x, wid = tid >> 5;
    int bos, eos;
    seq_range(P, s, bos, eos);
    const int nc = (eos - bos + P.BT - 1) / P.BT;
    const int base = seq_chunk_base(P, s);

    // S^T accumulators: warp w owns rows (k) 32w .. 32w+31, all BV columns (v)
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
                if (P.h0 && kk < P.K && vv < P.V) x = P.h0[(((size_t)s * P.Hv + hv) * P.V + vv) * P.K + kk];
                acc[mt][nt][e] = x;
            }

    auto issue = [&](int c, int buf) {
        const size_t u = (size_t)(base + c) * P.Hv + hv;
        cp_block_f16(Ws + buf * CT * LDD, LDD, P.W + u * CT * DT, CT, DT, tid, K2_THREADS);
        cp_block_f16(Kts + buf * CT * LDD, LDD, P.Kt + u * CT * DT, CT, DT, tid, K2_THREADS);
        // U slice: CT rows of BV halves
        for (int e = tid; e < CT * (BV / 8); e += K2_THREADS) {
            int r = e / (BV / 8), c8 = (e % (BV / 8)) * 8;
            cp_async16(Us + buf * CT * LDB + r * LDB + c8, P.U + u * CT * DT + r * DT + v0 + c8);
        }
        int len = eos - (bos + c * P.BT);
        len = len < P.BT ? len : P.BT;
        if (PC) {
            for (int e = tid; e < DT / 4; e += K2_THREADS)
                cp_async16(gC + buf * DT + 4 * e, P.gam + (u * CT + len - 1) * DT + 4 * e);
        } else if (tid == 0) {
            cp_async4(gC + buf * DT, P.gam + u * CT + len - 1);
        }
        cp_async_commit();
    };

    if (nc > 0) {
        issue(0, 0);
        cp_async_wait<0>();
    }
    for (int c = 0; c < nc; ++c) {
        const int buf = c & 1;
        const size_t u = (size_t)(base + c) * P.Hv + hv;
        // S^T -> fp16 shared copy (operand of the V_new product and source of h_n)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) Sts[acc_row(m0, mt, e) * LDB + acc_col(0, nt, e)] = __float2half_rn(acc[mt][nt][e]);
        __syncthreads();  // chunk c's operands (waited for at the end of the previous step) and S^T visible
        if (c + 1 < nc) issue(c + 1, buf ^ 1);
        // h_n[v][k] for this V slice (coalesced along k)
        {
            __half *hg = P.h + u * DT * DT;
            for (int e = tid; e < BV * DT; e += K2_THREADS) {
                int vv = e / DT, kk = e % DT;
                hg[(size_t)(v0 + vv) * DT + kk] = Sts[kk * LDB + vv];
            }
        }
        // V_new = U - W S^T : warp w owns token rows 16w .. 16w+15
        {
            float vn[1][NT][4];
            zero_acc(vn);
            warp_mma<1, NT, false, false>(vn, Ws + buf * CT * LDD, LDD, Sts, LDB, wid * 16, 0, DT);
            __half *vng = P.Vn + u * CT * DT;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    int r = acc_row(wid * 16, 0, e), cc = acc_col(0, nt, e);
                    const __half *up = Us + buf * CT * LDB + r * LDB + cc;
                    __half2 val = __floats2half2_rn(__half2float(up[0]) - vn[0][nt][e],
                                                    __half2float(up[1]) - vn[0][nt][e + 1]);
                    *reinterpret_cast<__half2 *>(Vns + r * LDB + cc) = val;
                    *reinterpret_cast<__half2 *>(vng + (size_t)r * DT + v0 + cc) = val;
                }
        }
        __syncthreads();
        // S^T <- Gamma_C S^T + K~^T V_new
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float G = expf(PC ? gC[buf * DT + acc_row(m0, mt, e)] : gC[buf * DT]);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) acc[mt][nt][e] *= G;
            }
        warp_mma<2, NT, true, false>(acc, Kts + buf * CT * LDD, LDD, Vns, LDB, m0, 0, CT);
        if (c + 1 < nc) cp_async_wait<0>();  // chunk c+1's operands landed (this thread's copies)
    }
}

template <int BV, bool PC>
static cudaError_t launch_k2_t(const Params &P, cudaStream_t stream) {
    constexpr int LDB = ScanLd<BV>::value;
    size_t smem = sizeof(__half) * (4 * CT * LDD + 2 * CT * LDB + DT * LDB + CT * LDB) + sizeof(float) * 2 * DT;
    cudaError_t e = cudaFuncSetAttribute(k2_fused_gdr_h<BV, PC>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int nvt = DT / BV;
    k2_fused_gdr_h<BV, PC><<<P.N * P.Hv * nvt, K2_THREADS, smem, stream>>>(P, nvt);
    return cudaGetLastError();
}

cudaError_t launch_k2(const Params &P, int bv, cudaStream_t stream) {
    switch (bv) {
        case 8: return P.per_channel ? launch_k2_t<8, true>(P, stream) : launch_k2_t<8, false>(P, stream);
        case 16: return P.per_channel ? launch_k2_t<16, true>(P, stream) : launch_k2_t<16, false>(P, stream);
        case 32: return P.per_channel ? launch_k2_t<32, true>(P, stream) : launch_k2_t<32, false>(P, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdr
