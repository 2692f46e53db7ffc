// k23_combine.cu -- exact combination of the per-segment scan summaries (fp32).
//
// Forward:  S_entry(0) = h0,                  S_entry(s+1) = S_entry(s) Phi_s + E_s
// Backward: dS_exit(last) = dht,              dS_exit(s-1) = dS_exit(s) Phi_s^T + F_s
// where E_s / F_s are the segment's zero-initialised local scans and Phi_s the product of its chunk
// transitions (k2_scan_tc.cu, k3_scan_tc.cu).  Rows of the state are independent, so a CTA owns 16 rows
// of one sequence x head; it walks the segments serially (only a handful per sequence).
#include "gdr_common.cuh"
#include "gdr_kernels.h"

namespace gdr {

constexpr int CB_THREADS = 256;
constexpr int CB_ROWS = 16;
constexpr int CB_LD = DT + 4;  // fp32 pitch of the transition tile (16-byte aligned rows)

template <bool FWD>
__global__ void __launch_bounds__(CB_THREADS) k23_combine(const Params P) {
    __shared__ __align__(16) float X[CB_ROWS][DT];
    extern __shared__ __align__(16) float Ph[];  // [DT][CB_LD]: Phi (forward) or Phi^T (backward)
    if (*P.status & ST_BAD_SEQLENS) return;
    const int s = blockIdx.x / P.Hv, hv = blockIdx.x % P.Hv, r0 = blockIdx.y * CB_ROWS;
    int bos, eos;
    seq_range(P, s, bos, eos);
    const int nc = (eos - bos + P.BT - 1) / P.BT;
    const int nss = (nc + P.Lseg - 1) / P.Lseg;  // segments holding chunks
    if (nss == 0) return;
    const int tid = threadIdx.x;
    const int r = tid / 16, k0 = (tid % 16) * 8;
    const size_t su0 = ((size_t)s * P.Hv + hv) * P.NS;
    float *out = FWD ? P.segSin : P.segdS;
    const float *init = FWD ? P.h0 : P.dht;

    // starting rows: h0 / dht (absent = 0)
    for (int e = tid; e < CB_ROWS * DT; e += CB_THREADS) {
        int rr = e / DT, k = e % DT, v = r0 + rr;
        float x = 0.f;
        if (init && v < P.V && k < P.K) x = init[(((size_t)s * P.Hv + hv) * P.V + v) * P.K + k];
        X[rr][k] = x;
    }
    __syncthreads();
    const int first = FWD ? 0 : nss - 1;
    for (int e = tid; e < CB_ROWS * DT; e += CB_THREADS) out[(su0 + first) * DT * DT + (size_t)(r0 + e / DT) * DT + e % DT] = X[e / DT][e % DT];

    for (int step = 0; step < nss - 1; ++step) {
        const int sg = FWD ? step : nss - 1 - step;          // segment whose summary is applied
        const int dst = FWD ? sg + 1 : sg - 1;
        const float *phi = P.segPhi + (su0 + sg) * DT * DT;
        const float *add = (FWD ? P.segE : P.segF) + (su0 + sg) * DT * DT;
        if (FWD) {
            for (int e = tid; e < DT * DT / 4; e += CB_THREADS) {
                int j = e / (DT / 4), k4 = (e % (DT / 4)) * 4;
                *reinterpret_cast<float4 *>(&Ph[j * CB_LD + k4]) = *reinterpret_cast<const float4 *>(phi + (size_t)j * DT + k4);
            }
        } else {
            for (int e = tid; e < DT * DT; e += CB_THREADS) {
                int k = e / DT, j = e % DT;  // read Phi[k][j] coalesced, store transposed
                Ph[j * CB_LD + k] = phi[(size_t)k * DT + j];
            }
        }
        __syncthreads();
        float y[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) y[t] = add[(size_t)(r0 + r) * DT + k0 + t];
        for (int j = 0; j < DT; ++j) {
            const float x = X[r][j];
            const float4 a = *reinterpret_cast<const float4 *>(&Ph[j * CB_LD + k0]);
            const float4 b = *reinterpret_cast<const float4 *>(&Ph[j * CB_LD + k0 + 4]);
            y[0] += x * a.x; y[1] += x * a.y; y[2] += x * a.z; y[3] += x * a.w;
            y[4] += x * b.x; y[5] += x * b.y; y[6] += x * b.z; y[7] += x * b.w;
        }
        __syncthreads();  // everyone done reading X and Ph
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            X[r][k0 + t] = y[t];
            out[(su0 + dst) * DT * DT + (size_t)(r0 + r) * DT + k0 + t] = y[t];
        }
        __syncthreads();
    }
}

cudaError_t launch_k23_combine(const Params &P, bool fwd, cudaStream_t stream) {
    size_t smem = sizeof(float) * DT * CB_LD;
    cudaError_t e;
    dim3 grid(P.N * P.Hv, DT / CB_ROWS);
    if (fwd) {
        e = cudaFuncSetAttribute(k23_combine<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        k23_combine<true><<<grid, CB_THREADS, smem, stream>>>(P);
    } else {
        e = cudaFuncSetAttribute(k23_combine<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        k23_combine<false><<<grid, CB_THREADS, smem, stream>>>(P);
    }
    return cudaGetLastError();
}

}  // namespace gdr
