// k23_combine.cu -- exact combination of the per-segment scan summaries (fp32).
//
// Forward:  S_entry(0) = h0,                  S_entry(s+1) = S_entry(s) Phi_s + E_s
// Backward: dS_exit(last) = dht,              dS_exit(s-1) = dS_exit(s) Phi_s^T + F_s
// where E_s / F_s are the segment's zero-initialised local scans and Phi_s the product of its chunk
// transitions (k2_scan_tc.cu writes Phi_s and Phi_s^T, k3_scan_tc.cu writes F_s).  Rows of the state are
// independent, so a CTA owns CB_ROWS rows of one sequence x head (one wave of CTAs for the usual head
// counts) and walks the segments serially, prefetching the next segment's transition and summary rows
// with cp.async while it multiplies by the current ones.
#include "gdr_common.cuh"
#include "gdr_kernels.h"

namespace gdr {

constexpr int CB_THREADS = 1024;  // 16 rows x 32 column quads x 2 slices of the reduction
constexpr int CB_ROWS = 16;
constexpr int CB_LD = DT + 4;  // fp32 pitch of a transition tile (16-byte aligned rows)

template <bool FWD>
__global__ void __launch_bounds__(CB_THREADS) k23_combine(const Params P) {
    __shared__ __align__(16) float X[CB_ROWS][DT];
    __shared__ __align__(16) float part[CB_ROWS][DT];  // partial sums of reduction slice 1
    extern __shared__ __align__(16) float dyn[];         // Ph [2][DT][CB_LD], Ad [2][CB_ROWS][DT]
    float *Ph = dyn, *Ad = dyn + 2 * DT * CB_LD;
    if (*P.status & ST_BAD_SEQLENS) return;
    const int s = blockIdx.x / P.Hv, hv = blockIdx.x % P.Hv, r0 = blockIdx.y * CB_ROWS;
    int bos, eos;
    seq_range(P, s, bos, eos);
    const int nc = (eos - bos + P.BT - 1) / P.BT;
    const int nss = (nc + P.Lseg - 1) / P.Lseg;  // segments holding chunks
    if (nss == 0) return;
    const int tid = threadIdx.x;
    const int js = tid >> 9;                                         // reduction slice: j in [64 js, 64 js + 64)
    const int r = (tid >> 5) & (CB_ROWS - 1), k0 = (tid & 31) * 4;  // 4 outputs per thread
    const size_t su0 = ((size_t)s * P.Hv + hv) * P.NS;
    float *out = FWD ? P.segSin : P.segdS;
    const float *init = FWD ? P.h0 : P.dht;
    const float *trans = FWD ? P.segPhi : P.segPhiT;  // row j of the matrix applied on the right
    const float *adds = FWD ? P.segE : P.segF;

    // the next step's transition and summary rows, in flight while the current step multiplies
    auto prefetch = [&](int step, int buf) {
        const int sg = FWD ? step : nss - 1 - step;
        const float *src = trans + (su0 + sg) * DT * DT;
        float *dst = Ph + buf * DT * CB_LD;
        for (int e = tid; e < DT * DT / 4; e += CB_THREADS) {
            int j = e / (DT / 4), k4 = (e % (DT / 4)) * 4;
            cp_async16(dst + j * CB_LD + k4, src + (size_t)j * DT + k4);
        }
        const float *asrc = adds + (su0 + sg) * DT * DT + (size_t)r0 * DT;
        float *adst = Ad + buf * CB_ROWS * DT;
        for (int e = tid; e < CB_ROWS * DT / 4; e += CB_THREADS) cp_async16(adst + 4 * e, asrc + 4 * e);
        cp_async_commit();
    };
    if (nss > 1) prefetch(0, 0);
    // starting rows: h0 / dht (absent = 0)
    for (int e = tid; e < CB_ROWS * DT; e += CB_THREADS) {
        int rr = e / DT, k = e % DT, v = r0 + rr;
        float x = 0.f;
        if (init && v < P.V && k < P.K) x = init[(((size_t)s * P.Hv + hv) * P.V + v) * P.K + k];
        X[rr][k] = x;
        out[(su0 + (FWD ? 0 : nss - 1)) * DT * DT + (size_t)v * DT + k] = x;
    }
    for (int step = 0; step < nss - 1; ++step) {
        const int buf = step & 1;
        const int sg = FWD ? step : nss - 1 - step;  // segment whose summary is applied
        const int dst = FWD ? sg + 1 : sg - 1;
        cp_async_wait<0>();
        __syncthreads();  // transition and summary of this step and X visible; previous step's readers done
        if (step + 1 < nss - 1) prefetch(step + 1, buf ^ 1);
        const float *ph = Ph + buf * DT * CB_LD;
        float4 y = js == 0 ? *reinterpret_cast<const float4 *>(Ad + buf * CB_ROWS * DT + r * DT + k0)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
        for (int j = 64 * js; j < 64 * js + 64; ++j) {
            const float x = X[r][j];
            const float4 a = *reinterpret_cast<const float4 *>(&ph[j * CB_LD + k0]);
            y.x += x * a.x;
            y.y += x * a.y;
            y.z += x * a.z;
            y.w += x * a.w;
        }
        if (js > 0) *reinterpret_cast<float4 *>(&part[r][k0]) = y;
        __syncthreads();  // partials written; everyone done reading X
        if (js == 0) {
            const float4 z = *reinterpret_cast<const float4 *>(&part[r][k0]);
            y.x += z.x;
            y.y += z.y;
            y.z += z.z;
            y.w += z.w;
            *reinterpret_cast<float4 *>(&X[r][k0]) = y;
            *reinterpret_cast<float4 *>(out + (su0 + dst) * DT * DT + (size_t)(r0 + r) * DT + k0) = y;
        }
    }
}

cudaError_t launch_k23_combine(const Params &P, bool fwd, cudaStream_t stream) {
    size_t smem = sizeof(float) * (2 * DT * CB_LD + 2 * CB_ROWS * DT);
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
