// k5_dg_reduce.cu -- closing step of the backward ("FlashQLA backward explained", section 1, step 4:
// the GQA group reduction and the reverse cumsum of dg).
//
// The chunk kernels produce the gradient of the chunk-local cumulative gate gamma_r = sum_{i<=r} g_i, so
// the gradient of the raw gate is its reverse cumulative sum inside the chunk,
//     dg_t = sum_{r >= t, r in the chunk} dgamma_r          (per key channel for the KDA gate),
// and with grouped-query attention each key head's dq / dk is the sum over the Hv / Hk value heads that
// read it.  One CTA per chunk x key head.
#include "gdr_common.cuh"
#include "gdr_kernels.h"

namespace gdr {

constexpr int K5_THREADS = 128;

template <bool PC>
__global__ void __launch_bounds__(K5_THREADS) k5_dg_reduce(const Params P) {
    if (*P.status & ST_BAD_SEQLENS) return;
    const int n = blockIdx.x, hk = blockIdx.y;
    ChunkInfo ci;
    if (!chunk_info(P, n, ci)) return;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int len = ci.len;

    // reverse cumsum of the gate gradient for each value head of this key head
    for (int hv = hk * P.G; hv < (hk + 1) * P.G; ++hv) {
        const size_t u = (size_t)n * P.Hv + hv;
        if (!PC) {
            if (wid == 0) {
                // lane l holds rows 2l, 2l+1; reverse inclusive scan over 64 rows
                float x0 = 2 * lane < len ? P.dgam[u * CT + 2 * lane] : 0.f;
                float x1 = 2 * lane + 1 < len ? P.dgam[u * CT + 2 * lane + 1] : 0.f;
                float s = x0 + x1;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    float y = __shfl_down_sync(0xffffffffu, s, o);
                    if (lane + o < 32) s += y;
                }
                // s = sum over pairs >= lane
                float r1 = s - x0;  // rows >= 2l+1
                if (2 * lane < len) P.dg[(size_t)(ci.tok0 + 2 * lane) * P.Hv + hv] = s;
                if (2 * lane + 1 < len) P.dg[(size_t)(ci.tok0 + 2 * lane + 1) * P.Hv + hv] = r1;
            }
        } else {
            for (int c = tid; c < P.K; c += K5_THREADS) {
                float run = 0.f;
                for (int r = len - 1; r >= 0; --r) {
                    run += P.dgam[(u * CT + r) * DT + c];
                    P.dg[((size_t)(ci.tok0 + r) * P.Hv + hv) * P.K + c] = run;
                }
            }
        }
    }
    // GQA: dq[t, hk] = sum over the group's value heads (only when Hv > Hk)
    if (P.G > 1) {
        for (int e = tid; e < len * P.K; e += K5_THREADS) {
            int r = e / P.K, c = e % P.K;
            size_t t = (size_t)ci.tok0 + r;
            float sq = 0.f, sk = 0.f;
            for (int hv = hk * P.G; hv < (hk + 1) * P.G; ++hv) {
                sq += P.dq_h[(t * P.Hv + hv) * P.K + c];
                sk += P.dk_h[(t * P.Hv + hv) * P.K + c];
            }
            store_scalar(P.dq, (t * P.Hk + hk) * P.K + c, sq, P.dqdk_dtype);
            store_scalar(P.dk, (t * P.Hk + hk) * P.K + c, sk, P.dqdk_dtype);
        }
    }
}

cudaError_t launch_k5(const Params &P, cudaStream_t stream) {
    dim3 grid(P.max_chunks, P.Hk);
    if (P.per_channel) k5_dg_reduce<true><<<grid, K5_THREADS, 0, stream>>>(P);
    else k5_dg_reduce<false><<<grid, K5_THREADS, 0, stream>>>(P);
    return cudaGetLastError();
}

}  // namespace gdr
