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

// four consecutive outputs (index i a multiple of 4 in a 16-byte aligned array): one 8- or 16-byte store
__device__ __forceinline__ void store4(void *p, size_t i, float4 x, int dt) {
    if (dt == F32) {
        *reinterpret_cast<float4 *>(reinterpret_cast<float *>(p) + i) = x;
    } else if (dt == BF16) {
        __nv_bfloat162 v[2] = {__floats2bfloat162_rn(x.x, x.y), __floats2bfloat162_rn(x.z, x.w)};
        *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(p) + i) = *reinterpret_cast<uint2 *>(v);
    } else {
        __half2 v[2] = {__floats2half2_rn(x.x, x.y), __floats2half2_rn(x.z, x.w)};
        *reinterpret_cast<uint2 *>(reinterpret_cast<__half *>(p) + i) = *reinterpret_cast<uint2 *>(v);
    }
}

// eight consecutive 16-bit values of type dt (one 16-byte load) as floats
__device__ __forceinline__ void load8_16(const char *p, int dt, float (&o)[8]) {
    if (dt == BF16) {
        Raw8<__nv_bfloat16> x;
        x.v = *reinterpret_cast<const uint4 *>(p);
        raw_get(x, o);
    } else {
        Raw8<__half> x;
        x.v = *reinterpret_cast<const uint4 *>(p);
        raw_get(x, o);
    }
}

template <bool PC>
__global__ void __launch_bounds__(K5_THREADS) k5_dg_reduce(const Params P) {
    if (*P.status & ST_BAD_SEQLENS) return;
    const int n = blockIdx.x, hk = blockIdx.y;
    ChunkInfo ci;
    if (!chunk_info(P, n, ci)) return;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int len = ci.len;
    __shared__ __align__(16) float dgt[PC ? CT : 1][DT];  // per-channel gate: one unit's d(gamma) rows

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
            // the unit's d(gamma) tile [CT][DT] (contiguous) into shared memory first, all loads in flight at
            // once, then one channel per thread walks the rows backwards over shared memory
            __syncthreads();  // (the previous head's readers are done with the tile)
            const float4 *src = reinterpret_cast<const float4 *>(P.dgam + u * CT * DT);
            for (int e = tid; e < len * (DT / 4); e += K5_THREADS) reinterpret_cast<float4 *>(&dgt[0][0])[e] = src[e];
            __syncthreads();
            for (int c = tid; c < P.K; c += K5_THREADS) {
                float run = 0.f;
                for (int r = len - 1; r >= 0; --r) {
                    run += dgt[r][c];
                    P.dg[((size_t)(ci.tok0 + r) * P.Hv + hv) * P.K + c] = run;
                }
            }
        }
    }
    // GQA: dq[t, hk] = sum over the group's value heads (when Hv > Hk and the gradient kernel wrote
    // per-value-head rows; the tcgen05 one sums in place), four channels per thread: the per-head rows are
    // aligned workspace rows (K a multiple of 8) in the output's type (fp32 for fp32 outputs, else the 16-bit
    // type), summed in fp32 in head order
    if (P.G > 1 && P.dq_h) {
        const int pdt = gqa_part_dtype(P);
        if (pdt == F32) {  // four channels per thread
            const int k4n = P.K / 4;
            for (int e = tid; e < len * k4n; e += K5_THREADS) {
                const int r = e / k4n, c = 4 * (e % k4n);
                const size_t t = (size_t)ci.tok0 + r;
                float4 sq = make_float4(0.f, 0.f, 0.f, 0.f), sk = sq;
                for (int hv = hk * P.G; hv < (hk + 1) * P.G; ++hv) {
                    const size_t i = (t * P.Hv + hv) * P.K + c;
                    const float4 a = *reinterpret_cast<const float4 *>(P.dq_h + i);
                    const float4 b = *reinterpret_cast<const float4 *>(P.dk_h + i);
                    sq.x += a.x, sq.y += a.y, sq.z += a.z, sq.w += a.w;
                    sk.x += b.x, sk.y += b.y, sk.z += b.z, sk.w += b.w;
                }
                store4(P.dq, (t * P.Hk + hk) * P.K + c, sq, P.dqdk_dtype);
                store4(P.dk, (t * P.Hk + hk) * P.K + c, sk, P.dqdk_dtype);
            }
        } else {  // 16-bit partials: eight channels (16 bytes) per thread
            const int k8n = P.K / 8;
            for (int e = tid; e < len * k8n; e += K5_THREADS) {
                const int r = e / k8n, c = 8 * (e % k8n);
                const size_t t = (size_t)ci.tok0 + r;
                float sq[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, sk[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                for (int hv = hk * P.G; hv < (hk + 1) * P.G; ++hv) {
                    const size_t i = (t * P.Hv + hv) * P.K + c;
                    float a[8], b[8];
                    load8_16(gqa_part(P.dq_h, i, P), pdt, a);
                    load8_16(gqa_part(P.dk_h, i, P), pdt, b);
#pragma unroll
                    for (int j = 0; j < 8; ++j) sq[j] += a[j], sk[j] += b[j];
                }
                store4(P.dq, (t * P.Hk + hk) * P.K + c, make_float4(sq[0], sq[1], sq[2], sq[3]), P.dqdk_dtype);
                store4(P.dq, (t * P.Hk + hk) * P.K + c + 4, make_float4(sq[4], sq[5], sq[6], sq[7]), P.dqdk_dtype);
                store4(P.dk, (t * P.Hk + hk) * P.K + c, make_float4(sk[0], sk[1], sk[2], sk[3]), P.dqdk_dtype);
                store4(P.dk, (t * P.Hk + hk) * P.K + c + 4, make_float4(sk[4], sk[5], sk[6], sk[7]), P.dqdk_dtype);
            }
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
