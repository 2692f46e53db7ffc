// k7_wy_inputs.cu -- inputs of the WY-gradient stage taken alone, as the per-chunk kernel's workspace tiles.
//
// The stage (MindSpeed-Ops chunk_kda_bwd.md: chunk_kda_bwd_wy_dqkg_fused) receives the chunk quantities
// that the full backward computes itself: the chunk-local cumulative gate g [T, H, K], the triangular matrix
// A [T, H, BT], the chunk states h and their gradients dh [NT, H, K, V] (fp32), V_new and its gradient dv
// [T, H, V], and dO.  One CTA per chunk x head writes them in the layout of the per-chunk gradient kernel:
// gamma [CT][DT] fp32 (rows past the chunk end repeat its last row, so in-chunk decays stay at most 1),
// T = A as a [r][i] tile, D = scale dO as a [r][v] tile, S_0 and dS_next as [v][k] tiles (transposed through
// shared memory), V_new^T and -dV_new^T as [v][c] tiles.  Padding is zero.
#include "gdr_common.cuh"
#include "gdr_kernels.h"
#include "tc_util.cuh"

namespace gdr {

constexpr int K7_THREADS = 256;

__device__ __forceinline__ float ld_any(const float *p) { return *p; }
__device__ __forceinline__ float ld_any(const __half *p) { return __half2float(*p); }
__device__ __forceinline__ float ld_any(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

// tile[b][a] (DT rows, C columns, fp16 core-matrix layout in shared memory) = mul * src[a * stride + b] for
// a < na, b < nb, zero elsewhere.  Consecutive threads take consecutive a (one source row each, 8 elements).
template <typename Ts>
__device__ void transpose_to_tile(unsigned char *tile, int C, const Ts *src, size_t stride, int na, int nb, float mul,
                                  int tid) {
    for (int e = tid; e < C * (DT / 8); e += K7_THREADS) {
        const int a = e % C, b8 = (e / C) * 8;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const int b = b8 + t;
            const float x = (a < na && b < nb) ? mul * ld_any(src + (size_t)a * stride + b) : 0.f;
            *reinterpret_cast<__half *>(tile + ctile_off(b, a, C)) = __float2half_rn(x);
        }
    }
}

// rows r < nr of a row-major source (columns < nc, times mul) as a [CT][C] fp16 tile in global memory
template <typename Ts>
__device__ void rows_to_tile(unsigned char *dst, int C, const Ts *src, size_t stride, int nr, int nc, float mul,
                             int tid) {
    for (int e = tid; e < CT * (C / 8); e += K7_THREADS) {
        const int r = e / (C / 8), c8 = (e % (C / 8)) * 8;
        float x[8];
#pragma unroll
        for (int t = 0; t < 8; ++t)
            x[t] = (r < nr && c8 + t < nc) ? mul * ld_any(src + (size_t)r * stride + c8 + t) : 0.f;
        *reinterpret_cast<uint4 *>(dst + ctile_off(r, c8, C)) = pack8_half(x);
    }
}

template <typename Tin>
__global__ void __launch_bounds__(K7_THREADS) k7_wy_inputs(const Params P, const Tin *A, const Tin *vnew,
                                                           const Tin *dvin, const float *h, const float *dh) {
    __shared__ __align__(16) unsigned char tile[DT * DT * 2];
    if (*P.status & ST_BAD_SEQLENS) return;
    const int n = blockIdx.x, hv = blockIdx.y;
    ChunkInfo ci;
    if (!chunk_info(P, n, ci)) return;
    const int tid = threadIdx.x, len = ci.len;
    const size_t u = (size_t)n * P.Hv + hv;

    // cumulative gate, rows past the end repeat the last row
    for (int e = tid; e < CT * DT; e += K7_THREADS) {
        const int r = e / DT, c = e % DT, rr = r < len ? r : len - 1;
        P.gam[u * CT * DT + e] = c < P.K ? P.g[((size_t)(ci.tok0 + rr) * P.Hv + hv) * P.K + c] : 0.f;
    }
    // T = A (the chunk's valid columns only) and D = scale dO
    rows_to_tile(reinterpret_cast<unsigned char *>(P.Tm + u * CT * CT), CT, A + ((size_t)ci.tok0 * P.Hv + hv) * P.BT,
                 (size_t)P.Hv * P.BT, len, len < P.BT ? len : P.BT, 1.f, tid);
    rows_to_tile(reinterpret_cast<unsigned char *>(P.Dt + u * CT * DT), DT,
                 reinterpret_cast<const Tin *>(P.dO) + ((size_t)ci.tok0 * P.Hv + hv) * P.V, (size_t)P.Hv * P.V, len,
                 P.V, P.scale, tid);
    // S_0 and dS_next: [K][V] fp32 per chunk -> [v][k] tiles
    for (int w = 0; w < 2; ++w) {
        const float *src = (w ? dh : h) + u * P.K * P.V;
        transpose_to_tile(tile, DT, src, (size_t)P.V, P.K, P.V, 1.f, tid);
        __syncthreads();
        uint4 *dst = reinterpret_cast<uint4 *>(w ? P.dh + u * DT * DT : P.h + u * DT * DT);
        for (int e = tid; e < DT * DT * 2 / 16; e += K7_THREADS) dst[e] = reinterpret_cast<const uint4 *>(tile)[e];
        __syncthreads();
    }
    // V_new^T and -dV_new^T: [c][v] rows -> [v][c] tiles
    for (int w = 0; w < 2; ++w) {
        const Tin *src = (w ? dvin : vnew) + ((size_t)ci.tok0 * P.Hv + hv) * P.V;
        transpose_to_tile(tile, CT, src, (size_t)P.Hv * P.V, len, P.V, w ? -1.f : 1.f, tid);
        __syncthreads();
        uint4 *dst = reinterpret_cast<uint4 *>(w ? P.dVn + u * DT * CT : P.Vn + u * DT * CT);
        for (int e = tid; e < DT * CT * 2 / 16; e += K7_THREADS) dst[e] = reinterpret_cast<const uint4 *>(tile)[e];
        __syncthreads();
    }
}

template <typename Tin>
static cudaError_t launch_k7_t(const Params &P, const void *A, const void *vnew, const void *dvin, const float *h,
                               const float *dh, cudaStream_t stream) {
    dim3 grid(P.max_chunks, P.Hv);
    k7_wy_inputs<Tin><<<grid, K7_THREADS, 0, stream>>>(P, reinterpret_cast<const Tin *>(A),
                                                       reinterpret_cast<const Tin *>(vnew),
                                                       reinterpret_cast<const Tin *>(dvin), h, dh);
    return cudaGetLastError();
}

cudaError_t launch_k7_wy_inputs(const Params &P, const void *A, const void *v_new, const void *dv_in, const float *h,
                                const float *dh, cudaStream_t stream) {
    if (P.qkv_dtype == F32) return launch_k7_t<float>(P, A, v_new, dv_in, h, dh, stream);
    if (P.qkv_dtype == BF16) return launch_k7_t<__nv_bfloat16>(P, A, v_new, dv_in, h, dh, stream);
    return launch_k7_t<__half>(P, A, v_new, dv_in, h, dh, stream);
}

}  // namespace gdr
