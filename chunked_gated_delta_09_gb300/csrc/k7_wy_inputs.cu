// k7_wy_inputs.cu -- inputs of the WY-gradient stage taken alone, as the per-chunk kernel's workspace tiles.
//
// The stage (MindSpeed-Ops chunk_kda_bwd.md: chunk_kda_bwd_wy_dqkg_fused) receives the chunk quantities
// that the full backward computes itself: the chunk-local cumulative gate g [T, H, K], the triangular matrix
// A [T, H, BT], the chunk states h and their gradients dh [NT, H, K, V] (fp32), V_new and its gradient dv
// [T, H, V], and dO.  Four CTAs per chunk x head (grid z: the gate, T and D; S_0; dS_next; V_new^T and
// -dV_new^T, about 60-100 KB of reads each, so that more reads are in flight per SM than one CTA's serial
// stages allow) write them in the layout of the per-chunk gradient kernel:
// gamma [CT][DT] fp32 (rows past the chunk end repeat its last row, so in-chunk decays stay at most 1),
// T = A as a [r][i] tile, D = scale dO as a [r][v] tile, S_0 and dS_next as [v][k] tiles (transposed through
// registers), V_new^T and -dV_new^T as [v][c] tiles.  Padding is zero.  No shared memory: every transposed
// tile row segment is assembled in a lane's registers from coalesced row reads and stored whole.
#include "gdr_common.cuh"
#include "gdr_kernels.h"
#include "tc_util.cuh"

namespace gdr {

constexpr int K7_THREADS = 256;
constexpr int K7_WARPS = K7_THREADS / 32;

__device__ __forceinline__ float ld_any(const float *p) { return *p; }
__device__ __forceinline__ float ld_any(const __half *p) { return __half2float(*p); }
__device__ __forceinline__ float ld_any(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

// 8 consecutive elements as floats: one 16-byte load for 16-bit types, two for fp32 (p 16-byte aligned)
__device__ __forceinline__ void ld8(const float *p, float (&x)[8]) {
    const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
    x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w, x[4] = b.x, x[5] = b.y, x[6] = b.z, x[7] = b.w;
}
template <typename T16>
__device__ __forceinline__ void ld8(const T16 *p, float (&x)[8]) {
    Raw8<T16> r;
    r.v = *reinterpret_cast<const uint4 *>(p);
    raw_get(r, x);
}

// Transposed tile: element (a, b) of a row-major source (rows a < na with row stride `stride` elements,
// columns b < nb) times mul goes to row b, column a of an fp16 core-matrix tile with DT rows and C columns;
// zero elsewhere.  A warp takes 8 source rows a0 .. a0 + 7 per step and lane l the columns b = l + 32 j
// (j < 4): every load instruction reads 32 consecutive elements of one row, and each lane then holds the
// 16-byte row segment (b, a0 .. a0 + 7) of the tile, so lanes 8m .. 8m + 7 store one whole core matrix.
template <typename Ts>
__device__ void transpose_to_tile(unsigned char *dst, int C, const Ts *src, size_t stride, int na, int nb, float mul,
                                  int wid, int lane) {
    for (int a0 = 8 * wid; a0 < C; a0 += 8 * K7_WARPS) {
        float x[4][8];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const int a = a0 + t;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int b = lane + 32 * j;
                x[j][t] = (a < na && b < nb) ? mul * ld_any(src + (size_t)a * stride + b) : 0.f;
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4 *>(dst + ctile_off(lane + 32 * j, a0, C)) = pack8_half(x[j]);
    }
}

// Rows r < nr of a row-major source (16-byte aligned rows; columns < nc, times mul) as a [CT][C] fp16 tile in
// global memory.  Consecutive threads take consecutive 8-column segments of a row (coalesced loads); a
// segment that crosses nc (only possible when nc is not a multiple of 8) is read element by element.
template <typename Ts>
__device__ void rows_to_tile(unsigned char *dst, int C, const Ts *src, size_t stride, int nr, int nc, float mul,
                             int tid) {
    for (int e = tid; e < CT * (C / 8); e += K7_THREADS) {
        const int r = e / (C / 8), c8 = (e % (C / 8)) * 8;
        float x[8];
        if (r < nr && c8 + 8 <= nc) {
            ld8(src + (size_t)r * stride + c8, x);
#pragma unroll
            for (int t = 0; t < 8; ++t) x[t] *= mul;
        } else {
#pragma unroll
            for (int t = 0; t < 8; ++t)
                x[t] = (r < nr && c8 + t < nc) ? mul * ld_any(src + (size_t)r * stride + c8 + t) : 0.f;
        }
        *reinterpret_cast<uint4 *>(dst + ctile_off(r, c8, C)) = pack8_half(x);
    }
}

template <typename Tin>
__global__ void __launch_bounds__(K7_THREADS) k7_wy_inputs(const Params P, const Tin *A, const Tin *vnew,
                                                           const Tin *dvin, const float *h, const float *dh) {
    if (*P.status & ST_BAD_SEQLENS) return;
    const int n = blockIdx.x, hv = blockIdx.y;
    ChunkInfo ci;
    if (!chunk_info(P, n, ci)) return;
    const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31, len = ci.len;
    const size_t u = (size_t)n * P.Hv + hv;
    const int part = blockIdx.z;

    if (part == 0) {
        // cumulative gate, rows past the end repeat the last row (g is only 4-byte aligned: scalar loads,
        // consecutive threads on consecutive channels; 16-byte stores into the workspace)
        for (int e = tid; e < CT * DT / 4; e += K7_THREADS) {
            const int r = e / (DT / 4), c4 = (e % (DT / 4)) * 4, rr = r < len ? r : len - 1;
            const float *src = P.g + ((size_t)(ci.tok0 + rr) * P.Hv + hv) * P.K;
            float4 o;
            o.x = c4 < P.K ? src[c4] : 0.f;
            o.y = c4 + 1 < P.K ? src[c4 + 1] : 0.f;
            o.z = c4 + 2 < P.K ? src[c4 + 2] : 0.f;
            o.w = c4 + 3 < P.K ? src[c4 + 3] : 0.f;
            reinterpret_cast<float4 *>(P.gam + u * CT * DT)[e] = o;
        }
        // T = A (the chunk's valid columns only) and D = scale dO
        rows_to_tile(reinterpret_cast<unsigned char *>(P.Tm + u * CT * CT), CT,
                     A + ((size_t)ci.tok0 * P.Hv + hv) * P.BT, (size_t)P.Hv * P.BT, len, len < P.BT ? len : P.BT, 1.f,
                     tid);
        rows_to_tile(reinterpret_cast<unsigned char *>(P.Dt + u * CT * DT), DT,
                     reinterpret_cast<const Tin *>(P.dO) + ((size_t)ci.tok0 * P.Hv + hv) * P.V, (size_t)P.Hv * P.V,
                     len, P.V, P.scale, tid);
    } else if (part == 1) {  // S_0: [K][V] fp32 per chunk -> a [v][k] tile
        transpose_to_tile(reinterpret_cast<unsigned char *>(P.h + u * DT * DT), DT, h + u * P.K * P.V, (size_t)P.V,
                          P.K, P.V, 1.f, wid, lane);
    } else if (part == 2) {  // dS_next, the same way
        transpose_to_tile(reinterpret_cast<unsigned char *>(P.dh + u * DT * DT), DT, dh + u * P.K * P.V, (size_t)P.V,
                          P.K, P.V, 1.f, wid, lane);
    } else {  // V_new^T and -dV_new^T: [c][v] rows -> [v][c] tiles
        transpose_to_tile(reinterpret_cast<unsigned char *>(P.Vn + u * DT * CT), CT,
                          vnew + ((size_t)ci.tok0 * P.Hv + hv) * P.V, (size_t)P.Hv * P.V, len, P.V, 1.f, wid, lane);
        transpose_to_tile(reinterpret_cast<unsigned char *>(P.dVn + u * DT * CT), CT,
                          dvin + ((size_t)ci.tok0 * P.Hv + hv) * P.V, (size_t)P.Hv * P.V, len, P.V, -1.f, wid, lane);
    }
}

template <typename Tin>
static cudaError_t launch_k7_t(const Params &P, const void *A, const void *vnew, const void *dvin, const float *h,
                               const float *dh, cudaStream_t stream) {
    dim3 grid(P.max_chunks, P.Hv, 4);  // the four parts of a chunk x head (see the kernel)
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
