// k6_fwd_output.cu -- forward output of one chunk: o = scale (diag(Gamma) Q S_0^T + (M (.) Q K^T) V_new).
//
// With the chunk quantities of the backward's preparation and state recompute (MindSpeed-Ops
// chunk_kda_bwd.md, input table: chunk states h and v_new; "FlashQLA backward explained", section 1),
// Q~ = Q (.) exp(gamma) and Aqk = M (.) Q K^T, the output of the chunk is
//     o^T = scale (S_0 Q~^T + V_new^T Aqk^T)        (V x C)
// i.e. two tcgen05 products accumulated into one tensor-memory region (M = 128 value rows, N = 64 chunk
// rows): A = the state tile [v][k] and V_new^T tile [v][c], B = the Q~ tile [r][k] and Aqk tile [r][j],
// all K-major.  One CTA of four warps per chunk x value head; the four tiles arrive by bulk copy; each
// thread owns one value row of the result and writes its 64 chunk rows (coalesced over the warp).
#include "gdr_common.cuh"
#include "gdr_kernels.h"
#include "tc_util.cuh"

namespace gdr {

constexpr int K6_THREADS = 128;

struct __align__(1024) K6Smem {
    unsigned char Qg[CT * DT * 2];   // Q~ [r][k]
    unsigned char H[DT * DT * 2];    // S_0 [v][k]
    unsigned char Aqk[CT * CT * 2];  // [r][j]
    unsigned char Vn[DT * CT * 2];   // V_new^T [v][c]
    uint64_t bar, lbar;
    uint32_t tslot;
};

template <typename To>
__global__ void __launch_bounds__(K6_THREADS) k6_fwd_output(const Params P) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    K6Smem &S = *reinterpret_cast<K6Smem *>(smem_raw);
    if (*P.status & ST_BAD_SEQLENS) return;
    const int n = blockIdx.x, hv = blockIdx.y;
    ChunkInfo ci;
    if (!chunk_info(P, n, ci)) return;
    const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
    const size_t u = (size_t)n * P.Hv + hv;

    if (wid == 0) tc::tmem_alloc(&S.tslot, 64);
    if (tid == 0) {
        tc::mbar_init(&S.bar, 1);
        tc::mbar_init(&S.lbar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        tc::mbar_expect_tx(&S.lbar, CT * DT * 2 + DT * DT * 2 + CT * CT * 2 + DT * CT * 2);
        tc::bulk_g2s(S.Qg, P.Qg + u * CT * DT, CT * DT * 2, &S.lbar);
        tc::bulk_g2s(S.H, P.h + u * DT * DT, DT * DT * 2, &S.lbar);
        tc::bulk_g2s(S.Aqk, P.Aqk + u * CT * CT, CT * CT * 2, &S.lbar);
        tc::bulk_g2s(S.Vn, P.Vn + u * DT * CT, DT * CT * 2, &S.lbar);
    }
    tc::fence_before();
    __syncthreads();  // barriers initialised, tensor-memory address visible
    tc::fence_after();
    const uint32_t tm = S.tslot;
    bool ok = true, loads_ok = true;
    if (tid == 0) {
        loads_ok = ok = tc::mbar_wait(&S.lbar, 0, P.spin);
        if (ok) {
            tc::gemm(tm, smem_u32(S.H), DT, false, smem_u32(S.Qg), DT, false, 128, 64, DT, false);
            tc::gemm(tm, smem_u32(S.Vn), CT, false, smem_u32(S.Aqk), CT, false, 128, 64, CT, true);
        }
        tc::commit(&S.bar);
    }
    const bool mma_ok = tc::mbar_wait(&S.bar, 0, P.spin);
    ok = mma_ok && ok;
    const bool lost = __syncthreads_or(!ok) != 0;
    tc::fence_after();
    if (!lost) {
        const int vrow = 32 * wid + lane;
        To *out = reinterpret_cast<To *>(P.o) + ((size_t)ci.tok0 * P.Hv + hv) * P.V + vrow;
        const size_t rs = (size_t)P.Hv * P.V;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float x[32];
            tc::ld32(tc::taddr(tm, 32 * h), x);
            if (vrow < P.V) {
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    const int r = 32 * h + t;
                    if (r < ci.len) out[(size_t)r * rs] = to_out_t<To>(P.scale * x[t]);
                }
            }
        }
    } else if (tid == 0) {
        flag_status(P.status, ST_TIMEOUT);
        // the loads and MMAs still tracked by a barrier that gave up complete before the CTA exits
        if (!loads_ok) tc::mbar_wait(&S.lbar, 0, DRAIN_LIMIT);
        if (!mma_ok) tc::mbar_wait(&S.bar, 0, DRAIN_LIMIT);
    }
    tc::fence_before();
    __syncthreads();
    if (wid == 0) {
        tc::fence_after();
        tc::tmem_dealloc(tm, 64);
    }
}

template <typename To>
static cudaError_t launch_k6_t(const Params &P, cudaStream_t stream) {
    const size_t smem = sizeof(K6Smem);
    cudaError_t e = smem_opt_in((const void *)k6_fwd_output<To>, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(P.max_chunks, P.Hv);
    k6_fwd_output<To><<<grid, K6_THREADS, smem, stream>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_k6_fwd_output(const Params &P, cudaStream_t stream) {
    if (P.qkv_dtype == F32) return launch_k6_t<float>(P, stream);
    if (P.qkv_dtype == BF16) return launch_k6_t<__nv_bfloat16>(P, stream);
    return launch_k6_t<__half>(P, stream);
}

}  // namespace gdr
