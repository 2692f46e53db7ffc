// k8_qr.cu -- per-chunk QR = Q~ - Aqk W for the factored state-gradient recurrence.
//
// The dh-gradient kernel of "FlashQLA backward explained" (section 3) factors the reverse recurrence with
// X = W (its Ab K), Y = K~ dS^T and QR = Q~ - Lower(P) X, so that a step needs no dV_new:
//     dS <- Gamma_C dS + D^T QR - Y^T W          (here, with dS as V x K: dS <- Gamma_C dS + D^T QR - (dS K~^T) W)
// which equals the unfactored step dS <- Gamma_C dS + D^T Q~ - dV_new^T W with dV_new = Aqk^T D + K~ dS^T.
// This kernel forms QR once per chunk x head (warp MMAs on core-matrix tiles) for the factored local pass of
// the state-gradient scan; the tile goes to a workspace region that no later kernel reads otherwise.
#include "gdr_common.cuh"
#include "gdr_kernels.h"
#include "tc_util.cuh"

namespace gdr {

constexpr int K8_THREADS = 256;

struct __align__(1024) K8Smem {
    unsigned char Aq[CT * CT * 2], W[CT * DT * 2], Qg[CT * DT * 2];
    uint64_t lbar;
};

__global__ void __launch_bounds__(K8_THREADS) k8_qr(const Params P, __half *QR) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    K8Smem &S = *reinterpret_cast<K8Smem *>(smem_raw);
    if (*P.status & ST_BAD_SEQLENS) return;
    const int n = blockIdx.x, hv = blockIdx.y;
    ChunkInfo ci;
    if (!chunk_info(P, n, ci)) return;
    const int tid = threadIdx.x, wid = tid >> 5;
    const size_t u = (size_t)n * P.Hv + hv;
    if (tid == 0) {
        tc::mbar_init(&S.lbar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        tc::mbar_expect_tx(&S.lbar, CT * CT * 2 + 2 * CT * DT * 2);
        tc::bulk_g2s(S.Aq, P.Aqk + u * CT * CT, CT * CT * 2, &S.lbar);
        tc::bulk_g2s(S.W, P.W + u * CT * DT, CT * DT * 2, &S.lbar);
        tc::bulk_g2s(S.Qg, P.Qg + u * CT * DT, CT * DT * 2, &S.lbar);
    }
    __syncthreads();  // barrier initialised
    const bool ok = tc::mbar_wait(&S.lbar, 0, P.spin);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) {
            flag_status(P.status, ST_TIMEOUT);
            tc::mbar_wait(&S.lbar, 0, DRAIN_LIMIT);  // the tiles land before the CTA exits
        }
        return;
    }
    // QR [r][k] = Q~ - Aqk W: warp w owns rows 16 (w % 4) .. +15 and columns 64 (w / 4) .. +63
    const int m0 = (wid & 3) * 16, n0 = (wid >> 2) * 64;
    float acc[1][8][4];
    zero_acc(acc);
    warp_mma_ct<1, 8, false, false>(acc, S.Aq, CT, S.W, DT, m0, n0, CT);
    unsigned char *dst = reinterpret_cast<unsigned char *>(QR + u * CT * DT);
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
            const int r = acc_row(m0, 0, e), c = acc_col(n0, nt, e);
            const uint32_t off = ctile_off(r, c, DT);
            const float2 qg = __half22float2(*reinterpret_cast<const __half2 *>(S.Qg + off));
            *reinterpret_cast<__half2 *>(dst + off) = __floats2half2_rn(qg.x - acc[0][nt][e], qg.y - acc[0][nt][e + 1]);
        }
}

cudaError_t launch_k8_qr(const Params &P, __half *QR, cudaStream_t stream) {
    const size_t smem = sizeof(K8Smem);
    cudaError_t e = smem_opt_in((const void *)k8_qr, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(P.max_chunks, P.Hv);
    k8_qr<<<grid, K8_THREADS, smem, stream>>>(P, QR);
    return cudaGetLastError();
}

}  // namespace gdr
