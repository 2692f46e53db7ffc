// k23_combine.cu -- exact combination of the per-segment scan summaries (fp32).
//
// Forward:  S_entry(0) = h0,                  S_entry(s+1) = S_entry(s) Phi_s + E_s
// Backward: dS_exit(last) = dht,              dS_exit(s-1) = dS_exit(s) Phi_s^T + F_s
// where E_s / F_s are the segment's zero-initialised local scans and Phi_s the product of its chunk
// transitions (k2_scan_tc.cu writes Phi_s and Phi_s^T, k3_scan_tc.cu writes F_s).  Rows of the state are
// independent, so a CTA owns CB_ROWS rows of one sequence x head (one wave of CTAs for the usual head
// counts) and walks the segments serially, prefetching the next segment's transition and summary rows
// while it multiplies by the current ones.  Each thread accumulates four columns of all
// the CTA's rows over one warp's slice of the reduction, so every transition element read from shared
// memory serves 16 rows; the slices are summed in a fixed order.  The prefetch is two bulk copies (the
// transition, 64 KB, and the CTA's summary rows, 8 KB, both contiguous) by one thread on the buffer's
// mbarrier.
#include "gdr_common.cuh"
#include "gdr_kernels.h"
#include "tc_util.cuh"

namespace gdr {

constexpr int CB_THREADS = 256;  // 8 warps = 8 slices of 16 reduction indices; lane = 4 output columns
constexpr int CB_ROWS = 16;      // rows of the state per CTA (all of them in every thread)
constexpr int CB_PP = DT + 4;    // fp32 pitch of a partial-sum row (16-byte reads without bank conflicts)

template <bool FWD>
__global__ void __launch_bounds__(CB_THREADS) k23_combine(const Params P) {
    __shared__ __align__(16) float XT[DT][CB_ROWS];  // the current rows, transposed: XT[j][r]
    __shared__ uint64_t pbar[2];                     // the two prefetch buffers' bulk copies
    extern __shared__ __align__(16) float dyn[];     // Ph [2][DT][DT], Ad [2][CB_ROWS][DT], part [8][CB_ROWS][CB_PP]
    float *Ph = dyn, *Ad = dyn + 2 * DT * DT, *part = Ad + 2 * CB_ROWS * DT;
    if (*P.status & ST_BAD_SEQLENS) return;
    const int s = blockIdx.x / P.Hv, hv = blockIdx.x % P.Hv, r0 = blockIdx.y * CB_ROWS;
    int bos, eos;
    seq_range(P, s, bos, eos);
    const int nc = (eos - bos + P.BT - 1) / P.BT;
    const int nss = (nc + P.Lseg - 1) / P.Lseg;  // segments holding chunks
    if (nss == 0) return;
    const int tid = threadIdx.x, w = tid >> 5, k0 = (tid & 31) * 4;
    const size_t su0 = ((size_t)s * P.Hv + hv) * P.NS;
    float *out = FWD ? P.segSin : P.segdS;
    const float *init = FWD ? P.h0 : P.dht;
    const float *trans = FWD ? P.segPhi : P.segPhiT;  // row j of the matrix applied on the right
    const float *adds = FWD ? P.segE : P.segF;

    // the next step's transition and summary rows, in flight while the current step multiplies (thread 0)
    auto prefetch = [&](int step, int buf) {
        const int sg = FWD ? step : nss - 1 - step;
        tc::mbar_expect_tx(&pbar[buf], (DT * DT + CB_ROWS * DT) * 4);
        tc::bulk_g2s(Ph + buf * DT * DT, trans + (su0 + sg) * DT * DT, DT * DT * 4, &pbar[buf]);
        tc::bulk_g2s(Ad + buf * CB_ROWS * DT, adds + (su0 + sg) * DT * DT + (size_t)r0 * DT, CB_ROWS * DT * 4,
                     &pbar[buf]);
    };
    if (tid == 0) {
        tc::mbar_init(&pbar[0], 1);
        tc::mbar_init(&pbar[1], 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncthreads();
    if (nss > 1 && tid == 0) prefetch(0, 0);
    // starting rows: h0 / dht (absent = 0)
    for (int e = tid; e < CB_ROWS * DT; e += CB_THREADS) {
        int rr = e / DT, k = e % DT, v = r0 + rr;
        float x = 0.f;
        if (init && v < P.V && k < P.K) x = init[(((size_t)s * P.Hv + hv) * P.V + v) * P.K + k];
        XT[k][rr] = x;
        out[(su0 + (FWD ? 0 : nss - 1)) * DT * DT + (size_t)v * DT + k] = x;
    }
    for (int step = 0; step < nss - 1; ++step) {
        const int buf = step & 1;
        const int sg = FWD ? step : nss - 1 - step;  // segment whose summary is applied
        const int dst = FWD ? sg + 1 : sg - 1;
        const bool landed = tc::mbar_wait(&pbar[buf], (uint32_t)(step >> 1) & 1u, P.spin);
        if (__syncthreads_or(!landed)) {  // (this step's rows, and XT, visible; last step's readers done)
            if (tid == 0) {  // the status is flagged whether or not the copies then land in time
                flag_status(P.status, ST_TIMEOUT);
                // this step's two copies are the only ones in flight: they land before the CTA exits
                tc::mbar_wait(&pbar[buf], (uint32_t)(step >> 1) & 1u, DRAIN_LIMIT);
            }
            return;
        }
        if (step + 1 < nss - 1 && tid == 0) prefetch(step + 1, buf ^ 1);
        // partial products of this warp's 16 reduction indices: all 16 rows x columns k0 .. k0+3
        const float *ph = Ph + buf * DT * DT;
        float acc[CB_ROWS][4];
#pragma unroll
        for (int r = 0; r < CB_ROWS; ++r) acc[r][0] = acc[r][1] = acc[r][2] = acc[r][3] = 0.f;
#pragma unroll 4
        for (int j = 16 * w; j < 16 * w + 16; ++j) {
            const float4 a = *reinterpret_cast<const float4 *>(ph + j * DT + k0);
#pragma unroll
            for (int r4 = 0; r4 < CB_ROWS; r4 += 4) {
                const float4 x = *reinterpret_cast<const float4 *>(&XT[j][r4]);
                const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[r4 + i][0] += xs[i] * a.x;
                    acc[r4 + i][1] += xs[i] * a.y;
                    acc[r4 + i][2] += xs[i] * a.z;
                    acc[r4 + i][3] += xs[i] * a.w;
                }
            }
        }
#pragma unroll
        for (int r = 0; r < CB_ROWS; ++r)
            *reinterpret_cast<float4 *>(part + (w * CB_ROWS + r) * CB_PP + k0) =
                make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
        __syncthreads();  // partials written; everyone done reading XT
        // sum the 8 slices in a fixed order, add the summary rows; lanes walk rows so that the transposed
        // writes hit distinct banks
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            const int r = tid & 15, kq = 4 * ((tid >> 4) + 16 * p);
            float4 y = *reinterpret_cast<const float4 *>(Ad + buf * CB_ROWS * DT + r * DT + kq);
#pragma unroll
            for (int ww = 0; ww < 8; ++ww) {
                const float4 z = *reinterpret_cast<const float4 *>(part + (ww * CB_ROWS + r) * CB_PP + kq);
                y.x += z.x;
                y.y += z.y;
                y.z += z.z;
                y.w += z.w;
            }
            XT[kq][r] = y.x;
            XT[kq + 1][r] = y.y;
            XT[kq + 2][r] = y.z;
            XT[kq + 3][r] = y.w;
            *reinterpret_cast<float4 *>(out + (su0 + dst) * DT * DT + (size_t)(r0 + r) * DT + kq) = y;
        }
    }
}

cudaError_t launch_k23_combine(const Params &P, bool fwd, cudaStream_t stream) {
    size_t smem = sizeof(float) * (2 * DT * DT + 2 * CB_ROWS * DT + 8 * CB_ROWS * CB_PP);
    cudaError_t e;
    dim3 grid(P.N * P.Hv, DT / CB_ROWS);
    if (fwd) {
        e = smem_opt_in((const void *)k23_combine<true>, smem);
        if (e != cudaSuccess) return e;
        k23_combine<true><<<grid, CB_THREADS, smem, stream>>>(P);
    } else {
        e = smem_opt_in((const void *)k23_combine<false>, smem);
        if (e != cudaSuccess) return e;
        k23_combine<false><<<grid, CB_THREADS, smem, stream>>>(P);
    }
    return cudaGetLastError();
}

}  // namespace gdr
