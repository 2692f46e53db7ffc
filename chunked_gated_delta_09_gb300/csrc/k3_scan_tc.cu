// k3_scan_tc.cu -- reverse scan of the state gradient on the 5th-generation tensor cores, segment-parallel.
//
// Per chunk, walking backwards ("FlashQLA backward explained", section 2: dS <- g_last dS + Q^T (dO g)
// - K^T (dV g), accumulated into dh0; section 1: dht optional, dh0 in fp32), with D = scale dO:
//     dV_new = Aqk^T D + K~ dS^T,     dS <- Gamma_C dS + D^T (Q (.) Gamma) - dV_new^T W
// i.e. dS <- dS M_n^T + R_n with the same transition M_n = Gamma_C I - W^T K~ as the forward, so the
// forward's segment products Phi_s serve here transposed:
//   local pass (LOCAL = true): every segment runs from dS = 0 at its end (-> F_s, the state gradient
//     at its start);
//   combine (k23_combine.cu): dS_exit(s-1) = dS_exit(s) Phi_s^T + F_s, exactly, in fp32;
//   final pass (LOCAL = false): every segment runs from its exact exit gradient and writes dh_n and
//     -dV_new^T; segment 0 also writes dh0.
// One CTA holds the 128 x 128 fp32 dS in tensor memory; each step issues two MMA groups.  Operand tiles
// arrive by bulk copy one chunk ahead; dh_n and -dV_new^T leave by bulk copy from the operand tiles.  The
// local pass, which stores neither, keeps its fp16 A operands (dS rows, -dV_new^T) in tensor memory.
// FACT (local pass only): the factored step of the dh-gradient kernel of section 3 of the same page,
// dS <- Gamma_C dS + D^T QR - (dS K~^T) W with QR = Q~ - Aqk W formed per chunk by k8_qr.cu, which needs
// neither Aqk nor dV_new inside the step (selected with GDR_DH_FACTORED=1).
#include "gdr_common.cuh"
#include "gdr_kernels.h"
#include "k2_scan_body.cuh"
#include "tc_util.cuh"

namespace gdr {

constexpr int SB_THREADS = 256;

struct __align__(1024) BwdSmem {
    unsigned char Aq[2][CT * CT * 2], D[2][CT * DT * 2], Kt[2][CT * DT * 2], Qg[2][CT * DT * 2], W[2][CT * DT * 2];
    unsigned char dSa[DT * DT * 2];  // dS rows as fp16 (A operand; dh_n)
    unsigned char dVa[DT * CT * 2];  // -dV_new^T [v][c] (A operand)
    float gam[2][DT];
    uint64_t bar, lbar[2];  // MMA completion, the two tile buffers' loads
    uint32_t tslot;
};

// The whole kernel for one CTA: bid is its (sequence x head x segment) index.
template <bool PC, bool LOCAL, bool FACT = false>
__device__ __forceinline__ void k3_scan_body(const Params &P, const int bid) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    BwdSmem &S = *reinterpret_cast<BwdSmem *>(smem_raw);
    if (*P.status & ST_BAD_SEQLENS) return;
    const int NS = P.NS;
    const int seg = bid % NS, hv = (bid / NS) % P.Hv, s = bid / (NS * P.Hv);
    int bos, eos;
    seq_range(P, s, bos, eos);
    const int nc = (eos - bos + P.BT - 1) / P.BT;
    const int c_lo = seg * P.Lseg, c_hi = min(nc, c_lo + P.Lseg);
    const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
    const int q = wid & 3, half = wid >> 2;
    const int row = 32 * q + lane;  // dS row (v) owned in the epilogues
    const size_t su = ((size_t)s * P.Hv + hv) * NS + seg;
    if (c_lo >= c_hi) {
        // no chunk in this segment: only an empty sequence's dh0 (= dht) remains to be written
        if (!LOCAL && seg == 0 && P.dh0) {
            for (int e = tid; e < P.V * P.K; e += SB_THREADS) {
                size_t o = ((size_t)s * P.Hv + hv) * P.V * P.K + e;
                P.dh0[o] = P.dht ? P.dht[o] : 0.f;
            }
        }
        return;
    }
    const int base = seq_chunk_base(P, s);

    if (wid == 0) tc::tmem_alloc(&S.tslot, 256);
    if (tid == 0) {
        tc::mbar_init(&S.bar, 1);
        tc::mbar_init(&S.lbar[0], 1);
        tc::mbar_init(&S.lbar[1], 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    auto chunk_len = [&](int c) {
        int len = eos - (bos + c * P.BT);
        return len < P.BT ? len : P.BT;
    };
    auto issue = [&](int c, int buf) {
        const size_t u = (size_t)(base + c) * P.Hv + hv;
        const uint32_t gbytes = PC ? DT * 4 : CT * 4;
        const float *gsrc = PC ? P.gam + (u * CT + chunk_len(c) - 1) * DT : P.gam + u * CT;
        tc::mbar_expect_tx(&S.lbar[buf], (FACT ? 0 : CT * CT * 2) + 4 * CT * DT * 2 + gbytes);
        if (!FACT) tc::bulk_g2s(S.Aq[buf], P.Aqk + u * CT * CT, CT * CT * 2, &S.lbar[buf]);
        tc::bulk_g2s(S.D[buf], P.Dt + u * CT * DT, CT * DT * 2, &S.lbar[buf]);
        tc::bulk_g2s(S.Kt[buf], P.Kt + u * CT * DT, CT * DT * 2, &S.lbar[buf]);
        tc::bulk_g2s(S.Qg[buf], (FACT ? P.QR : P.Qg) + u * CT * DT, CT * DT * 2, &S.lbar[buf]);  // QR if FACT
        tc::bulk_g2s(S.W[buf], P.W + u * CT * DT, CT * DT * 2, &S.lbar[buf]);
        tc::bulk_g2s(S.gam[buf], gsrc, gbytes, &S.lbar[buf]);
    };
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    // armed0 / armed1: a buffer's loads are in flight and not yet waited for (tracked by every thread alike)
    bool armed0 = ((c_hi - 1 - c_lo) & 1) == 0, armed1 = !armed0;
    if (tid == 0) issue(c_hi - 1, (c_hi - 1 - c_lo) & 1);
    const uint32_t tm = S.tslot;
    constexpr int T_S = 0, T_DV = 128;
    // local pass: dS rows as fp16 pairs (64 columns), then -dV_new^T over their first 32 once the product
    // that reads dS has completed
    constexpr int T_SA = 192;
    {
        const float *src = nullptr;
        if (!LOCAL) src = NS > 1 ? P.segdS + su * DT * DT : (P.dht ? P.dht + ((size_t)s * P.Hv + hv) * P.V * P.K : nullptr);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float v[32];
#pragma unroll
            for (int t = 0; t < 32; ++t) {
                int col = 64 * half + 32 * h + t;
                float x = 0.f;
                if (src) {
                    if (NS > 1) x = src[(size_t)row * DT + col];
                    else if (row < P.V && col < P.K) x = src[(size_t)row * P.K + col];
                }
                v[t] = x;
            }
            tc::st32(tc::taddr(tm, T_S + 64 * half + 32 * h), v);
        }
        tc::wait_st();
    }
    const uint32_t sdSa = smem_u32(S.dSa), sdVa = smem_u32(S.dVa);
    uint32_t parity = 0, lpar0 = 0, lpar1 = 0;
    bool lost = false;
    bool mma_ok = true;  // false: the last MMA commit's phase is still pending (the exit drains it)
    auto mma_done = [&]() {
        if (tid == 0) tc::commit(&S.bar);
        mma_ok = tc::mbar_wait(&S.bar, parity, P.spin);
        if (mma_ok) parity ^= 1u;
        lost = __syncthreads_or(!mma_ok) != 0;
        tc::fence_after();
    };

    for (int c = c_hi - 1; c >= c_lo && !lost; --c) {
        const int buf = (c - c_lo) & 1;
        const size_t u = (size_t)(base + c) * P.Hv + hv;
        bool ok = tc::mbar_wait(&S.lbar[buf], buf ? lpar1 : lpar0, P.spin);
        if (ok) {  // (a failed wait leaves the phase armed: the exit drains it)
            if (buf) lpar1 ^= 1u, armed1 = false;
            else lpar0 ^= 1u, armed0 = false;
        }
        if (!LOCAL && tid == 0) tc::bulk_wait_read();
        tc::fence_before();
        lost = __syncthreads_or(!ok) != 0;
        tc::fence_after();
        if (lost) break;
        if (c > c_lo) {
            if (tid == 0) issue(c - 1, buf ^ 1);
            if (buf) armed0 = true;
            else armed1 = true;
        }
        const float gl = PC ? 0.f : S.gam[buf][chunk_len(c) - 1];
        if (PC) {  // the per-channel chunk decay exp(gamma_C[c]), once per channel, in place of gamma_C
            if (tid < DT) S.gam[buf][tid] = expf(S.gam[buf][tid]);
            __syncthreads();
        }
        // epilogue 0: dS rows -> fp16 operand (= dh_n), then scale by Gamma_C in place
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int c0 = 64 * half + 32 * h;
            float v[32];
            tc::ld32(tc::taddr(tm, T_S + c0), v);
            if constexpr (LOCAL) {
                tc::st32_f16(tc::taddr(tm, T_SA + c0 / 2), v);
            } else {
#pragma unroll
                for (int j8 = 0; j8 < 32; j8 += 8) tc::st_tile8(S.dSa, row, c0 + j8, DT, v + j8);
            }
            if (PC) {
#pragma unroll
                for (int t = 0; t < 32; ++t) v[t] *= S.gam[buf][c0 + t];
            } else {
                const float G = expf(gl);
#pragma unroll
                for (int t = 0; t < 32; ++t) v[t] *= G;
            }
            tc::st32(tc::taddr(tm, T_S + c0), v);
        }
        tc::wait_st();
        tc::fence_smem_to_async();
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
        // MMA 1: dV_new^T = D^T Aqk + dS K~^T;  dh_n leaves by bulk copy
        if (tid == 0) {  // (FACT: only Y = dS K~^T)
            if (!FACT)
                tc::gemm(tm + T_DV, smem_u32(S.D[buf]), DT, true, smem_u32(S.Aq[buf]), CT, true, 128, 64, CT, false);
            if constexpr (LOCAL) {
                tc::gemm_ta(tm + T_DV, tm + T_SA, tc::op_rows(smem_u32(S.Kt[buf]), DT, false), 64, DT, !FACT);
            } else {
                tc::gemm(tm + T_DV, sdSa, DT, false, smem_u32(S.Kt[buf]), DT, false, 128, 64, DT, !FACT);
                tc::bulk_s2g(P.dh + u * DT * DT, S.dSa, DT * DT * 2);
            }
        }
        mma_done();
        if (lost) break;
        // epilogue 1: -dV_new^T -> fp16 operand
        {
            const int c0 = 32 * half;
            float v[32];
            tc::ld32(tc::taddr(tm, T_DV + c0), v);
#pragma unroll
            for (int t = 0; t < 32; ++t) v[t] = -v[t];
            if constexpr (LOCAL) {
                tc::st32_f16(tc::taddr(tm, T_SA + c0 / 2), v);
                tc::wait_st();
            } else {
#pragma unroll
                for (int j8 = 0; j8 < 32; j8 += 8) tc::st_tile8(S.dVa, row, c0 + j8, CT, v + j8);
            }
        }
        tc::fence_smem_to_async();
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
        // MMA 2: dS += D^T Q~ - dV_new^T W;  -dV_new^T leaves by bulk copy
        if (tid == 0) {
            tc::gemm(tm + T_S, smem_u32(S.D[buf]), DT, true, smem_u32(S.Qg[buf]), DT, true, 128, 128, CT, true);
            if constexpr (LOCAL) tc::gemm_ta(tm + T_S, tm + T_SA, tc::op_rows(smem_u32(S.W[buf]), DT, true), 128, CT, true);
            else tc::gemm(tm + T_S, sdVa, CT, false, smem_u32(S.W[buf]), DT, true, 128, 128, CT, true);
            if (!LOCAL) {
                tc::bulk_s2g(P.dVn + u * DT * CT, S.dVa, DT * CT * 2);
                tc::bulk_commit();
            }
        }
        mma_done();
    }
    // ---- local pass: F_s; final pass of segment 0: dh0
    if (!lost && (LOCAL || (seg == 0 && P.dh0))) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int c0 = 64 * half + 32 * h;
            float v[32];
            tc::ld32(tc::taddr(tm, T_S + c0), v);
            if (LOCAL) {
                float *dst = P.segF + su * DT * DT + (size_t)row * DT;
#pragma unroll
                for (int t = 0; t < 32; t += 4)
                    *reinterpret_cast<float4 *>(dst + c0 + t) = make_float4(v[t], v[t + 1], v[t + 2], v[t + 3]);
            } else if (row < P.V) {
                float *dst = P.dh0 + ((size_t)s * P.Hv + hv) * P.V * P.K + (size_t)row * P.K;
#pragma unroll
                for (int t = 0; t < 32; ++t)
                    if (c0 + t < P.K) dst[c0 + t] = v[t];
            }
        }
    }
    if (lost && tid == 0) {
        flag_status(P.status, ST_TIMEOUT);
        // drain: the MMAs of a commit whose wait gave up, and the tile loads still armed, complete before
        // the exit (every MMA is followed by its commit and wait, so nothing else can be in flight)
        if (!mma_ok) tc::mbar_wait(&S.bar, parity, DRAIN_LIMIT);
        if (armed0) tc::mbar_wait(&S.lbar[0], lpar0, DRAIN_LIMIT);
        if (armed1) tc::mbar_wait(&S.lbar[1], lpar1, DRAIN_LIMIT);
    }
    if (tid == 0) tc::bulk_wait();
    tc::fence_before();
    __syncthreads();
    if (wid == 0) {
        tc::fence_after();
        tc::tmem_dealloc(tm, 256);
    }
}

template <bool PC, bool LOCAL, bool FACT = false>
__global__ void __launch_bounds__(SB_THREADS, 1) k3_scan_tc(const Params P) {
    k3_scan_body<PC, LOCAL, FACT>(P, (int)blockIdx.x);
}

// One segment per sequence: the forward state recompute and the state-gradient scan do not depend on each
// other (both read only the WY preparation's tiles), so their single passes run as one grid, the first N Hv
// CTAs walking the forward recurrence and the rest the reverse one; with few sequences x heads each scan alone
// would leave most SMs idle.
template <bool PC>
__global__ void __launch_bounds__(SB_THREADS, 1) k23_scan_pair(const Params P) {
    const int n = P.N * P.Hv;
    if ((int)blockIdx.x < n) k2_scan_body<PC, false>(P, (int)blockIdx.x);
    else k3_scan_body<PC, false>(P, (int)blockIdx.x - n);
}

template <bool PC, bool LOCAL, bool FACT = false>
static cudaError_t launch_bwd_t(const Params &P, cudaStream_t stream) {
    size_t smem = sizeof(BwdSmem);
    cudaError_t e =
        smem_opt_in((const void *)k3_scan_tc<PC, LOCAL, FACT>, smem);
    if (e != cudaSuccess) return e;
    k3_scan_tc<PC, LOCAL, FACT><<<P.N * P.Hv * P.NS, SB_THREADS, smem, stream>>>(P);
    return cudaGetLastError();
}

template <bool PC>
static cudaError_t launch_pair_t(const Params &P, cudaStream_t stream) {
    const size_t smem = sizeof(BwdSmem) > sizeof(FwdSmem<false>) ? sizeof(BwdSmem) : sizeof(FwdSmem<false>);
    cudaError_t e = smem_opt_in((const void *)k23_scan_pair<PC>, smem);
    if (e != cudaSuccess) return e;
    k23_scan_pair<PC><<<2 * P.N * P.Hv, SB_THREADS, smem, stream>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_k23_scan_pair(const Params &P, cudaStream_t stream) {
    if (P.NS != 1) return cudaErrorInvalidValue;
    static_assert(SB_THREADS == SC_THREADS, "one block shape for both scans");
    return P.per_channel ? launch_pair_t<true>(P, stream) : launch_pair_t<false>(P, stream);
}

cudaError_t launch_k3_scan(const Params &P, bool local, cudaStream_t stream) {
    if (local && P.QR)
        return P.per_channel ? launch_bwd_t<true, true, true>(P, stream) : launch_bwd_t<false, true, true>(P, stream);
    if (local) return P.per_channel ? launch_bwd_t<true, true>(P, stream) : launch_bwd_t<false, true>(P, stream);
    return P.per_channel ? launch_bwd_t<true, false>(P, stream) : launch_bwd_t<false, false>(P, stream);
}

}  // namespace gdr
