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
//     dV_new; segment 0 also writes dh0.
// One CTA holds the 128 x 128 fp32 dS in tensor memory; each step issues two MMA groups.
#include "gdr_common.cuh"
#include "gdr_kernels.h"
#include "tc_util.cuh"

namespace gdr {

constexpr int SB_THREADS = 256;
constexpr uint32_t SB_WAIT_LIMIT = 1u << 24;

template <typename Tin>
struct __align__(1024) BwdSmem {
    unsigned char Aq[2][CT * CT * 2], D[2][CT * DT * 2], Kt[2][CT * DT * 2], Qg[2][CT * DT * 2], W[2][CT * DT * 2];
    unsigned char dSa[DT * DT * 2];  // dS rows as fp16 (A operand)
    unsigned char dVa[DT * CT * 2];  // -dV_new^T [v][c] (A operand)
    Tin Draw[CT * DT];               // raw dO slice of the next chunk
    float gC[2][DT];
    uint64_t bar;
    uint32_t tslot;
};

__device__ __forceinline__ void cp_tile_sb(unsigned char *tile, const __half *src, int cols, int tid) {
    const int wid = tid >> 5, lane = tid & 31;
    const int cpr = cols / 8;  // 16-byte chunks per row
    for (int it = wid; it < (CT / 8) * (cpr / 4); it += SB_THREADS / 32) {
        int r = 8 * (it / (cpr / 4)) + (lane & 7), c8 = 8 * (4 * (it % (cpr / 4)) + (lane >> 3));
        cp_async16(tile + tc::tile_off(r, c8, cols), src + (size_t)r * cols + c8);
    }
}

template <typename Tin, bool PC, bool LOCAL>
__global__ void __launch_bounds__(SB_THREADS, 1) k3_scan_tc(const Params P) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    BwdSmem<Tin> &S = *reinterpret_cast<BwdSmem<Tin> *>(smem_raw);
    if (*P.status & ST_BAD_SEQLENS) return;
    const int NS = P.NS;
    const int seg = blockIdx.x % NS, hv = (blockIdx.x / NS) % P.Hv, s = blockIdx.x / (NS * P.Hv);
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
    const Tin *dOp = reinterpret_cast<const Tin *>(P.dO);
    constexpr int EPC = 16 / sizeof(Tin);  // input elements per 16-byte copy

    if (wid == 0) tc::tmem_alloc(&S.tslot, 256);
    if (tid == 0) {
        tc::mbar_init(&S.bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    // raw dO slice of chunk c: rows past the chunk and columns past V zero-fill.  Each thread later
    // converts exactly the copies it issued (lane % 8 -> row inside a core matrix).
    auto for_my_d = [&](auto &&fn) {
#pragma unroll
        for (int i = 0; i < (CT * DT / 8) / SB_THREADS; ++i) {
            int it = wid + (SB_THREADS / 32) * i;
            int r = 8 * (it >> 2) + (lane & 7), c8 = 8 * (4 * (it & 3) + (lane >> 3));
            fn(r, c8);
        }
    };
    auto issue = [&](int c, int buf) {
        const size_t u = (size_t)(base + c) * P.Hv + hv;
        cp_tile_sb(S.Aq[buf], P.Aqk + u * CT * CT, CT, tid);
        cp_tile_sb(S.Kt[buf], P.Kt + u * CT * DT, DT, tid);
        cp_tile_sb(S.Qg[buf], P.Qg + u * CT * DT, DT, tid);
        cp_tile_sb(S.W[buf], P.W + u * CT * DT, DT, tid);
        const int tok0 = bos + c * P.BT;
        int len = eos - tok0;
        len = len < P.BT ? len : P.BT;
        for_my_d([&](int r, int c8) {
#pragma unroll
            for (int h = 0; h < 8 / EPC; ++h) {
                int cc = c8 + h * EPC;
                bool ok = r < len && cc + EPC <= P.V;
                const Tin *src = ok ? dOp + ((size_t)(tok0 + r) * P.Hv + hv) * P.V + cc : dOp;
                cp_async16_zfill(S.Draw + r * DT + cc, src, ok ? 16 : 0);
            }
        });
        if (PC) {
            if (tid < DT / 4) cp_async16(&S.gC[buf][4 * tid], P.gam + (u * CT + len - 1) * DT + 4 * tid);
        } else if (tid == 0) {
            cp_async4(&S.gC[buf][0], P.gam + u * CT + len - 1);
        }
        cp_async_commit();
    };
    auto convert_d = [&](int buf) {
        for_my_d([&](int r, int c8) {
            float x[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) x[j] = to_f32(S.Draw[r * DT + c8 + j]) * P.scale;
            tc::st_tile8(S.D[buf], r, c8, DT, x);
        });
    };
    issue(c_hi - 1, (c_hi - 1 - c_lo) & 1);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tm = S.tslot;
    constexpr int T_S = 0, T_DV = 128;
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
    uint32_t parity = 0;
    bool lost = false;
    auto mma_done = [&]() {
        if (tid == 0) tc::commit(&S.bar);
        bool ok = tc::mbar_wait(&S.bar, parity, SB_WAIT_LIMIT);
        parity ^= 1u;
        lost = __syncthreads_or(!ok) != 0;
        tc::fence_after();
    };
    cp_async_wait<0>();
    convert_d((c_hi - 1 - c_lo) & 1);

    for (int c = c_hi - 1; c >= c_lo && !lost; --c) {
        const int buf = (c - c_lo) & 1;
        const size_t u = (size_t)(base + c) * P.Hv + hv;
        tc::fence_smem_to_async();
        tc::fence_before();
        __syncthreads();  // chunk c's operands (and its converted D) visible; previous MMAs finished
        tc::fence_after();
        // epilogue 0: dS rows -> fp16 operand (+ dh_n), then scale by Gamma_C in place
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int c0 = 64 * half + 32 * h;
            float v[32];
            tc::ld32(tc::taddr(tm, T_S + c0), v);
#pragma unroll
            for (int j8 = 0; j8 < 32; j8 += 8) tc::st_tile8(S.dSa, row, c0 + j8, DT, v + j8);
            if (!LOCAL) {
                uint4 pk[4];
                __half2 *h2 = reinterpret_cast<__half2 *>(pk);
#pragma unroll
                for (int t = 0; t < 16; ++t) h2[t] = __floats2half2_rn(v[2 * t], v[2 * t + 1]);
                uint4 *dst = reinterpret_cast<uint4 *>(P.dh + u * DT * DT + (size_t)row * DT + c0);
#pragma unroll
                for (int t = 0; t < 4; ++t) dst[t] = pk[t];
            }
#pragma unroll
            for (int t = 0; t < 32; ++t) v[t] *= expf(PC ? S.gC[buf][c0 + t] : S.gC[buf][0]);
            tc::st32(tc::taddr(tm, T_S + c0), v);
        }
        tc::wait_st();
        tc::fence_smem_to_async();
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
        if (c > c_lo) issue(c - 1, buf ^ 1);
        // MMA 1: dV_new^T = D^T Aqk + dS K~^T
        if (tid == 0) {
            tc::gemm(tm + T_DV, smem_u32(S.D[buf]), DT, true, smem_u32(S.Aq[buf]), CT, true, 128, 64, CT, false);
            tc::gemm(tm + T_DV, sdSa, DT, false, smem_u32(S.Kt[buf]), DT, false, 128, 64, DT, true);
        }
        mma_done();
        if (lost) break;
        // epilogue 1: dV_new (+ global), -dV_new^T -> fp16 operand
        {
            const int c0 = 32 * half;
            float v[32];
            tc::ld32(tc::taddr(tm, T_DV + c0), v);
            if (!LOCAL) {
                __half *dg = P.dVn + u * CT * DT;
#pragma unroll
                for (int t = 0; t < 32; ++t) dg[(size_t)(c0 + t) * DT + row] = __float2half_rn(v[t]);
            }
#pragma unroll
            for (int t = 0; t < 32; ++t) v[t] = -v[t];
#pragma unroll
            for (int j8 = 0; j8 < 32; j8 += 8) tc::st_tile8(S.dVa, row, c0 + j8, CT, v + j8);
        }
        tc::fence_smem_to_async();
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
        // MMA 2: dS += D^T Q~ - dV_new^T W
        if (tid == 0) {
            tc::gemm(tm + T_S, smem_u32(S.D[buf]), DT, true, smem_u32(S.Qg[buf]), DT, true, 128, 128, CT, true);
            tc::gemm(tm + T_S, sdVa, CT, false, smem_u32(S.W[buf]), DT, true, 128, 128, CT, true);
        }
        mma_done();
        if (c > c_lo) {
            cp_async_wait<0>();
            convert_d(buf ^ 1);
        }
    }
    cp_async_wait<0>();
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
    if (lost && tid == 0) flag_status(P.status, ST_TIMEOUT);
    tc::fence_before();
    __syncthreads();
    if (wid == 0) {
        tc::fence_after();
        tc::tmem_dealloc(tm, 256);
    }
}

template <typename Tin, bool PC, bool LOCAL>
static cudaError_t launch_bwd_t(const Params &P, cudaStream_t stream) {
    size_t smem = sizeof(BwdSmem<Tin>);
    cudaError_t e = cudaFuncSetAttribute(k3_scan_tc<Tin, PC, LOCAL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k3_scan_tc<Tin, PC, LOCAL><<<P.N * P.Hv * P.NS, SB_THREADS, smem, stream>>>(P);
    return cudaGetLastError();
}

template <typename Tin>
static cudaError_t launch_bwd_d(const Params &P, bool local, cudaStream_t stream) {
    if (local) return P.per_channel ? launch_bwd_t<Tin, true, true>(P, stream) : launch_bwd_t<Tin, false, true>(P, stream);
    return P.per_channel ? launch_bwd_t<Tin, true, false>(P, stream) : launch_bwd_t<Tin, false, false>(P, stream);
}

cudaError_t launch_k3_scan(const Params &P, bool local, cudaStream_t stream) {
    if (P.qkv_dtype == F32) return launch_bwd_d<float>(P, local, stream);
    if (P.qkv_dtype == BF16) return launch_bwd_d<__nv_bfloat16>(P, local, stream);
    return launch_bwd_d<__half>(P, local, stream);
}

}  // namespace gdr
