// k2_scan_body.cuh -- forward state recompute on the 5th-generation tensor cores, segment-parallel.
//
// Per chunk the state update is linear in the state ("FlashQLA backward explained", section 1, step 2:
// fused_gdr_h rebuilds the chunk states h):
//     V_new = U - W S^T,      S <- Gamma_C S + V_new^T K~        (K~ = K (.) exp(gamma_C - gamma))
// i.e. S <- S M_n + U^T K~ with the transition M_n = Gamma_C I - W^T K~ (K x K).  A sequence is cut into
// segments of Lseg chunks so that sequences x heads x segments CTAs fill the GPU:
//   local pass (LOCAL = true): every segment runs from a zero state (-> E_s) and, in a second CTA, the
//     rows of the transition product Phi_s = prod M_n run from the identity (the same update without U);
//     the two chains are independent and their CTAs share an SM (half the tensor memory each), so each
//     one's products run while the other's epilogues do;
//   combine (k23_combine.cu): S_entry(s+1) = S_entry(s) Phi_s + E_s, exactly, in fp32;
//   final pass (LOCAL = false): every segment runs from its exact entry state and writes h_n and V_new
//     (in the forward pass, OUT = true, it writes the chunk outputs o instead; see k2_scan_body).
// This is the state-passing correction that the page's context-parallel path applies across devices
// (section 3: partition states corrected with an all-gather), done inside one GPU.
//
// One CTA holds the whole 128 x 128 fp32 state (and Phi) in tensor memory; each step issues two MMA
// groups: V_new^T = S W^T (M = 128 state rows, N = 64 tokens) and S += V_new^T K~ (N = 128).  Operand
// tiles arrive by bulk copy one chunk ahead; h_n and V_new^T leave by bulk copy from the operand tiles.
// The local pass, which stores neither, keeps its fp16 A operands (the state or transition rows, V_new^T or
// -(Phi W^T)) in tensor memory instead of shared memory: the products then read only their B tiles from
// shared memory.
#pragma once

#include "gdr_common.cuh"
#include "gdr_kernels.h"
#include "tc_util.cuh"

namespace gdr {

constexpr int SC_THREADS = 256;

// OUT (the forward's final pass): W[buf] holds the W tile and then the Q~ tile, and Aq the Aqk tiles.
template <bool LOCAL, bool OUT = false>
struct __align__(1024) FwdSmem {
    unsigned char W[2][(OUT ? 2 : 1) * CT * DT * 2], Kt[2][CT * DT * 2], U[2][CT * DT * 2];  // U^T tiles [v][c]
    unsigned char Sa[LOCAL ? 16 : DT * DT * 2];   // state rows as fp16 (A operand; h_n): final pass only
    unsigned char Vna[LOCAL ? 16 : DT * CT * 2];  // V_new^T [v][c] (A operand): final pass only
    unsigned char Aq[OUT ? 2 : 1][OUT ? CT * CT * 2 : 16];
    float gam[2][DT];                             // gate row block of the chunk (scalar: first CT used)
    uint64_t bar, lbar[2];  // MMA completion, the two tile buffers' loads
    uint32_t tslot;
};

// The whole kernel for one CTA: bid is its (sequence x head x segment) index (the launch that pairs the two
// final passes runs it with the CTA index of its first half); local pass: phi selects the transition chain
// (else the state chain).  OUT (final pass of the forward): the chunk's output
// o^T = scale (S_0 Q~^T + V_new^T Aqk^T) is formed in the same steps (S_0 Q~^T in the product that takes
// S_0 W^T, as its second 64 columns; V_new^T Aqk^T after S += V_new^T K~) and written, while h_n and V_new,
// which only the backward reads, are not.
template <bool PC, bool LOCAL, bool OUT = false>
__device__ __forceinline__ void k2_scan_body(const Params &P, const int bid, const bool phi = false) {
    static_assert(!(LOCAL && OUT), "the output comes from the final pass");
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    FwdSmem<LOCAL, OUT> &S = *reinterpret_cast<FwdSmem<LOCAL, OUT> *>(smem_raw);
    if (*P.status & ST_BAD_SEQLENS) return;
    const int NS = P.NS;
    const int seg = bid % NS, hv = (bid / NS) % P.Hv, s = bid / (NS * P.Hv);
    int bos, eos;
    seq_range(P, s, bos, eos);
    const int nc = (eos - bos + P.BT - 1) / P.BT;
    const int c_lo = seg * P.Lseg, c_hi = min(nc, c_lo + P.Lseg);
    if (c_lo >= c_hi) {  // segment without chunks; the forward's final state of an empty sequence is h0
        if (!LOCAL && P.ht && nc == 0 && seg == 0) {
            const int hv0 = (bid / NS) % P.Hv;
            float *dst = P.ht + ((size_t)s * P.Hv + hv0) * P.V * P.K;
            const float *src = P.h0 ? P.h0 + ((size_t)s * P.Hv + hv0) * P.V * P.K : nullptr;
            for (int e = threadIdx.x; e < P.V * P.K; e += SC_THREADS) dst[e] = src ? src[e] : 0.f;
        }
        return;
    }
    const int base = seq_chunk_base(P, s);
    const size_t su = ((size_t)s * P.Hv + hv) * NS + seg;
    const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
    const int q = wid & 3, half = wid >> 2;
    const int row = 32 * q + lane;  // state row (v) / transition row (k') owned in the epilogues

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
    // one thread: bulk-load chunk c's operand tiles and gate row into buffer `buf`
    auto issue = [&](int c, int buf) {
        const size_t u = (size_t)(base + c) * P.Hv + hv;
        const uint32_t gbytes = PC ? DT * 4 : CT * 4;
        const float *gsrc = PC ? P.gam + (u * CT + chunk_len(c) - 1) * DT : P.gam + u * CT;
        tc::mbar_expect_tx(&S.lbar[buf], (phi ? 2 : 3) * CT * DT * 2 + gbytes + (OUT ? CT * DT * 2 + CT * CT * 2 : 0));
        tc::bulk_g2s(S.W[buf], P.W + u * CT * DT, CT * DT * 2, &S.lbar[buf]);
        tc::bulk_g2s(S.Kt[buf], P.Kt + u * CT * DT, CT * DT * 2, &S.lbar[buf]);
        if (!phi) tc::bulk_g2s(S.U[buf], P.U + u * CT * DT, CT * DT * 2, &S.lbar[buf]);  // (the transition: no U)
        if (OUT) {  // Q~ right after W (one 128-row B operand), and Aqk
            tc::bulk_g2s(S.W[buf] + CT * DT * 2, P.Qg + u * CT * DT, CT * DT * 2, &S.lbar[buf]);
            tc::bulk_g2s(S.Aq[buf], P.Aqk + u * CT * CT, CT * CT * 2, &S.lbar[buf]);
        }
        tc::bulk_g2s(S.gam[buf], gsrc, gbytes, &S.lbar[buf]);
    };
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    // armed0 / armed1: a buffer's loads are in flight and not yet waited for (tracked by every thread alike)
    bool armed0 = true, armed1 = false;
    if (tid == 0) issue(c_lo, 0);
    const uint32_t tm = S.tslot;
    // the chain's rows (state, or transition in the local pass's second CTA), then V_new^T (resp. Phi W^T)
    constexpr int T_S = 0, T_VN = 128, T_O = 192;  // (T_O: the output o^T, OUT only)
    // local pass: the fp16 A operands, packed two per column: the chain's rows (64 columns), then V_new^T (resp.
    // -(Phi W^T)) over their first 32 columns once the first product has completed
    constexpr int T_SA = 192;

    // ---- initial rows: zero state or identity transition (local pass), the exact entry state (final pass)
    {
        const float *src = nullptr;
        if (!LOCAL) src = NS > 1 ? P.segSin + su * DT * DT : (P.h0 ? P.h0 + ((size_t)s * P.Hv + hv) * P.V * P.K : nullptr);
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
                } else if (LOCAL && phi) {
                    x = col == row ? 1.f : 0.f;
                }
                v[t] = x;
            }
            tc::st32(tc::taddr(tm, T_S + 64 * half + 32 * h), v);
        }
        tc::wait_st();
    }
    const uint32_t sSa = smem_u32(S.Sa), sVna = smem_u32(S.Vna);
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

    for (int c = c_lo; c < c_hi && !lost; ++c) {
        const int buf = (c - c_lo) & 1;
        const size_t u = (size_t)(base + c) * P.Hv + hv;
        // chunk c's tiles landed; the previous step's bulk stores no longer read Sa / Vna
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
        if (c + 1 < c_hi) {
            if (tid == 0) issue(c + 1, buf ^ 1);
            if (buf) armed0 = true;
            else armed1 = true;
        }
        const float gl = PC ? 0.f : S.gam[buf][chunk_len(c) - 1];
        if (PC) {  // the per-channel chunk decay exp(gamma_C[c]), once per channel, in place of gamma_C
            if (tid < DT) S.gam[buf][tid] = expf(S.gam[buf][tid]);
            __syncthreads();
        }
        // epilogue 0: the chain's rows -> fp16 operand (= h_n), then scale by Gamma_C in place
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int c0 = 64 * half + 32 * h;
            float v[32];
            tc::ld32(tc::taddr(tm, T_S + c0), v);
            if constexpr (LOCAL) {
                tc::st32_f16(tc::taddr(tm, T_SA + c0 / 2), v);
            } else {
#pragma unroll
                for (int j8 = 0; j8 < 32; j8 += 8) tc::st_tile8(S.Sa, row, c0 + j8, DT, v + j8);
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
        // MMA 1: V_new^T (pre) = S W^T   [transition: Phi W^T];  h_n leaves by bulk copy
        if (tid == 0) {
            if constexpr (LOCAL) {
                tc::gemm_ta(tm + T_VN, tm + T_SA, tc::op_rows(smem_u32(S.W[buf]), DT, false), 64, DT, false);
            } else {  // (OUT: N = 128 over [W ; Q~], the second half = S_0 Q~^T at T_O)
                tc::gemm(tm + T_VN, sSa, DT, false, smem_u32(S.W[buf]), DT, false, 128, OUT ? 128 : 64, DT, false);
                if (!OUT) tc::bulk_s2g(P.h + u * DT * DT, S.Sa, DT * DT * 2);
            }
        }
        mma_done();
        if (lost) break;
        // epilogue 1: V_new^T = U^T - S W^T  (transition rows: -(Phi W^T)) -> fp16 operand
        {
            const int c0 = 32 * half;
            float v[32];
            tc::ld32(tc::taddr(tm, T_VN + c0), v);
            if (LOCAL && phi) {
#pragma unroll
                for (int t = 0; t < 32; ++t) v[t] = -v[t];
            } else {
#pragma unroll
                for (int j8 = 0; j8 < 32; j8 += 8) {  // U^T row segment: 16-byte reads of the [v][c] tile
                    const __half2 *u2 =
                        reinterpret_cast<const __half2 *>(S.U[buf] + tc::tile_off(row, c0 + j8, CT));
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const float2 f = __half22float2(u2[t]);
                        v[j8 + 2 * t] = f.x - v[j8 + 2 * t];
                        v[j8 + 2 * t + 1] = f.y - v[j8 + 2 * t + 1];
                    }
                }
            }
            if constexpr (LOCAL) {
                tc::st32_f16(tc::taddr(tm, T_SA + c0 / 2), v);
                tc::wait_st();
            } else {
#pragma unroll
                for (int j8 = 0; j8 < 32; j8 += 8) tc::st_tile8(S.Vna, row, c0 + j8, CT, v + j8);
            }
        }
        tc::fence_smem_to_async();
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
        // MMA 2: S += V_new^T K~   [transition: Phi += (-(Phi W^T)) K~];  V_new^T leaves by bulk copy
        if (tid == 0) {
            if constexpr (LOCAL) {
                tc::gemm_ta(tm + T_S, tm + T_SA, tc::op_rows(smem_u32(S.Kt[buf]), DT, true), 128, CT, true);
            } else {
                tc::gemm(tm + T_S, sVna, CT, false, smem_u32(S.Kt[buf]), DT, true, 128, 128, CT, true);
                if (OUT) {
                    tc::gemm(tm + T_O, sVna, CT, false, smem_u32(S.Aq[buf]), CT, false, 128, 64, CT, true);
                } else {
                    tc::bulk_s2g(P.Vn + u * DT * CT, S.Vna, DT * CT * 2);
                    tc::bulk_commit();
                }
            }
        }
        mma_done();
        if constexpr (OUT) {
            // o rows of this chunk: each thread holds one value row and 32 chunk rows.  The four lanes of a quad
            // (value rows 4g .. 4g + 3) transpose each block of 4 chunk rows among themselves (two swap rounds),
            // so that lane j writes chunk row 4b + j of the four value rows with one 8-byte store (V is a
            // multiple of 8)
            if (lost) break;
            const int c0 = 32 * half, len = chunk_len(c), j = lane & 3;
            float v[32];
            tc::ld32(tc::taddr(tm, T_O + c0), v);
            const size_t rs = (size_t)P.Hv * P.V;
            const size_t o0 = ((size_t)(bos + c * P.BT) * P.Hv + hv) * P.V + (row & ~3);
#pragma unroll
            for (int b = 0; b < 32; b += 4) {
#pragma unroll
                for (int sw = 2; sw >= 1; sw >>= 1) {
                    const bool up = (j & sw) != 0;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if (i & sw) continue;
                        const float recv = __shfl_xor_sync(0xffffffffu, up ? v[b + i] : v[b + i + sw], sw);
                        if (up) v[b + i] = recv;
                        else v[b + i + sw] = recv;
                    }
                }
                const int r = c0 + b + j;  // v[b .. b + 3]: value rows (row & ~3) .. + 3 at chunk row r
                if (r < len && row < P.V) {
                    const size_t oi = o0 + (size_t)r * rs;
                    const float x0 = P.scale * v[b], x1 = P.scale * v[b + 1], x2 = P.scale * v[b + 2],
                                x3 = P.scale * v[b + 3];
                    if (P.qkv_dtype == BF16) {
                        const __nv_bfloat162 p0 = __floats2bfloat162_rn(x0, x1), p1 = __floats2bfloat162_rn(x2, x3);
                        *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(P.o) + oi) =
                            make_uint2(*reinterpret_cast<const uint32_t *>(&p0), *reinterpret_cast<const uint32_t *>(&p1));
                    } else if (P.qkv_dtype == F16) {
                        const __half2 p0 = __floats2half2_rn(x0, x1), p1 = __floats2half2_rn(x2, x3);
                        *reinterpret_cast<uint2 *>(reinterpret_cast<__half *>(P.o) + oi) =
                            make_uint2(*reinterpret_cast<const uint32_t *>(&p0), *reinterpret_cast<const uint32_t *>(&p1));
                    } else {
                        *reinterpret_cast<float4 *>(reinterpret_cast<float *>(P.o) + oi) = make_float4(x0, x1, x2, x3);
                    }
                }
            }
        }
    }
    // ---- local pass: segment summaries E_s (state CTA), Phi_s and Phi_s^T (transition CTA), fp32
    if (LOCAL && !lost) {
        float *dst = (phi ? P.segPhi : P.segE) + su * DT * DT + (size_t)row * DT;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int c0 = 64 * half + 32 * h;
            float v[32];
            tc::ld32(tc::taddr(tm, T_S + c0), v);
#pragma unroll
            for (int t = 0; t < 32; t += 4)
                *reinterpret_cast<float4 *>(dst + c0 + t) = make_float4(v[t], v[t + 1], v[t + 2], v[t + 3]);
            if (phi) {  // Phi^T, so that the backward combine also reads rows
                float *dT = P.segPhiT + su * DT * DT + row;
#pragma unroll
                for (int t = 0; t < 32; ++t) dT[(size_t)(c0 + t) * DT] = v[t];
            }
        }
    }
    if (!LOCAL && !lost && P.ht && c_hi == nc) {  // forward: the final state of the sequence
        float *dst = P.ht + ((size_t)s * P.Hv + hv) * P.V * P.K + (size_t)row * P.K;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int c0 = 64 * half + 32 * h;
            float v[32];
            tc::ld32(tc::taddr(tm, T_S + c0), v);
            if (row < P.V) {
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

}  // namespace gdr
