// k4_intra_grad_tc.cu -- per-chunk gradients on the 5th-generation tensor cores (scalar gate).
//
// Same mathematics as k4_intra_grad.cu (the WY-gradient stage of MindSpeed-Ops chunk_kda_bwd.md,
// "implementation principle", with the scalar gate of "FlashQLA backward explained", section 2): every
// matrix product is a tcgen05.mma (fp16 operands from shared memory, fp32 accumulators in tensor memory)
// issued by one thread, completion tracked by an mbarrier with a bounded wait, results read back with
// tcgen05.ld.
//
// Layout of the work:
//  * persistent CTAs (one per SM, 16 warps) take the items (chunk n, value head hv), item = n Hv + hv, by
//    key-head group: the value heads that share a key head run on one CTA one after the other (groups
//    round-robin), the first storing the key head's dq / dk rows and the others adding to them;
//  * products with a chunk x feature result are computed transposed (feature x chunk, M = 128), so each
//    epilogue thread owns one feature row and 16 chunk columns; chunk x chunk products use M = 64;
//  * the feature-major copies K^T, V^T, Q^T that those epilogues need come from products with a 64 x 64
//    identity tile: one tensor-memory load replaces 16 scattered 2-byte shared-memory reads;
//  * each buffer is refilled for the CTA's next item as soon as its last reader is done: S_0, dS_next, D,
//    V_new^T, -dV_new^T after phase 1 and T after phase 4 (bulk copies: one barrier phase per item for the
//    first group, one on a second barrier for T); for 16-bit inputs V after phase 1, Q after phase 2 and K
//    after phase 5, each by one TMA tensor load (a 4-D tensor map over [tokens, heads, features] whose box of
//    8-element rows lands as a column-block-major core-matrix tile: core matrix (r/8, c/8) at
//    ((c/8) 8 + r/8) 128), converted to fp16 in place when the item starts (rows past the chunk's end and
//    columns past K or V set to zero).
//
// Five MMA phases, each followed by an epilogue that produces the next phase's operands:
//   1: dk_SC^T = dS^T V_new^T, dW^T = -S0^T dV^T, TdU^T = dV^T T, K^T, P0 = D V_new^T, dT2 = dV V^T,
//      dq_inter^T = S0^T D^T
//   2: dq_intra^T = K^T P^T, dk_O^T = Q^T P, TdW^T = dW^T T, Q^T, KK = K K^T, dT1 = dW K^T
//   3: X = dT T^T        4: dA' = T^T X        5: dk_Ar^T = K^T E^T, dk_Ac^T = K^T E
// The WY part of dbeta, sum_k (T^T dW)_jk Gamma_j k_jk + sum_v (T^T dU)_jv v_jv, equals the column sum
// sum_i T_ij (Gamma_j dT1_ij + dT2_ij) of two chunk x chunk products, so it is taken there.  The epilogues of
// M = 64 products spread each row's 16 columns over both half-warps.
#include <type_traits>

#include "gdr_common.cuh"
#include "gdr_kernels.h"
#include "tc_util.cuh"

namespace gdr {

constexpr int K4T_THREADS = 512;
// MMA issue: lane 0 of warps 0..3 issues the products of a phase's group 1 (one product each, committed to
// its mbarrier), lane 0 of warps 4..7 those of group 2; an issuer without a product commits empty.  No warp
// is held up by more than one product's issue before its own epilogue work.
constexpr int K4T_ISSUERS = 4;
constexpr uint32_t K4T_TMEM_COLS = 512;

// tensor-memory column map, 64 columns per region (C_* regions use the M = 64 lane layout)
constexpr int R_DKSC = 0, R_DWT = 64, R_TDU = 128, R_KT = 256, C_G1 = 320, C_DT2 = 384,
              R_DQI = 448;                                                              // phase 1
constexpr int R_DQA = 0, R_DKO = 64, R_TDW = 128, R_QT = 192, C_DT1 = 320;              // phase 2
constexpr int C_X = 0, C_KK = 256;                                                      // phase 3
constexpr int C_DA = 64;                                                                // phase 4
constexpr int R_DKAR = 128, R_DKAC = 192;                                               // phase 5

struct __align__(1024) K4TSmem {
    unsigned char Q[CT * DT * 2], K[CT * DT * 2], V[CT * DT * 2], D[CT * DT * 2];
    unsigned char Vn[DT * CT * 2], dVn[DT * CT * 2];  // V_new^T and -dV_new^T, tiles [v][c]
    unsigned char H[DT * DT * 2], dH[DT * DT * 2];    // [v][k] tiles: S_0 and dS_next
    unsigned char T[CT * CT * 2];
    unsigned char Pm[CT * CT * 2];   // P, later X
    unsigned char dWT[DT * CT * 2];  // dW^T [k][r]
    unsigned char dT[CT * CT * 2];   // dT, later E
    unsigned char I[CT * CT * 2];    // identity
    float gam[CT], G[CT], GC[CT], beta[CT];
    float scal[4][CT];  // the next item's per-token record (beta, exp(gamma), exp(gamma_C - gamma), gamma)
    // partial sums in fixed slots, added in a fixed order at the end (run-to-run reproducible):
    // dbeta: 4 row quarters (WY term), 4 column quarters (A term); dgamma rows: 4 lane quarters; last row:
    // 16 warps
    // (two sets, by item parity: an item's sums are added during the next item's first MMA phase)
    float db_wy[2][4][CT], db_a[2][4][CT], dg_q[2][4][CT], last_w[2][16];
    int red_u, red_len, red_tok0, red_hv, red_b;  // the item whose sums are pending (red_u < 0: none), its set
    uint64_t bar, bar2, lbar, tbar;  // MMA groups 1 and 2 of a phase; bulk loads (T on its own barrier)
    uint64_t kbar, qbar, vbar;       // tensor-map loads of the raw k, q, v rows
    uint32_t tslot;
};

__device__ __forceinline__ void st2(__nv_bfloat16 *p, float lo, float hi) {
    *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(lo, hi);
}
__device__ __forceinline__ void st2(__half *p, float lo, float hi) {
    *reinterpret_cast<__half2 *>(p) = __floats2half2_rn(lo, hi);
}
__device__ __forceinline__ void st2(float *p, float lo, float hi) { *reinterpret_cast<float2 *>(p) = make_float2(lo, hi); }
// add a pair to memory (a reduction in the element's own type; no value is returned)
__device__ __forceinline__ void red2(__nv_bfloat16 *p, float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    asm volatile("red.global.add.noftz.bf16x2 [%0], %1;\n" ::"l"(p), "r"(*reinterpret_cast<const uint32_t *>(&v))
                 : "memory");
}
__device__ __forceinline__ void red2(__half *p, float lo, float hi) {
    const __half2 v = __floats2half2_rn(lo, hi);
    asm volatile("red.global.add.noftz.f16x2 [%0], %1;\n" ::"l"(p), "r"(*reinterpret_cast<const uint32_t *>(&v))
                 : "memory");
}
__device__ __forceinline__ void red2(float *p, float lo, float hi) {
    asm volatile("red.global.add.f32 [%0], %1;\n" ::"l"(p), "f"(lo) : "memory");
    asm volatile("red.global.add.f32 [%0], %1;\n" ::"l"(p + 1), "f"(hi) : "memory");
}
template <bool ADD, typename To>
__device__ __forceinline__ void pairs16_t(To *p, size_t rs, int n, bool act, const float (&x)[16]) {
    const bool odd = (threadIdx.x & 1) != 0;
    To *q = odd ? p - 1 + rs : p;  // the pair's even column, on the first row this lane writes
#pragma unroll
    for (int t = 0; t < 16; t += 2) {
        const float recv = __shfl_xor_sync(0xffffffffu, odd ? x[t] : x[t + 1], 1);
        if (act && t + (odd ? 1 : 0) < n) {
            if (ADD) red2(q + (size_t)t * rs, odd ? recv : x[t], odd ? x[t + 1] : recv);
            else st2(q + (size_t)t * rs, odd ? recv : x[t], odd ? x[t + 1] : recv);
        }
    }
}
// x[t] -> element (t, 0) of a row-major output with row stride rs (elements), for the first n rows.  Lanes
// 2m and 2m + 1 hold adjacent columns; the even lane writes rows 0, 2, .. and the odd lane rows 1, 3, .. of
// both columns with one 2-element store each.  Every lane of the warp calls it (shuffles); act says whether
// this lane's column exists (the same for both lanes of a pair: the feature sizes are even).
// ADD: added to what is there instead (same lanes, same addresses).
template <bool ADD = false>
__device__ __forceinline__ void store_pairs16(void *p, int dt, size_t rs, int n, bool act, const float (&x)[16]) {
    if (dt == BF16) pairs16_t<ADD>(reinterpret_cast<__nv_bfloat16 *>(p), rs, n, act, x);
    else if (dt == F16) pairs16_t<ADD>(reinterpret_cast<__half *>(p), rs, n, act, x);
    else pairs16_t<ADD>(reinterpret_cast<float *>(p), rs, n, act, x);
}
// A key head's dq / dk row block: the group's first value head stores it, the others add to it.  One CTA
// runs a group's items in head order and a given element is always written by the same thread, so the
// additions follow the stores in program order and the sum's order is fixed (run-to-run identical).
__device__ __forceinline__ void put_pairs16(bool add, void *p, int dt, size_t rs, int n, bool act, const float (&x)[16]) {
    if (add) store_pairs16<true>(p, dt, rs, n, act, x);
    else store_pairs16<false>(p, dt, rs, n, act, x);
}
__device__ __forceinline__ size_t esize(int dt) { return dt == F32 ? 4 : 2; }
// 8 consecutive floats of a 16-byte aligned shared array as two vector loads
__device__ __forceinline__ void lds8(const float *p, float (&v)[8]) {
    const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
    v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
}

// Tensor maps of the 16-bit inputs (unused for fp32 inputs): 4-D over (8-element column chunk, token, column
// block, head), box (8, 64, K/8 or V/8, 1).
// GRP: grouped-query attention (several value heads per key head), whose groups are summed in place.
template <typename Tin, bool GRP>
__global__ void __launch_bounds__(K4T_THREADS, 1)
    k4_intra_grad_tc(const Params P, const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmq,
                     const __grid_constant__ CUtensorMap tmv) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    K4TSmem &S = *reinterpret_cast<K4TSmem *>(smem_raw);
    if (*P.status & ST_BAD_SEQLENS) return;
    const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
    // Items go out by key-head group: the G value heads that read one key head are consecutive items (item =
    // n Hv + hv, hv = hk G + i), and a CTA runs a whole group in head order before its next group (groups
    // round-robin over the CTAs), so the group's dq / dk are summed in place in the outputs.
    const int n_items = P.max_chunks * P.Hv, G = GRP ? P.G : 1;
    auto valid_from = [&](int it) -> int {  // it: the first item of a group
        ChunkInfo t;
        while (it < n_items && !chunk_info(P, it / P.Hv, t)) it += (int)gridDim.x * G;
        return it;
    };
    auto next_item = [&](int it) -> int {
        return (it + 1) % G != 0 ? it + 1 : valid_from(it + 1 + ((int)gridDim.x - 1) * G);
    };
    int item = valid_from((int)blockIdx.x * G);
    if (item >= n_items) return;
    // 16-bit inputs are fetched raw ahead of time and converted in place; fp32 inputs are staged directly
    constexpr bool kRaw = sizeof(Tin) == 2;
    constexpr int PER = CT * (DT / 8) / K4T_THREADS;  // 16-byte chunks per thread per input tile

    if (wid == 0) tc::tmem_alloc(&S.tslot, K4T_TMEM_COLS);
    if (tid == 0) {
        tc::mbar_init(&S.bar, K4T_ISSUERS);
        tc::mbar_init(&S.bar2, K4T_ISSUERS);
        tc::mbar_init(&S.lbar, 1);
        tc::mbar_init(&S.tbar, 1);
        tc::mbar_init(&S.kbar, 1);
        tc::mbar_init(&S.qbar, 1);
        tc::mbar_init(&S.vbar, 1);
        S.red_u = -1;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    for (int e = tid; e < CT * CT / 8; e += K4T_THREADS) {
        const int r = e >> 3, c8 = (e & 7) * 8;
        float x[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) x[t] = (c8 + t == r) ? 1.f : 0.f;
        tc::st_tile8(S.I, r, c8, CT, x);
    }
    tc::fence_smem_to_async();
    tc::fence_before();
    __syncthreads();  // barriers initialised, identity written, tensor-memory address visible
    tc::fence_after();
    const uint32_t tm = S.tslot;
    const uint32_t sQ = smem_u32(S.Q), sK = smem_u32(S.K), sV = smem_u32(S.V), sD = smem_u32(S.D);
    const uint32_t sVn = smem_u32(S.Vn), sdVn = smem_u32(S.dVn), sH = smem_u32(S.H), sdH = smem_u32(S.dH);
    const uint32_t sT = smem_u32(S.T), sPm = smem_u32(S.Pm), sdWT = smem_u32(S.dWT), sdT = smem_u32(S.dT);
    const uint32_t sI = smem_u32(S.I);
    unsigned char *Xs = S.Pm, *Es = S.dT;
    const uint32_t sX = sPm, sE = sdT;

    // workspace tiles of an item: everything the first phase reads, then T (read until phase 4)
    auto issue_ws1 = [&](size_t un) {
        tc::mbar_expect_tx(&S.lbar, 2 * DT * DT * 2 + CT * DT * 2 + 2 * DT * CT * 2 + 4 * CT * 4);
        tc::bulk_g2s(&S.scal[0][0], P.sc + un * 4 * CT, 4 * CT * 4, &S.lbar);
        tc::bulk_g2s(S.H, P.h + un * DT * DT, DT * DT * 2, &S.lbar);
        tc::bulk_g2s(S.dH, P.dh + un * DT * DT, DT * DT * 2, &S.lbar);
        tc::bulk_g2s(S.D, P.Dt + un * CT * DT, CT * DT * 2, &S.lbar);
        tc::bulk_g2s(S.Vn, P.Vn + un * DT * CT, DT * CT * 2, &S.lbar);
        tc::bulk_g2s(S.dVn, P.dVn + un * DT * CT, DT * CT * 2, &S.lbar);
    };
    auto issue_ws2 = [&](size_t un) {
        tc::mbar_expect_tx(&S.tbar, CT * CT * 2);
        tc::bulk_g2s(S.T, P.Tm + un * CT * CT, CT * CT * 2, &S.tbar);
    };
    // input rows of an item (key head for q / k, value head for v); which: 0 = k, 1 = q, 2 = v
    auto input_src = [&](int it, int which, const Tin *&src, size_t &st, int &nc, int &len_) {
        ChunkInfo c2;
        chunk_info(P, it / P.Hv, c2);
        const int hv2 = it % P.Hv, hk2 = hv2 / P.G;
        len_ = c2.len;
        if (which == 2) {
            src = reinterpret_cast<const Tin *>(P.v) + ((size_t)c2.tok0 * P.Hv + hv2) * P.V;
            st = (size_t)P.Hv * P.V;
            nc = P.V;
        } else {
            src = reinterpret_cast<const Tin *>(which == 0 ? P.k : P.q) + ((size_t)c2.tok0 * P.Hk + hk2) * P.K;
            st = (size_t)P.Hk * P.K;
            nc = P.K;
        }
    };
    // raw rows of an item into their (column-block-major) tile slot: one tensor-map load by the loader thread
    auto fetch_raw = [&](int it, int which, unsigned char *dst) {
        ChunkInfo c2;
        chunk_info(P, it / P.Hv, c2);
        const int hv2 = it % P.Hv;
        const int ncb = (which == 2 ? P.V : P.K) >> 3;
        uint64_t *bar = which == 0 ? &S.kbar : which == 1 ? &S.qbar : &S.vbar;
        const CUtensorMap *map = which == 0 ? &tmk : which == 1 ? &tmq : &tmv;
        tc::mbar_expect_tx(bar, (uint32_t)(8 * CT * ncb * 2));
        tc::tma_load_4d(dst, map, 0, c2.tok0, 0, which == 2 ? hv2 : hv2 / P.G, bar);
    };
    // this thread's chunks of a landed tile: 16-bit input -> fp16 in place; rows past len and columns past nc
    // become zero (the box also covers the next sequence's rows and, for K or V < 128, leaves columns unset)
    auto convert_raw = [&](unsigned char *dst, int len_, int nc) {
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int e = tid + K4T_THREADS * i, cb = e >> 6, r = e & (CT - 1);
            uint4 *p = reinterpret_cast<uint4 *>(dst + cb * (CT * 16) + r * 16);
            if (r < len_ && 8 * cb < nc) {
                if constexpr (std::is_same<Tin, __nv_bfloat16>::value) {
                    Raw8<Tin> x;
                    x.v = *p;
                    float f[8];
                    raw_get(x, f);
                    *p = pack8_half(f);
                }
            } else {
                *p = make_uint4(0u, 0u, 0u, 0u);
            }
        }
    };
    // fp32 inputs: staged straight into the column-block-major tile (rows past len, columns past nc zero)
    auto stage_f32 = [&](int it, int which, unsigned char *dst) {
        const Tin *src;
        size_t st;
        int nc, ln;
        input_src(it, which, src, st, nc, ln);
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int e = tid + K4T_THREADS * i, cb = e >> 6, r = e & (CT - 1);
            float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (r < ln && 8 * cb < nc) load8(reinterpret_cast<const float *>(src) + (size_t)r * st + 8 * cb, f);
            *reinterpret_cast<uint4 *>(dst + cb * (CT * 16) + r * 16) = pack8_half(f);
        }
    };

    if (tid == 0) {
        issue_ws1(item);
        issue_ws2(item);
    }
    if (kRaw && tid == 0) {
        fetch_raw(item, 0, S.K);
        fetch_raw(item, 1, S.Q);
        fetch_raw(item, 2, S.V);
    }
    uint32_t lpar = 0, tpar = 0, mpar = 0, mpar2 = 0, kpar = 0, qpar = 0, vpar = 0;
    bool lost = false, okq = true;
    // Barrier phases this thread has not yet seen complete: loads armed and not waited for (the same for every
    // thread: the arming points are passed by all), and MMA commits whose wait gave up.  A wait that gives up
    // leaves its parity unflipped; the exit drains every pending phase before the CTA releases its memory.
    bool l_pend = true, t_pend = true, m_pend = false, m2_pend = false;
    bool k_pend = kRaw, q_pend = kRaw, v_pend = kRaw;  // tensor-map loads of the raw input rows
    // Each phase: the issuers issue group 1 (committed to bar) and, in phases 1 and 2, group 2 (committed to
    // bar2); every thread waits (bounded) for group 1 itself, and the outcomes of all waits since the last
    // agreement are agreed at the next block-wide barrier (publish_tiles or the end of the item); the
    // epilogue starts on group 1's results while group 2 still runs.
    auto finish_phase = [&](bool fail) {
        const bool ok = tc::mbar_wait(&S.bar, mpar, P.spin);
        if (ok) mpar ^= 1u;
        m_pend = !ok;
        okq &= ok && !fail;
        tc::fence_after();
    };
    auto wait_group2 = [&]() -> bool {  // per thread; the outcome is agreed at the next publish_tiles
        const bool ok = tc::mbar_wait(&S.bar2, mpar2, P.spin);
        if (ok) mpar2 ^= 1u;
        m2_pend = !ok;
        tc::fence_after();
        return ok;
    };
    // threads < CT: dbeta and d(gamma) of the pending item from its partial set, added in a fixed order
    auto reduce_pending = [&]() {
        const int ru = S.red_u, rlen = S.red_len, b = S.red_b;
        if (ru < 0) return;
        float x = (S.dg_q[b][0][tid] + S.dg_q[b][1][tid]) + (S.dg_q[b][2][tid] + S.dg_q[b][3][tid]);
        if (tid == rlen - 1) {
            float l = 0.f;
#pragma unroll
            for (int w = 0; w < 16; ++w) l += S.last_w[b][w];
            x += l;
        }
        P.dgam[(size_t)ru * CT + tid] = tid < rlen ? x : 0.f;
        float bb = (S.db_wy[b][0][tid] + S.db_wy[b][1][tid]) + (S.db_wy[b][2][tid] + S.db_wy[b][3][tid]);
        bb += (S.db_a[b][0][tid] + S.db_a[b][1][tid]) + (S.db_a[b][2][tid] + S.db_a[b][3][tid]);
        if (tid < rlen) P.dbeta[(size_t)(S.red_tok0 + tid) * P.Hv + S.red_hv] = bb;
    };
    auto publish_tiles = [&](bool ok) {  // make epilogue-written tiles visible to the next phase's MMAs
        tc::fence_smem_to_async();
        tc::fence_before();
        lost = __syncthreads_or(!ok || !okq || lost) != 0;
        okq = true;
        tc::fence_after();
    };

    // Epilogue ownership: warp w reads lane quarter q = w % 4 and the 16 columns c0 = 16 (w / 4) of a region.
    const int q = wid & 3, c0 = 16 * (wid >> 2);
    const int k = 32 * q + lane;    // feature row in M = 128 regions
    const int r64 = 16 * q + lane;  // chunk row in M = 64 regions (lanes 0..15)
    const bool own64 = lane < 16;
    const bool iss1 = lane == 0 && wid < K4T_ISSUERS;                            // group-1 issuer
    const bool iss2 = lane == 0 && wid >= K4T_ISSUERS && wid < 2 * K4T_ISSUERS;  // group-2 issuer
    const int slot = wid & (K4T_ISSUERS - 1);
    const bool loader = tid == 32 * 2 * K4T_ISSUERS;  // issues the bulk copies (lane 0 of the first non-issuing warp)
    // M = 64 epilogues after split_rows16: row i64, columns jh .. jh + 7
    const int i64 = 16 * q + (lane & 15), jh = c0 + 8 * (lane >> 4);

    while (item < n_items && !lost) {
        const int n = item / P.Hv, hv = item % P.Hv, hk = hv / P.G;
        ChunkInfo ci;
        chunk_info(P, n, ci);
        const size_t u = (size_t)item;  // = n Hv + hv
        const int len = ci.len, rl = len - 1;
        const int next = next_item(item);
        const bool has_next = next < n_items;
        const int nrow = len - c0 < 0 ? 0 : (len - c0 > 16 ? 16 : len - c0);  // valid rows among c0 .. c0+15
        // partial-sum set of this item: the parity of its place in the CTA's sequence (invalid items only trail
        // the list)
        const int pb = ((item / G - (int)blockIdx.x) / (int)gridDim.x * G + item % G) & 1;

        // ---- inputs as fp16 tiles (the workspace tiles are on their way by bulk copy)
        if constexpr (kRaw) {  // (Q, first read in phase 2, is converted while phase 1 runs)
            const bool okk = tc::mbar_wait(&S.kbar, kpar, P.spin), okv = tc::mbar_wait(&S.vbar, vpar, P.spin);
            if (okk) kpar ^= 1u, k_pend = false;
            if (okv) vpar ^= 1u, v_pend = false;
            okq &= okk && okv;  // agreed at the barrier below
            convert_raw(S.K, len, P.K);
            convert_raw(S.V, len, P.V);
        } else {
            stage_f32(item, 0, S.K);
            stage_f32(item, 1, S.Q);
            stage_f32(item, 2, S.V);
        }
        // every thread waits for the workspace tiles itself (the epilogues read some of them directly); the
        // per-token record came with them
        bool fail = false;
        if (tc::mbar_wait(&S.lbar, lpar, P.spin)) lpar ^= 1u, l_pend = false;
        else fail = true;
        if (tc::mbar_wait(&S.tbar, tpar, P.spin)) tpar ^= 1u, t_pend = false;
        else fail = true;
        tc::fence_smem_to_async();
        tc::fence_before();
        lost = __syncthreads_or(!okq || lost) != 0;  // (also orders the previous item's partial sums)
        okq = true;
        tc::fence_after();

        // ---------------- phase 1
        if (iss1) {
            if (!fail) {
                if (slot == 0) tc::gemm_ops(tm + R_KT, tc::op_cols(sK, CT, true), tc::op_rows(sI, CT, false), 128, 64, CT, false);
                else if (slot == 1) tc::gemm(tm + R_DWT, sH, DT, true, sdVn, CT, true, 128, 64, DT, false);
                else if (slot == 2) tc::gemm(tm + R_DKSC, sdH, DT, true, sVn, CT, true, 128, 64, DT, false);
                else tc::gemm(tm + R_TDU, sdVn, CT, false, sT, CT, true, 128, 64, CT, false);
            }
            tc::commit(&S.bar);
        }
        if constexpr (kRaw) {  // published to phase 2 by the tile barrier after the first epilogue
            const bool okq2 = tc::mbar_wait(&S.qbar, qpar, P.spin);
            if (okq2) qpar ^= 1u, q_pend = false;
            okq &= okq2;
            convert_raw(S.Q, len, P.K);
        }
        if (tid < CT) {
            reduce_pending();  // the previous item's sums, while phase 1 runs
            // the record into the arrays the later epilogues read (the first reads it in place; the next
            // item's record lands over it after the first tile barrier)
            S.beta[tid] = S.scal[0][tid];
            S.G[tid] = S.scal[1][tid];
            S.GC[tid] = S.scal[2][tid];
            S.gam[tid] = S.scal[3][tid];
        }
        finish_phase(fail);
        if (iss2) {  // group 2 once group 1 is done: it runs during group 1's epilogue
            if (!fail) {
                if (slot == 0) tc::gemm(tm + C_G1, sD, DT, false, sVn, CT, true, 64, 64, DT, false);
                else if (slot == 1) tc::gemm_ops(tm + C_DT2, tc::op_rows(sdVn, CT, true), tc::op_cols(sV, CT, false), 64, 64, DT, false);
                else if (slot == 2) tc::gemm(tm + R_DQI, sH, DT, true, sD, DT, false, 128, 64, DT, false);
            }
            tc::commit(&S.bar2);
        }
        float dk[16], dg[16], kreg[16];
        float lastpart = 0.f;
        {
            float g[16], g2[16];
            // dW^T -> dWT tile (the stored dV tile is negated, so the product already is dW^T)
            tc::ld16x2(tc::taddr(tm, R_KT + c0), kreg, tc::taddr(tm, R_DWT + c0), g);
            tc::st_tile8(S.dWT, k, c0, CT, g);
            tc::st_tile8(S.dWT, k, c0 + 8, CT, g + 8);
            // dk_SC = exp(gamma_C - gamma_j) (V_new dS)_j
            tc::ld16x2(tc::taddr(tm, R_DKSC + c0), g, tc::taddr(tm, R_TDU + c0), g2);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float gc[8];
                lds8(S.scal[2] + c0 + 8 * h, gc);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int t = 8 * h + u;
                    const float x = g[t] * gc[u];
                    const float kx = kreg[t] * x;
                    dk[t] = x;
                    dg[t] = -kx;
                    lastpart += kx;
                }
            }
            // TdU^T -> dv (rows c0.., column k)   (negated dV tile)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float bv[8];
                lds8(S.scal[0] + c0 + 8 * h, bv);
#pragma unroll
                for (int u = 0; u < 8; ++u) g2[8 * h + u] *= -bv[u];
            }
            store_pairs16(reinterpret_cast<char *>(P.dv) +
                              (((size_t)(ci.tok0 + c0) * P.Hv + hv) * P.V + k) * esize(P.dv_dtype),
                          P.dv_dtype, (size_t)P.Hv * P.V, nrow, k < P.V, g2);
        }
        {
            // last row: Gamma_C <S_0, dS_next> + sum_j k_j (.) dk_SC_j.  Warp w takes the 8-column chunk
            // 4 (w % 4) + lane / 8 over rows 32 (w / 4) .. +31; a quarter-warp reads the 8 rows of one core
            // matrix (16-byte reads, no bank conflicts)
            const int cc8 = 8 * (4 * (wid & 3) + (lane >> 3));
            float hd = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t off = tc::tile_off(32 * (wid >> 2) + 8 * j + (lane & 7), cc8, DT);
                const uint4 av = *reinterpret_cast<const uint4 *>(S.H + off);
                const uint4 bv = *reinterpret_cast<const uint4 *>(S.dH + off);
                const __half2 *a2 = reinterpret_cast<const __half2 *>(&av);
                const __half2 *b2 = reinterpret_cast<const __half2 *>(&bv);
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const float2 a = __half22float2(a2[t]), b = __half22float2(b2[t]);
                    hd += a.x * b.x + a.y * b.y;
                }
            }
            float tot = lastpart + S.scal[1][rl] * hd;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
            if (lane == 0) S.last_w[pb][wid] = tot;
        }
        const bool ok1 = wait_group2();
        {
            // P = (D V_new^T) (.) M  -> Pm tile (row i, columns jh .. jh + 7)
            float g[16], x[8];
            tc::ld16(tc::taddr(tm, C_G1 + c0), g);
            tc::split_rows16(g, x);
            const float gr = S.scal[3][i64];
            float gj[8];
            lds8(S.scal[3] + jh, gj);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const int j = jh + t;
                x[t] = j <= i64 ? x[t] * __expf(gr - gj[t]) : 0.f;
            }
            tc::st_tile8(S.Pm, i64, jh, CT, x);
        }
        publish_tiles(ok1);
        if (lost) break;

        // ---------------- phase 2
        if (iss1) {
            if (slot == 0) tc::gemm_ops(tm + R_QT, tc::op_cols(sQ, CT, true), tc::op_rows(sI, CT, false), 128, 64, CT, false);
            else if (slot == 1) tc::gemm_ops(tm + R_DQA, tc::op_cols(sK, CT, true), tc::op_rows(sPm, CT, false), 128, 64, CT, false);
            tc::commit(&S.bar);
        }
        // S_0, dS_next, D, V_new^T, -dV_new^T and V are not read again in this item (after the MMA issue, so
        // that no issuer waits behind the copies)
        if (has_next) {
            if (loader) issue_ws1(next);
            l_pend = true;
            if (kRaw) {
                if (loader) fetch_raw(next, 2, S.V);
                v_pend = true;
            }
        }
        finish_phase(false);
        if (iss2) {
            if (slot == 0) tc::gemm_ops(tm + R_DKO, tc::op_cols(sQ, CT, true), tc::op_rows(sPm, CT, true), 128, 64, CT, false);
            else if (slot == 1) tc::gemm(tm + R_TDW, sdWT, CT, false, sT, CT, true, 128, 64, CT, false);
            else if (slot == 2) tc::gemm_ops(tm + C_DT1, tc::op_rows(sdWT, CT, true), tc::op_cols(sK, CT, false), 64, 64, DT, false);
            tc::commit(&S.bar2);
        }
        bool ok2;
        {
            float a[16], b[16], qreg[16];
            tc::ld16(tc::taddr(tm, R_QT + c0), qreg);
            // dq = Gamma (.) dq_inter + dq_intra
            tc::ld16x2(tc::taddr(tm, R_DQI + c0), a, tc::taddr(tm, R_DQA + c0), b);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float gv[8];
                lds8(S.G + c0 + 8 * h, gv);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int t = 8 * h + u;
                    a[t] = gv[u] * a[t] + b[t];
                    dg[t] += qreg[t] * a[t];
                }
            }
            put_pairs16(GRP && hv % G != 0,
                        reinterpret_cast<char *>(P.dq) + (((size_t)(ci.tok0 + c0) * P.Hk + hk) * P.K + k) * esize(P.dqdk_dtype),
                        P.dqdk_dtype, (size_t)P.Hk * P.K, nrow, k < P.K, a);
            ok2 = wait_group2();
            // dk_O
            tc::ld16x2(tc::taddr(tm, R_DKO + c0), b, tc::taddr(tm, R_TDW + c0), a);
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                dk[t] += b[t];
                dg[t] -= kreg[t] * b[t];
            }
            // TdW^T -> dk_W
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float gv[8], bv[8];
                lds8(S.G + c0 + 8 * h, gv);
                lds8(S.beta + c0 + 8 * h, bv);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int t = 8 * h + u;
                    const float x = bv[u] * gv[u] * a[t];
                    dk[t] += x;
                    dg[t] += kreg[t] * x;
                }
            }
            // s = Gamma_j dT1 + dT2 (dT2 came negated); dT = beta_j s -> dT tile; dbeta_j (WY part) =
            // sum_i T_ij s_ij over this warp's 16 rows
            tc::ld16x2(tc::taddr(tm, C_DT1 + c0), a, tc::taddr(tm, C_DT2 + c0), b);
            float x[8], y[8], tr[8];
            tc::split_rows16(a, x);
            tc::split_rows16(b, y);
            {
                const uint4 tv = *reinterpret_cast<const uint4 *>(S.T + tc::tile_off(i64, jh, CT));
                const __half2 *t2 = reinterpret_cast<const __half2 *>(&tv);
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const float2 f = __half22float2(t2[t]);
                    tr[2 * t] = f.x;
                    tr[2 * t + 1] = f.y;
                }
            }
            {
                float gv[8], bv[8];
                lds8(S.G + jh, gv);
                lds8(S.beta + jh, bv);
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const float sv = gv[t] * x[t] - y[t];
                    x[t] = bv[t] * sv;
                    tr[t] *= sv;
                }
            }
            tc::st_tile8(S.dT, i64, jh, CT, x);
            const float s = tc::half_transpose_sum8(tr);
            if ((lane & 8) == 0) S.db_wy[pb][q][jh + (lane & 7)] = s;
        }
        publish_tiles(ok2);
        if (lost) break;

        // ---------------- phase 3: X = dT T^T
        if (iss1) {
            if (slot == 0) tc::gemm(tm + C_X, sdT, CT, false, sT, CT, false, 64, 64, CT, false);
            else if (slot == 1) tc::gemm_ops(tm + C_KK, tc::op_cols(sK, CT, false), tc::op_cols(sK, CT, false), 64, 64, DT, false);
            tc::commit(&S.bar);
        }
        if (has_next && kRaw) {  // Q is not read again in this item
            if (loader) fetch_raw(next, 1, S.Q);
            q_pend = true;
        }
        finish_phase(false);
        {
            float a[16];
            tc::ld16(tc::taddr(tm, C_X + c0), a);
            if (own64) {
                tc::st_tile8(Xs, r64, c0, CT, a);
                tc::st_tile8(Xs, r64, c0 + 8, CT, a + 8);
            }
        }
        publish_tiles(true);
        if (lost) break;

        // ---------------- phase 4: dA' = T^T X; dA = strict_lower(-dA'); E = beta L dA
        if (iss1) {
            if (slot == 0) tc::gemm(tm + C_DA, sT, CT, true, sX, CT, true, 64, 64, CT, false);
            tc::commit(&S.bar);
        }
        finish_phase(false);
        if (has_next) {  // T is not read again in this item
            if (loader) issue_ws2(next);
            t_pend = true;
        }
        {
            float a[16], kk[16], x[8], y[8];
            tc::ld16x2(tc::taddr(tm, C_DA + c0), a, tc::taddr(tm, C_KK + c0), kk);
            tc::split_rows16(a, x);
            tc::split_rows16(kk, y);
            const int i = i64;
            const float gi = S.gam[i], bi = S.beta[i];
            float rb = 0.f, gj[8];
            lds8(S.gam + jh, gj);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const int j = jh + t;
                float e = 0.f;
                if (j < i) {
                    const float L = __expf(gi - gj[t]);
                    const float dA = -x[t];
                    rb += dA * L * y[t];
                    e = bi * L * dA;
                }
                x[t] = e;
            }
            tc::st_tile8(Es, i, jh, CT, x);
            rb += __shfl_xor_sync(0xffffffffu, rb, 16);
            if (lane < 16) S.db_a[pb][wid >> 2][i] = rb;
        }
        publish_tiles(true);
        if (lost) break;

        // ---------------- phase 5: dk_Ar^T = K^T E^T (+), dk_Ac^T = K^T E (-)
        if (iss1) {
            if (slot == 0) tc::gemm_ops(tm + R_DKAR, tc::op_cols(sK, CT, true), tc::op_rows(sE, CT, false), 128, 64, CT, false);
            else if (slot == 1) tc::gemm_ops(tm + R_DKAC, tc::op_cols(sK, CT, true), tc::op_rows(sE, CT, true), 128, 64, CT, false);
            tc::commit(&S.bar);
        }
        finish_phase(false);
        if (has_next && kRaw) {  // K is not read again in this item
            if (loader) fetch_raw(next, 0, S.K);
            k_pend = true;
        }
        {
            float a[16], b[16];
            tc::ld16x2(tc::taddr(tm, R_DKAR + c0), a, tc::taddr(tm, R_DKAC + c0), b);
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                dk[t] += a[t] + b[t];
                dg[t] += kreg[t] * (a[t] - b[t]);
            }
            put_pairs16(GRP && hv % G != 0,
                        reinterpret_cast<char *>(P.dk) + (((size_t)(ci.tok0 + c0) * P.Hk + hk) * P.K + k) * esize(P.dqdk_dtype),
                        P.dqdk_dtype, (size_t)P.Hk * P.K, nrow, k < P.K, dk);
            // gate gradient: column sums over the feature rows
            const float s = tc::warp_transpose_sum16(dg);
            if (lane < 16) S.dg_q[pb][q][c0 + lane] = s;
        }
        if (tid == 0) {  // its sums are added during the next item's first phase (or after the loop)
            S.red_u = (int)u;
            S.red_len = len;
            S.red_tok0 = ci.tok0;
            S.red_hv = hv;
            S.red_b = pb;
        }
        tc::fence_before();
        item = next;
    }
    lost = __syncthreads_or(!okq || lost) != 0;
    if (!lost && tid < CT) reduce_pending();  // the last item's sums
    if (lost) {
        if (tid == 0) flag_status(P.status, ST_TIMEOUT);
        // every barrier phase this thread saw pending completes before the CTA releases its shared and
        // tensor memory: the MMAs of a commit whose wait gave up, the loads armed and not waited for
        if (m_pend) tc::mbar_wait(&S.bar, mpar, DRAIN_LIMIT);
        if (m2_pend) tc::mbar_wait(&S.bar2, mpar2, DRAIN_LIMIT);
        if (l_pend) tc::mbar_wait(&S.lbar, lpar, DRAIN_LIMIT);
        if (t_pend) tc::mbar_wait(&S.tbar, tpar, DRAIN_LIMIT);
        if (k_pend) tc::mbar_wait(&S.kbar, kpar, DRAIN_LIMIT);
        if (q_pend) tc::mbar_wait(&S.qbar, qpar, DRAIN_LIMIT);
        if (v_pend) tc::mbar_wait(&S.vbar, vpar, DRAIN_LIMIT);
    }
    tc::fence_before();
    __syncthreads();
    if (wid == 0) {
        tc::fence_after();
        tc::tmem_dealloc(tm, K4T_TMEM_COLS);
    }
}


template <typename Tin, bool GRP>
static cudaError_t launch_k4_tc_t(const Params &P, cudaStream_t stream) {
    size_t smem = sizeof(K4TSmem);
    cudaError_t e = smem_opt_in((const void *)k4_intra_grad_tc<Tin, GRP>, smem);
    if (e != cudaSuccess) return e;
    int nsm = 0;
    if ((e = device_sm_count(&nsm)) != cudaSuccess) return e;
    const long groups = (long)P.max_chunks * P.Hk;  // the G items of a key-head group run on one CTA
    if (groups == 0) return cudaSuccess;
    CUtensorMap mk, mq, mv;
    memset(&mk, 0, sizeof(mk));
    memset(&mq, 0, sizeof(mq));
    memset(&mv, 0, sizeof(mv));
    if (sizeof(Tin) == 2) {
        const long long tokens = (long long)P.B * P.T;
        if ((e = encode_rows_map(&mk, P.k, P.qkv_dtype, tokens, P.Hk, P.K)) != cudaSuccess) return e;
        if ((e = encode_rows_map(&mq, P.q, P.qkv_dtype, tokens, P.Hk, P.K)) != cudaSuccess) return e;
        if ((e = encode_rows_map(&mv, P.v, P.qkv_dtype, tokens, P.Hv, P.V)) != cudaSuccess) return e;
    }
    const int grid = (int)(groups < nsm ? groups : nsm);  // one persistent CTA per SM
    k4_intra_grad_tc<Tin, GRP><<<grid, K4T_THREADS, smem, stream>>>(P, mk, mq, mv);
    return cudaGetLastError();
}

template <bool GRP>
static cudaError_t launch_k4_tc_g(const Params &P, cudaStream_t stream) {
    if (P.qkv_dtype == F32) return launch_k4_tc_t<float, GRP>(P, stream);
    if (P.qkv_dtype == BF16) return launch_k4_tc_t<__nv_bfloat16, GRP>(P, stream);
    return launch_k4_tc_t<__half, GRP>(P, stream);
}

cudaError_t launch_k4_tc(const Params &P, cudaStream_t stream) {
    return P.G > 1 ? launch_k4_tc_g<true>(P, stream) : launch_k4_tc_g<false>(P, stream);
}

}  // namespace gdr
