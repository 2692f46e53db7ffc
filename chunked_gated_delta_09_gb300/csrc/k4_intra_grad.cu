// k4_intra_grad.cu -- per-chunk gradients with warp-level tensor-core MMAs (one CTA per chunk x head).
//
// Given the state entering the chunk S_0 = h_n, the adjoint of the state leaving it dS_next = dh_n,
// V_new, dV_new and T from the two scans and the WY preparation, this kernel produces the chunk's dq,
// dk, dv, dbeta and the gradient of the chunk-local cumulative gate.  It follows the WY-gradient stage
// of MindSpeed-Ops chunk_kda_bwd.md ("implementation principle": the inter-chunk products
// dq = dO h^T, dk = v_new dh^T, dw = -(dv h^T), then the WY corrections with g, beta and A, and the
// gradient through the triangular inverse dA = -A (dA_pre A) of the dA post kernels).  With
// D = scale dO, M[r, j] = exp(gamma_r - gamma_j) [j <= r], L the strict part of M, K~ = K (.) exp(gamma_C - gamma):
//   P      = (D V_new^T) (.) M
//   dq     = diag(Gamma) D S_0 + P K
//   dk     = P^T Q + K~-rowscale (V_new dS_next) + diag(beta Gamma) T^T dW + E K + E^T K
//   dW     = -dV_new S_0,   dT = dW (diag(beta Gamma) K)^T + dV_new (diag(beta) V)^T
//   dv     = diag(beta) T^T dV_new
//   dA     = strict_lower(-T^T dT T^T),   E = diag(beta) (L (.) dA)
//   dbeta  = rowsum(T^T dW (.) Gamma K) + rowsum(T^T dV_new (.) V) + rowsum(dA (.) L (.) K K^T)
//   dgamma = q (.) dq - k (.) (P^T Q + K~ term) + k (.) (W term + E K - E^T K), plus, on the last row,
//            Gamma_C <S_0, dS_next> + sum_j k_j (.) (K~ term)_j
// (for the scalar gate the dgamma row is summed over channels).  The per-channel (KDA) gate turns each
// decayed C x C product into a per-channel sum that the owner of each output element evaluates directly;
// this kernel serves that gate (the scalar gate runs on k4_intra_grad_tc.cu).  Every decay factor is
// exp of a non-positive argument (a later minus an earlier cumulative log-decay, or a cumulative log-decay
// itself) and is taken with the fast hardware exponential (relative error about 1e-6, below the fp16
// rounding of the operand tiles).
//
// All operands live in shared memory as core-matrix tiles (ctile_off); the workspace tiles arrive by
// bulk copy.  The workspace holds V_new^T and -dV_new^T (tiles [v][c]).
#include "gdr_common.cuh"
#include "gdr_kernels.h"
#include "tc_util.cuh"

namespace gdr {

constexpr int K4_THREADS = 512;
// warp tiling: 16 warps, four row blocks of 16 rows x four column blocks
constexpr int NK = 4;  // C x K tiles: 16 x 32 per warp (four n8 tiles)
constexpr int NC = 2;  // C x C tiles: 16 x 16 per warp (two n8 tiles)
constexpr int GKS = DT + 4;  // row stride (floats) of the per-channel gate tile: 4 mod 32, so that the rows a
                             // fragment's lanes read (several rows, consecutive columns) fall on distinct banks

// Per-channel decayed products on the accumulator layout of a 16 x (8 NK) warp tile (rows r0 = m0 + lane / 4
// and r0 + 8, column pairs c = n0 + 8 nt + 2 (lane % 4) + {0, 1}), A a C x C and X a C x DT fp16 tile, g the
// per-channel cumulative gate [CT] rows at stride GKS:
//   LOWER:  acc[r][c] += sum_{j <= r (INCL) or j < r} A[r][j] X[j][c] exp(g[r][c] - g[j][c])
//   else:   acc[r][c] += sum_{i >= r (INCL) or i > r} A[i][r] X[i][c] exp(g[i][c] - g[r][c])
// Sub-chunk factorisation: the warp's rows form one 16-row block of the chunk.  The terms from the other
// blocks (j below the block for LOWER, i above it otherwise) share a reference row ref on the block boundary
// between them (ref = m0, resp. m0 + 16), and exp(g[r] - g[j]) = exp(g[r] - g[ref]) exp(g[ref] - g[j]) with both
// factors at most 1 (g is non-increasing along the chunk): those terms are one warp MMA over the rescaled
// X~[j][c] = X[j][c] exp(g[ref][c] - g[j][c]) (built straight into the B fragments), times exp(g[r][c] -
// g[ref][c]) per output element.  The 16 x 16 diagonal block splits once more at its middle row: its cross 8 x 8
// quarter the same way, and only the two 8 x 8 triangles term by term, where one pass over the inner index
// serves all 16 elements of a thread and terms outside a row's range are dropped by selection, never by a zero
// factor.
template <bool LOWER, bool INCL>
__device__ __forceinline__ void decayed_acc(float (&acc)[1][NK][4], const unsigned char *A, const unsigned char *X,
                                            const float *g, int m0, int n0, int lane) {
    const int r0 = m0 + (lane >> 2), cq = n0 + 2 * (lane & 3);
    // ---- off-diagonal blocks on the tensor cores
    const int ks_lo = LOWER ? 0 : m0 / 16 + 1, ks_hi = LOWER ? m0 / 16 : CT / 16;  // 16-row k-steps [lo, hi)
    if (ks_lo < ks_hi) {
        const int ref = LOWER ? m0 : m0 + 16;
        float off[1][NK][4];
        zero_acc(off);
        const int bn = lane >> 2;                 // B fragment: column n = n0 + 8 nt + lane / 4
        const int bk = 2 * (lane & 3);            // B fragment: k rows bk, bk + 1 and bk + 8, bk + 9
        float gref_b[NK];
#pragma unroll
        for (int nt = 0; nt < NK; ++nt) gref_b[nt] = g[ref * GKS + n0 + 8 * nt + bn];
        const int r8 = lane & 7, mat = lane >> 3;
        for (int ks = ks_lo; ks < ks_hi; ++ks) {
            const int k0 = 16 * ks;
            uint32_t a[4];
            if (LOWER) ldsm_x4(a, A + ctile_off(m0 + (lane & 15), k0 + (lane >> 4) * 8, CT));
            else ldsm_x4_t(a, A + ctile_off(k0 + r8 + (mat >> 1) * 8, m0 + (mat & 1) * 8, CT));
#pragma unroll
            for (int nt = 0; nt < NK; ++nt) {
                const int c = n0 + 8 * nt + bn;
                float v[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int j = k0 + bk + (q & 1) + 8 * (q >> 1);
                    const float x = ctile_get(X, j, c, DT);
                    // exponent <= 0 on both sides of the reference row
                    v[q] = x * __expf(LOWER ? gref_b[nt] - g[j * GKS + c] : g[j * GKS + c] - gref_b[nt]);
                }
                const __half2 b0 = __floats2half2_rn(v[0], v[1]), b1 = __floats2half2_rn(v[2], v[3]);
                mma16816(off[0][nt], a, *reinterpret_cast<const uint32_t *>(&b0), *reinterpret_cast<const uint32_t *>(&b1));
            }
        }
#pragma unroll
        for (int nt = 0; nt < NK; ++nt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int c = cq + 8 * nt + h;
                const float gr = g[ref * GKS + c];
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int r = r0 + 8 * rr;
                    const float gx = g[r * GKS + c];
                    acc[0][nt][2 * rr + h] += off[0][nt][2 * rr + h] * __expf(LOWER ? gx - gr : gr - gx);
                }
            }
    }
    // ---- the diagonal block: its cross quarter (the warp's upper 8 rows against its lower 8 for LOWER, the
    // reverse otherwise) by the same factorisation around the block's middle row mid = m0 + 8, one k = 8 MMA
    // with the other half's fragment rows left zero; the two 8 x 8 triangles term by term
    const int mid = m0 + 8;
    {
        const int bn = lane >> 2, bk = 2 * (lane & 3);
        uint32_t a0 = 0u, a1 = 0u;
        if (LOWER) a1 = *reinterpret_cast<const uint32_t *>(A + ctile_off(mid + bn, m0 + bk, CT));  // A[r0 + 8][m0 + bk..]
        else a0 = pack_half2(ctile_get(A, mid + bk, r0, CT), ctile_get(A, mid + bk + 1, r0, CT));  // A[mid + bk..][r0]
        float off[NK][4];
#pragma unroll
        for (int nt = 0; nt < NK; ++nt) {
            off[nt][0] = off[nt][1] = off[nt][2] = off[nt][3] = 0.f;
            const int c = n0 + 8 * nt + bn;
            const float gm = g[mid * GKS + c];
            const int j = LOWER ? m0 + bk : mid + bk;  // k rows of the B fragment
            const float v0 = ctile_get(X, j, c, DT) * __expf(LOWER ? gm - g[j * GKS + c] : g[j * GKS + c] - gm);
            const float v1 = ctile_get(X, j + 1, c, DT) * __expf(LOWER ? gm - g[(j + 1) * GKS + c] : g[(j + 1) * GKS + c] - gm);
            mma1688(off[nt], a0, a1, pack_half2(v0, v1));
        }
#pragma unroll
        for (int nt = 0; nt < NK; ++nt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int c = cq + 8 * nt + h;
                const float gm = g[mid * GKS + c];
                if (LOWER) acc[0][nt][2 + h] += off[nt][2 + h] * __expf(g[(r0 + 8) * GKS + c] - gm);  // rows r0 + 8
                else acc[0][nt][h] += off[nt][h] * __expf(gm - g[r0 * GKS + c]);                    // rows r0
            }
    }
    // The two 8 x 8 triangles, term by term.  Row r0 = m0 + g (and r0 + 8 in the other half, with the same
    // terms) has own_n terms, t in order k = 0, 1, .. (t = k below the diagonal, t = 7 - k above it); the lane
    // of row 7 - g in the same column quad (lane ^ 28) has the complement, NPAIR in all.  The two share them
    // evenly: a lane with more than NH terms keeps its first NH and its partner takes the rest (into pacc,
    // returned by one shuffle per accumulator), so every lane runs NH iterations instead of 8.
    constexpr int NPAIR = INCL ? 9 : 7, NH = (NPAIR + 1) / 2;
    const int gq = lane >> 2;
    const int own_n = LOWER ? (INCL ? gq + 1 : gq) : (INCL ? 8 - gq : 7 - gq);
    const int par_n = NPAIR - own_n, own_cap = own_n < NH ? own_n : NH;
    float pacc[NK][4];
#pragma unroll
    for (int nt = 0; nt < NK; ++nt) pacc[nt][0] = pacc[nt][1] = pacc[nt][2] = pacc[nt][3] = 0.f;
#pragma unroll 1  // (rolled: fewer live registers, fewer spills)
    for (int i = 0; i < NH; ++i) {
        const bool mine = i < own_cap;
        const int k = mine ? i : NH + (i - own_n);
        const bool valid = mine || k < par_n;
        const float wm = mine ? 1.f : 0.f, wp = 1.f - wm;
        const int row = m0 + (mine ? gq : 7 - gq);  // this term's row in the first half (second: row + 8)
        const int t = valid ? (LOWER ? k : 7 - k) : 0;  // (k reaches 8 on a spare iteration: keep rows in the tile)
        const int j0 = m0 + t, j1 = mid + t;
        const float a0 = valid ? (LOWER ? ctile_get(A, row, j0, CT) : ctile_get(A, j0, row, CT)) : 0.f;
        const float a1 = valid ? (LOWER ? ctile_get(A, row + 8, j1, CT) : ctile_get(A, j1, row + 8, CT)) : 0.f;
#pragma unroll
        for (int nt = 0; nt < NK; ++nt) {
            const float2 x0 = __half22float2(*reinterpret_cast<const __half2 *>(X + ctile_off(j0, cq + 8 * nt, DT)));
            const float2 x1 = __half22float2(*reinterpret_cast<const __half2 *>(X + ctile_off(j1, cq + 8 * nt, DT)));
            const float2 g0 = *reinterpret_cast<const float2 *>(g + j0 * GKS + cq + 8 * nt);
            const float2 g1 = *reinterpret_cast<const float2 *>(g + j1 * GKS + cq + 8 * nt);
            const float2 r0g = *reinterpret_cast<const float2 *>(g + row * GKS + cq + 8 * nt);
            const float2 r1g = *reinterpret_cast<const float2 *>(g + (row + 8) * GKS + cq + 8 * nt);
            // (an invalid term has a = 0 and its exponent may be positive: it is selected away, never multiplied)
            const float e00 = __expf(LOWER ? r0g.x - g0.x : g0.x - r0g.x);
            const float e01 = __expf(LOWER ? r0g.y - g0.y : g0.y - r0g.y);
            const float e10 = __expf(LOWER ? r1g.x - g1.x : g1.x - r1g.x);
            const float e11 = __expf(LOWER ? r1g.y - g1.y : g1.y - r1g.y);
            const float y0 = valid ? a0 * x0.x * e00 : 0.f, y1 = valid ? a0 * x0.y * e01 : 0.f;
            const float y2 = valid ? a1 * x1.x * e10 : 0.f, y3 = valid ? a1 * x1.y * e11 : 0.f;
            // (y finite: a 0 / 1 weight routes it to this lane's sums or the partner's)
            acc[0][nt][0] = fmaf(wm, y0, acc[0][nt][0]);
            acc[0][nt][1] = fmaf(wm, y1, acc[0][nt][1]);
            acc[0][nt][2] = fmaf(wm, y2, acc[0][nt][2]);
            acc[0][nt][3] = fmaf(wm, y3, acc[0][nt][3]);
            pacc[nt][0] = fmaf(wp, y0, pacc[nt][0]);
            pacc[nt][1] = fmaf(wp, y1, pacc[nt][1]);
            pacc[nt][2] = fmaf(wp, y2, pacc[nt][2]);
            pacc[nt][3] = fmaf(wp, y3, pacc[nt][3]);
        }
    }
#pragma unroll
    for (int nt = 0; nt < NK; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[0][nt][e] += __shfl_xor_sync(0xffffffffu, pacc[nt][e], 28);
}

struct __align__(1024) K4Smem {
    unsigned char Qs[CT * DT * 2], Ks[CT * DT * 2], Vs[CT * DT * 2], Ds[CT * DT * 2];
    unsigned char VnT[DT * CT * 2], NdVT[DT * CT * 2];  // V_new^T, -dV_new^T  [v][c]
    unsigned char Hs[DT * DT * 2], dHs[DT * DT * 2];    // [v][k]
    unsigned char Ts[CT * CT * 2], Pms[CT * CT * 2];
    float gam[CT];
    float G[CT], GC[CT];  // exp(gamma), exp(gamma_C - gamma) (scalar gate)
    float beta[CT];
    // partial sums in fixed slots, added in a fixed order (results do not depend on warp timing)
    float dbp[8][CT];    // dbeta: [0..3] from dA (by column block), [4..7] from T^T dW / T^T dV_new (by K block)
    float dgp[4][CT];    // scalar gate: per-row gate-gradient sums by K block
    float lrs[32];       // scalar gate: last-row terms, [w] from dk_SC and [16 + w] from <S_0, dS_next>
    float lrp[8][DT];    // per-channel gate: last-row terms, [0..3] from dk_SC (by row block), [4..7] from
                         // <S_0, dS_next> (by row quarter)
    uint64_t lbar;
};

// Store a warp's accumulator tile (16 rows x 8 NT columns of a C x K block) as an output gradient row block
// (column pairs).
template <int NT>
__device__ __forceinline__ void store_ck(const float (&a)[1][NT][4], int m0, int n0, int len, int ncols, void *base,
                                         size_t row_stride, int dt) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
            int r = acc_row(m0, 0, e), c = acc_col(n0, nt, e);  // c is even and ncols a multiple of 8
            if (r < len && c < ncols) store_pair(base, (size_t)r * row_stride + c, a[0][nt][e], a[0][nt][e + 1], dt);
        }
}

// WY = true: the WY-gradient stage taken alone (MindSpeed-Ops chunk_kda_bwd.md,
// chunk_kda_bwd_wy_dqkg_fused): no intra-chunk attention terms (P, dq_intra, dk_O) and no terms through A_kk
// (E, dk_Ar, dk_Ac, the A part of dbeta); instead dA = strict_lower(-T^T dT T^T) is written out, and the
// gradient of the cumulative gate goes straight to dg (no reverse cumsum follows).
template <typename Tin, bool PC, bool WY>
__global__ void __launch_bounds__(K4_THREADS, 1) k4_intra_grad(const Params P) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    K4Smem &S = *reinterpret_cast<K4Smem *>(smem_raw);
    float *gamK = reinterpret_cast<float *>(smem_raw + sizeof(K4Smem));  // [CT] rows at stride GKS, per-channel only
    // per-channel gate: the decayed key Gram tile (from the WY preparation), fetched with the item's other tiles
    unsigned char *Kds = reinterpret_cast<unsigned char *>(gamK + CT * GKS);
    constexpr bool kKd = PC && !WY;
    // buffers reused once their first owner is done
    unsigned char *dWs = S.Ds;     // dW [r][k]          after dq
    unsigned char *KGb = S.Qs;     // beta Gamma K       after dk_O (per-channel)
    unsigned char *dTs = S.Pms;    // dT                 after dk_O
    unsigned char *Xs = S.VnT;     // dT T^T (C x C)     after dk_SC
    unsigned char *Es = S.Pms;     // E                  after X

    if (*P.status & ST_BAD_SEQLENS) return;
    const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
    // Persistent CTAs take the items (chunk n, value head hv), item = n Hv + hv, round-robin.  The workspace
    // tiles of a CTA's next item are bulk-copied into each buffer as soon as the current item is done with
    // it (three groups, all counted on one barrier phase per item), so their transfer overlaps the compute.
    const int n_items = P.max_chunks * P.Hv;
    auto valid_from = [&](int it) -> int {
        ChunkInfo t;
        while (it < n_items && !chunk_info(P, it / P.Hv, t)) it += gridDim.x;
        return it;
    };
    constexpr uint32_t kBytesHdH = 2 * DT * DT * 2, kBytesDdV = CT * DT * 2 + DT * CT * 2,
                       kBytesTVn = CT * CT * 2 + DT * CT * 2 + (kKd ? CT * CT * 2 : 0);
    auto issue_HdH = [&](size_t un) {  // expects the whole item's bytes, so it comes first
        tc::mbar_expect_tx(&S.lbar, kBytesHdH + kBytesDdV + kBytesTVn);
        tc::bulk_g2s(S.Hs, P.h + un * DT * DT, DT * DT * 2, &S.lbar);
        tc::bulk_g2s(S.dHs, P.dh + un * DT * DT, DT * DT * 2, &S.lbar);
    };
    auto issue_DdV = [&](size_t un) {
        tc::bulk_g2s(S.Ds, P.Dt + un * CT * DT, CT * DT * 2, &S.lbar);
        tc::bulk_g2s(S.NdVT, P.dVn + un * DT * CT, DT * CT * 2, &S.lbar);
    };
    auto issue_TVn = [&](size_t un) {
        tc::bulk_g2s(S.Ts, P.Tm + un * CT * CT, CT * CT * 2, &S.lbar);
        tc::bulk_g2s(S.VnT, P.Vn + un * DT * CT, DT * CT * 2, &S.lbar);
        if (kKd) tc::bulk_g2s(Kds, P.Kd + un * CT * CT, CT * CT * 2, &S.lbar);
    };
    int item = valid_from(blockIdx.x);
    if (item >= n_items) return;
    if (tid == 0) {
        tc::mbar_init(&S.lbar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        issue_HdH(item);
        issue_DdV(item);
        issue_TVn(item);
    }
    uint32_t parity = 0;
    while (item < n_items) {
        const int n = item / P.Hv, hv = item % P.Hv, hk = hv / P.G;
        ChunkInfo ci;
        chunk_info(P, n, ci);
        const size_t u = (size_t)item;  // = n Hv + hv
        const int len = ci.len;
        const int next = valid_from(item + gridDim.x);
        const bool has_next = next < n_items;

        // ---- stage the inputs as fp16 tiles (the workspace tiles are already on their way); the per-channel gate
        // tile (workspace, contiguous) by asynchronous 16-byte copies issued first, so that they overlap
        if (PC) {
            for (int e = 4 * tid; e < CT * DT; e += 4 * K4_THREADS)
                cp_async16(gamK + (e / DT) * GKS + e % DT, P.gam + u * CT * DT + e);
            cp_async_commit();
        }
        const Tin *kp = reinterpret_cast<const Tin *>(P.k) + ((size_t)ci.tok0 * P.Hk + hk) * P.K;
        const Tin *qp = reinterpret_cast<const Tin *>(P.q) + ((size_t)ci.tok0 * P.Hk + hk) * P.K;
        const Tin *vp = reinterpret_cast<const Tin *>(P.v) + ((size_t)ci.tok0 * P.Hv + hv) * P.V;
        {
            unsigned char *const dst[3] = {S.Ks, S.Qs, S.Vs};
            const Tin *const src[3] = {kp, qp, vp};
            const size_t st[3] = {(size_t)P.Hk * P.K, (size_t)P.Hk * P.K, (size_t)P.Hv * P.V};
            const int nc[3] = {P.K, P.K, P.V};
            const float mul[3] = {1.f, 1.f, 1.f};
            stage_ct_n<Tin, K4_THREADS, 3>(dst, src, st, nc, mul, len, tid);
        }
        if (tid < CT) {
            S.beta[tid] = tid < len ? load_scalar(P.beta, (size_t)(ci.tok0 + tid) * P.Hv + hv, P.beta_dtype) : 0.f;
            if (!PC) S.gam[tid] = P.gam[u * CT + tid];
        }
        if (PC) cp_async_wait<0>();
        __syncthreads();  // barrier initialised (first item); the gate tile landed
        if (!PC && tid < CT) {
            S.G[tid] = __expf(S.gam[tid]);
            S.GC[tid] = __expf(S.gam[len - 1] - S.gam[tid]);
        }
        const bool loaded = tc::mbar_wait(&S.lbar, parity, P.spin);
        if (__syncthreads_or(!loaded)) {
            if (tid == 0) {
                flag_status(P.status, ST_TIMEOUT);
                tc::mbar_wait(&S.lbar, parity, DRAIN_LIMIT);  // this item's tiles land before the CTA exits
            }
            return;
        }
        parity ^= 1u;

        // C x K tiling: warp w owns rows m0 .. m0+15 and columns n0 .. n0+31
        const int m0 = (wid & 3) * 16, n0 = (wid >> 2) * (NK * 8);
        // C x C tiling: rows cm0 .. cm0+15, columns cn0 .. cn0+15
        const int cm0 = (wid & 3) * 16, cn0 = (wid >> 2) * (NC * 8);
        auto G_ = [&](int r, int c) -> float { return PC ? gamK[r * GKS + c] : S.gam[r]; };
        auto Kv = [&](int r, int c) -> float { return ctile_get(S.Ks, r, c, DT); };
        const int rl = len - 1;
        auto row_dbeta = [&](int r) -> float {
            float x = 0.f;
#pragma unroll
            for (int i = WY ? 4 : 0; i < 8; ++i) x += S.dbp[i][r];
            return x;
        };

        // ---- S1: P = (D V_new^T) (.) causal mask (.) [scalar: decay]
        if (!WY) {
            float g1[1][NC][4];
            zero_acc(g1);
            warp_mma_ct<1, NC, false, false>(g1, S.Ds, DT, S.VnT, CT, cm0, cn0, DT);
#pragma unroll
            for (int nt = 0; nt < NC; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    int r = acc_row(cm0, 0, e), j = acc_col(cn0, nt, e);
                    float x = 0.f;
                    if (j <= r) x = PC ? g1[0][nt][e] : g1[0][nt][e] * __expf(S.gam[r] - S.gam[j]);
                    ctile_set(S.Pms, r, j, CT, x);
                }
        }
        __syncthreads();

        // gate-gradient contributions: per element for the per-channel gate, per row for the scalar gate
        float dgam[1][PC ? NK : 1][4];
        float rsg[2] = {0.f, 0.f};
        float dk[1][NK][4];
        zero_acc(dgam);
        auto add_dg = [&](int nt, int e, float x) {
            if (PC) dgam[0][PC ? nt : 0][e] += x;
            else rsg[e >> 1] += x;
        };
        // ---- S2: dq = Gamma (.) (D S_0) + P K   [per-channel: decayed sum per element]
        {
            float dq[1][NK][4];
            zero_acc(dq);
            warp_mma_ct<1, NK, false, false>(dq, S.Ds, DT, S.Hs, DT, m0, n0, DT);
#pragma unroll
            for (int nt = 0; nt < NK; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    dq[0][nt][e] *= PC ? __expf(G_(acc_row(m0, 0, e), acc_col(n0, nt, e))) : S.G[acc_row(m0, 0, e)];
            if (WY) {
            } else if (!PC) {
                warp_mma_ct<1, NK, false, false>(dq, S.Pms, CT, S.Ks, DT, m0, n0, CT);
            } else {
                decayed_acc<true, true>(dq, S.Pms, S.Ks, gamK, m0, n0, lane);
            }
#pragma unroll
            for (int nt = 0; nt < NK; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    int r = acc_row(m0, 0, e), c = acc_col(n0, nt, e);
                    add_dg(nt, e, ctile_get(S.Qs, r, c, DT) * dq[0][nt][e]);
                }
            if (P.G == 1)
                store_ck(dq, m0, n0, len, P.K, reinterpret_cast<char *>(P.dq) + ((size_t)ci.tok0 * P.Hk + hk) * P.K *
                         (P.dqdk_dtype == F32 ? 4 : 2), (size_t)P.Hk * P.K, P.dqdk_dtype);
            else
                store_ck(dq, m0, n0, len, P.K, gqa_part(P.dq_h, ((size_t)ci.tok0 * P.Hv + hv) * P.K, P), (size_t)P.Hv * P.K,
                         gqa_part_dtype(P));
        }
        // ---- S3: dk_O = P^T Q
        {
            zero_acc(dk);
            if (WY) {
            } else if (!PC) {
                warp_mma_ct<1, NK, true, false>(dk, S.Pms, CT, S.Qs, DT, m0, n0, CT);
            } else {
                decayed_acc<false, true>(dk, S.Pms, S.Qs, gamK, m0, n0, lane);
            }
#pragma unroll
            for (int nt = 0; nt < NK; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    int r = acc_row(m0, 0, e), c = acc_col(n0, nt, e);
                    add_dg(nt, e, -(Kv(r, c) * dk[0][nt][e]));
                }
        }
        __syncthreads();  // Ds, Pms, Qs free

        // ---- S4: dk_SC = exp(gamma_C - gamma) (.) (V_new dS_next); last-row gate terms
        {
            float t[1][NK][4];
            zero_acc(t);
            warp_mma_ct<1, NK, true, false>(t, S.VnT, CT, S.dHs, DT, m0, n0, DT);
            float part = 0.f, colp[PC ? NK : 1][2];
#pragma unroll
            for (int nt = 0; nt < (PC ? NK : 1); ++nt) colp[nt][0] = colp[nt][1] = 0.f;
#pragma unroll
            for (int nt = 0; nt < NK; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    int r = acc_row(m0, 0, e), c = acc_col(n0, nt, e);
                    float x = t[0][nt][e] * (PC ? __expf(G_(rl, c) - G_(r, c)) : S.GC[r]);
                    float kx = Kv(r, c) * x;
                    dk[0][nt][e] += x;
                    add_dg(nt, e, -(kx));
                    if (PC) colp[PC ? nt : 0][e & 1] += kx;
                    else part += kx;
                }
            if (!PC) {
                float s = part;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                if (lane == 0) S.lrs[wid] = s;
            } else {
                // column sums over the warp's 16 rows: lanes that differ in lane / 4 share columns
#pragma unroll
                for (int nt = 0; nt < (PC ? NK : 1); ++nt)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        float s = colp[nt][h];
                        s += __shfl_xor_sync(0xffffffffu, s, 4);
                        s += __shfl_xor_sync(0xffffffffu, s, 8);
                        s += __shfl_xor_sync(0xffffffffu, s, 16);
                        if (lane < 4) S.lrp[wid & 3][acc_col(n0, nt, h)] = s;
                    }
            }
            // Gamma_C <S_0, dS_next> per channel (summed over channels for the scalar gate).  Warp w takes the
            // 8-column chunk 4 (w % 4) + lane / 8 over rows 32 (w / 4) .. +31; the 8 lanes of a quarter-warp read
            // the 8 rows of one core matrix (16-byte reads, no bank conflicts)
            {
                const int c8 = 8 * (4 * (wid & 3) + (lane >> 3));
                float acc8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t off = ctile_off(32 * (wid >> 2) + 8 * j + (lane & 7), c8, DT);
                    const __half2 *a2 = reinterpret_cast<const __half2 *>(S.Hs + off);
                    const __half2 *b2 = reinterpret_cast<const __half2 *>(S.dHs + off);
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        float2 a = __half22float2(a2[t]), b = __half22float2(b2[t]);
                        acc8[2 * t] += a.x * b.x;
                        acc8[2 * t + 1] += a.y * b.y;
                    }
                }
                if (PC) {
                    // lanes that differ in lane % 8 hold the same column chunk
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        float s = acc8[t];
                        s += __shfl_xor_sync(0xffffffffu, s, 1);
                        s += __shfl_xor_sync(0xffffffffu, s, 2);
                        s += __shfl_xor_sync(0xffffffffu, s, 4);
                        if ((lane & 7) == 0) S.lrp[4 + (wid >> 2)][c8 + t] = s * __expf(G_(rl, c8 + t));
                    }
                } else {
                    float s = 0.f;
#pragma unroll
                    for (int t = 0; t < 8; ++t) s += acc8[t];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                    if (lane == 0) S.lrs[16 + wid] = s * __expf(S.gam[rl]);
                }
            }
        }
        // ---- S5: dW = -dV_new S_0 (the stored tile is -dV_new^T)  -> dWs;  per-channel: beta Gamma K -> KGb
        {
            float t[1][NK][4];
            zero_acc(t);
            warp_mma_ct<1, NK, true, false>(t, S.NdVT, CT, S.Hs, DT, m0, n0, DT);
#pragma unroll
            for (int nt = 0; nt < NK; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    int r = acc_row(m0, 0, e), c = acc_col(n0, nt, e);
                    *reinterpret_cast<__half2 *>(dWs + ctile_off(r, c, DT)) = __floats2half2_rn(t[0][nt][e], t[0][nt][e + 1]);
                }
            if (PC) {  // 8 columns of one row per step; the 8 lanes of a quarter-warp take the 8 rows of a core matrix
                for (int e = tid; e < CT * DT / 8; e += K4_THREADS) {
                    const int r = e & (CT - 1), c8 = 8 * (e >> 6);
                    const uint4 kv = *reinterpret_cast<const uint4 *>(S.Ks + ctile_off(r, c8, DT));
                    const float4 ga = *reinterpret_cast<const float4 *>(gamK + r * GKS + c8);
                    const float4 gb = *reinterpret_cast<const float4 *>(gamK + r * GKS + c8 + 4);
                    const float gv[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
                    const __half2 *k2 = reinterpret_cast<const __half2 *>(&kv);
                    const float b = S.beta[r];
                    float f[8];
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const float2 kf = __half22float2(k2[t]);
                        f[2 * t] = b * __expf(gv[2 * t]) * kf.x;
                        f[2 * t + 1] = b * __expf(gv[2 * t + 1]) * kf.y;
                    }
                    *reinterpret_cast<uint4 *>(KGb + ctile_off(r, c8, DT)) = pack8_half(f);
                }
            }
        }
        __syncthreads();
        if (tid == 0 && has_next) {  // H and dH are read for the last time in S4 / S5
            tc::fence_smem_to_async();
            issue_HdH(next);
        }

        // ---- S6: dT = dW (beta Gamma K)^T + dV_new (beta V)^T  -> dTs
        {
            float a[1][NC][4], b[1][NC][4];
            zero_acc(a);
            zero_acc(b);
            warp_mma_ct<1, NC, false, true>(a, dWs, DT, PC ? KGb : S.Ks, DT, cm0, cn0, DT);
            warp_mma_ct<1, NC, true, true>(b, S.NdVT, CT, S.Vs, DT, cm0, cn0, DT);  // = -(dV_new V^T)
#pragma unroll
            for (int nt = 0; nt < NC; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    int r = acc_row(cm0, 0, e), j = acc_col(cn0, nt, e);
                    float x = (PC ? a[0][nt][e] : a[0][nt][e] * S.beta[j] * S.G[j]) - b[0][nt][e] * S.beta[j];
                    ctile_set(dTs, r, j, CT, x);
                }
        }
        // ---- S7: T^T dW -> dk_W, dbeta, dgamma
        float rowb[2] = {0.f, 0.f};  // dbeta partials for rows m0 + lane/4 and +8
        {
            float t[1][NK][4];
            zero_acc(t);
            warp_mma_ct<1, NK, true, false>(t, S.Ts, CT, dWs, DT, m0, n0, CT);
#pragma unroll
            for (int nt = 0; nt < NK; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    int r = acc_row(m0, 0, e), c = acc_col(n0, nt, e);
                    float Gm = PC ? __expf(G_(r, c)) : S.G[r];
                    float kv = Kv(r, c);
                    float x = S.beta[r] * Gm * t[0][nt][e];
                    dk[0][nt][e] += x;
                    add_dg(nt, e, kv * x);
                    rowb[e >> 1] += t[0][nt][e] * kv * Gm;
                }
        }
        // ---- S8: T^T dV_new -> dv, dbeta  (negated tile: product is -T^T dV_new)
        {
            float t[1][NK][4];
            zero_acc(t);
            warp_mma_ct<1, NK, true, true>(t, S.Ts, CT, S.NdVT, CT, m0, n0, CT);
#pragma unroll
            for (int nt = 0; nt < NK; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    int r = acc_row(m0, 0, e), c = acc_col(n0, nt, e);
                    float x = -t[0][nt][e];
                    rowb[e >> 1] += x * ctile_get(S.Vs, r, c, DT);
                    t[0][nt][e] = S.beta[r] * x;
                }
            store_ck(t, m0, n0, len, P.V, reinterpret_cast<char *>(P.dv) + ((size_t)ci.tok0 * P.Hv + hv) * P.V *
                     (P.dv_dtype == F32 ? 4 : 2), (size_t)P.Hv * P.V, P.dv_dtype);
        }
        __syncthreads();  // dTs complete; D (as dW) and -dV_new^T read for the last time
        if (tid == 0 && has_next) {
            tc::fence_smem_to_async();
            issue_DdV(next);
        }

        // ---- S9: X = dT T^T -> Xs
        {
            float x[1][NC][4];
            zero_acc(x);
            warp_mma_ct<1, NC, false, true>(x, dTs, CT, S.Ts, CT, cm0, cn0, CT);
#pragma unroll
            for (int nt = 0; nt < NC; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    int r = acc_row(cm0, 0, e), j = acc_col(cn0, nt, e);
                    *reinterpret_cast<__half2 *>(Xs + ctile_off(r, j, CT)) = __floats2half2_rn(x[0][nt][e], x[0][nt][e + 1]);
                }
        }
        __syncthreads();
        // ---- S10: dA = strict_lower(-T^T X); dbeta from A; E = beta (.) L (.) dA -> Es
        {
            float da[1][NC][4], kk[1][NC][4];
            zero_acc(da);
            warp_mma_ct<1, NC, true, false>(da, S.Ts, CT, Xs, CT, cm0, cn0, CT);
            if (WY) {  // the stage's output: dA [token][chunk position], strictly lower, fp32
#pragma unroll
                for (int nt = 0; nt < NC; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; e += 2) {
                        const int i = acc_row(cm0, 0, e), j = acc_col(cn0, nt, e);  // j even
                        if (i < len && j < P.BT) {
                            float2 x = make_float2(j < i ? -da[0][nt][e] : 0.f, j + 1 < i ? -da[0][nt][e + 1] : 0.f);
                            *reinterpret_cast<float2 *>(P.dA_out + ((size_t)(ci.tok0 + i) * P.Hv + hv) * P.BT + j) = x;
                        }
                    }
            }
            if (!PC && !WY) {
                zero_acc(kk);
                warp_mma_ct<1, NC, false, true>(kk, S.Ks, DT, S.Ks, DT, cm0, cn0, DT);
            }
            float rb[2] = {0.f, 0.f};
#pragma unroll
            for (int nt = 0; nt < NC; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    int i = acc_row(cm0, 0, e), j = acc_col(cn0, nt, e);
                    float dA = j < i ? -da[0][nt][e] : 0.f;
                    float L = 1.f, kkd = 0.f;
                    if (!WY && j < i) {
                        if (!PC) {
                            L = __expf(S.gam[i] - S.gam[j]);
                            kkd = L * kk[0][nt][e];
                        } else {  // the decayed key Gram, formed by the WY preparation
                            kkd = ctile_get(Kds, i, j, CT);
                        }
                    }
                    rb[e >> 1] += dA * kkd;
                    if (!WY) ctile_set(Es, i, j, CT, S.beta[i] * (PC ? 1.f : L) * dA);
                }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float s = rb[h];
                s += __shfl_xor_sync(0xffffffffu, s, 1);
                s += __shfl_xor_sync(0xffffffffu, s, 2);
                if ((lane & 3) == 0) S.dbp[wid >> 2][cm0 + (lane >> 2) + 8 * h] = s;
            }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float s = rowb[h];
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            if ((lane & 3) == 0) S.dbp[4 + (wid >> 2)][m0 + (lane >> 2) + 8 * h] = s;
        }
        __syncthreads();
        if (tid == 0 && has_next) {  // T, V_new^T (as X) and the decayed key Gram read for the last time in S10
            tc::fence_smem_to_async();
            issue_TVn(next);
        }
        // ---- S11: dk_Ar = E K (+), dk_Ac = E^T K (-)
        if (!WY) {
            float a[1][NK][4], b[1][NK][4];
            zero_acc(a);
            zero_acc(b);
            if (!PC) {
                warp_mma_ct<1, NK, false, false>(a, Es, CT, S.Ks, DT, m0, n0, CT);
                warp_mma_ct<1, NK, true, false>(b, Es, CT, S.Ks, DT, m0, n0, CT);
            } else {
                decayed_acc<true, false>(a, Es, S.Ks, gamK, m0, n0, lane);
                decayed_acc<false, false>(b, Es, S.Ks, gamK, m0, n0, lane);
            }
#pragma unroll
            for (int nt = 0; nt < NK; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    int r = acc_row(m0, 0, e), c = acc_col(n0, nt, e);
                    float kv = Kv(r, c);
                    dk[0][nt][e] += a[0][nt][e] + b[0][nt][e];
                    add_dg(nt, e, kv * (a[0][nt][e] - b[0][nt][e]));
                }
        }
        // ---- dk out
        if (P.G == 1)
            store_ck(dk, m0, n0, len, P.K, reinterpret_cast<char *>(P.dk) + ((size_t)ci.tok0 * P.Hk + hk) * P.K *
                     (P.dqdk_dtype == F32 ? 4 : 2), (size_t)P.Hk * P.K, P.dqdk_dtype);
        else
            store_ck(dk, m0, n0, len, P.K, gqa_part(P.dk_h, ((size_t)ci.tok0 * P.Hv + hv) * P.K, P), (size_t)P.Hv * P.K,
                     gqa_part_dtype(P));

        // ---- gate gradient of the cumulative gate
        if (!PC) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float s = rsg[h];
                s += __shfl_xor_sync(0xffffffffu, s, 1);
                s += __shfl_xor_sync(0xffffffffu, s, 2);
                if ((lane & 3) == 0) S.dgp[wid >> 2][m0 + (lane >> 2) + 8 * h] = s;
            }
            __syncthreads();
            if (tid < CT) {
                float x = (S.dgp[0][tid] + S.dgp[1][tid]) + (S.dgp[2][tid] + S.dgp[3][tid]);
                if (tid == rl) {
                    float l = 0.f;
#pragma unroll
                    for (int i = 0; i < 32; ++i) l += S.lrs[i];
                    x += l;
                }
                P.dgam[u * CT + tid] = tid < len ? x : 0.f;
                if (tid < len) P.dbeta[(size_t)(ci.tok0 + tid) * P.Hv + hv] = row_dbeta(tid);
            }
        } else {
            __syncthreads();
#pragma unroll
            for (int nt = 0; nt < NK; ++nt)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {  // column pairs c, c + 1 (c even)
                    const int r = acc_row(m0, 0, e), c = acc_col(n0, nt, e);
                    float x[2] = {dgam[0][PC ? nt : 0][e], dgam[0][PC ? nt : 0][e + 1]};
                    if (r == rl) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            float l = 0.f;
#pragma unroll
                            for (int i = 0; i < 8; ++i) l += S.lrp[i][c + h];
                            x[h] += l;
                        }
                    }
                    if (WY) {  // gradient of the cumulative gate, straight to the output
#pragma unroll
                        for (int h = 0; h < 2; ++h)
                            if (r < len && c + h < P.K) P.dg[((size_t)(ci.tok0 + r) * P.Hv + hv) * P.K + c + h] = x[h];
                    } else {
                        *reinterpret_cast<float2 *>(P.dgam + (u * CT + r) * DT + c) =
                            r < len ? make_float2(x[0], x[1]) : make_float2(0.f, 0.f);
                    }
                }
            if (tid < len) P.dbeta[(size_t)(ci.tok0 + tid) * P.Hv + hv] = row_dbeta(tid);
        }
        __syncthreads();  // the next item overwrites the staged inputs and the partial-sum slots
        item = next;
    }
}

template <typename Tin, bool PC, bool WY = false>
static cudaError_t launch_k4_t(const Params &P, cudaStream_t stream) {
    static_assert(sizeof(K4Smem) + sizeof(float) * CT * GKS + CT * CT * 2 <= 227 * 1024,
                  "the per-channel kernel's shared memory exceeds the 227 KB a CTA can have");
    size_t smem = sizeof(K4Smem) + (PC ? sizeof(float) * CT * GKS : 0) + (PC && !WY ? CT * CT * 2 : 0);
    cudaError_t e = smem_opt_in((const void *)k4_intra_grad<Tin, PC, WY>, smem);
    if (e != cudaSuccess) return e;
    int nsm = 0;
    if ((e = device_sm_count(&nsm)) != cudaSuccess) return e;
    const long items = (long)P.max_chunks * P.Hv;
    if (items == 0) return cudaSuccess;
    const int grid = (int)(items < nsm ? items : nsm);  // one persistent CTA per SM
    k4_intra_grad<Tin, PC, WY><<<grid, K4_THREADS, smem, stream>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_k4(const Params &P, cudaStream_t stream) {
    if (P.qkv_dtype == F32) return P.per_channel ? launch_k4_t<float, true>(P, stream) : launch_k4_t<float, false>(P, stream);
    if (P.qkv_dtype == BF16)
        return P.per_channel ? launch_k4_t<__nv_bfloat16, true>(P, stream) : launch_k4_t<__nv_bfloat16, false>(P, stream);
    return P.per_channel ? launch_k4_t<__half, true>(P, stream) : launch_k4_t<__half, false>(P, stream);
}

// The WY-gradient stage alone (per-channel gate, dq / dk in fp32).
cudaError_t launch_k4_wy(const Params &P, cudaStream_t stream) {
    if (P.qkv_dtype == F32) return launch_k4_t<float, true, true>(P, stream);
    if (P.qkv_dtype == BF16) return launch_k4_t<__nv_bfloat16, true, true>(P, stream);
    return launch_k4_t<__half, true, true>(P, stream);
}

}  // namespace gdr
