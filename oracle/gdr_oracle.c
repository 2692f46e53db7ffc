/*
 * gdr_oracle.c -- fp64 CPU oracle for the gated delta rule forward and its exact backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, the smoke check and the CPU-baseline leg of the benchmark
 * load this file's library.  The CUDA product path never calls, links or includes it, and it shares
 * no code with the CUDA sources.
 *
 * What it computes (one unit = one packed sequence x one value head; the recurrence is the one stated
 * for Gated DeltaNet, "FlashQLA backward explained" (gtnt.cn/news/163832) section 1, which lists the
 * six gradients dq, dk, dv, dg, db, dh0 of one backward call):
 *
 *   S_t = e^{g_t} S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,       S in R^{V x K}, S_0 = h0
 *   o_t = scale * S_t q_t
 *   L   = sum_t <o_t, dO_t> + <S_T, dht>
 *
 * Per-channel (KDA) gate: e^{g_t} becomes diag(e^{g_t}) acting on the K index, S_{t-1} diag(e^{g_t}),
 * g given as [T, H, K] fp32 "gate log values" (MindSpeed-Ops chunk_kda_bwd.md, input table).
 *
 * The backward is the hand-derived reverse-mode adjoint of the token recurrence, not of any chunked
 * form: with S' = e^{g_t} S_{t-1}, u = S' k_t, delta = v_t - u and y = dS k_t,
 *   dS  += scale dO_t q_t^T          (output of step t)
 *   dq_t = scale S_t^T dO_t
 *   dv_t = b_t y,   db_t = delta . y,   dk_t = b_t (dS^T delta - S'^T y)
 *   dS'  = dS - b_t y k_t^T,  dg_t = <dS', S'>_F  (KDA: column sums of dS' (.) S'),  dS = e^{g_t} dS'
 * dg is the gradient with respect to the raw per-token log-gate (the chunk-local cumulative sum that
 * a chunked kernel works with is never formed here).  GQA: value head hv reads key head hv / (Hv/Hk)
 * and dq/dk are summed over the value heads of each key head group.
 *
 * The forward keeps a checkpoint of S every CKPT tokens; the backward recomputes the states of one
 * checkpoint segment at a time.  Everything is double precision, plain loops, OpenMP over
 * (sequence, key head) groups so that the GQA sums never race.
 *
 * The `mutation` argument plants one deliberate mistake (1..8) so that the tests can show that the
 * finite-difference pins catch each of them; 0 is the correct oracle.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define CKPT 64

typedef struct {
    int num_seqs;
    const int64_t *cu; /* [num_seqs+1] token offsets into the packed token axis */
    int Hk, Hv, K, V, per_channel;
    double scale;
    const double *q, *k, *v, *beta, *g, *h0;
} prob_t;

/* Strided views of one token of one head. */
static inline const double *qk_row(const double *x, const prob_t *p, int64_t t, int hk) {
    return x + ((size_t)t * p->Hk + hk) * p->K;
}
static inline const double *v_row(const double *x, const prob_t *p, int64_t t, int hv) {
    return x + ((size_t)t * p->Hv + hv) * p->V;
}
static inline const double *g_row(const prob_t *p, int64_t t, int hv) {
    return p->g + ((size_t)t * p->Hv + hv) * (p->per_channel ? p->K : 1);
}

/* S <- S' = gate(S): scalar gate multiplies every entry, per-channel gate scales column c by e^{g[c]}. */
static void apply_gate(double *S, const double *gt, const prob_t *p) {
    int V = p->V, K = p->K;
    if (p->per_channel) {
        for (int i = 0; i < V; ++i)
            for (int c = 0; c < K; ++c) S[(size_t)i * K + c] *= exp(gt[c]);
    } else {
        double e = exp(gt[0]);
        for (size_t i = 0; i < (size_t)V * K; ++i) S[i] *= e;
    }
}

/* One forward step in place: S <- S' + b (v - S' k) k^T, with S' = gate(S). */
static void step_forward(double *S, double *u, const double *kt, const double *vt, double bt,
                         const double *gt, const prob_t *p) {
    int V = p->V, K = p->K;
    apply_gate(S, gt, p);
    for (int i = 0; i < V; ++i) {
        double acc = 0.0;
        for (int c = 0; c < K; ++c) acc += S[(size_t)i * K + c] * kt[c];
        u[i] = acc;
    }
    for (int i = 0; i < V; ++i) {
        double d = bt * (vt[i] - u[i]);
        for (int c = 0; c < K; ++c) S[(size_t)i * K + c] += d * kt[c];
    }
}

/*
 * Forward of all units.  Outputs (each may be NULL):
 *   o      [T, Hv, V]        o_t = scale S_t q_t
 *   hT     [N, Hv, V, K]     final state of each sequence
 *   states [NC, Hv, V, K]    the state entering each chunk of BTs tokens, chunks enumerated
 *                            sequence-major then chunk ascending (NC = sum_s ceil(L_s / BTs))
 */
int gdr_oracle_fwd(int num_seqs, const int64_t *cu, int Hk, int Hv, int K, int V, int per_channel,
                   double scale, const double *q, const double *k, const double *v, const double *beta,
                   const double *g, const double *h0, double *o, double *hT, int BTs, double *states,
                   int nthreads) {
    if (num_seqs < 0 || Hk <= 0 || Hv <= 0 || Hv % Hk || K <= 0 || V <= 0) return 1;
    prob_t P = {num_seqs, cu, Hk, Hv, K, V, per_channel, scale, q, k, v, beta, g, h0};
    const prob_t *p = &P;
    int G = Hv / Hk;
    /* chunk offsets for the optional chunk-state export */
    int64_t *coff = (int64_t *)calloc((size_t)num_seqs + 1, sizeof(int64_t));
    for (int s = 0; s < num_seqs; ++s) {
        int64_t L = cu[s + 1] - cu[s];
        coff[s + 1] = coff[s] + (BTs > 0 ? (L + BTs - 1) / BTs : 0);
    }
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t unit = 0; unit < (int64_t)num_seqs * Hv; ++unit) {
        int s = (int)(unit / Hv), hv = (int)(unit % Hv), hk = hv / G;
        double *S = (double *)malloc(sizeof(double) * V * K);
        double *u = (double *)malloc(sizeof(double) * V);
        if (h0) memcpy(S, h0 + ((size_t)s * Hv + hv) * V * K, sizeof(double) * V * K);
        else memset(S, 0, sizeof(double) * V * K);
        for (int64_t t = cu[s]; t < cu[s + 1]; ++t) {
            int64_t r = t - cu[s];
            if (states && BTs > 0 && r % BTs == 0)
                memcpy(states + ((size_t)(coff[s] + r / BTs) * Hv + hv) * V * K, S, sizeof(double) * V * K);
            const double *kt = qk_row(k, p, t, hk), *vt = v_row(v, p, t, hv);
            step_forward(S, u, kt, vt, beta[(size_t)t * Hv + hv], g_row(p, t, hv), p);
            if (o) {
                const double *qt = qk_row(q, p, t, hk);
                double *ot = o + ((size_t)t * Hv + hv) * V;
                for (int i = 0; i < V; ++i) {
                    double acc = 0.0;
                    for (int c = 0; c < K; ++c) acc += S[(size_t)i * K + c] * qt[c];
                    ot[i] = scale * acc;
                }
            }
        }
        if (hT) memcpy(hT + ((size_t)s * Hv + hv) * V * K, S, sizeof(double) * V * K);
        free(S);
        free(u);
    }
    free(coff);
    return 0;
}

/*
 * Backward of all units.  dq, dk [T, Hk, K]; dv [T, Hv, V]; dbeta [T, Hv]; dg [T, Hv] or [T, Hv, K];
 * dh0 [N, Hv, V, K] (may be NULL).  dO [T, Hv, V]; dht [N, Hv, V, K] or NULL (= zero).
 * All outputs are overwritten.
 */
int gdr_oracle_bwd(int num_seqs, const int64_t *cu, int Hk, int Hv, int K, int V, int per_channel,
                   double scale, const double *q, const double *k, const double *v, const double *beta,
                   const double *g, const double *h0, const double *dO, const double *dht, double *dq,
                   double *dk, double *dv, double *dbeta, double *dg, double *dh0, int mutation,
                   int nthreads) {
    if (num_seqs < 0 || Hk <= 0 || Hv <= 0 || Hv % Hk || K <= 0 || V <= 0) return 1;
    prob_t P = {num_seqs, cu, Hk, Hv, K, V, per_channel, scale, q, k, v, beta, g, h0};
    const prob_t *p = &P;
    int G = Hv / Hk;
    int64_t Ttot = num_seqs > 0 ? cu[num_seqs] : 0;
    size_t VK = (size_t)V * K;
    int GK = per_channel ? K : 1;
    memset(dq, 0, sizeof(double) * Ttot * Hk * K);
    memset(dk, 0, sizeof(double) * Ttot * Hk * K);
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t grp = 0; grp < (int64_t)num_seqs * Hk; ++grp) {
        int s = (int)(grp / Hk), hk = (int)(grp % Hk);
        int64_t bos = cu[s], L = cu[s + 1] - cu[s];
        int64_t nck = (L + CKPT - 1) / CKPT;
        double *ck = (double *)malloc(sizeof(double) * VK * (size_t)(nck > 0 ? nck : 1));
        double *seg = (double *)malloc(sizeof(double) * VK * (CKPT + 1));
        double *dS = (double *)malloc(sizeof(double) * VK);
        double *Sp = (double *)malloc(sizeof(double) * VK);
        double *u = (double *)malloc(sizeof(double) * V);
        double *y = (double *)malloc(sizeof(double) * V);
        double *del = (double *)malloc(sizeof(double) * V);
        double *gk = (double *)malloc(sizeof(double) * K);
        for (int hv = hk * G; hv < (hk + 1) * G; ++hv) {
            /* forward: checkpoints ck[j] = state before token j*CKPT of this sequence */
            double *S = seg;
            if (h0) memcpy(S, h0 + ((size_t)s * Hv + hv) * VK, sizeof(double) * VK);
            else memset(S, 0, sizeof(double) * VK);
            for (int64_t r = 0; r < L; ++r) {
                if (r % CKPT == 0) memcpy(ck + (size_t)(r / CKPT) * VK, S, sizeof(double) * VK);
                int64_t t = bos + r;
                step_forward(S, u, qk_row(k, p, t, hk), v_row(v, p, t, hv), beta[(size_t)t * Hv + hv],
                             g_row(p, t, hv), p);
            }
            /* backward seed */
            if (dht && mutation != 1) memcpy(dS, dht + ((size_t)s * Hv + hv) * VK, sizeof(double) * VK);
            else memset(dS, 0, sizeof(double) * VK);
            for (int64_t j = nck - 1; j >= 0; --j) {
                int64_t r0 = j * CKPT, r1 = (j + 1) * CKPT < L ? (j + 1) * CKPT : L;
                /* seg[i] = state before token r0+i, i = 0..r1-r0 (seg[r1-r0] = state after r1-1) */
                memcpy(seg, ck + (size_t)j * VK, sizeof(double) * VK);
                for (int64_t r = r0; r < r1; ++r) {
                    int64_t t = bos + r;
                    double *nx = seg + (size_t)(r - r0 + 1) * VK;
                    memcpy(nx, seg + (size_t)(r - r0) * VK, sizeof(double) * VK);
                    step_forward(nx, u, qk_row(k, p, t, hk), v_row(v, p, t, hv), beta[(size_t)t * Hv + hv],
                                 g_row(p, t, hv), p);
                }
                for (int64_t r = r1 - 1; r >= r0; --r) {
                    int64_t t = bos + r;
                    const double *St = seg + (size_t)(r - r0 + 1) * VK; /* S_t */
                    const double *Sm = seg + (size_t)(r - r0) * VK;     /* S_{t-1} */
                    const double *qt = qk_row(q, p, t, hk), *kt = qk_row(k, p, t, hk);
                    const double *vt = v_row(v, p, t, hv), *dot = v_row(dO, p, t, hv);
                    const double *gt = g_row(p, t, hv);
                    double bt = beta[(size_t)t * Hv + hv];
                    /* output of step t */
                    for (int i = 0; i < V; ++i)
                        for (int c = 0; c < K; ++c) dS[(size_t)i * K + c] += scale * dot[i] * qt[c];
                    /* dq_t = scale S_t^T dO_t  (mutation 3: S_{t-1}; mutation 7: S_t without transpose) */
                    double *dqt = dq + ((size_t)t * Hk + hk) * K;
                    const double *Sq = (mutation == 3) ? Sm : St;
                    for (int c = 0; c < K; ++c) {
                        double acc = 0.0;
                        for (int i = 0; i < V; ++i)
                            acc += (mutation == 7 ? Sq[(size_t)c * K + i] : Sq[(size_t)i * K + c]) * dot[i];
                        dqt[c] += scale * acc;
                    }
                    /* S' = gate(S_{t-1}), u = S' k, delta = v - u, y = dS k */
                    memcpy(Sp, Sm, sizeof(double) * VK);
                    apply_gate(Sp, gt, p);
                    for (int i = 0; i < V; ++i) {
                        double a = 0.0, b = 0.0;
                        for (int c = 0; c < K; ++c) {
                            a += Sp[(size_t)i * K + c] * kt[c];
                            b += dS[(size_t)i * K + c] * kt[c];
                        }
                        u[i] = a;
                        y[i] = b;
                        del[i] = vt[i] - u[i];
                    }
                    double *dvt = dv + ((size_t)t * Hv + hv) * V;
                    double db = 0.0;
                    for (int i = 0; i < V; ++i) {
                        dvt[i] = bt * y[i];
                        db += (mutation == 5 ? vt[i] : del[i]) * y[i];
                    }
                    dbeta[(size_t)t * Hv + hv] = db;
                    double *dkt = dk + ((size_t)t * Hk + hk) * K;
                    double sgn = (mutation == 2) ? 1.0 : -1.0;
                    for (int c = 0; c < K; ++c) {
                        double a = 0.0, b = 0.0;
                        for (int i = 0; i < V; ++i) {
                            a += dS[(size_t)i * K + c] * del[i];
                            b += Sp[(size_t)i * K + c] * y[i];
                        }
                        dkt[c] += bt * (a + sgn * b);
                    }
                    /* dg from <dS', S'> before dS' overwrites dS (mutation 6 uses dS instead of dS') */
                    if (mutation == 6) {
                        for (int c = 0; c < GK; ++c) gk[c] = 0.0;
                        for (int i = 0; i < V; ++i)
                            for (int c = 0; c < K; ++c)
                                gk[per_channel ? c : 0] += dS[(size_t)i * K + c] * Sp[(size_t)i * K + c];
                    }
                    /* dS' = dS - b y k^T */
                    for (int i = 0; i < V; ++i)
                        for (int c = 0; c < K; ++c) dS[(size_t)i * K + c] -= bt * y[i] * kt[c];
                    if (mutation != 6) {
                        for (int c = 0; c < GK; ++c) gk[c] = 0.0;
                        for (int i = 0; i < V; ++i)
                            for (int c = 0; c < K; ++c)
                                gk[per_channel ? c : 0] += dS[(size_t)i * K + c] * Sp[(size_t)i * K + c];
                    }
                    double *dgt = dg + ((size_t)t * Hv + hv) * GK;
                    for (int c = 0; c < GK; ++c) dgt[c] = gk[c];
                    /* dS_{t-1} = gate^T(dS')  (mutation 4 drops the gate; mutation 8 gates the V side) */
                    if (mutation == 8 && per_channel) {
                        for (int i = 0; i < V; ++i)
                            for (int c = 0; c < K; ++c) dS[(size_t)i * K + c] *= exp(gt[i < K ? i : 0]);
                    } else if (mutation != 4) {
                        apply_gate(dS, gt, p);
                    }
                }
            }
            if (dh0) memcpy(dh0 + ((size_t)s * Hv + hv) * VK, dS, sizeof(double) * VK);
        }
        free(ck);
        free(seg);
        free(dS);
        free(Sp);
        free(u);
        free(y);
        free(del);
        free(gk);
    }
    return 0;
}

int gdr_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
