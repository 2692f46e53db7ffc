/*
 * gdr_bwd.h -- C ABI of the GB300 chunked gated delta rule backward (libgdrbwd.so).
 *
 * The operation: backward pass of chunked Gated DeltaNet, the call that returns the six gradients
 * dq, dk, dv, dg, db and dh0 in one pass ("FlashQLA backward explained", gtnt.cn/news/163832,
 * section 1, step 3).  Per (sequence, value head) the forward it differentiates is
 *
 *     S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T ,   S in R^{V x K}
 *     o_t = scale * S_t q_t
 *
 * with the loss L = sum_t <o_t, dO_t> + <S_T, dht>.  With the per-channel (KDA) gate, exp(g_t) becomes
 * diag(exp(g_t)) acting on the K index of S, and g is given per key channel (MindSpeed-Ops
 * chunk_kda_bwd.md, input table: g [B, T, H, K] fp32 "gate log values").
 *
 * Entry conventions ("FlashQLA backward explained", section 1, "three entry conventions"): dh0 is
 * accumulated and returned in fp32; dht is optional and absent means zero.  Unlike that library, this
 * API takes the RAW per-token log-gate g (not its chunk-local cumulative sum) and returns dg with
 * respect to the raw gate; the chunk cumsum and the closing reverse cumsum happen inside.
 *
 * Tensor layouts (all row-major, last axis contiguous; q, k, v, dO, dq, dk, dv 16-byte aligned, the
 * others 4-byte aligned):
 *   q, k      [B, T, Hk, K]     qkv_dtype
 *   v, dO     [B, T, Hv, V]     qkv_dtype
 *   beta      [B, T, Hv]        beta_dtype
 *   g         [B, T, Hv]        fp32 (gate_per_channel = 0)   or  [B, T, Hv, K] fp32 (= 1)
 *   h0, dht   [N, Hv, V, K]     fp32, S[v][k] ordering; N = B (dense) or num_seqs (varlen)
 *   dq, dk    [B, T, Hk, K]     dqdk_dtype
 *   dv        [B, T, Hv, V]     dv_dtype
 *   dbeta     [B, T, Hv]        fp32
 *   dg        same shape as g   fp32
 *   dh0       [N, Hv, V, K]     fp32
 * Varlen (MindSpeed-Ops chunk_kda_bwd.md, input table: cu_seqlens [N+1], chunk_indices [NT, 2]):
 * B must be 1, T is the packed total and cu_seqlens (int32, device) holds N+1 non-decreasing token
 * offsets with cu_seqlens[0] = 0 and cu_seqlens[N] = T.  Chunks never cross a sequence boundary.
 * GQA: value head hv reads key head hv / (Hv / Hk); dq and dk are summed over the Hv / Hk value heads
 * of each key head.
 *
 * Ownership: every tensor pointer is a device pointer owned by the caller.  The plan is a host object
 * owned by the library (create/destroy).  The workspace is device memory owned by the caller, at
 * least gdr_bwd_workspace_bytes() bytes, 256-byte aligned; the library never allocates device memory.
 *
 * Errors: every call returns a gdr_status and never aborts or throws.  Arguments are checked on the
 * host before anything is launched; a failed check returns GDR_ERR_INVALID_ARG (or
 * GDR_ERR_UNSUPPORTED for a valid but unimplemented combination) and launches nothing.  Kernels
 * report device-side problems (malformed cu_seqlens, an expired bounded wait) in a status word in the
 * workspace, which gdr_bwd_get_status() reads.
 */
#ifndef GDR_BWD_H_
#define GDR_BWD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDR_OK = 0,
    GDR_ERR_INVALID_ARG = 1, /* bad shape, dtype, null required pointer, misalignment */
    GDR_ERR_UNSUPPORTED = 2, /* valid request outside what this build implements */
    GDR_ERR_CUDA = 3,        /* a CUDA runtime call or a launch failed */
    GDR_ERR_OOM = 4,         /* host allocation of the plan failed */
    GDR_ERR_TIMEOUT = 5,     /* a device-side bounded wait expired (read by gdr_bwd_get_status) */
    GDR_ERR_DEVICE = 6       /* a kernel flagged malformed device input: cu_seqlens that are not
                                non-decreasing from 0 to T, or an input value that the fp16
                                tensor-core operands cannot hold (|x| > 65504, inf, nan) */
} gdr_status;

typedef enum { GDR_F32 = 0, GDR_BF16 = 1, GDR_F16 = 2 } gdr_dtype;

/* Problem description.  Sizes: K and V multiples of 8 in [8, 128]; BT in {16, 32, 64}; Hv a multiple
 * of Hk; B * T at most 2^30 tokens. */
typedef struct {
    int B, T, Hk, Hv, K, V, BT;
    int num_seqs;          /* 0: dense [B, T, ...]; > 0: varlen with B == 1 and cu_seqlens[num_seqs + 1] */
    int gate_per_channel;  /* 0: g [B, T, Hv]; 1: KDA gate g [B, T, Hv, K] */
    float scale;           /* output scale; <= 0 selects 1 / sqrt(K) */
    gdr_dtype qkv_dtype;   /* storage type of q, k, v and dO */
    gdr_dtype beta_dtype;  /* storage type of beta */
    gdr_dtype dqdk_dtype;  /* storage type of dq and dk */
    gdr_dtype dv_dtype;    /* storage type of dv */
    int has_h0, has_dht;   /* whether h0 / dht are given (absent means zero) */
} gdr_bwd_desc;

/* Device pointers for one call.  h0, dht and cu_seqlens may be NULL when the descriptor says they
 * are absent.  dh0 may be NULL (not returned). */
typedef struct {
    const void *q, *k, *v, *beta, *g, *h0, *dO, *dht;
    const int32_t *cu_seqlens;
    void *dq, *dk, *dv, *dbeta, *dg, *dh0;
} gdr_bwd_args;

typedef struct gdr_bwd_plan gdr_bwd_plan;

/* Validate a descriptor and build a plan (host only; no device memory).  The plan sizes its
 * segment-parallel scans for the current device's SM count (queried once per device; 152, GB300's
 * count, when no device can be queried), so build it with the device current that will run it.
 * The environment variable GDR_SPIN_LIMIT (a positive integer, read here) lowers the number of polls
 * after which a device-side wait gives up; it exists so that tests can make a real wait run out.
 * Returns GDR_ERR_INVALID_ARG for bad sizes, GDR_ERR_OOM if the host allocation fails. */
gdr_status gdr_bwd_create(const gdr_bwd_desc *desc, gdr_bwd_plan **out);

/* Bytes of device workspace that gdr_bwd_run needs for this plan (0 for a NULL plan). */
size_t gdr_bwd_workspace_bytes(const gdr_bwd_plan *plan);

/* Queue the whole backward on `stream` (a cudaStream_t; NULL is the legacy default stream).
 * Asynchronous: it never synchronises.  Outputs are fully overwritten.  The workspace must not be
 * used by another call that may run concurrently. */
gdr_status gdr_bwd_run(gdr_bwd_plan *plan, const gdr_bwd_args *args, void *workspace, size_t ws_bytes,
                       void *stream);

/* Number of stages and the kernels behind them: 0 varlen chunk bookkeeping, 1 WY preparation,
 * 2 forward state recompute, 3 state-gradient scan, 4 per-chunk gradients (with GQA, the tcgen05 kernel of
 * the scalar gate also sums each key head's group of value heads), 5 gate reverse cumsum and, after the
 * per-channel gate's kernel, the GQA reduction. */
#define GDR_BWD_NUM_STAGES 6

/* Same as gdr_bwd_run, and records events[0] before the first stage and events[i + 1] after stage i
 * (events: GDR_BWD_NUM_STAGES + 1 cudaEvent_t handles created by the caller, all on `stream`'s device).
 * A stage that has nothing to do (stage 0 for dense input) records its event right after the previous
 * one.  When the plan scans every sequence as one segment, stages 2 and 3 run as one launch, timed as
 * stage 2 (stage 3 then records its event right after).  Used to time each kernel on the stream it runs
 * on.  NULL events -> GDR_ERR_INVALID_ARG. */
gdr_status gdr_bwd_run_profiled(gdr_bwd_plan *plan, const gdr_bwd_args *args, void *workspace, size_t ws_bytes,
                                void *stream, void *const *events);

/* Number of kernel launches one gdr_bwd_run of this plan queues (0 for a NULL plan). */
int gdr_bwd_launch_count(const gdr_bwd_plan *plan);

/* Synchronise `stream` and read the device status word that the last run on this workspace left:
 * GDR_OK, GDR_ERR_TIMEOUT (a bounded wait gave up; that CTA released its memory only after every copy
 * and tensor-core operation it had started completed) or GDR_ERR_DEVICE (malformed cu_seqlens, or an
 * input value outside fp16 range).  Also clears the word.  After either error the outputs are not
 * valid. */
gdr_status gdr_bwd_get_status(gdr_bwd_plan *plan, void *workspace, void *stream);

/* No counterpart on the pages.  The whole backward without a caller-provided workspace, for callers
 * that cannot allocate device memory when they need it (a plugin that may only use the tensors it is
 * given, a fixed device-memory budget, a loop that cannot afford cudaMalloc's implicit synchronisation).
 * Its scratch memory is one file-scope __device__ array of GDR_BWD_NOALLOC_MAX_WORKSPACE bytes, which
 * every GPU that loads the library holds until the process exits.  It allocates nothing and calls no
 * allocating routine.  Plans whose gdr_bwd_workspace_bytes() exceeds the maximum are rejected with
 * GDR_ERR_UNSUPPORTED before anything is launched.  The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress) with that device current; make that first call before any
 * stream capture starts.  All calls share the array: calls that overlap on the GPU race.  Their device
 * status word is read with gdr_bwd_get_status_noalloc. */
#define GDR_BWD_NOALLOC_MAX_WORKSPACE (64u << 20)
gdr_status gdr_bwd_run_noalloc(gdr_bwd_plan *plan, const gdr_bwd_args *args, void *stream);

/* No counterpart on the pages.  The device status word of the last gdr_bwd_run_noalloc on the current
 * device (it lives in the shared array, so gdr_bwd_get_status cannot reach it): synchronises `stream`,
 * returns GDR_OK, GDR_ERR_TIMEOUT or GDR_ERR_DEVICE as gdr_bwd_get_status does, and clears the word.
 * GDR_ERR_UNSUPPORTED for a plan beyond the array's size; allocates nothing. */
gdr_status gdr_bwd_get_status_noalloc(gdr_bwd_plan *plan, void *stream);

/* ---- Forward pass (the output and final state that the backward above differentiates).
 * Per sequence and value head, S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T and
 * o_t = scale S_t q_t, computed chunkwise: the WY preparation and the state recompute of the backward,
 * whose final pass also forms per chunk o = scale (diag(Gamma) Q S_0^T + (M (.) Q K^T) V_new) ("FlashQLA backward explained",
 * section 1: the forward whose saved state the backward recomputes; MindSpeed-Ops chunk_kda_bwd.md, input
 * table: the chunk states h and v_new).  The per-channel gate acts on the K index as in the backward.
 * Uses the backward's plan and workspace (gdr_bwd_workspace_bytes); dO, dht and the gradient fields of
 * the descriptor are ignored.
 *   q, k      [B, T, Hk, K]  qkv_dtype       v [B, T, Hv, V] qkv_dtype     beta [B, T, Hv] beta_dtype
 *   g         fp32 [B, T, Hv] or [B, T, Hv, K] (raw log-gate)                h0 fp32 [N, Hv, V, K] or NULL
 *   o         [B, T, Hv, V] in qkv_dtype, fully overwritten
 *   ht        fp32 [N, Hv, V, K] final state per sequence and value head, or NULL (not returned)
 * All device pointers are caller-owned; q, k, v and o 16-byte aligned, the others 4-byte aligned.
 * Asynchronous on `stream`; GDR_ERR_INVALID_ARG for null required pointers, misalignment or a small
 * workspace; device-side problems are read with gdr_bwd_get_status as for the backward. */
typedef struct {
    const void *q, *k, *v, *beta, *g, *h0;
    const int32_t *cu_seqlens;
    void *o;
    float *ht;
} gdr_fwd_args;
gdr_status gdr_fwd_run(gdr_bwd_plan *plan, const gdr_fwd_args *args, void *workspace, size_t ws_bytes,
                       void *stream);

/* Number of kernel launches one gdr_fwd_run of this plan queues (0 for a NULL plan). */
int gdr_fwd_launch_count(const gdr_bwd_plan *plan);

/* ---- The WY-gradient stage taken alone (MindSpeed-Ops chunk_kda_bwd.md: chunk_kda_bwd_wy_dqkg_fused;
 * signature, input / output tables and "implementation principle").  For the per-channel (KDA) gate
 * only: the plan must have gate_per_channel = 1, Hk == Hv (= H), dqdk_dtype GDR_F32, beta_dtype and
 * dv_dtype equal to qkv_dtype; otherwise GDR_ERR_UNSUPPORTED.  Per chunk and head it returns the gradients
 * that flow through the chunk's state terms and its WY factors W = A diag(beta) (K (.) exp(g)),
 * U = A diag(beta) V, with h, dh, v_new, dv and do held fixed (the intra-chunk Q K^T terms and the terms
 * through A_kk are left to later stages, which receive dA):
 *   inputs  q, k [B, T, H, K]; v, v_new, do, dv [B, T, H, V]; beta [B, T, H]; A [B, T, H, BT]  (qkv_dtype)
 *           g  fp32 [B, T, H, K]   chunk-local cumulative log gate
 *           h, dh fp32 [B, NT, H, K, V]   state entering each chunk / gradient of the state leaving it
 *           (varlen: B = 1 and NT = total chunks, numbered sequence-major)
 *   outputs dq, dk fp32 [B, T, H, K]; dv_out [B, T, H, V] (qkv_dtype); db fp32 [B, T, H];
 *           dg fp32 [B, T, H, K] (with respect to the cumulative gate); dA fp32 [B, T, H, BT], the gradient
 *           with respect to A_kk where A = (I + A_kk)^-1 (strictly lower; other entries are zero).
 * scale multiplies dq; all pointers are device, caller-owned; q, k, v, v_new, do, dv, A, dq, dk, dv_out and
 * dA 16-byte aligned, the others 4-byte aligned.  Uses the plan's workspace; asynchronous on `stream`. */
typedef struct {
    const void *q, *k, *v, *v_new, *beta, *A, *dO, *dv;
    const float *g, *h, *dh;
    const int32_t *cu_seqlens;
    float *dq, *dk;
    void *dv_out;
    float *db, *dg, *dA;
} gdr_wy_args;
gdr_status gdr_wy_bwd_run(gdr_bwd_plan *plan, const gdr_wy_args *args, void *workspace, size_t ws_bytes,
                          void *stream);

/* Free the plan (NULL is accepted). */
void gdr_bwd_destroy(gdr_bwd_plan *plan);

/* Varlen chunk bookkeeping on the device (MindSpeed-Ops chunk_kda_bwd.md, input table: chunk_indices
 * [NT, 2] with NT = ceil(T / chunk_size)).  For the N sequences of cu_seqlens (device int32 [N+1]),
 * writes chunk_offsets[s] = number of chunks before sequence s (chunk_offsets[N] = total), and
 * chunk_indices[n] = (s, c) for the n-th chunk, sequence-major then chunk ascending; entries from the
 * total up to max_chunks - 1 are set to (-1, -1).  max_chunks must be at least the total, e.g.
 * T / BT + N.  Returns GDR_ERR_INVALID_ARG for null pointers, N < 1 or BT < 1; launches one kernel. */
gdr_status gdr_chunk_indices(const int32_t *cu_seqlens, int num_seqs, int BT, int max_chunks,
                             int32_t *chunk_indices, int32_t *chunk_offsets, void *stream);

/* Static description of a status code. */
const char *gdr_status_string(gdr_status status);

#ifdef __cplusplus
}
#endif

#endif /* GDR_BWD_H_ */
