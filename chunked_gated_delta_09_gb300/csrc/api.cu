// api.cu -- the C ABI of libgdrbwd.so: argument checks, workspace layout and the launch sequence
//   K0 chunk bookkeeping (varlen) -> K1 WY prep -> K2 state recompute -> K3 state-gradient scan
//   -> K4 per-chunk gradients -> K5 gate reverse cumsum + GQA reduction
// all queued on the caller's stream.  No device memory is allocated here.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <new>
#include <unordered_map>

#include "../../include/gdr_bwd.h"
#include "gdr_common.cuh"
#include "gdr_kernels.h"

using namespace gdr;

struct gdr_bwd_plan {
    gdr_bwd_desc d;
    int G, N, dense, nts, max_chunks;
    int k4_tc;  // per-chunk gradients on tcgen05 (scalar gate); the per-channel gate uses the mma.sync kernel
    int dh_factored;  // factored local pass of the state-gradient scan (QR = Q~ - Aqk W), GDR_DH_FACTORED=1
    int NS, Lseg;  // segment-parallel scans: segments per sequence and chunks per segment
    uint32_t spin;  // polls of a bounded device wait (GDR_SPIN_LIMIT, a test knob; default 2^24)
    long long tokens;  // B * T
    // workspace byte offsets
    size_t o_status, o_cidx, o_coff, o_gam, o_T, o_Aqk, o_W, o_U, o_Kt, o_Qg, o_Dt, o_h, o_dh, o_Vn, o_dVn, o_dgam, o_dqh,
        o_dkh, o_seg, o_sc, o_kd, total;
};

namespace gdr {

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
std::mutex g_attr_mu;
std::unordered_map<const void *, uint64_t> g_attr_set;  // kernel -> bit mask of devices already opted in
}  // namespace

cudaError_t device_sm_count(int *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev);
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n <= 0) {
        if ((e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        g_sm_count[dev].store(n, std::memory_order_relaxed);
    }
    *out = n;
    return cudaSuccess;
}

cudaError_t smem_opt_in(const void *kernel, size_t bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev >= 0 && dev < kMaxDevices ? (1ull << dev) : 0;
    {
        std::lock_guard<std::mutex> lock(g_attr_mu);
        auto it = g_attr_set.find(kernel);
        if (bit && it != g_attr_set.end() && (it->second & bit)) return cudaSuccess;
    }
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    if (bit) {
        std::lock_guard<std::mutex> lock(g_attr_mu);
        g_attr_set[kernel] |= bit;
    }
    return cudaSuccess;
}

namespace {
// cuTensorMapEncodeTiled from the driver, looked up once through the runtime (no link against libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}
}  // namespace

// byte strides (heads cols 2, 16, cols 2) for the dimensions (token, column block, head); the innermost
// dimension is the 8 contiguous elements of a column block
cudaError_t encode_rows_map(CUtensorMap *map, const void *base, int dtype, long long tokens, int heads, int cols) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[4] = {8, (cuuint64_t)tokens, (cuuint64_t)(cols / 8), (cuuint64_t)heads};
    const cuuint64_t strides[3] = {(cuuint64_t)heads * cols * 2, 16, (cuuint64_t)cols * 2};
    const cuuint32_t box[4] = {8, (cuuint32_t)CT, (cuuint32_t)(cols / 8), 1};
    const cuuint32_t estride[4] = {1, 1, 1, 1};
    const CUresult r = enc(map, dtype == BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                           const_cast<void *>(base), dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_rows_map_sw128(CUtensorMap *map, const void *base, int dtype, long long tokens, int heads,
                                  int cols) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)heads, (cuuint64_t)tokens};
    const cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)heads * cols * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)CT};
    const cuuint32_t estride[3] = {1, 1, 1};
    const CUresult r = enc(map, dtype == BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                           const_cast<void *>(base), dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace gdr

namespace {

// SM count that sizes the segment-parallel scans: the current device's, or GB300's 152 when no device
// can be queried (a plan built on a host without a GPU).
int plan_sm_count() {
    int n = 0;
    if (gdr::device_sm_count(&n) != cudaSuccess || n <= 0) {
        cudaGetLastError();  // clear the query's error
        return 152;
    }
    return n;
}

bool valid_dtype(int d) { return d == GDR_F32 || d == GDR_BF16 || d == GDR_F16; }

size_t align_up(size_t x) { return (x + 255) & ~size_t(255); }

void layout(gdr_bwd_plan &p) {
    const gdr_bwd_desc &d = p.d;
    size_t units = (size_t)p.max_chunks * d.Hv;
    size_t gw = d.gate_per_channel ? DT : 1;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = align_up(off + bytes);
        return o;
    };
    p.o_status = take(256);
    p.o_cidx = take(sizeof(int32_t) * 2 * (size_t)p.max_chunks);
    p.o_coff = take(sizeof(int32_t) * ((size_t)p.N + 1));
    p.o_gam = take(sizeof(float) * units * CT * gw);
    p.o_T = take(sizeof(__half) * units * CT * CT);
    p.o_Aqk = take(sizeof(__half) * units * CT * CT);
    p.o_W = take(sizeof(__half) * units * CT * DT);
    p.o_U = take(sizeof(__half) * units * CT * DT);
    p.o_Kt = take(sizeof(__half) * units * CT * DT);
    p.o_Qg = take(sizeof(__half) * units * CT * DT);
    p.o_Dt = take(sizeof(__half) * units * CT * DT);
    p.o_h = take(sizeof(__half) * units * DT * DT);
    p.o_dh = take(sizeof(__half) * units * DT * DT);
    p.o_Vn = take(sizeof(__half) * units * CT * DT);
    p.o_dVn = take(sizeof(__half) * units * CT * DT);
    p.o_dgam = take(sizeof(float) * units * CT * gw);
    // per-value-head dq / dk for the group sum in the closing kernel: only the mma.sync gradient kernel
    // writes them (the tcgen05 one sums each key head's group in place)
    size_t per_head = p.G > 1 && !p.k4_tc ? sizeof(float) * (size_t)p.tokens * d.Hv * d.K : 0;
    p.o_dqh = take(per_head);
    p.o_dkh = take(per_head);
    size_t seg_units = p.NS > 1 ? (size_t)p.N * d.Hv * p.NS : 0;
    p.o_seg = take(6 * sizeof(float) * seg_units * DT * DT);
    p.o_sc = take(d.gate_per_channel ? 0 : sizeof(float) * units * 4 * CT);
    p.o_kd = take(d.gate_per_channel ? sizeof(__half) * units * CT * CT : 0);
    p.total = off;
}

bool aligned(const void *ptr, size_t a) { return ((uintptr_t)ptr % a) == 0; }

}  // namespace

extern "C" {

const char *gdr_status_string(gdr_status s) {
    switch (s) {
        case GDR_OK: return "ok";
        case GDR_ERR_INVALID_ARG: return "invalid argument";
        case GDR_ERR_UNSUPPORTED: return "unsupported configuration";
        case GDR_ERR_CUDA: return "CUDA error";
        case GDR_ERR_OOM: return "out of host memory";
        case GDR_ERR_TIMEOUT: return "device wait timed out";
        case GDR_ERR_DEVICE: return "device reported malformed input";
    }
    return "unknown status";
}

gdr_status gdr_bwd_create(const gdr_bwd_desc *desc, gdr_bwd_plan **out) {
    if (!desc || !out) return GDR_ERR_INVALID_ARG;
    *out = nullptr;
    const gdr_bwd_desc &d = *desc;
    if (d.B < 1 || d.T < 0 || d.Hk < 1 || d.Hv < 1 || d.Hv % d.Hk != 0) return GDR_ERR_INVALID_ARG;
    if (d.K < 8 || d.K > DT || d.K % 8 || d.V < 8 || d.V > DT || d.V % 8) return GDR_ERR_INVALID_ARG;
    if (d.BT != 16 && d.BT != 32 && d.BT != 64) return GDR_ERR_INVALID_ARG;
    if (d.num_seqs < 0 || (d.num_seqs > 0 && d.B != 1)) return GDR_ERR_INVALID_ARG;
    if (d.gate_per_channel != 0 && d.gate_per_channel != 1) return GDR_ERR_INVALID_ARG;
    if (!valid_dtype(d.qkv_dtype) || !valid_dtype(d.beta_dtype) || !valid_dtype(d.dqdk_dtype) ||
        !valid_dtype(d.dv_dtype))
        return GDR_ERR_INVALID_ARG;
    if (d.has_h0 != 0 && d.has_h0 != 1) return GDR_ERR_INVALID_ARG;
    if (d.has_dht != 0 && d.has_dht != 1) return GDR_ERR_INVALID_ARG;
    long long tokens = (long long)d.B * d.T;
    if (tokens > (1LL << 30) || (long long)tokens * d.Hv * DT > (1LL << 40)) return GDR_ERR_UNSUPPORTED;
    gdr_bwd_plan *p = new (std::nothrow) gdr_bwd_plan();
    if (!p) return GDR_ERR_OOM;
    p->d = d;
    if (!(p->d.scale > 0.f)) p->d.scale = 1.0f / sqrtf((float)d.K);
    p->G = d.Hv / d.Hk;
    p->dense = d.num_seqs == 0;
    p->N = p->dense ? d.B : d.num_seqs;
    p->nts = (d.T + d.BT - 1) / d.BT;
    p->tokens = tokens;
    long long mc = p->dense ? (long long)d.B * p->nts : (long long)d.T / d.BT + d.num_seqs;
    if (mc > (1LL << 30)) {
        delete p;
        return GDR_ERR_UNSUPPORTED;
    }
    p->max_chunks = (int)mc;
    {
        // segments: at most one wave of (sequence x head x segment) CTAs, at least 4 chunks each; among those,
        // the count that minimises the scans' estimated time in chunk steps (measured on GB300): one segment
        // walks all chunks once; ns > 1 segments walk 2 ceil(chunks / ns) steps (local and final passes), plus
        // about 12 steps of fixed cost (two more launches, the segment summaries written and read) and 3.5 per
        // serial combine step
        long long units = (long long)p->N * d.Hv;
        long long maxnc = p->dense ? p->nts : ((long long)d.T + d.BT - 1) / d.BT;
        long long maxns = units > 0 ? plan_sm_count() / units : 1;
        maxns = maxns < (maxnc + 3) / 4 ? maxns : (maxnc + 3) / 4;
        long long ns = 1;
        double best = (double)maxnc;
        for (long long k = 2; k <= maxns; ++k) {
            const double c = 2.0 * (double)((maxnc + k - 1) / k) + 12.0 + 3.5 * (double)(k - 1);
            if (c < best) best = c, ns = k;
        }
        const char *env = getenv("GDR_NSEG");
        if (env && atoi(env) > 0) ns = atoi(env);
        if (ns < 1) ns = 1;
        p->NS = (int)ns;
        p->Lseg = maxnc > 0 ? (int)((maxnc + ns - 1) / ns) : 1;
    }
    // per-chunk gradients: the tcgen05 kernel for the scalar gate, the mma.sync kernel for the per-channel
    // gate; GDR_K4_TC=0 routes the scalar gate to the mma.sync kernel as well
    const char *k4tc = getenv("GDR_K4_TC");
    p->k4_tc = !d.gate_per_channel && !(k4tc && atoi(k4tc) == 0);
    const char *fact = getenv("GDR_DH_FACTORED");
    p->dh_factored = fact && atoi(fact) != 0;
    // bounded device waits give up after this many polls; tests lower it to make a real wait run out
    const char *spin = getenv("GDR_SPIN_LIMIT");
    p->spin = (spin && atol(spin) > 0) ? (uint32_t)atol(spin) : WAIT_LIMIT_DEFAULT;
    layout(*p);
    *out = p;
    return GDR_OK;
}

size_t gdr_bwd_workspace_bytes(const gdr_bwd_plan *plan) { return plan ? plan->total : 0; }

void gdr_bwd_destroy(gdr_bwd_plan *plan) { delete plan; }

// Sizes and workspace regions of a plan (inputs and outputs are set by the caller).
static void fill_common(const gdr_bwd_plan *plan, char *ws, Params &P) {
    const gdr_bwd_desc &d = plan->d;
    memset(&P, 0, sizeof(P));
    P.B = d.B;
    P.T = d.T;
    P.Hk = d.Hk;
    P.Hv = d.Hv;
    P.K = d.K;
    P.V = d.V;
    P.BT = d.BT;
    P.G = plan->G;
    P.N = plan->N;
    P.per_channel = d.gate_per_channel;
    P.dense = plan->dense;
    P.max_chunks = plan->max_chunks;
    P.nts = plan->nts;
    P.scale = d.scale;
    P.qkv_dtype = d.qkv_dtype;
    P.beta_dtype = d.beta_dtype;
    P.dqdk_dtype = d.dqdk_dtype;
    P.dv_dtype = d.dv_dtype;
    P.spin = plan->spin;
    P.status = reinterpret_cast<int *>(ws + plan->o_status);
    P.chunk_idx = reinterpret_cast<int32_t *>(ws + plan->o_cidx);
    P.chunk_off = reinterpret_cast<int32_t *>(ws + plan->o_coff);
    P.gam = reinterpret_cast<float *>(ws + plan->o_gam);
    P.sc = plan->d.gate_per_channel ? nullptr : reinterpret_cast<float *>(ws + plan->o_sc);
    P.Kd = plan->d.gate_per_channel ? reinterpret_cast<__half *>(ws + plan->o_kd) : nullptr;
    P.Tm = reinterpret_cast<__half *>(ws + plan->o_T);
    P.Aqk = reinterpret_cast<__half *>(ws + plan->o_Aqk);
    P.W = reinterpret_cast<__half *>(ws + plan->o_W);
    P.U = reinterpret_cast<__half *>(ws + plan->o_U);
    P.Kt = reinterpret_cast<__half *>(ws + plan->o_Kt);
    P.Qg = reinterpret_cast<__half *>(ws + plan->o_Qg);
    P.Dt = reinterpret_cast<__half *>(ws + plan->o_Dt);
    P.h = reinterpret_cast<__half *>(ws + plan->o_h);
    P.dh = reinterpret_cast<__half *>(ws + plan->o_dh);
    P.Vn = reinterpret_cast<__half *>(ws + plan->o_Vn);
    P.dVn = reinterpret_cast<__half *>(ws + plan->o_dVn);
    P.dgam = reinterpret_cast<float *>(ws + plan->o_dgam);
    P.dq_h = plan->G > 1 && !plan->k4_tc ? reinterpret_cast<float *>(ws + plan->o_dqh) : nullptr;
    P.dk_h = plan->G > 1 && !plan->k4_tc ? reinterpret_cast<float *>(ws + plan->o_dkh) : nullptr;
    P.NS = plan->NS;
    P.Lseg = plan->Lseg;
    if (plan->NS > 1) {
        size_t one = (size_t)plan->N * d.Hv * plan->NS * DT * DT;
        float *seg = reinterpret_cast<float *>(ws + plan->o_seg);
        P.segE = seg;
        P.segPhi = seg + one;
        P.segPhiT = seg + 2 * one;
        P.segF = seg + 3 * one;
        P.segSin = seg + 4 * one;
        P.segdS = seg + 5 * one;
    }
}

static gdr_status run_impl(gdr_bwd_plan *plan, const gdr_bwd_args *a, void *workspace, size_t ws_bytes, void *stream_,
                           void *const *events) {
    if (!plan || !a) return GDR_ERR_INVALID_ARG;
    const gdr_bwd_desc &d = plan->d;
    cudaStream_t stream = (cudaStream_t)stream_;
    if (!a->q || !a->k || !a->v || !a->beta || !a->g || !a->dO) return GDR_ERR_INVALID_ARG;
    if (!a->dq || !a->dk || !a->dv || !a->dbeta || !a->dg) return GDR_ERR_INVALID_ARG;
    if ((d.has_h0 && !a->h0) || (d.has_dht && !a->dht)) return GDR_ERR_INVALID_ARG;
    if (!plan->dense && !a->cu_seqlens) return GDR_ERR_INVALID_ARG;
    const void *vec[] = {a->q, a->k, a->v, a->dO, a->dq, a->dk, a->dv};
    for (const void *ptr : vec)
        if (!aligned(ptr, 16)) return GDR_ERR_INVALID_ARG;
    const void *nat[] = {a->beta, a->g, a->dbeta, a->dg, a->h0, a->dht, a->dh0, a->cu_seqlens};
    for (const void *ptr : nat)
        if (ptr && !aligned(ptr, 4)) return GDR_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256) || ws_bytes < plan->total) return GDR_ERR_INVALID_ARG;

    char *ws = reinterpret_cast<char *>(workspace);
    Params P;
    fill_common(plan, ws, P);
    P.q = a->q;
    P.k = a->k;
    P.v = a->v;
    P.beta = a->beta;
    P.dO = a->dO;
    P.g = reinterpret_cast<const float *>(a->g);
    P.h0 = d.has_h0 ? reinterpret_cast<const float *>(a->h0) : nullptr;
    P.dht = d.has_dht ? reinterpret_cast<const float *>(a->dht) : nullptr;
    P.cu = plan->dense ? nullptr : a->cu_seqlens;
    P.dq = a->dq;
    P.dk = a->dk;
    P.dv = a->dv;
    P.dbeta = reinterpret_cast<float *>(a->dbeta);
    P.dg = reinterpret_cast<float *>(a->dg);
    P.dh0 = reinterpret_cast<float *>(a->dh0);

    auto mark = [&](int i) -> bool {
        return !events || cudaEventRecord((cudaEvent_t)events[i], stream) == cudaSuccess;
    };
    if (cudaMemsetAsync(P.status, 0, sizeof(int), stream) != cudaSuccess) return GDR_ERR_CUDA;
    if (!mark(0)) return GDR_ERR_CUDA;
    cudaError_t e = cudaSuccess;
    if (!plan->dense) {
        e = launch_k0(a->cu_seqlens, plan->N, d.BT, plan->max_chunks, d.T, P.chunk_idx, P.chunk_off, P.status, stream);
        if (e != cudaSuccess) return GDR_ERR_CUDA;
    }
    if (!mark(1)) return GDR_ERR_CUDA;
    const bool any_chunks = plan->max_chunks > 0;
    if (any_chunks && (e = launch_k1(P, stream)) != cudaSuccess) return GDR_ERR_CUDA;
    if (!mark(2)) return GDR_ERR_CUDA;
    if (any_chunks && plan->NS == 1) {
        // one segment: both scans in one launch (timed as the forward-scan stage; the next stage is empty)
        if ((e = launch_k23_scan_pair(P, stream)) != cudaSuccess) return GDR_ERR_CUDA;
        if (!mark(3) || !mark(4)) return GDR_ERR_CUDA;
    } else {
    if (any_chunks && plan->NS > 1) {
        if ((e = launch_k2_scan(P, true, stream)) != cudaSuccess) return GDR_ERR_CUDA;
        if ((e = launch_k23_combine(P, true, stream)) != cudaSuccess) return GDR_ERR_CUDA;
    }
    if (any_chunks && (e = launch_k2_scan(P, false, stream)) != cudaSuccess) return GDR_ERR_CUDA;
    if (!mark(3)) return GDR_ERR_CUDA;
    if (any_chunks && plan->NS > 1) {
        if (plan->dh_factored) {  // QR into the U^T region, which the forward scan no longer needs
            P.QR = P.U;
            if ((e = launch_k8_qr(P, P.QR, stream)) != cudaSuccess) return GDR_ERR_CUDA;
        }
        if ((e = launch_k3_scan(P, true, stream)) != cudaSuccess) return GDR_ERR_CUDA;
        P.QR = nullptr;
        if ((e = launch_k23_combine(P, false, stream)) != cudaSuccess) return GDR_ERR_CUDA;
    }
    if ((e = launch_k3_scan(P, false, stream)) != cudaSuccess) return GDR_ERR_CUDA;
    if (!mark(4)) return GDR_ERR_CUDA;
    }
    if (any_chunks && (e = (plan->k4_tc ? launch_k4_tc(P, stream) : launch_k4(P, stream))) != cudaSuccess)
        return GDR_ERR_CUDA;
    if (!mark(5)) return GDR_ERR_CUDA;
    if (any_chunks && (e = launch_k5(P, stream)) != cudaSuccess) return GDR_ERR_CUDA;
    if (!mark(6)) return GDR_ERR_CUDA;
    return GDR_OK;
}

gdr_status gdr_bwd_run(gdr_bwd_plan *plan, const gdr_bwd_args *a, void *workspace, size_t ws_bytes, void *stream) {
    return run_impl(plan, a, workspace, ws_bytes, stream, nullptr);
}

gdr_status gdr_bwd_run_profiled(gdr_bwd_plan *plan, const gdr_bwd_args *a, void *workspace, size_t ws_bytes,
                                void *stream, void *const *events) {
    if (!events) return GDR_ERR_INVALID_ARG;
    for (int i = 0; i <= GDR_BWD_NUM_STAGES; ++i)
        if (!events[i]) return GDR_ERR_INVALID_ARG;
    return run_impl(plan, a, workspace, ws_bytes, stream, events);
}

int gdr_bwd_launch_count(const gdr_bwd_plan *plan) {
    if (!plan) return 0;
    int n = plan->dense ? 0 : 1;  // K0
    if (plan->max_chunks == 0) return n + 1;  // the state-gradient scan alone (it writes dh0)
    if (plan->NS == 1) return n + 4;          // K1, both scans in one launch, K4, K5
    // K1, the two final scans, K4, K5; the local scans and combines (and QR)
    return n + 5 + 4 + (plan->dh_factored ? 1 : 0);
}

gdr_status gdr_fwd_run(gdr_bwd_plan *plan, const gdr_fwd_args *a, void *workspace, size_t ws_bytes, void *stream_) {
    if (!plan || !a) return GDR_ERR_INVALID_ARG;
    const gdr_bwd_desc &d = plan->d;
    cudaStream_t stream = (cudaStream_t)stream_;
    if (!a->q || !a->k || !a->v || !a->beta || !a->g || !a->o) return GDR_ERR_INVALID_ARG;
    if (d.has_h0 && !a->h0) return GDR_ERR_INVALID_ARG;
    if (!plan->dense && !a->cu_seqlens) return GDR_ERR_INVALID_ARG;
    const void *vec[] = {a->q, a->k, a->v, a->o};
    for (const void *ptr : vec)
        if (!aligned(ptr, 16)) return GDR_ERR_INVALID_ARG;
    const void *nat[] = {a->beta, a->g, a->h0, a->ht, a->cu_seqlens};
    for (const void *ptr : nat)
        if (ptr && !aligned(ptr, 4)) return GDR_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256) || ws_bytes < plan->total) return GDR_ERR_INVALID_ARG;

    Params P;
    fill_common(plan, reinterpret_cast<char *>(workspace), P);
    P.q = a->q;
    P.k = a->k;
    P.v = a->v;
    P.beta = a->beta;
    P.g = reinterpret_cast<const float *>(a->g);
    P.h0 = d.has_h0 ? reinterpret_cast<const float *>(a->h0) : nullptr;
    P.cu = plan->dense ? nullptr : a->cu_seqlens;
    P.o = a->o;
    P.ht = a->ht;
    P.Kd = nullptr;  // the decayed key Gram serves only the backward's dbeta
    // the forward: chunk bookkeeping, WY preparation without dO, the state recompute, whose final pass also
    // writes each chunk's output and the final state
    if (cudaMemsetAsync(P.status, 0, sizeof(int), stream) != cudaSuccess) return GDR_ERR_CUDA;
    if (!plan->dense &&
        launch_k0(a->cu_seqlens, plan->N, d.BT, plan->max_chunks, d.T, P.chunk_idx, P.chunk_off, P.status, stream) !=
            cudaSuccess)
        return GDR_ERR_CUDA;
    const bool any_chunks = plan->max_chunks > 0;
    if (any_chunks && launch_k1(P, stream) != cudaSuccess) return GDR_ERR_CUDA;
    if (any_chunks && plan->NS > 1) {
        if (launch_k2_scan(P, true, stream) != cudaSuccess) return GDR_ERR_CUDA;
        if (launch_k23_combine(P, true, stream) != cudaSuccess) return GDR_ERR_CUDA;
    }
    if ((any_chunks || P.ht) && launch_k2_scan_out(P, stream) != cudaSuccess) return GDR_ERR_CUDA;
    return GDR_OK;
}

gdr_status gdr_wy_bwd_run(gdr_bwd_plan *plan, const gdr_wy_args *a, void *workspace, size_t ws_bytes,
                          void *stream_) {
    if (!plan || !a) return GDR_ERR_INVALID_ARG;
    const gdr_bwd_desc &d = plan->d;
    cudaStream_t stream = (cudaStream_t)stream_;
    if (!d.gate_per_channel || d.Hk != d.Hv || d.dqdk_dtype != GDR_F32 || d.beta_dtype != d.qkv_dtype ||
        d.dv_dtype != d.qkv_dtype)
        return GDR_ERR_UNSUPPORTED;
    const void *req[] = {a->q, a->k, a->v, a->v_new, a->beta, a->A, a->dO, a->dv, a->g, a->h, a->dh,
                         a->dq, a->dk, a->dv_out, a->db, a->dg, a->dA};
    for (const void *ptr : req)
        if (!ptr) return GDR_ERR_INVALID_ARG;
    if (!plan->dense && !a->cu_seqlens) return GDR_ERR_INVALID_ARG;
    const void *vec[] = {a->q, a->k, a->v, a->v_new, a->dO, a->dv, a->A, a->dq, a->dk, a->dv_out, a->dA};
    for (const void *ptr : vec)
        if (!aligned(ptr, 16)) return GDR_ERR_INVALID_ARG;
    const void *nat[] = {a->beta, a->g, a->h, a->dh, a->db, a->dg, a->cu_seqlens};
    for (const void *ptr : nat)
        if (ptr && !aligned(ptr, 4)) return GDR_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256) || ws_bytes < plan->total) return GDR_ERR_INVALID_ARG;

    Params P;
    fill_common(plan, reinterpret_cast<char *>(workspace), P);
    P.q = a->q;
    P.k = a->k;
    P.v = a->v;
    P.beta = a->beta;
    P.dO = a->dO;
    P.g = a->g;
    P.cu = plan->dense ? nullptr : a->cu_seqlens;
    P.dq = a->dq;
    P.dk = a->dk;
    P.dv = a->dv_out;
    P.dbeta = a->db;
    P.dg = a->dg;
    P.dA_out = a->dA;
    if (cudaMemsetAsync(P.status, 0, sizeof(int), stream) != cudaSuccess) return GDR_ERR_CUDA;
    if (!plan->dense &&
        launch_k0(a->cu_seqlens, plan->N, d.BT, plan->max_chunks, d.T, P.chunk_idx, P.chunk_off, P.status, stream) !=
            cudaSuccess)
        return GDR_ERR_CUDA;
    if (plan->max_chunks == 0) return GDR_OK;
    if (launch_k7_wy_inputs(P, a->A, a->v_new, a->dv, a->h, a->dh, stream) != cudaSuccess) return GDR_ERR_CUDA;
    if (launch_k4_wy(P, stream) != cudaSuccess) return GDR_ERR_CUDA;
    return GDR_OK;
}

int gdr_fwd_launch_count(const gdr_bwd_plan *plan) {
    if (!plan) return 0;
    int n = plan->dense ? 0 : 1;                             // K0
    n += 1;                                                  // the final scan pass (output, final state)
    if (plan->max_chunks > 0) n += 1;                        // K1
    if (plan->max_chunks > 0 && plan->NS > 1) n += 2;        // local scan and combine
    return n;
}

gdr_status gdr_bwd_get_status(gdr_bwd_plan *plan, void *workspace, void *stream_) {
    if (!plan || !workspace) return GDR_ERR_INVALID_ARG;
    cudaStream_t stream = (cudaStream_t)stream_;
    int word = 0;
    int *dev = reinterpret_cast<int *>(reinterpret_cast<char *>(workspace) + plan->o_status);
    if (cudaStreamSynchronize(stream) != cudaSuccess) return GDR_ERR_CUDA;
    if (cudaMemcpy(&word, dev, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return GDR_ERR_CUDA;
    if (cudaMemset(dev, 0, sizeof(int)) != cudaSuccess) return GDR_ERR_CUDA;
    if (word & ST_TIMEOUT) return GDR_ERR_TIMEOUT;
    if (word & (ST_BAD_SEQLENS | ST_RANGE)) return GDR_ERR_DEVICE;
    return GDR_OK;
}

gdr_status gdr_chunk_indices(const int32_t *cu_seqlens, int num_seqs, int BT, int max_chunks, int32_t *chunk_indices,
                             int32_t *chunk_offsets, void *stream) {
    if (!cu_seqlens || !chunk_indices || !chunk_offsets || num_seqs < 1 || BT < 1 || max_chunks < 0)
        return GDR_ERR_INVALID_ARG;
    if (launch_k0(cu_seqlens, num_seqs, BT, max_chunks, -1, chunk_indices, chunk_offsets, nullptr,
                  (cudaStream_t)stream) != cudaSuccess)
        return GDR_ERR_CUDA;
    return GDR_OK;
}

}  // extern "C"
