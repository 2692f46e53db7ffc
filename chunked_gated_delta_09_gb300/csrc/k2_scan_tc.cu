// k2_scan_tc.cu -- launches of the forward state recompute (the kernel body is k2_scan_body.cuh).
#include "k2_scan_body.cuh"

namespace gdr {

// Local pass: two CTAs per (sequence x head x segment), the state chain (even) and the transition chain
// (odd), two per SM.
// OUT: the forward's final pass, which also writes the output (and not h_n, V_new).
template <bool PC, bool LOCAL, bool OUT>
__global__ void __launch_bounds__(SC_THREADS, LOCAL ? 2 : 1) k2_scan_tc(const Params P) {
    if (LOCAL) k2_scan_body<PC, LOCAL>(P, (int)blockIdx.x >> 1, (blockIdx.x & 1) != 0);
    else k2_scan_body<PC, LOCAL, OUT>(P, (int)blockIdx.x);
}

template <bool PC, bool LOCAL, bool OUT = false>
static cudaError_t launch_fwd_t(const Params &P, cudaStream_t stream) {
    size_t smem = sizeof(FwdSmem<LOCAL, OUT>);
    cudaError_t e = smem_opt_in((const void *)k2_scan_tc<PC, LOCAL, OUT>, smem);
    if (e != cudaSuccess) return e;
    k2_scan_tc<PC, LOCAL, OUT><<<P.N * P.Hv * P.NS * (LOCAL ? 2 : 1), SC_THREADS, smem, stream>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_k2_scan(const Params &P, bool local, cudaStream_t stream) {
    if (local) return P.per_channel ? launch_fwd_t<true, true>(P, stream) : launch_fwd_t<false, true>(P, stream);
    return P.per_channel ? launch_fwd_t<true, false>(P, stream) : launch_fwd_t<false, false>(P, stream);
}

cudaError_t launch_k2_scan_out(const Params &P, cudaStream_t stream) {
    return P.per_channel ? launch_fwd_t<true, false, true>(P, stream) : launch_fwd_t<false, false, true>(P, stream);
}

}  // namespace gdr
