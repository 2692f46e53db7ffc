// k0_chunk_indices.cu -- varlen chunk bookkeeping on the device.
//
// Definition (MindSpeed-Ops chunk_kda_bwd.md, input table: cu_seqlens [N+1] cumulative lengths,
// chunk_indices [NT, 2] with NT = ceil(T / chunk_size)): sequence s covers tokens [cu[s], cu[s+1]) and
// is cut into ceil(L_s / BT) chunks that never cross its ends.  Chunks are numbered sequence-major,
// chunk ascending: chunk_offsets[s] counts the chunks of all earlier sequences, chunk_indices[n] =
// (s, c).  Everything is integer arithmetic, so the result is exact.
#include "gdr_common.cuh"
#include "gdr_kernels.h"

namespace gdr {

constexpr int K0_THREADS = 1024;

// One block.  Pass 1: block-wide scan of per-sequence chunk counts, tile by tile.  Pass 2: every
// chunk slot binary-searches its sequence in chunk_offsets.
__global__ void __launch_bounds__(K0_THREADS) k0_chunk_indices(const int32_t *__restrict__ cu, int N, int BT,
                                                                 int max_chunks, int expect_total_tokens,
                                                                 int32_t *__restrict__ chunk_idx,
                                                                 int32_t *__restrict__ chunk_off, int *status) {
    __shared__ int warp_sums[K0_THREADS / 32];
    __shared__ int carry;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (tid == 0) {
        carry = 0;
        chunk_off[0] = 0;
        bool bad = cu[0] != 0 || (expect_total_tokens >= 0 && cu[N] != expect_total_tokens);
        if (bad && status) flag_status(status, ST_BAD_SEQLENS);
    }
    __syncthreads();
    for (int base = 0; base < N; base += K0_THREADS) {
        int s = base + tid;
        int cnt = 0;
        if (s < N) {
            int L = cu[s + 1] - cu[s];
            if (L < 0) {
                if (status) flag_status(status, ST_BAD_SEQLENS);
                L = 0;
            }
            cnt = (L + BT - 1) / BT;
        }
        // inclusive warp scan
        int x = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sums[wid] = x;
        __syncthreads();
        if (wid == 0) {
            int w = warp_sums[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            warp_sums[lane] = w;  // inclusive over warps
        }
        __syncthreads();
        int incl = x + (wid > 0 ? warp_sums[wid - 1] : 0) + carry;
        if (s < N) chunk_off[s + 1] = incl;
        __syncthreads();
        if (tid == K0_THREADS - 1) carry = incl;
        __syncthreads();
    }
    __threadfence_block();
    __syncthreads();
    const int total = chunk_off[N];
    if (tid == 0 && total > max_chunks && status) flag_status(status, ST_BAD_SEQLENS);
    for (int n = tid; n < max_chunks; n += K0_THREADS) {
        int s = -1, c = -1;
        if (n < total) {
            // largest s with chunk_off[s] <= n (chunk_off is non-decreasing)
            int lo = 0, hi = N - 1;
            while (lo < hi) {
                int mid = (lo + hi + 1) >> 1;
                if (chunk_off[mid] <= n) lo = mid;
                else hi = mid - 1;
            }
            s = lo;
            c = n - chunk_off[s];
        }
        chunk_idx[2 * n] = s;
        chunk_idx[2 * n + 1] = c;
    }
}

cudaError_t launch_k0(const int32_t *cu, int N, int BT, int max_chunks, int expect_total_tokens, int32_t *chunk_idx,
                      int32_t *chunk_off, int *status, cudaStream_t stream) {
    k0_chunk_indices<<<1, K0_THREADS, 0, stream>>>(cu, N, BT, max_chunks, expect_total_tokens, chunk_idx, chunk_off,
                                                   status);
    return cudaGetLastError();
}

}  // namespace gdr
