// gdr_kernels.h -- host-side launchers of the backward kernels (internal to libgdrbwd.so).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace gdr {

struct Params;

// Opt a kernel in to `bytes` of dynamic shared memory, once per (kernel, device); later calls return at once.
cudaError_t smem_opt_in(const void *kernel, size_t bytes);
// Streaming-multiprocessor count of the current device (queried once per device).
cudaError_t device_sm_count(int *out);
// Tensor map of a 16-bit input [tokens][heads][cols] (dtype BF16 or F16) for loads of a chunk's rows of one
// head: 4-D over (8-element column chunk, token, column block, head), box (8, 64, cols / 8, 1), so that one
// box lands as a column-block-major core-matrix tile (core matrix (r/8, c/8) at ((c/8) 8 + r/8) 128 bytes).
// Rows past the tensor's end read as zero.  cols must be a multiple of 8 and base 16-byte aligned.
cudaError_t encode_rows_map(CUtensorMap *map, const void *base, int dtype, long long tokens, int heads, int cols);
// The same input for loads of 64-column halves of a chunk's rows with the 128-byte swizzle: 3-D over (column,
// head, token), box (64, 1, 64), so that one box lands as 64 rows of 128 bytes whose 16-byte chunks are permuted
// within each row (chunk j of row r at position j ^ (r % 8)); the destination must be 1024-byte aligned.
// Columns past cols and rows past the tensor's end read as zero.
cudaError_t encode_rows_map_sw128(CUtensorMap *map, const void *base, int dtype, long long tokens, int heads,
                                  int cols);

// K0: varlen chunk bookkeeping (one block).  expect_total_tokens < 0 skips the cu[N] == T check.
cudaError_t launch_k0(const int32_t *cu, int N, int BT, int max_chunks, int expect_total_tokens, int32_t *chunk_idx,
                      int32_t *chunk_off, int *status, cudaStream_t stream);
// K1: chunk-local WY preparation (gate cumsum, A_kk inverse, W, U, decayed copies of K and Q).
cudaError_t launch_k1(const Params &P, cudaStream_t stream);
// K2 / K3: forward state recompute (fused_gdr_h) and reverse state-gradient scan, segment-parallel on
// the tensor cores: local (zero-start) pass or final (exact-start) pass.
cudaError_t launch_k2_scan(const Params &P, bool local, cudaStream_t stream);
// The forward's final pass with the output fused in (writes o and ht; no h_n, V_new).
cudaError_t launch_k2_scan_out(const Params &P, cudaStream_t stream);
cudaError_t launch_k3_scan(const Params &P, bool local, cudaStream_t stream);
// With one segment per sequence: both scans' single passes as one grid (forward CTAs first).
cudaError_t launch_k23_scan_pair(const Params &P, cudaStream_t stream);
// Exact fp32 combination of segment summaries (forward entry states / backward exit gradients).
cudaError_t launch_k23_combine(const Params &P, bool fwd, cudaStream_t stream);
// K4: per-chunk gradients dq, dk, dv, dbeta and the cumulative-gate gradient.
cudaError_t launch_k4(const Params &P, cudaStream_t stream);
// K4 on the 5th-generation tensor cores (scalar gate only).
cudaError_t launch_k4_tc(const Params &P, cudaStream_t stream);
// K5: reverse cumsum of the gate gradient and GQA reduction of dq / dk.
cudaError_t launch_k5(const Params &P, cudaStream_t stream);
// the WY-gradient stage taken alone: its inputs as workspace tiles, then the per-chunk kernel in that mode
cudaError_t launch_k7_wy_inputs(const Params &P, const void *A, const void *v_new, const void *dv_in, const float *h,
                                const float *dh, cudaStream_t stream);
cudaError_t launch_k4_wy(const Params &P, cudaStream_t stream);
// QR = Q~ - Aqk W per chunk for the factored local pass of the state-gradient scan
cudaError_t launch_k8_qr(const Params &P, __half *QR, cudaStream_t stream);

}  // namespace gdr
