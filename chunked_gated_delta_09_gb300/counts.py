"""FLOP and byte conventions used to report throughput and roofline fractions.

FLOPs are counted from the chunked algorithm (2 m n k per matrix product) per chunk x value head, with
C = BT tokens per chunk:
    F_chunk = 16 C K V + 18 C^2 K + 10 C^2 V + (14/3) C^3
  16 C K V : state recompute 4, state-gradient scan 6, inter-chunk dq / dk / dW products 6
  18 C^2 K : K K^T 2, W 2, Q K^T 2, intra dq / dk 4, dT 2, T^T dW 2, dA -> dk 4
  10 C^2 V : U 2, local dV 2, dO V_new^T 2, dT 2, T^T dU 2
  C^3      : triangular inverse 2/3, dA = -T^T dT T^T 4
Every started chunk counts as a full one.  Element-wise work (exp, masks, cumsums) is not counted.

Algorithmic bytes are the least any implementation must move: each input read once and each output
written once (q, k, v, dO, beta, g, h0, dht, cu_seqlens in; dq, dk, dv, dbeta, dg, dh0 out).

Stage bytes (:func:`stage_bytes`) are what each kernel stage of this implementation must read and write
given the split of the path into stages: its share of the inputs and outputs plus the workspace tiles it
consumes or produces (fp16 tiles padded to 64 chunk rows and 128 features).  They decide which roofline
(tensor or HBM) binds each stage.
"""
from __future__ import annotations

import torch


def flops_per_chunk(C: int, K: int, V: int) -> float:
    return 16.0 * C * K * V + 18.0 * C * C * K + 10.0 * C * C * V + (14.0 / 3.0) * C ** 3


def chunk_units(prob) -> int:
    return prob.n_chunks() * prob.Hv


def total_flops(prob) -> float:
    return chunk_units(prob) * flops_per_chunk(prob.BT, prob.K, prob.V)


def _nbytes(dtype: torch.dtype) -> int:
    return torch.empty((), dtype=dtype).element_size()


def algorithmic_bytes(prob) -> int:
    T = prob.B * prob.T
    gk = prob.K if prob.per_channel else 1
    ib = _nbytes(prob.qkv_dtype)
    state = prob.N * prob.Hv * prob.V * prob.K * 4
    inputs = (2 * T * prob.Hk * prob.K * ib + 2 * T * prob.Hv * prob.V * ib
              + T * prob.Hv * _nbytes(prob.beta_dtype) + T * prob.Hv * gk * 4
              + (state if prob.h0 is not None else 0) + (state if prob.dht is not None else 0)
              + (4 * (prob.num_seqs + 1) if prob.cu_seqlens is not None else 0))
    outputs = (2 * T * prob.Hk * prob.K * _nbytes(prob.dqdk_dtype) + T * prob.Hv * prob.V * _nbytes(prob.dv_dtype)
               + T * prob.Hv * 4 + T * prob.Hv * gk * 4 + state)
    return int(inputs + outputs)


def gradient_stage_algorithmic_bytes(prob) -> int:
    """The least the per-chunk gradient stage must move, whatever the split of the path: the inputs it
    differentiates read once (q, k, v, dO, beta, g) and its outputs written once (dq, dk, dv, dbeta).  The
    dominant kernel's roofline is taken against these bytes, not against the workspace tiles this design
    passes between its stages."""
    T = prob.B * prob.T
    ib = _nbytes(prob.qkv_dtype)
    gk = prob.K if prob.per_channel else 1
    return int(2 * T * prob.Hk * prob.K * ib + 2 * T * prob.Hv * prob.V * ib + T * prob.Hv * _nbytes(prob.beta_dtype)
               + T * prob.Hv * gk * 4 + 2 * T * prob.Hk * prob.K * _nbytes(prob.dqdk_dtype)
               + T * prob.Hv * prob.V * _nbytes(prob.dv_dtype) + T * prob.Hv * 4)


def stage_flops(prob) -> list:
    """The FLOP convention split over the six kernel stages (chunk bookkeeping, WY preparation, state
    recompute, state-gradient scan, per-chunk gradients, gate cumsum / GQA reduction); sums to
    :func:`total_flops`."""
    C, K, V = prob.BT, prob.K, prob.V
    per = [0.0,
           6.0 * C * C * K + 2.0 * C * C * V + (2.0 / 3.0) * C ** 3,
           4.0 * C * K * V,
           6.0 * C * K * V + 2.0 * C * C * V,
           6.0 * C * K * V + 12.0 * C * C * K + 6.0 * C * C * V + 4.0 * C ** 3,
           0.0]
    u = chunk_units(prob)
    return [u * x for x in per]


# Segments per sequence of the segment-parallel scans, chosen as the library's plan does: enough
# sequence x head x segment CTAs to fill the 152 SMs, at least 4 chunks per segment.
NUM_SMS = 152


def scan_segments(prob) -> int:
    """The segment count the library's plan picks (the same estimate of the scans' time in chunk steps)."""
    units = prob.N * prob.Hv
    maxnc = (prob.T + prob.BT - 1) // prob.BT if prob.cu_seqlens is None else \
        (prob.B * prob.T + prob.BT - 1) // prob.BT
    maxns = NUM_SMS // units if units > 0 else 1
    maxns = min(maxns, (maxnc + 3) // 4)
    ns, best = 1, float(maxnc)
    for k in range(2, maxns + 1):
        c = 2.0 * ((maxnc + k - 1) // k) + 12.0 + 3.5 * (k - 1)
        if c < best:
            ns, best = k, c
    return ns


def stage_bytes(prob) -> list:
    """Bytes each of the six stages reads plus writes (see the module docstring), summed over all units."""
    CT, DT = 64, 128
    tile_ck, tile_cc, tile_kk = CT * DT * 2, CT * CT * 2, DT * DT * 2  # fp16 workspace tiles
    u = chunk_units(prob)
    C, K, V = prob.BT, prob.K, prob.V
    ib, bb = _nbytes(prob.qkv_dtype), _nbytes(prob.beta_dtype)
    gk = K if prob.per_channel else 1
    G = prob.Hv // prob.Hk
    oq, ov = _nbytes(prob.dqdk_dtype), _nbytes(prob.dv_dtype)
    state = prob.N * prob.Hv * V * K * 4
    ns = scan_segments(prob)
    seg = 6 * prob.N * prob.Hv * ns * DT * DT * 4 if ns > 1 else 0  # segment summaries, all passes
    k0 = 0 if prob.cu_seqlens is None else 4 * (prob.num_seqs + 1) + 8 * u // prob.Hv + 4 * (prob.num_seqs + 1)
    rec = 0 if prob.per_channel else 4 * CT * 4  # scalar gate: per-token record for the gradient kernel
    k1 = u * (2 * C * K * ib + 2 * C * V * ib + C * bb + C * gk * 4          # q, k, v, dO, beta, g
              + CT * gk * 4 + 2 * tile_cc + 5 * tile_ck + rec)                # gamma, T, Aqk, W, U, K~, Q~, D
    k2 = u * ((3 * tile_ck) * (2 if ns > 1 else 1) + tile_kk + tile_ck) \
        + (state if prob.h0 is not None else 0) + seg // 2                      # W, U, K~ (+ local pass); h, V_new
    k3 = u * ((tile_cc + 4 * tile_ck) * (2 if ns > 1 else 1) + tile_kk + tile_ck) \
        + (state if prob.dht is not None else 0) + state + seg // 2             # Aqk, D, K~, Q~, W; dh, dV_new; dh0
    dqdk_out = 2 * C * K * oq  # (with GQA: each value head's rows, added in place or per-head partials)
    scal_in = rec if rec else C * bb + CT * gk * 4  # the record, else beta and gamma
    k4 = u * (2 * tile_kk + 3 * tile_ck + tile_cc + 2 * C * K * ib + C * V * ib + scal_in   # reads
              + dqdk_out + C * V * ov + C * 4 + CT * gk * 4)                               # writes
    # GQA group sum in the closing kernel: only after the per-channel (mma.sync) gradient kernel, which writes
    # per-value-head partials; the scalar gate's tcgen05 kernel sums each group in place
    gsum = G > 1 and prob.per_channel
    k5 = u * (CT * gk * 4 + C * gk * 4) + (u * 2 * C * K * oq + (u // G) * 2 * C * K * oq if gsum else 0)
    return [float(k0), float(k1), float(k2), float(k3), float(k4), float(k5)]


def forward_flops_per_chunk(C: int, K: int, V: int) -> float:
    """The forward by the same convention: WY preparation (K K^T, Q K^T, W 2 C^2 K each; U 2 C^2 V; the
    inverse 2/3 C^3), state recompute 4 C K V, output (Q~ S_0^T 2 C K V, Aqk V_new 2 C^2 V)."""
    return 6.0 * C * K * V + 6.0 * C * C * K + 4.0 * C * C * V + (2.0 / 3.0) * C ** 3


def forward_total_flops(prob) -> float:
    return chunk_units(prob) * forward_flops_per_chunk(prob.BT, prob.K, prob.V)


def forward_algorithmic_bytes(prob) -> int:
    """Inputs q, k, v, beta, g, h0 read once; outputs o and the final state written once."""
    T = prob.B * prob.T
    gk = prob.K if prob.per_channel else 1
    ib = _nbytes(prob.qkv_dtype)
    state = prob.N * prob.Hv * prob.V * prob.K * 4
    return int(2 * T * prob.Hk * prob.K * ib + T * prob.Hv * prob.V * ib + T * prob.Hv * _nbytes(prob.beta_dtype)
               + T * prob.Hv * gk * 4 + (state if prob.h0 is not None else 0)
               + T * prob.Hv * prob.V * ib + state)


def wy_stage_flops_per_chunk(C: int, K: int, V: int) -> float:
    """The WY-gradient stage taken alone: D S_0, V_new dS, dV S_0 (2 C K V each); dT from dW and dV
    (2 C^2 K + 2 C^2 V); T^T dW (2 C^2 K), T^T dV (2 C^2 V); dT T^T and T^T X (2 C^3 each)."""
    return 6.0 * C * K * V + 4.0 * C * C * K + 4.0 * C * C * V + 4.0 * C ** 3


def wy_stage_bytes(B, T, H, K, V, BT, ib) -> int:
    """Its inputs read once and outputs written once: q, k, v, v_new, do, dv, beta, A (ib bytes each), g and
    the fp32 states h, dh; dq, dk, db, dg, dA (fp32) and dv (ib)."""
    NT = B * ((T + BT - 1) // BT)
    tok = B * T * H
    return int(tok * (2 * K + 4 * V + 1 + BT) * ib + tok * K * 4 + 2 * NT * H * K * V * 4
               + tok * (2 * K + 1 + K + BT) * 4 + tok * V * ib)
