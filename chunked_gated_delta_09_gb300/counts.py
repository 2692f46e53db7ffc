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
