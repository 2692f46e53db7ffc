"""Seeded synthetic inputs for the gated delta rule backward.

This module is shared by the CUDA path's tests and benchmark and by the oracle's tests.  It holds
none of the method's arithmetic: it draws random tensors, applies the input recipe (per-token L2
normalisation of q and k, sigmoid for beta, logsigmoid for the gate, as in the KDA op's usage example,
MindSpeed-Ops chunk_kda_bwd.md, "usage example"), casts to the storage dtypes and, for the oracle,
upcasts the rounded values to fp64.

Recipe: values are drawn in fp32 on the CPU with ``torch.Generator().manual_seed(seed)`` in the fixed
order lengths (varlen only), q, k, v, beta, g, h0, dO, dht, then cast.  The oracle and the GPU see the
same rounded values.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch


def l2_normalise(x: torch.Tensor) -> torch.Tensor:
    """Per-token L2 normalisation of the last axis (input recipe, done before the cast)."""
    return x / torch.sqrt((x * x).sum(-1, keepdim=True) + 1e-6)


@dataclasses.dataclass
class Problem:
    """One backward problem: shapes, dtypes and CPU tensors in their storage dtypes.

    Dense: q, k [B, T, Hk, K]; v, dO [B, T, Hv, V]; beta [B, T, Hv]; g [B, T, Hv] or [B, T, Hv, K].
    Varlen: B == 1, T is the packed total and ``cu_seqlens`` (int32 [N+1]) splits it.
    h0, dht: fp32 [N, Hv, V, K] (N = B when dense) or None (zero).
    """
    name: str
    B: int
    T: int
    Hk: int
    Hv: int
    K: int
    V: int
    BT: int
    per_channel: bool
    scale: float
    qkv_dtype: torch.dtype
    beta_dtype: torch.dtype
    dqdk_dtype: torch.dtype
    dv_dtype: torch.dtype
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    beta: torch.Tensor
    g: torch.Tensor
    dO: torch.Tensor
    h0: Optional[torch.Tensor] = None
    dht: Optional[torch.Tensor] = None
    cu_seqlens: Optional[torch.Tensor] = None
    seed: int = 0

    @property
    def num_seqs(self) -> int:
        return 0 if self.cu_seqlens is None else int(self.cu_seqlens.numel() - 1)

    @property
    def N(self) -> int:
        """Number of independent sequences (state tensors have this leading size)."""
        return self.B if self.cu_seqlens is None else self.num_seqs

    def seq_lengths(self):
        if self.cu_seqlens is None:
            return [self.T] * self.B
        c = self.cu_seqlens.tolist()
        return [c[i + 1] - c[i] for i in range(len(c) - 1)]

    def cu_packed(self) -> np.ndarray:
        """int64 token offsets of every sequence on the packed [B*T] token axis."""
        if self.cu_seqlens is None:
            return np.arange(self.B + 1, dtype=np.int64) * self.T
        return self.cu_seqlens.numpy().astype(np.int64)

    def packed_f64(self) -> dict:
        """fp64 numpy copies of the rounded inputs on the packed token axis."""
        def f(x, tail):
            if x is None:
                return None
            return x.to(torch.float64).reshape(-1, *tail).numpy().copy()
        gt = (self.Hv, self.K) if self.per_channel else (self.Hv,)
        return dict(cu=self.cu_packed(), q=f(self.q, (self.Hk, self.K)), k=f(self.k, (self.Hk, self.K)),
                    v=f(self.v, (self.Hv, self.V)), beta=f(self.beta, (self.Hv,)), g=f(self.g, gt),
                    dO=f(self.dO, (self.Hv, self.V)),
                    h0=None if self.h0 is None else self.h0.to(torch.float64).numpy().copy(),
                    dht=None if self.dht is None else self.dht.to(torch.float64).numpy().copy())

    def unpack(self, out: dict) -> dict:
        """Reshape packed [B*T, ...] results back to [B, T, ...]."""
        res = {}
        for key, val in out.items():
            if key == "dh0":
                res[key] = val
            else:
                res[key] = val.reshape(self.B, self.T, *val.shape[1:])
        return res

    def n_chunks(self) -> int:
        return sum((L + self.BT - 1) // self.BT for L in self.seq_lengths())

    def nbytes_inputs(self) -> int:
        ts = [self.q, self.k, self.v, self.beta, self.g, self.dO, self.h0, self.dht, self.cu_seqlens]
        return sum(t.numel() * t.element_size() for t in ts if t is not None)


def make_problem(name="custom", *, B=1, T=64, Hk=1, Hv=1, K=32, V=32, BT=64, per_channel=False,
                 scale=None, qkv_dtype=torch.bfloat16, beta_dtype=torch.float32,
                 dqdk_dtype=None, dv_dtype=None, has_h0=True, has_dht=True, seq_lens=None,
                 seed=0, h0_std=0.1, dht_std=0.1, g_shift=0.0, beta_zero=False,
                 gate_zero=False) -> Problem:
    """Draw one seeded problem.

    seq_lens: list of sequence lengths => varlen (B must be 1, T becomes their sum).
    g_shift: added to the raw log-gate before logsigmoid (tests use it to vary decay strength).
    beta_zero / gate_zero: special cases (beta = 0, g = 0) used by the invariant tests.
    """
    gen = torch.Generator().manual_seed(seed)
    cu = None
    if seq_lens is not None:
        assert B == 1
        seq_lens = [int(x) for x in seq_lens]
        cu = torch.tensor([0] + list(np.cumsum(seq_lens)), dtype=torch.int32)
        T = int(sum(seq_lens))
        N = len(seq_lens)
    else:
        N = B
    if scale is None:
        scale = 1.0 / math.sqrt(K)
    if dqdk_dtype is None:
        dqdk_dtype = qkv_dtype
    if dv_dtype is None:
        dv_dtype = qkv_dtype

    def rn(*shape):
        return torch.randn(*shape, generator=gen, dtype=torch.float32)

    q = l2_normalise(rn(B, T, Hk, K)).to(qkv_dtype)
    k = l2_normalise(rn(B, T, Hk, K)).to(qkv_dtype)
    v = rn(B, T, Hv, V).to(qkv_dtype)
    beta = torch.sigmoid(rn(B, T, Hv))
    if beta_zero:
        beta = torch.zeros_like(beta)
    beta = beta.to(beta_dtype)
    gshape = (B, T, Hv, K) if per_channel else (B, T, Hv)
    g = torch.nn.functional.logsigmoid(rn(*gshape) + g_shift)
    if gate_zero:
        g = torch.zeros_like(g)
    h0 = h0_std * rn(N, Hv, V, K) if has_h0 else None
    dO = rn(B, T, Hv, V).to(qkv_dtype)
    dht = dht_std * rn(N, Hv, V, K) if has_dht else None
    return Problem(name=name, B=B, T=T, Hk=Hk, Hv=Hv, K=K, V=V, BT=BT, per_channel=per_channel,
                   scale=float(scale), qkv_dtype=qkv_dtype, beta_dtype=beta_dtype,
                   dqdk_dtype=dqdk_dtype, dv_dtype=dv_dtype, q=q, k=k, v=v, beta=beta, g=g, dO=dO,
                   h0=h0, dht=dht, cu_seqlens=cu, seed=seed)


def varlen_lengths(seed: int, n: int = 8, lo: int = 512, hi: int = 8192):
    """Sequence lengths drawn uniformly from the integers [lo, hi] (inclusive) with a seeded generator."""
    gen = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (n,), generator=gen).tolist()


# The five workloads: tiny fp32, T=8192 bf16, T=32768 bf16 (headline), GQA + varlen bf16, KDA fp16.
WORKLOADS = ("tiny_fp32", "gdn_t8k_bf16", "gdn_t32k_bf16", "gqa_varlen_bf16", "kda_t2k_fp16")


def workload(name: str) -> Problem:
    if name == "tiny_fp32":
        return make_problem(name, B=1, T=128, Hk=2, Hv=2, K=32, V=32, BT=64,
                            qkv_dtype=torch.float32, has_h0=True, has_dht=False, seed=1001)
    if name == "gdn_t8k_bf16":
        return make_problem(name, B=1, T=8192, Hk=16, Hv=16, K=128, V=128, BT=64,
                            qkv_dtype=torch.bfloat16, has_h0=True, has_dht=True, seed=1002)
    if name == "gdn_t32k_bf16":
        return make_problem(name, B=1, T=32768, Hk=16, Hv=16, K=128, V=128, BT=64,
                            qkv_dtype=torch.bfloat16, has_h0=True, has_dht=True, seed=1003)
    if name == "gqa_varlen_bf16":
        lens = varlen_lengths(1004)
        return make_problem(name, B=1, Hk=16, Hv=32, K=128, V=128, BT=64, seq_lens=lens,
                            qkv_dtype=torch.bfloat16, has_h0=True, has_dht=False, seed=1004)
    if name == "kda_t2k_fp16":
        return make_problem(name, B=1, T=2048, Hk=32, Hv=32, K=128, V=128, BT=64, per_channel=True,
                            qkv_dtype=torch.float16, beta_dtype=torch.float16,
                            dqdk_dtype=torch.float32, dv_dtype=torch.float16,
                            has_h0=False, has_dht=False, seed=1005)
    raise KeyError(name)
