"""Torch-facing wrapper of the C ABI: the same calls, with torch tensors for device memory and streams.

Every step of the forward and the backward runs in libgdrbwd.so's kernels; this module only checks
tensor placement, allocates outputs and workspace with torch, and passes raw pointers.  A missing
library raises.  :class:`ChunkGatedDeltaRule` joins the two as a torch.autograd.Function.
"""
from __future__ import annotations

import ctypes
import math
from typing import Optional

import torch

from . import _lib
from ._lib import GdrBwdArgs, GdrBwdDesc, GdrError, GdrFwdArgs, GdrWyArgs

_DT = {torch.float32: _lib.GDR_F32, torch.bfloat16: _lib.GDR_BF16, torch.float16: _lib.GDR_F16}


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


class GdrBwdPlan:
    """Owns one gdr_bwd_plan (host object).  Create once per problem shape, run many times."""

    def __init__(self, *, B, T, Hk, Hv, K, V, BT=64, num_seqs=0, per_channel=False, scale=None,
                 qkv_dtype=torch.bfloat16, beta_dtype=torch.float32, dqdk_dtype=None, dv_dtype=None,
                 has_h0=False, has_dht=False):
        self.lib = _lib.load()
        self.desc = GdrBwdDesc(B=B, T=T, Hk=Hk, Hv=Hv, K=K, V=V, BT=BT, num_seqs=num_seqs,
                               gate_per_channel=int(per_channel),
                               scale=float(scale) if scale else 0.0,
                               qkv_dtype=_DT[qkv_dtype], beta_dtype=_DT[beta_dtype],
                               dqdk_dtype=_DT[dqdk_dtype or qkv_dtype], dv_dtype=_DT[dv_dtype or qkv_dtype],
                               has_h0=int(has_h0), has_dht=int(has_dht))
        self.shape = dict(B=B, T=T, Hk=Hk, Hv=Hv, K=K, V=V, BT=BT, num_seqs=num_seqs, per_channel=per_channel)
        self.scale = float(scale) if scale else 1.0 / math.sqrt(K)
        self.dqdk_dtype = dqdk_dtype or qkv_dtype
        self.dv_dtype = dv_dtype or qkv_dtype
        self.handle = ctypes.c_void_p()
        st = self.lib.gdr_bwd_create(ctypes.byref(self.desc), ctypes.byref(self.handle))
        if st != _lib.GDR_OK:
            raise GdrError(st, "gdr_bwd_create")

    @property
    def workspace_bytes(self) -> int:
        return int(self.lib.gdr_bwd_workspace_bytes(self.handle))

    def alloc_workspace(self, device="cuda") -> torch.Tensor:
        return torch.empty(max(self.workspace_bytes, 256), dtype=torch.uint8, device=device)

    def alloc_outputs(self, device="cuda") -> dict:
        s = self.shape
        N = s["B"] if s["num_seqs"] == 0 else s["num_seqs"]
        B, T, Hk, Hv, K, V = s["B"], s["T"], s["Hk"], s["Hv"], s["K"], s["V"]
        gshape = (B, T, Hv, K) if s["per_channel"] else (B, T, Hv)
        return dict(dq=torch.empty(B, T, Hk, K, dtype=self.dqdk_dtype, device=device),
                    dk=torch.empty(B, T, Hk, K, dtype=self.dqdk_dtype, device=device),
                    dv=torch.empty(B, T, Hv, V, dtype=self.dv_dtype, device=device),
                    dbeta=torch.empty(B, T, Hv, dtype=torch.float32, device=device),
                    dg=torch.empty(gshape, dtype=torch.float32, device=device),
                    dh0=torch.empty(N, Hv, V, K, dtype=torch.float32, device=device))

    def run(self, *, q, k, v, beta, g, dO, h0=None, dht=None, cu_seqlens=None, out: dict, workspace,
            stream=None):
        """Queue gdr_bwd_run on `stream` (default: torch's current stream).  Asynchronous."""
        args = GdrBwdArgs(q=_ptr(q), k=_ptr(k), v=_ptr(v), beta=_ptr(beta), g=_ptr(g), h0=_ptr(h0), dO=_ptr(dO),
                          dht=_ptr(dht), cu_seqlens=_ptr(cu_seqlens), dq=_ptr(out["dq"]), dk=_ptr(out["dk"]),
                          dv=_ptr(out["dv"]), dbeta=_ptr(out["dbeta"]), dg=_ptr(out["dg"]),
                          dh0=_ptr(out.get("dh0")))
        st = self.lib.gdr_bwd_run(self.handle, ctypes.byref(args), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream_ptr(stream))
        if st != _lib.GDR_OK:
            raise GdrError(st, "gdr_bwd_run")

    def run_profiled(self, events, *, q, k, v, beta, g, dO, h0=None, dht=None, cu_seqlens=None, out: dict,
                     workspace, stream=None):
        """As :meth:`run`, recording ``events`` (NUM_STAGES + 1 torch.cuda.Event with timing, already
        recorded once so that their handles exist) around each kernel stage."""
        args = GdrBwdArgs(q=_ptr(q), k=_ptr(k), v=_ptr(v), beta=_ptr(beta), g=_ptr(g), h0=_ptr(h0), dO=_ptr(dO),
                          dht=_ptr(dht), cu_seqlens=_ptr(cu_seqlens), dq=_ptr(out["dq"]), dk=_ptr(out["dk"]),
                          dv=_ptr(out["dv"]), dbeta=_ptr(out["dbeta"]), dg=_ptr(out["dg"]),
                          dh0=_ptr(out.get("dh0")))
        arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
        st = self.lib.gdr_bwd_run_profiled(self.handle, ctypes.byref(args), _ptr(workspace),
                                           workspace.numel() * workspace.element_size(), _stream_ptr(stream), arr)
        if st != _lib.GDR_OK:
            raise GdrError(st, "gdr_bwd_run_profiled")

    def run_noalloc(self, *, q, k, v, beta, g, dO, h0=None, dht=None, cu_seqlens=None, out: dict, stream=None):
        """Queue gdr_bwd_run_noalloc: the same backward with the library's own static scratch array
        instead of a workspace (plans up to NOALLOC_MAX_WORKSPACE bytes of workspace)."""
        args = GdrBwdArgs(q=_ptr(q), k=_ptr(k), v=_ptr(v), beta=_ptr(beta), g=_ptr(g), h0=_ptr(h0), dO=_ptr(dO),
                          dht=_ptr(dht), cu_seqlens=_ptr(cu_seqlens), dq=_ptr(out["dq"]), dk=_ptr(out["dk"]),
                          dv=_ptr(out["dv"]), dbeta=_ptr(out["dbeta"]), dg=_ptr(out["dg"]),
                          dh0=_ptr(out.get("dh0")))
        st = self.lib.gdr_bwd_run_noalloc(self.handle, ctypes.byref(args), _stream_ptr(stream))
        if st != _lib.GDR_OK:
            raise GdrError(st, "gdr_bwd_run_noalloc")

    def alloc_forward_outputs(self, device="cuda", qkv_dtype=None) -> dict:
        s = self.shape
        N = s["B"] if s["num_seqs"] == 0 else s["num_seqs"]
        dt = qkv_dtype or {v: k for k, v in _DT.items()}[self.desc.qkv_dtype]
        return dict(o=torch.empty(s["B"], s["T"], s["Hv"], s["V"], dtype=dt, device=device),
                    ht=torch.empty(N, s["Hv"], s["V"], s["K"], dtype=torch.float32, device=device))

    def run_forward(self, *, q, k, v, beta, g, h0=None, cu_seqlens=None, out: dict, workspace, stream=None):
        """Queue gdr_fwd_run (o and, if ``out`` has it, the final state ht) on `stream`.  Asynchronous."""
        args = GdrFwdArgs(q=_ptr(q), k=_ptr(k), v=_ptr(v), beta=_ptr(beta), g=_ptr(g), h0=_ptr(h0),
                          cu_seqlens=_ptr(cu_seqlens), o=_ptr(out["o"]), ht=_ptr(out.get("ht")))
        st = self.lib.gdr_fwd_run(self.handle, ctypes.byref(args), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream_ptr(stream))
        if st != _lib.GDR_OK:
            raise GdrError(st, "gdr_fwd_run")

    @property
    def forward_launch_count(self) -> int:
        return int(self.lib.gdr_fwd_launch_count(self.handle))

    @property
    def launch_count(self) -> int:
        return int(self.lib.gdr_bwd_launch_count(self.handle))

    def get_status(self, workspace, stream=None) -> int:
        return int(self.lib.gdr_bwd_get_status(self.handle, _ptr(workspace), _stream_ptr(stream)))

    def get_status_noalloc(self, stream=None) -> int:
        """Status word of the last :meth:`run_noalloc` on the current device (gdr_bwd_get_status_noalloc)."""
        return int(self.lib.gdr_bwd_get_status_noalloc(self.handle, _stream_ptr(stream)))

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value:
            self.lib.gdr_bwd_destroy(h)
            self.handle = ctypes.c_void_p()


def _check_cuda(**tensors):
    for name, t in tensors.items():
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor (the backward has no CPU path)")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")


def gdr_bwd(q, k, v, beta, g, dO, h0=None, dht=None, cu_seqlens=None, *, scale=None, BT=64,
            dqdk_dtype=None, dv_dtype=None, stream=None, check_status=False) -> dict:
    """Backward of the chunked gated delta rule on CUDA tensors.

    q, k [B, T, Hk, K]; v, dO [B, T, Hv, V]; beta [B, T, Hv]; g [B, T, Hv] or [B, T, Hv, K] (raw fp32
    log-gate); h0, dht fp32 [N, Hv, V, K] or None; cu_seqlens int32 [N+1] (varlen, B == 1) or None.
    Returns dict(dq, dk, dv, dbeta, dg, dh0).
    """
    _check_cuda(q=q, k=k, v=v, beta=beta, g=g, dO=dO, h0=h0, dht=dht, cu_seqlens=cu_seqlens)
    B, T, Hk, K = q.shape
    Hv, V = v.shape[2], v.shape[3]
    per_channel = g.dim() == 4
    num_seqs = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
    plan = GdrBwdPlan(B=B, T=T, Hk=Hk, Hv=Hv, K=K, V=V, BT=BT, num_seqs=num_seqs, per_channel=per_channel,
                      scale=scale, qkv_dtype=q.dtype, beta_dtype=beta.dtype, dqdk_dtype=dqdk_dtype,
                      dv_dtype=dv_dtype, has_h0=h0 is not None, has_dht=dht is not None)
    out = plan.alloc_outputs(q.device)
    ws = plan.alloc_workspace(q.device)
    plan.run(q=q, k=k, v=v, beta=beta, g=g, dO=dO, h0=h0, dht=dht, cu_seqlens=cu_seqlens, out=out,
             workspace=ws, stream=stream)
    if check_status:
        st = plan.get_status(ws, stream)
        if st != _lib.GDR_OK:
            raise GdrError(st, "gdr_bwd_get_status")
    return out


def gdr_fwd(q, k, v, beta, g, h0=None, cu_seqlens=None, *, scale=None, BT=64, stream=None,
            check_status=False):
    """Forward of the chunked gated delta rule on CUDA tensors (shapes as :func:`gdr_bwd`).

    Returns (o [B, T, Hv, V] in q's dtype, ht fp32 [N, Hv, V, K], the final state per sequence).
    """
    _check_cuda(q=q, k=k, v=v, beta=beta, g=g, h0=h0, cu_seqlens=cu_seqlens)
    B, T, Hk, K = q.shape
    Hv, V = v.shape[2], v.shape[3]
    num_seqs = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
    plan = GdrBwdPlan(B=B, T=T, Hk=Hk, Hv=Hv, K=K, V=V, BT=BT, num_seqs=num_seqs, per_channel=g.dim() == 4,
                      scale=scale, qkv_dtype=q.dtype, beta_dtype=beta.dtype, has_h0=h0 is not None)
    out = plan.alloc_forward_outputs(q.device)
    ws = plan.alloc_workspace(q.device)
    plan.run_forward(q=q, k=k, v=v, beta=beta, g=g, h0=h0, cu_seqlens=cu_seqlens, out=out, workspace=ws,
                     stream=stream)
    if check_status:
        st = plan.get_status(ws, stream)
        if st != _lib.GDR_OK:
            raise GdrError(st, "gdr_bwd_get_status")
    return out["o"], out["ht"]


class ChunkGatedDeltaRule(torch.autograd.Function):
    """o, ht = forward(q, k, v, beta, g, h0, cu_seqlens, scale, BT): the chunked gated delta rule with its
    exact backward, both on the GPU kernels.  Gradients flow to q, k, v, beta, g (raw log-gate) and h0;
    the backward recomputes the chunk states from the inputs (nothing but the inputs is saved)."""

    @staticmethod
    def forward(ctx, q, k, v, beta, g, h0=None, cu_seqlens=None, scale=None, BT=64):
        for t in (q, k, v, beta, g, h0):
            if t is not None and not t.is_contiguous():
                raise ValueError("inputs must be contiguous")
        B, T, Hk, K = q.shape
        Hv, V = v.shape[2], v.shape[3]
        num_seqs = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
        plan = GdrBwdPlan(B=B, T=T, Hk=Hk, Hv=Hv, K=K, V=V, BT=BT, num_seqs=num_seqs, per_channel=g.dim() == 4,
                          scale=scale, qkv_dtype=q.dtype, beta_dtype=beta.dtype, has_h0=h0 is not None,
                          has_dht=True)
        out = plan.alloc_forward_outputs(q.device)
        ws = plan.alloc_workspace(q.device)
        plan.run_forward(q=q, k=k, v=v, beta=beta, g=g, h0=h0, cu_seqlens=cu_seqlens, out=out, workspace=ws)
        ctx.plan = plan  # the workspace is released here; the backward takes a fresh one
        ctx.save_for_backward(q, k, v, beta, g, h0, cu_seqlens)
        return out["o"], out["ht"]

    @staticmethod
    def backward(ctx, do, dht):
        q, k, v, beta, g, h0, cu_seqlens = ctx.saved_tensors
        plan = ctx.plan
        if do is None:
            do = torch.zeros(*q.shape[:2], v.shape[2], v.shape[3], dtype=q.dtype, device=q.device)
        if dht is None:
            N = q.shape[0] if cu_seqlens is None else cu_seqlens.numel() - 1
            dht = torch.zeros(N, v.shape[2], v.shape[3], q.shape[3], dtype=torch.float32, device=q.device)
        do, dht = do.contiguous(), dht.contiguous().float()
        ws = plan.alloc_workspace(q.device)
        out = plan.alloc_outputs(q.device)
        plan.run(q=q, k=k, v=v, beta=beta, g=g, dO=do.to(q.dtype), h0=h0, dht=dht, cu_seqlens=cu_seqlens,
                 out=out, workspace=ws)
        return (out["dq"], out["dk"], out["dv"], out["dbeta"].to(beta.dtype), out["dg"],
                out["dh0"] if h0 is not None else None, None, None, None)


def chunk_gated_delta_rule(q, k, v, beta, g, h0=None, cu_seqlens=None, *, scale=None, BT=64):
    """Differentiable chunked gated delta rule: returns (o, ht); see :class:`ChunkGatedDeltaRule`."""
    _check_cuda(q=q, k=k, v=v, beta=beta, g=g, h0=h0, cu_seqlens=cu_seqlens)
    return ChunkGatedDeltaRule.apply(q, k, v, beta, g, h0, cu_seqlens, scale, BT)


def gdr_wy_bwd(q, k, v, v_new, g, beta, A, h, do, dh, dv, scale=None, cu_seqlens=None, chunk_size=64,
               stream=None, check_status=False):
    """The WY-gradient stage taken alone (gdr_wy_bwd_run; per-channel gate), with the argument order and
    return order (dq, dk, dv, db, dg, dA) of the operation it follows.  q, k [B, T, H, K]; v, v_new, do, dv
    [B, T, H, V]; beta [B, T, H]; A [B, T, H, BT] (one dtype: fp16, bf16 or fp32); g fp32 [B, T, H, K]
    (chunk-local cumulative gate); h, dh fp32 [B, NT, H, K, V]; cu_seqlens int32 [N+1] (B == 1) or None."""
    _check_cuda(q=q, k=k, v=v, v_new=v_new, g=g, beta=beta, A=A, h=h, do=do, dh=dh, dv=dv, cu_seqlens=cu_seqlens)
    B, T, H, K = q.shape
    V = v.shape[3]
    if A.shape[-1] != chunk_size:
        raise ValueError("chunk_size must equal A.shape[-1]")
    num_seqs = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
    plan = GdrBwdPlan(B=B, T=T, Hk=H, Hv=H, K=K, V=V, BT=chunk_size, num_seqs=num_seqs, per_channel=True,
                      scale=scale, qkv_dtype=q.dtype, beta_dtype=q.dtype, dqdk_dtype=torch.float32,
                      dv_dtype=q.dtype)
    dev = q.device
    out = dict(dq=torch.empty(B, T, H, K, dtype=torch.float32, device=dev),
               dk=torch.empty(B, T, H, K, dtype=torch.float32, device=dev),
               dv=torch.empty(B, T, H, V, dtype=q.dtype, device=dev),
               db=torch.empty(B, T, H, dtype=torch.float32, device=dev),
               dg=torch.empty(B, T, H, K, dtype=torch.float32, device=dev),
               dA=torch.empty(B, T, H, chunk_size, dtype=torch.float32, device=dev))
    ws = plan.alloc_workspace(dev)
    args = GdrWyArgs(q=_ptr(q), k=_ptr(k), v=_ptr(v), v_new=_ptr(v_new), beta=_ptr(beta), A=_ptr(A), dO=_ptr(do),
                     dv=_ptr(dv), g=_ptr(g), h=_ptr(h), dh=_ptr(dh), cu_seqlens=_ptr(cu_seqlens),
                     dq=_ptr(out["dq"]), dk=_ptr(out["dk"]), dv_out=_ptr(out["dv"]), db=_ptr(out["db"]),
                     dg=_ptr(out["dg"]), dA=_ptr(out["dA"]))
    st = plan.lib.gdr_wy_bwd_run(plan.handle, ctypes.byref(args), _ptr(ws), ws.numel(), _stream_ptr(stream))
    if st != _lib.GDR_OK:
        raise GdrError(st, "gdr_wy_bwd_run")
    if check_status:
        st = plan.get_status(ws, stream)
        if st != _lib.GDR_OK:
            raise GdrError(st, "gdr_bwd_get_status")
    return out["dq"], out["dk"], out["dv"], out["db"], out["dg"], out["dA"]


def chunk_indices(cu_seqlens: torch.Tensor, BT: int, max_chunks: Optional[int] = None, stream=None):
    """Device chunk bookkeeping through gdr_chunk_indices: returns (chunk_indices [max_chunks, 2],
    chunk_offsets [N+1]) as int32 CUDA tensors; unused rows are (-1, -1)."""
    _check_cuda(cu_seqlens=cu_seqlens)
    if cu_seqlens.dtype != torch.int32:
        raise ValueError("cu_seqlens must be int32")
    N = cu_seqlens.numel() - 1
    if max_chunks is None:
        max_chunks = int(cu_seqlens[-1].item()) // BT + N
    idx = torch.empty(max(max_chunks, 1), 2, dtype=torch.int32, device=cu_seqlens.device)
    off = torch.empty(N + 1, dtype=torch.int32, device=cu_seqlens.device)
    st = _lib.load().gdr_chunk_indices(_ptr(cu_seqlens), N, BT, max_chunks, _ptr(idx), _ptr(off),
                                       _stream_ptr(stream))
    if st != _lib.GDR_OK:
        raise GdrError(st, "gdr_chunk_indices")
    return idx[:max_chunks], off


def problem_to_device(prob, device="cuda") -> dict:
    """Copy a seeded :class:`inputs.Problem` to the device (argument marshalling for tests and bench)."""
    def d(t):
        return None if t is None else t.to(device).contiguous()
    return dict(q=d(prob.q), k=d(prob.k), v=d(prob.v), beta=d(prob.beta), g=d(prob.g), dO=d(prob.dO),
                h0=d(prob.h0), dht=d(prob.dht), cu_seqlens=d(prob.cu_seqlens))


def plan_for(prob) -> GdrBwdPlan:
    return GdrBwdPlan(B=prob.B, T=prob.T, Hk=prob.Hk, Hv=prob.Hv, K=prob.K, V=prob.V, BT=prob.BT,
                      num_seqs=prob.num_seqs, per_channel=prob.per_channel, scale=prob.scale,
                      qkv_dtype=prob.qkv_dtype, beta_dtype=prob.beta_dtype, dqdk_dtype=prob.dqdk_dtype,
                      dv_dtype=prob.dv_dtype, has_h0=prob.h0 is not None, has_dht=prob.dht is not None)
