"""Helpers shared by the GPU parity tests: run the CUDA path, run the oracle, compare."""
from __future__ import annotations

import dataclasses
import json
import os

import numpy as np
import torch

import oracle
from chunked_gated_delta_09_gb300 import ops

# relative L2 bars: 2e-2 for bf16 / fp16 outputs, 5e-3 for fp32 outputs
TOL = {torch.float32: 5e-3, torch.bfloat16: 2e-2, torch.float16: 2e-2}


def out_dtypes(prob):
    return dict(dq=prob.dqdk_dtype, dk=prob.dqdk_dtype, dv=prob.dv_dtype, dbeta=torch.float32,
                dg=torch.float32, dh0=torch.float32)


def run_gpu(prob, plan=None, device="cuda"):
    plan = plan or ops.plan_for(prob)
    d = ops.problem_to_device(prob, device)
    out = plan.alloc_outputs(device)
    ws = plan.alloc_workspace(device)
    plan.run(out=out, workspace=ws, **d)
    st = plan.get_status(ws)
    assert st == 0, f"device status {st}"
    torch.cuda.synchronize()
    return {k: v.float().cpu().to(torch.float64).numpy() for k, v in out.items()}


def rel_l2(got, ref):
    """||got - ref|| / ||ref|| (the relative L2 error of the parity bars)."""
    nr = np.linalg.norm(ref)
    diff = np.linalg.norm(got - ref)
    return diff / nr if nr > 0 else (0.0 if diff == 0 else np.inf)


# A reference that is (numerically) zero has no meaningful relative error; it is compared absolutely instead:
# ||got - ref|| <= ZERO_REF_ABS * (the largest magnitude among the problem's inputs).  "Numerically zero"
# means a norm below that same absolute bar: exactly zero (dk and dv when every beta is 0) or below what an
# fp32 output can hold (the forward's final state with beta = 0 is h0 exp(sum g), about 1e-45 after 128
# tokens of g ~ logsigmoid(randn), under fp32's smallest normal 1.2e-38).
ZERO_REF_ABS = 1e-6


def input_scale(prob):
    """Largest |x| over the problem's inputs q, k, v, dO, h0, dht (the scale of an absolute bar)."""
    ts = [prob.q, prob.k, prob.v, prob.dO, prob.h0, prob.dht]
    return max(float(t.abs().max()) for t in ts if t is not None and t.numel() > 0)


def parity_error(got, ref, bar, prob):
    """(error, bar) of one output: relative L2 against `bar`, or, for a numerically zero reference, the
    absolute L2 difference against ZERO_REF_ABS times the input scale."""
    abs_bar = ZERO_REF_ABS * input_scale(prob)
    if np.linalg.norm(ref) > abs_bar:
        return rel_l2(got, ref), bar
    return float(np.linalg.norm(got - ref)), abs_bar


def compare(prob, got, ref, keys=None, slices=None):
    """Return {name: (rel_l2, tol)} and assert every output is within its tolerance."""
    res = {}
    for name, dt in out_dtypes(prob).items():
        if keys is not None and name not in keys:
            continue
        g, r = got[name], ref[name]
        if slices and name in slices:
            g = g[slices[name]]
        assert g.shape == r.shape, (name, g.shape, r.shape)
        assert np.all(np.isfinite(g)), f"{name} has non-finite values"
        res[name] = parity_error(g, r, TOL[dt], prob)
    log = os.environ.get("GDR_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"case": prob.name, **{k: v[0] for k, v in res.items()}}) + "\n")
    bad = {k: v for k, v in res.items() if not v[0] <= v[1]}
    assert not bad, f"{prob.name}: outside tolerance {bad} (all: {res})"
    return res


def head_subset(prob, hks):
    """The same problem restricted to key heads `hks` and the value heads that read them."""
    G = prob.Hv // prob.Hk
    hvs = [hk * G + j for hk in hks for j in range(G)]
    sub = dataclasses.replace(
        prob, name=prob.name + f"[hk{hks}]", Hk=len(hks), Hv=len(hvs),
        q=prob.q[:, :, hks].contiguous(), k=prob.k[:, :, hks].contiguous(), v=prob.v[:, :, hvs].contiguous(),
        beta=prob.beta[:, :, hvs].contiguous(), g=prob.g[:, :, hvs].contiguous(),
        dO=prob.dO[:, :, hvs].contiguous(),
        h0=None if prob.h0 is None else prob.h0[:, hvs].contiguous(),
        dht=None if prob.dht is None else prob.dht[:, hvs].contiguous())
    slices = dict(dq=(slice(None), slice(None), hks), dk=(slice(None), slice(None), hks),
                  dv=(slice(None), slice(None), hvs), dbeta=(slice(None), slice(None), hvs),
                  dg=(slice(None), slice(None), hvs), dh0=(slice(None), hvs))
    return sub, slices
