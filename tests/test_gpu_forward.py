"""Parity of the CUDA forward pass (gdr_fwd_run through the C ABI) with the fp64 token-recurrence oracle.

The forward returns o (in the input dtype) and the final state ht (fp32); the bars are those of the
backward outputs of the same dtypes (relative L2 2e-2 for bf16 / fp16, 5e-3 for fp32).  The autograd
Function that joins forward and backward is checked against the oracle's gradients.
"""
import json
import os
import zlib

import numpy as np
import pytest
import torch

import oracle
from chunked_gated_delta_09_gb300 import ops
from chunked_gated_delta_09_gb300.inputs import make_problem, workload
from parity_util import TOL, compare, parity_error
from test_gpu_parity import SMALL

pytestmark = pytest.mark.gpu


def run_forward_gpu(prob, device="cuda"):
    plan = ops.plan_for(prob)
    d = ops.problem_to_device(prob, device)
    out = plan.alloc_forward_outputs(device)
    ws = plan.alloc_workspace(device)
    plan.run_forward(q=d["q"], k=d["k"], v=d["v"], beta=d["beta"], g=d["g"], h0=d.get("h0"),
                     cu_seqlens=d.get("cu_seqlens"), out=out, workspace=ws)
    assert plan.get_status(ws) == 0
    torch.cuda.synchronize()
    return {k: v.float().cpu().to(torch.float64).numpy() for k, v in out.items()}


def oracle_forward(prob):
    a = prob.packed_f64()
    o, hT, _ = oracle.forward(a["cu"], prob.Hk, prob.Hv, prob.K, prob.V, prob.per_channel, prob.scale,
                              a["q"], a["k"], a["v"], a["beta"], a["g"], a["h0"])
    return {"o": o.reshape(prob.B, prob.T, prob.Hv, prob.V), "ht": hT}


def check_forward(prob, got, ref):
    bars = {"o": TOL[prob.qkv_dtype], "ht": TOL[torch.float32]}
    res = {}
    for key, bar in bars.items():
        g, r = got[key], ref[key]
        assert g.shape == r.shape, (key, g.shape, r.shape)
        assert np.all(np.isfinite(g)), f"{key} has non-finite values"
        res[key] = parity_error(g, r, bar, prob)
    log = os.environ.get("GDR_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"case": "fwd:" + prob.name, **{k: v[0] for k, v in res.items()}}) + "\n")
    bad = {k: v for k, v in res.items() if not v[0] <= v[1]}
    assert not bad, f"{prob.name}: outside tolerance {bad} (all: {res})"


@pytest.mark.parametrize("name", sorted(SMALL))
def test_forward_small_cases_match_oracle(name):
    prob = make_problem(name, seed=zlib.crc32(name.encode()) % 1000, **SMALL[name])
    check_forward(prob, run_forward_gpu(prob), oracle_forward(prob))


@pytest.mark.parametrize("BT", [16, 32, 64])
@pytest.mark.parametrize("per_channel", [False, True], ids=["scalar", "kda"])
def test_forward_chunk_size_invariance(BT, per_channel):
    prob = make_problem(f"fwd_bt{BT}", B=1, Hk=1, Hv=2, K=64, V=64, BT=BT, per_channel=per_channel,
                        seq_lens=[100, 0, 37], seed=78)
    check_forward(prob, run_forward_gpu(prob), oracle_forward(prob))


@pytest.mark.parametrize("nseg", [1, 3])
def test_forward_segment_counts(nseg, monkeypatch):
    monkeypatch.setenv("GDR_NSEG", str(nseg))
    prob = make_problem(f"fwd_nseg{nseg}", B=1, Hk=1, Hv=2, K=64, V=64, seq_lens=[700, 64, 130, 1], seed=89)
    check_forward(prob, run_forward_gpu(prob), oracle_forward(prob))


@pytest.mark.parametrize("name", ["tiny_fp32", "kda_t2k_fp16", "gdn_t8k_bf16", "gdn_t32k_bf16", "gqa_varlen_bf16"])
def test_forward_workloads(name):
    prob = workload(name)
    check_forward(prob, run_forward_gpu(prob), oracle_forward(prob))


@pytest.mark.parametrize("per_channel", [False, True], ids=["scalar", "kda"])
def test_autograd_function_matches_oracle_gradients(per_channel):
    """loss = <o, dO> + <ht, dht> through ChunkGatedDeltaRule.apply and torch.autograd; the gradients of
    q, k, v, beta, g and h0 equal the oracle's."""
    prob = make_problem("autograd", Hk=1, Hv=2, K=64, V=64, per_channel=per_channel, seq_lens=[150, 70],
                        seed=17)
    d = ops.problem_to_device(prob, "cuda")
    leaves = {n: d[n].clone().requires_grad_(True) for n in ("q", "k", "v", "beta", "g", "h0")}
    o, ht = ops.chunk_gated_delta_rule(leaves["q"], leaves["k"], leaves["v"], leaves["beta"], leaves["g"],
                                       leaves["h0"], d["cu_seqlens"], scale=prob.scale, BT=prob.BT)
    loss = (o.float() * d["dO"].float()).sum() + (ht * d["dht"]).sum()
    loss.backward()
    ref = oracle.problem_backward(prob)
    got = {"dq": leaves["q"].grad, "dk": leaves["k"].grad, "dv": leaves["v"].grad, "dbeta": leaves["beta"].grad,
           "dg": leaves["g"].grad, "dh0": leaves["h0"].grad}
    got = {k: v.float().cpu().to(torch.float64).numpy() for k, v in got.items()}
    compare(prob, got, ref)
