"""Device-side failure reporting, exercised without faulting the GPU.

* Bounded waits: the plan's poll limit (GDR_SPIN_LIMIT, read when the plan is built) is lowered to one
  poll, so real waits for bulk copies and tensor-core work run out.  The run must report
  GDR_ERR_TIMEOUT through gdr_bwd_get_status, every CTA must drain what it started before exiting (the
  context stays usable), and the next run with the normal limit must match the oracle.
* Malformed cu_seqlens (not non-decreasing) must be reported as GDR_ERR_DEVICE, with every kernel after
  the bookkeeping doing nothing.
* Input values that the fp16 tensor-core operands cannot hold (|x| > 65504) must be reported as
  GDR_ERR_DEVICE rather than returned as silently wrong gradients.
"""
import pytest
import torch

import oracle
from chunked_gated_delta_09_gb300 import _lib, ops
from chunked_gated_delta_09_gb300.inputs import make_problem
from parity_util import compare, run_gpu

pytestmark = pytest.mark.gpu


def _run_status(prob, plan):
    dev = ops.problem_to_device(prob, "cuda")
    out = plan.alloc_outputs("cuda")
    ws = plan.alloc_workspace("cuda")
    plan.run(out=out, workspace=ws, **dev)
    st = plan.get_status(ws)
    torch.cuda.synchronize()
    return st


@pytest.mark.parametrize("per_channel", [False, True], ids=["scalar", "kda"])
def test_a_wait_that_runs_out_reports_timeout_and_the_next_run_is_exact(per_channel, monkeypatch):
    prob = make_problem("spin", B=1, T=4096, Hk=4, Hv=4, K=128, V=128, per_channel=per_channel, seed=17)
    monkeypatch.setenv("GDR_SPIN_LIMIT", "1")
    short = ops.plan_for(prob)
    statuses = [_run_status(prob, short) for _ in range(3)]
    assert set(statuses) <= {_lib.GDR_OK, _lib.GDR_ERR_TIMEOUT}, statuses
    assert _lib.GDR_ERR_TIMEOUT in statuses, statuses
    monkeypatch.delenv("GDR_SPIN_LIMIT")
    compare(prob, run_gpu(prob), oracle.problem_backward(prob))


def test_malformed_cu_seqlens_reports_device_error():
    prob = make_problem("badcu", Hk=1, Hv=2, K=64, V=64, seq_lens=[100, 37, 64], seed=4)
    prob.cu_seqlens = torch.tensor([0, 100, 60, 201], dtype=torch.int32)  # not non-decreasing
    assert _run_status(prob, ops.plan_for(prob)) == _lib.GDR_ERR_DEVICE


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "fp32"])
def test_inputs_beyond_fp16_range_report_device_error(dtype):
    prob = make_problem("range", B=1, T=200, Hk=1, Hv=2, K=64, V=64, qkv_dtype=dtype, seed=8)
    prob.v = prob.v.clone()
    prob.v[0, 77, 1, 5] = 1.0e5
    assert _run_status(prob, ops.plan_for(prob)) == _lib.GDR_ERR_DEVICE
    # the same problem within range is accepted
    ok = make_problem("range_ok", B=1, T=200, Hk=1, Hv=2, K=64, V=64, qkv_dtype=dtype, seed=8)
    assert _run_status(ok, ops.plan_for(ok)) == _lib.GDR_OK
