"""gdr_bwd_run_noalloc, the entry point for callers that cannot allocate device memory (it keeps its
scratch in the library's own static device array instead of a caller workspace), must give the same
gradients as gdr_bwd_run on two calls in a row.  The backward is bit-reproducible run to run (fixed-slot
partial sums, no atomics in the arithmetic), so the comparison is bit for bit; before the checked calls a
problem of another shape runs through the same array, so that anything read from a previous call's
leftovers would show.  This file is collected last on purpose."""
import pytest
import torch

from chunked_gated_delta_09_gb300 import GdrError, _lib, ops
from chunked_gated_delta_09_gb300.inputs import make_problem

pytestmark = pytest.mark.gpu


def _fresh_outputs(plan):
    out = plan.alloc_outputs("cuda")
    for t in out.values():
        t.fill_(float("nan"))
    return out


def test_noalloc_matches_the_workspace_entry_point_on_two_calls():
    prob = make_problem("noalloc", B=1, Hk=2, Hv=4, K=64, V=64, seq_lens=[100, 37, 64, 1], seed=321)
    plan = ops.plan_for(prob)
    assert plan.workspace_bytes <= _lib.NOALLOC_MAX_WORKSPACE
    dev = ops.problem_to_device(prob, "cuda")
    ref = _fresh_outputs(plan)
    ws = plan.alloc_workspace("cuda")
    plan.run(out=ref, workspace=ws, **dev)
    assert plan.get_status(ws) == 0
    # another shape (more heads, dense, larger K) through the shared array first
    other = make_problem("noalloc_other", B=2, T=300, Hk=3, Hv=3, K=128, V=128, seed=5)
    oplan = ops.plan_for(other)
    oplan.run_noalloc(out=_fresh_outputs(oplan), **ops.problem_to_device(other, "cuda"))
    assert oplan.get_status_noalloc() == _lib.GDR_OK
    for call in range(2):
        out = _fresh_outputs(plan)
        plan.run_noalloc(out=out, **dev)
        assert plan.get_status_noalloc() == _lib.GDR_OK
        torch.cuda.synchronize()
        for name in ref:
            assert torch.equal(out[name], ref[name]), (call, name)


def test_noalloc_status_reports_malformed_cu_seqlens():
    prob = make_problem("noalloc_bad", Hk=1, Hv=2, K=64, V=64, seq_lens=[100, 37, 64], seed=6)
    plan = ops.plan_for(prob)
    dev = ops.problem_to_device(prob, "cuda")
    dev["cu_seqlens"] = torch.tensor([0, 100, 60, 201], dtype=torch.int32, device="cuda")  # decreasing
    plan.run_noalloc(out=_fresh_outputs(plan), **dev)
    assert plan.get_status_noalloc() == _lib.GDR_ERR_DEVICE
    # the word was cleared: a good call afterwards reports success
    good = ops.problem_to_device(prob, "cuda")
    plan.run_noalloc(out=_fresh_outputs(plan), **good)
    assert plan.get_status_noalloc() == _lib.GDR_OK


def test_noalloc_rejects_plans_beyond_its_scratch():
    plan = ops.GdrBwdPlan(B=1, T=32768, Hk=16, Hv=16, K=128, V=128, has_h0=True, has_dht=True)
    assert plan.workspace_bytes > _lib.NOALLOC_MAX_WORKSPACE
    x = torch.empty(16, device="cuda")
    with pytest.raises(GdrError) as ei:
        plan.run_noalloc(q=x, k=x, v=x, beta=x, g=x, dO=x, h0=x, dht=x,
                         out={n: x for n in ("dq", "dk", "dv", "dbeta", "dg", "dh0")})
    assert ei.value.status == _lib.GDR_ERR_UNSUPPORTED
    assert plan.get_status_noalloc() == _lib.GDR_ERR_UNSUPPORTED
