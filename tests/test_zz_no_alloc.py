"""gdr_bwd_run_noalloc, the entry point for callers that cannot allocate device memory (it keeps its
scratch in the library's own static device array instead of a caller workspace), must give the same
gradients as gdr_bwd_run on two calls in a row.  This file is collected last on purpose."""
import ctypes

import pytest
import torch

from chunked_gated_delta_09_gb300 import GdrError, _lib, ops
from chunked_gated_delta_09_gb300.inputs import make_problem
from parity_util import TOL, out_dtypes, rel_l2

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
    ref = {k: v.double().cpu().numpy() for k, v in ref.items()}
    for call in range(2):
        out = _fresh_outputs(plan)
        plan.run_noalloc(out=out, **dev)
        torch.cuda.synchronize()
        for name, dt in out_dtypes(prob).items():
            got = out[name].double().cpu().numpy()
            err = rel_l2(got, ref[name])
            assert err <= TOL[dt], (call, name, err)


def test_noalloc_rejects_plans_beyond_its_scratch():
    plan = ops.GdrBwdPlan(B=1, T=32768, Hk=16, Hv=16, K=128, V=128, has_h0=True, has_dht=True)
    assert plan.workspace_bytes > _lib.NOALLOC_MAX_WORKSPACE
    x = torch.empty(16, device="cuda")
    with pytest.raises(GdrError) as ei:
        plan.run_noalloc(q=x, k=x, v=x, beta=x, g=x, dO=x, h0=x, dht=x,
                         out={n: x for n in ("dq", "dk", "dv", "dbeta", "dg", "dh0")})
    assert ei.value.status == _lib.GDR_ERR_UNSUPPORTED
