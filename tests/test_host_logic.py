"""Host-side logic: input recipe, workloads, FLOP / byte conventions, the binding's refusal to run
without a GPU."""
import math

import pytest
import torch

from chunked_gated_delta_09_gb300 import counts
from chunked_gated_delta_09_gb300.inputs import WORKLOADS, make_problem, varlen_lengths, workload


def test_generator_is_deterministic_and_follows_the_recipe():
    a = make_problem(B=1, T=100, Hk=2, Hv=4, K=32, V=16, seed=3)
    b = make_problem(B=1, T=100, Hk=2, Hv=4, K=32, V=16, seed=3)
    for n in ("q", "k", "v", "beta", "g", "dO", "h0", "dht"):
        assert torch.equal(getattr(a, n), getattr(b, n)), n
    nq = a.q.float().pow(2).sum(-1).sqrt()
    assert torch.allclose(nq, torch.ones_like(nq), atol=1e-2)
    assert (a.beta > 0).all() and (a.beta < 1).all()
    assert (a.g < 0).all()
    assert a.q.dtype == torch.bfloat16 and a.beta.dtype == torch.float32 and a.g.dtype == torch.float32


def test_workload_shapes():
    lens = varlen_lengths(1004)
    assert len(lens) == 8 and all(512 <= x <= 8192 for x in lens)
    shapes = {
        "tiny_fp32": (1, 128, 2, 2, 32, 32),
        "gdn_t8k_bf16": (1, 8192, 16, 16, 128, 128),
        "gdn_t32k_bf16": (1, 32768, 16, 16, 128, 128),
        "gqa_varlen_bf16": (1, sum(lens), 16, 32, 128, 128),
        "kda_t2k_fp16": (1, 2048, 32, 32, 128, 128),
    }
    for name in WORKLOADS:
        if name == "gdn_t32k_bf16":
            continue  # large; its shape is the T=8192 one with T=32768
        p = workload(name)
        assert (p.B, p.T, p.Hk, p.Hv, p.K, p.V) == shapes[name], name
    kda = workload("kda_t2k_fp16")
    assert kda.g.shape == (1, 2048, 32, 128) and kda.dqdk_dtype == torch.float32
    assert kda.dv_dtype == torch.float16 and kda.h0 is None and kda.dht is None


def test_flop_and_byte_conventions_for_the_headline_shape():
    assert counts.flops_per_chunk(64, 128, 128) == pytest.approx(32.68e6, rel=1e-3)
    # the headline T=32768, H=16, K=V=128 bf16 workload, built cheaply with the same shapes
    p = make_problem(B=1, T=32768, Hk=16, Hv=16, K=128, V=128, seed=0)
    assert counts.chunk_units(p) == 8192
    assert counts.total_flops(p) == pytest.approx(2.677e11, rel=1e-3)
    assert counts.algorithmic_bytes(p) == pytest.approx(951e6, rel=5e-3)


def test_binding_refuses_cpu_tensors():
    from chunked_gated_delta_09_gb300 import gdr_bwd
    p = make_problem(B=1, T=8, Hk=1, Hv=1, K=8, V=8, seed=0)
    with pytest.raises(ValueError):
        gdr_bwd(p.q, p.k, p.v, p.beta, p.g, p.dO, p.h0, p.dht)


def test_stage_flops_sum_to_the_total():
    p = make_problem(B=1, T=1000, Hk=2, Hv=4, K=64, V=32, BT=32, seed=0)
    assert sum(counts.stage_flops(p)) == pytest.approx(counts.total_flops(p), rel=1e-12)


def test_stage_bytes_of_the_per_chunk_gradient_stage():
    """Per chunk x head unit at the T=32768 bf16 shape the gradient stage reads S_0, dS_next (2 x 32 KB),
    V_new^T, -dV_new^T, D (3 x 16 KB), T (8 KB), q, k, v (3 x 16 KB) and the per-token record of the scalar
    gate (beta, exp(gamma), exp(gamma_C - gamma), gamma: 1 KB) and writes dq, dk, dv (3 x 16 KB), dbeta and
    d(gamma) (256 B each)."""
    from chunked_gated_delta_09_gb300 import counts
    from chunked_gated_delta_09_gb300.inputs import workload
    p = workload("gdn_t32k_bf16")
    per_unit = 2 * 32768 + 3 * 16384 + 8192 + 3 * 16384 + 1024 + 3 * 16384 + 2 * 256
    sb = counts.stage_bytes(p)
    assert sb[4] == 8192 * per_unit
    assert counts.scan_segments(p) == 9
    assert all(b > 0 for b in sb[1:])
    # the gradient stage sits below the ridge: HBM-bound at any peaks with ratio above 80 FLOP per byte
    assert counts.stage_flops(p)[4] / sb[4] < 80


def test_factored_scan_adds_one_launch(monkeypatch):
    """GDR_DH_FACTORED=1 adds the per-chunk QR kernel to a segmented plan (host-only plan creation)."""
    from chunked_gated_delta_09_gb300 import ops
    kw = dict(B=1, T=32768, Hk=16, Hv=16, K=128, V=128)
    base = ops.GdrBwdPlan(**kw).launch_count
    monkeypatch.setenv("GDR_DH_FACTORED", "1")
    assert ops.GdrBwdPlan(**kw).launch_count == base + 1


def test_single_segment_runs_both_scans_in_one_launch():
    """A short sequence (32 chunks per head here) is scanned as one segment, and then the forward and the
    state-gradient scans share one launch: K1, the scan pair, K4, K5 (host-only plan creation)."""
    from chunked_gated_delta_09_gb300 import counts, ops
    from chunked_gated_delta_09_gb300.inputs import workload
    assert counts.scan_segments(workload("kda_t2k_fp16")) == 1
    assert ops.GdrBwdPlan(B=1, T=2048, Hk=32, Hv=32, K=128, V=128, per_channel=True).launch_count == 4
    # a long one is segmented: K1, two local scans, two combines, two final scans, K4, K5
    assert counts.scan_segments(workload("gdn_t32k_bf16")) == 9
    assert ops.GdrBwdPlan(B=1, T=32768, Hk=16, Hv=16, K=128, V=128).launch_count == 9
