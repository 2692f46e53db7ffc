"""Parity of the CUDA path (through the C ABI) with the fp64 oracle on the same seeded inputs.

Small cases span several chunk tiles and ragged tails and cover every supported variant; the five
named workloads run at full size, the two longest ones on a sample of whole heads (every token of
the sampled heads is compared).  Bars: relative L2 <= 2e-2 for bf16 / fp16 outputs, <= 5e-3 for fp32.
"""
import zlib

import pytest
import torch

import oracle
from chunked_gated_delta_09_gb300.inputs import make_problem, workload
from parity_util import compare, head_subset, run_gpu

pytestmark = pytest.mark.gpu

SMALL = {
    "dense_ragged_bf16": dict(B=2, T=300, Hk=2, Hv=2, K=64, V=64),
    "gqa_varlen_bf16": dict(Hk=2, Hv=4, K=64, V=64, seq_lens=[1, 63, 64, 65, 0, 200]),
    "kda_fp16": dict(B=1, T=200, Hk=2, Hv=2, K=128, V=128, per_channel=True, qkv_dtype=torch.float16,
                     beta_dtype=torch.float16, dqdk_dtype=torch.float32, dv_dtype=torch.float16),
    "kda_varlen_bf16": dict(Hk=1, Hv=2, K=64, V=64, per_channel=True, seq_lens=[70, 5, 130]),
    "fp32_all": dict(B=1, T=150, Hk=1, Hv=2, K=32, V=32, qkv_dtype=torch.float32),
    "fp16_scalar": dict(B=1, T=256, Hk=2, Hv=2, K=128, V=128, qkv_dtype=torch.float16),
    "single_token": dict(B=3, T=1, Hk=1, Hv=1, K=32, V=32),
    "no_h0_no_dht": dict(B=1, T=130, Hk=1, Hv=1, K=128, V=128, has_h0=False, has_dht=False),
    "k64_v32": dict(B=1, T=100, Hk=1, Hv=1, K=64, V=32),
    "k128_v64_gqa4": dict(B=1, T=129, Hk=1, Hv=4, K=128, V=64),
    # three value heads per key head, fp16 throughout: the group's dq / dk summed in place in fp16
    "fp16_gqa3": dict(B=1, T=200, Hk=2, Hv=6, K=64, V=64, qkv_dtype=torch.float16),
    "strong_decay": dict(B=1, T=256, Hk=1, Hv=2, K=128, V=128, g_shift=-3.0),
    "weak_decay": dict(B=1, T=256, Hk=1, Hv=2, K=128, V=128, g_shift=4.0),
    # per-channel gate with strong decay: chunk-wide cumulative gates far below the fp32 exponent range, so
    # any decay factor formed as a ratio of cumulative gates (rather than a difference inside one exp) would
    # overflow or lose the result
    "kda_strong_decay": dict(B=1, T=256, Hk=1, Hv=2, K=128, V=128, per_channel=True, g_shift=-3.0),
    "beta_zero": dict(B=1, T=128, Hk=1, Hv=1, K=64, V=64, beta_zero=True),
    "gate_zero": dict(B=1, T=128, Hk=1, Hv=1, K=64, V=64, gate_zero=True),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_cases_match_oracle(name):
    prob = make_problem(name, seed=zlib.crc32(name.encode()) % 1000, **SMALL[name])
    compare(prob, run_gpu(prob), oracle.problem_backward(prob))


@pytest.mark.parametrize("BT", [16, 32, 64])
@pytest.mark.parametrize("per_channel", [False, True], ids=["scalar", "kda"])
def test_chunk_size_invariance(BT, per_channel):
    """Every supported chunk size computes the same gradient (the oracle has no chunks at all)."""
    prob = make_problem(f"bt{BT}", B=1, Hk=1, Hv=2, K=64, V=64, BT=BT, per_channel=per_channel,
                        seq_lens=[100, 37], seed=77)
    compare(prob, run_gpu(prob), oracle.problem_backward(prob))


def test_varlen_single_sequence_equals_dense():
    dense = make_problem("dense", B=1, T=333, Hk=2, Hv=2, K=64, V=64, seed=5)
    var = make_problem("var", B=1, Hk=2, Hv=2, K=64, V=64, seq_lens=[333], seed=5)
    a, b = run_gpu(dense), run_gpu(var)
    for key in a:
        assert (a[key] == b[key]).all(), key


@pytest.mark.parametrize("per_channel", [False, True], ids=["scalar", "kda"])
def test_run_to_run_bit_identical(per_channel):
    """Every reduction sums in a fixed order: two runs of one problem give the same bits."""
    prob = make_problem("repeat", Hk=2, Hv=4, K=128, V=128, per_channel=per_channel,
                        seq_lens=[700, 33, 190], seed=91)
    a, b = run_gpu(prob), run_gpu(prob)
    for key in a:
        assert (a[key] == b[key]).all(), key


@pytest.mark.parametrize("name", ["tiny_fp32", "kda_t2k_fp16", "gdn_t8k_bf16"])
def test_workload_full(name):
    prob = workload(name)
    compare(prob, run_gpu(prob), oracle.problem_backward(prob))


@pytest.mark.parametrize("name,hks", [("gdn_t32k_bf16", [0, 7, 11, 15]), ("gqa_varlen_bf16", [0, 5, 10, 15])])
def test_workload_sampled_heads(name, hks):
    prob = workload(name)
    got = run_gpu(prob)
    sub, slices = head_subset(prob, hks)
    compare(prob, got, oracle.problem_backward(sub), slices=slices)


@pytest.mark.parametrize("nseg", [1, 2, 3, 7])
@pytest.mark.parametrize("per_channel", [False, True], ids=["scalar", "kda"])
def test_segment_parallel_scan_matches_oracle(nseg, per_channel, monkeypatch):
    """The scans split each sequence into segments and combine exactly; any segment count gives the
    oracle's gradients (varlen sequences of different lengths, some shorter than a segment)."""
    monkeypatch.setenv("GDR_NSEG", str(nseg))
    prob = make_problem(f"nseg{nseg}", B=1, Hk=1, Hv=2, K=64, V=64, per_channel=per_channel,
                        seq_lens=[700, 64, 130, 1], seed=88)
    compare(prob, run_gpu(prob), oracle.problem_backward(prob))


@pytest.mark.parametrize("name", ["dense_ragged_bf16", "gqa_varlen_bf16", "fp16_scalar", "fp32_all"])
def test_scalar_gate_on_mma_sync_kernel(name, monkeypatch):
    """The scalar gate normally runs on the tcgen05 per-chunk kernel; the warp-MMA kernel (which serves the
    per-channel gate) computes the same gradients for it when selected."""
    monkeypatch.setenv("GDR_K4_TC", "0")
    prob = make_problem(name, seed=zlib.crc32(name.encode()) % 1000, **SMALL[name])
    compare(prob, run_gpu(prob), oracle.problem_backward(prob))


@pytest.mark.parametrize("nseg", [2, 3, 7])
@pytest.mark.parametrize("per_channel", [False, True], ids=["scalar", "kda"])
def test_factored_state_gradient_local_pass(nseg, per_channel, monkeypatch):
    """The factored local pass of the state-gradient scan (QR = Q~ - Aqk W; dS <- Gamma_C dS + D^T QR -
    (dS K~^T) W) gives the oracle's gradients like the unfactored one."""
    monkeypatch.setenv("GDR_NSEG", str(nseg))
    monkeypatch.setenv("GDR_DH_FACTORED", "1")
    prob = make_problem(f"fact_nseg{nseg}", B=1, Hk=1, Hv=2, K=64, V=64, per_channel=per_channel,
                        seq_lens=[700, 64, 130, 1], seed=90)
    compare(prob, run_gpu(prob), oracle.problem_backward(prob))


def test_factored_state_gradient_on_the_t8k_workload(monkeypatch):
    monkeypatch.setenv("GDR_DH_FACTORED", "1")
    prob = workload("gdn_t8k_bf16")
    compare(prob, run_gpu(prob), oracle.problem_backward(prob))


@pytest.mark.parametrize("offset", [0, 1], ids=["aligned16", "aligned4"])
def test_per_channel_gate_tensor_alignment(offset):
    """The per-channel gate may be only 4-byte aligned (the C ABI's rule for it): the WY preparation then
    copies its rows 4 bytes at a time instead of 16.  Either way the gradients match the oracle."""
    from chunked_gated_delta_09_gb300 import ops
    prob = make_problem("kda_gate_align", B=1, T=200, Hk=1, Hv=2, K=64, V=64, per_channel=True, seed=31)
    plan = ops.plan_for(prob)
    dev = ops.problem_to_device(prob, "cuda")
    g = dev["g"]
    store = torch.empty(g.numel() + 4, dtype=g.dtype, device="cuda")
    shifted = store[offset:offset + g.numel()].view_as(g)
    shifted.copy_(g)
    assert (shifted.data_ptr() % 16 == 0) == (offset == 0)
    dev["g"] = shifted
    out = plan.alloc_outputs("cuda")
    ws = plan.alloc_workspace("cuda")
    plan.run(out=out, workspace=ws, **dev)
    assert plan.get_status(ws) == 0
    torch.cuda.synchronize()
    got = {k: v.float().cpu().to(torch.float64).numpy() for k, v in out.items()}
    compare(prob, got, oracle.problem_backward(prob))
