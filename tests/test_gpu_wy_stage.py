"""Parity of the WY-gradient stage taken alone (gdr_wy_bwd_run through the C ABI) with its fp64 oracle
(oracle/wy_stage.py), on inputs drawn like the usage example of the operation it follows (randn tensors,
logsigmoid gates, sigmoid beta) except that g is a chunk-local cumulative gate and A a true
(I + A_kk)^-1 per chunk.  Bars: relative L2 <= 5e-3 for the fp32 outputs (dq, dk, db, dg, dA) and for dv
in fp32, <= 2e-2 for dv in fp16 / bf16."""
import numpy as np
import pytest
import torch

from chunked_gated_delta_09_gb300 import ops
from oracle import wy_stage
from parity_util import rel_l2

pytestmark = pytest.mark.gpu


def make_wy_inputs(B, T, H, K, V, BT, dtype, seq_lens=None, seed=0):
    gen = torch.Generator().manual_seed(seed)
    if seq_lens is not None:
        assert B == 1
        T = sum(seq_lens)
        cu = np.concatenate([[0], np.cumsum(seq_lens)]).astype(np.int64)
    else:
        cu = np.arange(B + 1, dtype=np.int64) * T
    rn = lambda *s: torch.randn(*s, generator=gen)
    q, k = rn(B, T, H, K), rn(B, T, H, K)
    v, v_new, do, dv = rn(B, T, H, V), rn(B, T, H, V), rn(B, T, H, V), rn(B, T, H, V)
    beta = torch.sigmoid(rn(B, T, H))
    graw = torch.nn.functional.logsigmoid(rn(B, T, H, K)).reshape(B * T, H, K)
    g = torch.empty_like(graw)
    A = torch.zeros(B * T, H, BT)
    chunks = []
    for s in range(len(cu) - 1):
        for c0 in range(int(cu[s]), int(cu[s + 1]), BT):
            c1 = min(c0 + BT, int(cu[s + 1]))
            chunks.append((c0, c1))
            g[c0:c1] = torch.cumsum(graw[c0:c1], dim=0)
            C = c1 - c0
            Akk = torch.tril(0.2 * rn(H, C, C), -1)
            A[c0:c1, :, :C] = torch.linalg.inv(torch.eye(C) + Akk).permute(1, 0, 2)
    NT = len(chunks)
    h, dh = rn(NT, H, K, V), rn(NT, H, K, V)
    t = dict(q=q, k=k, v=v, v_new=v_new, do=do, dv=dv, beta=beta, A=A.reshape(B, T, H, BT))
    t = {n: x.to(dtype) for n, x in t.items()}
    t.update(g=g.reshape(B, T, H, K), h=h.reshape(B if seq_lens is None else 1, -1, H, K, V), dh=dh.reshape(B if seq_lens is None else 1, -1, H, K, V))
    return t, cu


@pytest.mark.parametrize("case", [
    dict(B=2, T=150, H=2, K=64, V=64, BT=64, dtype=torch.float16),
    dict(B=1, T=200, H=2, K=128, V=128, BT=64, dtype=torch.float32),
    dict(B=1, T=0, H=2, K=64, V=32, BT=16, dtype=torch.float16, seq_lens=[70, 5, 130]),
    dict(B=1, T=300, H=1, K=32, V=64, BT=16, dtype=torch.bfloat16),
    dict(B=1, T=2048, H=32, K=128, V=128, BT=64, dtype=torch.float16),  # the operation's model shape
    # feature sizes that leave lanes of a warp without a column, ragged chunks of 1 and 33 tokens
    dict(B=1, T=0, H=3, K=40, V=24, BT=32, dtype=torch.bfloat16, seq_lens=[33, 64, 1, 95]),
], ids=["dense_fp16", "fp32", "varlen_bt16_fp16", "bt16_bf16", "model_shape_fp16", "varlen_bt32_k40_v24_bf16"])
def test_wy_stage_matches_oracle(case):
    case = dict(case)
    dtype, seq_lens = case.pop("dtype"), case.pop("seq_lens", None)
    t, cu = make_wy_inputs(dtype=dtype, seq_lens=seq_lens, seed=23, **case)
    B, H, K, V, BT = case["B"], case["H"], case["K"], case["V"], case["BT"]
    T = t["q"].shape[1]
    scale = K ** -0.5
    dev = {n: x.cuda().contiguous() for n, x in t.items()}
    cu_dev = None if seq_lens is None else torch.tensor(cu, dtype=torch.int32, device="cuda")
    got = ops.gdr_wy_bwd(dev["q"], dev["k"], dev["v"], dev["v_new"], dev["g"], dev["beta"], dev["A"], dev["h"],
                         dev["do"], dev["dh"], dev["dv"], scale=scale, cu_seqlens=cu_dev, chunk_size=BT,
                         check_status=True)
    torch.cuda.synchronize()
    f = lambda x, *tail: x.to(torch.float64).reshape(-1, *tail).numpy()
    ref = wy_stage.wy_stage(cu, H, K, V, BT, scale, f(t["q"], H, K), f(t["k"], H, K), f(t["v"], H, V),
                            f(t["v_new"], H, V), f(t["g"], H, K), f(t["beta"], H), f(t["A"], H, BT),
                            f(t["h"], H, K, V), f(t["do"], H, V), f(t["dh"], H, K, V), f(t["dv"], H, V))
    names = ("dq", "dk", "dv", "db", "dg", "dA")
    res = {}
    for name, x in zip(names, got):
        g_ = x.float().cpu().to(torch.float64).numpy().reshape(ref[name].shape)
        assert np.all(np.isfinite(g_)), name
        bar = 2e-2 if (name == "dv" and dtype != torch.float32) else 5e-3
        res[name] = (rel_l2(g_, ref[name]), bar)
    bad = {n: v for n, v in res.items() if not v[0] <= v[1]}
    assert not bad, f"outside tolerance {bad} (all {res})"
