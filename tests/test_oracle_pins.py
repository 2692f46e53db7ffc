"""Pins for the fp64 oracle, independent of the oracle itself.

Each test checks the oracle against something the mathematics fixes: central finite differences of
the token forward, exact symbolic derivatives (sympy), hand-derived closed forms, the beta = 0 and
g = beta = 0 special cases, the orthonormal-key reduction to causal linear attention (computed with
plain matmuls), linearity in the cotangents, the GQA and varlen decompositions, and an independent
chunkwise WY forward.  A planted-mistake test shows that each of eight plausible slips in the
backward fails the finite-difference pin.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import oracle.wy_forward as wy
from oracle.chunk_index import enumerate_chunks
from chunked_gated_delta_09_gb300.inputs import make_problem

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
NAMES = dict(q="dq", k="dk", v="dv", beta="dbeta", g="dg", h0="dh0")


def _args(p, a):
    return (a["cu"], p.Hk, p.Hv, p.K, p.V, p.per_channel, p.scale, a["q"], a["k"], a["v"], a["beta"],
            a["g"], a["h0"], a["dO"], a["dht"])


def _fd_grads(p, a, eps=1e-6):
    """Central finite differences of L = <o, dO> + <S_T, dht> for every input element."""
    out = {}
    for nm in NAMES:
        x = a[nm]
        if x is None:
            continue
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            b = dict(a)
            xp = x.copy()
            xp[idx] += eps
            b[nm] = xp
            lp = oracle.loss(*_args(p, b))
            xm = x.copy()
            xm[idx] -= eps
            b[nm] = xm
            lm = oracle.loss(*_args(p, b))
            fd[idx] = (lp - lm) / (2 * eps)
        out[NAMES[nm]] = fd
    return out


def _rel(a, b):
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


FD_CASES = [
    dict(B=1, T=9, Hk=1, Hv=1, K=4, V=4),
    dict(B=2, T=6, Hk=1, Hv=2, K=4, V=4),                 # batch + GQA
    dict(B=1, Hk=2, Hv=2, K=4, V=4, seq_lens=[5, 9]),      # varlen pair
    dict(B=1, T=1, Hk=1, Hv=1, K=4, V=4),                 # a single token
    dict(B=1, T=16, Hk=1, Hv=1, K=4, V=3, has_h0=False, has_dht=False),
]


@pytest.mark.parametrize("per_channel", [False, True], ids=["scalar", "kda"])
@pytest.mark.parametrize("case", range(len(FD_CASES)))
def test_backward_matches_finite_differences(case, per_channel):
    p = make_problem(per_channel=per_channel, qkv_dtype=torch.float64, seed=100 + case,
                     **FD_CASES[case])
    a = p.packed_f64()
    got = oracle.backward(*_args(p, a))
    fd = _fd_grads(p, a)
    for key, ref in fd.items():
        assert _rel(got[key], ref) < 1e-6, (key, _rel(got[key], ref))
    if a["h0"] is None:
        # h0 absent = zero: dh0 is still the gradient at h0 = 0
        b = dict(a)
        b["h0"] = np.zeros((p.N, p.Hv, p.V, p.K))
        fd0 = _fd_grads(p, b)["dh0"]
        assert _rel(got["dh0"], fd0) < 1e-6


@pytest.mark.parametrize("mutation", range(1, 9))
def test_planted_mistakes_fail_the_finite_difference_pin(mutation):
    per_channel = mutation == 8
    p = make_problem(B=1, T=7, Hk=1, Hv=1, K=4, V=4, per_channel=per_channel,
                     qkv_dtype=torch.float64, seed=7)
    a = p.packed_f64()
    fd = _fd_grads(p, a)
    good = oracle.backward(*_args(p, a))
    bad = oracle.backward(*_args(p, a), mutation=mutation)
    assert max(_rel(good[key], fd[key]) for key in fd) < 1e-6
    assert max(_rel(bad[key], fd[key]) for key in fd) > 1e-3


@pytest.mark.parametrize("per_channel", [False, True], ids=["scalar", "kda"])
def test_backward_matches_symbolic_derivatives(per_channel):
    """Exact derivatives of the unrolled recurrence by sympy, T = 3, K = V = 2."""
    sp = pytest.importorskip("sympy")
    T, K, V = 3, 2, 2
    rng = np.random.default_rng(5)
    vals = dict(q=rng.normal(size=(T, K)), k=rng.normal(size=(T, K)) * 0.5, v=rng.normal(size=(T, V)),
                beta=rng.uniform(0.1, 0.9, size=T),
                g=rng.uniform(-1, 0, size=(T, K) if per_channel else T),
                h0=rng.normal(size=(V, K)) * 0.3, dO=rng.normal(size=(T, V)), dht=rng.normal(size=(V, K)))
    scale = 0.7
    sym = {}

    def mk(name, shape):
        arr = np.empty(shape, dtype=object)
        for idx in np.ndindex(shape):
            arr[idx] = sp.Symbol(f"{name}_{'_'.join(map(str, idx))}")
        sym[name] = arr
        return arr

    q, k, v = mk("q", (T, K)), mk("k", (T, K)), mk("v", (T, V))
    beta = mk("beta", (T,))
    g = mk("g", (T, K) if per_channel else (T,))
    h0 = mk("h0", (V, K))
    S = sp.Matrix(h0.tolist())
    Lexpr = 0
    for t in range(T):
        kt = sp.Matrix(k[t].tolist())
        if per_channel:
            Sp = S * sp.diag(*[sp.exp(g[t, c]) for c in range(K)])
        else:
            Sp = sp.exp(g[t]) * S
        S = Sp + beta[t] * (sp.Matrix(v[t].tolist()) - Sp * kt) * kt.T
        o = scale * S * sp.Matrix(q[t].tolist())
        Lexpr += sum(o[i] * vals["dO"][t, i] for i in range(V))
    Lexpr += sum(S[i, c] * vals["dht"][i, c] for i in range(V) for c in range(K))
    subs = {}
    for name, arr in sym.items():
        for idx in np.ndindex(arr.shape):
            subs[arr[idx]] = sp.Float(float(vals[name][idx]), 30)
    cu = np.array([0, T])
    got = oracle.backward(cu, 1, 1, K, V, per_channel, scale, vals["q"][:, None], vals["k"][:, None],
                          vals["v"][:, None], vals["beta"][:, None],
                          vals["g"][:, None], vals["h0"][None, None], vals["dO"][:, None],
                          vals["dht"][None, None])
    gmap = dict(q=got["dq"][:, 0], k=got["dk"][:, 0], v=got["dv"][:, 0], beta=got["dbeta"][:, 0],
                g=got["dg"][:, 0], h0=got["dh0"][0, 0])
    for name, arr in sym.items():
        for idx in np.ndindex(arr.shape):
            exact = float(sp.diff(Lexpr, arr[idx]).evalf(30, subs=subs))
            assert abs(gmap[name][idx] - exact) <= 1e-12 * max(1.0, abs(exact)), (name, idx)


def test_single_token_closed_form():
    """T = 1, K = V = 1 worked by hand: S1 = e^g s0 (1 - b k^2) + b v k, o = scale S1 q."""
    q, k, v, b, g, s0, dO, dht, scale = 0.8, -0.6, 1.3, 0.4, -0.25, 0.5, -0.9, 0.3, 0.5
    e = np.exp(g)
    S1 = e * s0 * (1 - b * k * k) + b * v * k
    a = scale * q * dO + dht                      # dL/dS1
    want = dict(dq=scale * S1 * dO, dv=a * b * k, dbeta=a * k * (v - e * s0 * k),
                dk=a * b * (v - 2 * e * s0 * k), dg=a * e * s0 * (1 - b * k * k),
                dh0=a * e * (1 - b * k * k))
    arr = lambda x: np.array(x, dtype=np.float64).reshape(1, 1, 1)
    got = oracle.backward(np.array([0, 1]), 1, 1, 1, 1, False, scale, arr(q), arr(k), arr(v),
                          np.array([[b]]), np.array([[g]]), arr(s0).reshape(1, 1, 1, 1), arr(dO),
                          arr(dht).reshape(1, 1, 1, 1))
    for key, val in want.items():
        assert abs(float(got[key].ravel()[0]) - val) < 1e-14, key


@pytest.mark.parametrize("per_channel", [False, True], ids=["scalar", "kda"])
@pytest.mark.parametrize("BT", [1, 4, 16, 64])
def test_chunkwise_wy_forward_matches_token_forward(BT, per_channel):
    p = make_problem(B=1, Hk=1, Hv=2, K=8, V=6, per_channel=per_channel, qkv_dtype=torch.float64,
                     seq_lens=[37, 64, 5, 70], seed=11)
    a = p.packed_f64()
    args = (a["cu"], p.Hk, p.Hv, p.K, p.V, per_channel, p.scale, a["q"], a["k"], a["v"], a["beta"],
            a["g"], a["h0"])
    o1, hT1, st1 = oracle.forward(*args, BTs=BT)
    o2, hT2, st2 = wy.forward(*args, BT)
    assert np.abs(o1 - o2).max() < 1e-10
    assert np.abs(hT1 - hT2).max() < 1e-10
    assert np.abs(st1 - st2).max() < 1e-10


@pytest.mark.parametrize("per_channel", [False, True], ids=["scalar", "kda"])
def test_beta_zero_state_only_decays(per_channel):
    p = make_problem(B=1, T=20, Hk=1, Hv=1, K=4, V=5, per_channel=per_channel, qkv_dtype=torch.float64,
                     beta_zero=True, seed=3)
    a = p.packed_f64()
    _, hT, states = oracle.forward(a["cu"], 1, 1, p.K, p.V, per_channel, p.scale, a["q"], a["k"], a["v"],
                                   a["beta"], a["g"], a["h0"], BTs=1)
    h0 = a["h0"][0, 0]
    for t in range(1, 20):
        if per_channel:
            want = states[t - 1, 0] * np.exp(a["g"][t - 1, 0])[None, :]
        else:
            want = states[t - 1, 0] * np.exp(a["g"][t - 1, 0])
        assert np.allclose(states[t, 0], want, rtol=1e-13, atol=1e-15)
    gsum = a["g"][:, 0].sum(0)
    want_T = h0 * (np.exp(gsum)[None, :] if per_channel else np.exp(gsum))
    assert np.allclose(hT[0, 0], want_T, rtol=1e-12, atol=1e-15)


def test_gate_zero_beta_zero_closed_forms():
    """g = 0, beta = 0: S_t = S_0 for every t, so the gradients have the closed forms below."""
    T, K, V = 12, 4, 5
    p = make_problem(B=1, T=T, Hk=1, Hv=1, K=K, V=V, qkv_dtype=torch.float64, beta_zero=True,
                     gate_zero=True, seed=9)
    a = p.packed_f64()
    got = oracle.backward(*_args(p, a))
    S0 = a["h0"][0, 0]
    q, k, v, dO = a["q"][:, 0], a["k"][:, 0], a["v"][:, 0], a["dO"][:, 0]
    dht = a["dht"][0, 0]
    s = p.scale
    assert np.allclose(got["dq"][:, 0], s * dO @ S0, atol=1e-14)
    assert np.allclose(got["dh0"][0, 0], dht + s * dO.T @ q, atol=1e-13)
    assert np.abs(got["dk"]).max() == 0.0 and np.abs(got["dv"]).max() == 0.0
    for t in range(T):
        dSt = dht + s * dO[t:].T @ q[t:]          # adjoint of S_t, including o_t
        assert np.isclose(got["dbeta"][t, 0], (v[t] - S0 @ k[t]) @ (dSt @ k[t]), atol=1e-13)
        assert np.isclose(got["dg"][t, 0], np.sum(dSt * S0), atol=1e-13)


def test_orthonormal_keys_reduce_to_causal_linear_attention():
    """g = 0, beta = 1, h0 = 0 and orthonormal keys: S_t = sum_{j<=t} v_j k_j^T exactly, so o, dq and
    dv are those of causal linear attention, computed here with plain matmuls."""
    T, K, V = 8, 8, 6
    rng = np.random.default_rng(2)
    Qm, _ = np.linalg.qr(rng.normal(size=(K, K)))
    k = Qm[:T]
    q, v, dO = rng.normal(size=(T, K)), rng.normal(size=(T, V)), rng.normal(size=(T, V))
    scale = 0.3
    cu = np.array([0, T])
    ones, zeros = np.ones((T, 1)), np.zeros((T, 1))
    o, _, _ = oracle.forward(cu, 1, 1, K, V, False, scale, q[:, None], k[:, None], v[:, None], ones, zeros)
    got = oracle.backward(cu, 1, 1, K, V, False, scale, q[:, None], k[:, None], v[:, None], ones, zeros,
                          None, dO[:, None], None)
    causal = np.tril(np.ones((T, T)))
    P = (q @ k.T) * causal
    assert np.allclose(o[:, 0], scale * P @ v, atol=1e-12)
    assert np.allclose(got["dq"][:, 0], scale * ((dO @ v.T) * causal) @ k, atol=1e-12)
    assert np.allclose(got["dv"][:, 0], scale * P.T @ dO, atol=1e-12)


@pytest.mark.parametrize("per_channel", [False, True], ids=["scalar", "kda"])
def test_gradients_are_linear_in_the_cotangents(per_channel):
    p1 = make_problem(B=1, T=30, Hk=1, Hv=2, K=6, V=5, per_channel=per_channel, qkv_dtype=torch.float64,
                      seed=21)
    p2 = make_problem(B=1, T=30, Hk=1, Hv=2, K=6, V=5, per_channel=per_channel, qkv_dtype=torch.float64,
                      seed=22)
    a1, a2 = p1.packed_f64(), p2.packed_f64()
    a2 = dict(a1, dO=a2["dO"], dht=a2["dht"])
    a12 = dict(a1, dO=a1["dO"] + a2["dO"], dht=a1["dht"] + a2["dht"])
    g1, g2, g12 = (oracle.backward(*_args(p1, x)) for x in (a1, a2, a12))
    for key in ("dq", "dk", "dv", "dbeta", "dg", "dh0"):
        assert np.allclose(g12[key], g1[key] + g2[key], rtol=1e-10, atol=1e-12), key


def test_gqa_sums_over_the_value_heads_of_a_key_head():
    p = make_problem(B=1, T=25, Hk=1, Hv=3, K=4, V=4, qkv_dtype=torch.float64, seed=31)
    a = p.packed_f64()
    full = oracle.backward(*_args(p, a))
    dq = np.zeros_like(full["dq"])
    dk = np.zeros_like(full["dk"])
    for hv in range(3):
        sl = slice(hv, hv + 1)
        one = oracle.backward(a["cu"], 1, 1, 4, 4, False, p.scale, a["q"], a["k"], a["v"][:, sl],
                              a["beta"][:, sl], a["g"][:, sl], a["h0"][:, sl], a["dO"][:, sl],
                              a["dht"][:, sl])
        dq += one["dq"]
        dk += one["dk"]
        for key in ("dv", "dbeta", "dg", "dh0"):
            ref = full[key][:, sl] if key != "dh0" else full[key][:, sl]
            assert np.allclose(one[key], ref, rtol=1e-12, atol=1e-14)
    assert np.allclose(full["dq"], dq, rtol=1e-12, atol=1e-14)
    assert np.allclose(full["dk"], dk, rtol=1e-12, atol=1e-14)


def test_varlen_equals_separate_sequences():
    lens = [7, 13, 1]
    p = make_problem(B=1, Hk=1, Hv=2, K=4, V=4, qkv_dtype=torch.float64, seq_lens=lens, seed=41)
    a = p.packed_f64()
    full = oracle.backward(*_args(p, a))
    for s, (b0, b1) in enumerate(zip(a["cu"][:-1], a["cu"][1:])):
        sl = slice(int(b0), int(b1))
        one = oracle.backward(np.array([0, b1 - b0]), 1, 2, 4, 4, False, p.scale, a["q"][sl], a["k"][sl],
                              a["v"][sl], a["beta"][sl], a["g"][sl], a["h0"][s:s + 1], a["dO"][sl],
                              a["dht"][s:s + 1])
        for key in ("dq", "dk", "dv", "dbeta", "dg"):
            assert np.allclose(one[key], full[key][sl], rtol=1e-12, atol=1e-14), key
        assert np.allclose(one["dh0"][0], full["dh0"][s], rtol=1e-12, atol=1e-14)


def test_chunk_index_enumeration_matches_golden():
    with open(os.path.join(GOLDEN, "chunk_indices.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        idx, off = enumerate_chunks(c["cu_seqlens"], c["BT"])
        assert [list(x) for x in idx] == c["chunk_indices"]
        assert off == c["chunk_offsets"]


# ---------------------------------------------------------------- the WY-gradient stage taken alone (row f4)
def _wy_inputs(seed, C, K, V):
    rng = np.random.default_rng(seed)
    q, k = rng.standard_normal((C, K)), rng.standard_normal((C, K))
    v, v_new, do, dv = (rng.standard_normal((C, V)) for _ in range(4))
    g = np.cumsum(-np.log1p(np.exp(-rng.standard_normal((C, K)))), axis=0)  # cumulative logsigmoid
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(C)))
    A_kk = np.tril(0.3 * rng.standard_normal((C, C)), -1)
    h, dh = rng.standard_normal((K, V)), rng.standard_normal((K, V))
    return dict(q=q, k=k, v=v, v_new=v_new, g=g, beta=beta, A_kk=A_kk, h=h, do=do, dh=dh, dv=dv)


@pytest.mark.parametrize("C,K,V", [(5, 3, 4), (1, 2, 2), (4, 4, 3)])
def test_wy_stage_gradients_match_finite_differences(C, K, V):
    """Every output of the WY-stage oracle (dq, dk, dv, db, dg, and dA through A = (I + A_kk)^-1) is the
    central finite difference of its defining scalar, element by element."""
    from oracle import wy_stage
    x = _wy_inputs(11 + C, C, K, V)
    scale = 0.7

    def loss(d):
        A = np.linalg.inv(np.eye(C) + d["A_kk"])
        return wy_stage.chunk_loss(d["q"], d["k"], d["v"], d["v_new"], d["g"], d["beta"], A, d["h"], d["do"],
                                   d["dh"], d["dv"], scale)

    A = np.linalg.inv(np.eye(C) + x["A_kk"])
    got = wy_stage.chunk_grads(x["q"], x["k"], x["v"], x["v_new"], x["g"], x["beta"], A, x["h"], x["do"],
                               x["dh"], x["dv"], scale)
    eps = 1e-6
    for name, key in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("beta", "db"), ("g", "dg"), ("A_kk", "dA")):
        fd = np.zeros_like(x[name])
        for idx in np.ndindex(*x[name].shape):
            if name == "A_kk" and idx[1] >= idx[0]:
                continue  # A_kk is strictly lower
            xp = {kk: vv.copy() for kk, vv in x.items()}
            xm = {kk: vv.copy() for kk, vv in x.items()}
            xp[name][idx] += eps
            xm[name][idx] -= eps
            fd[idx] = (loss(xp) - loss(xm)) / (2 * eps)
        err = np.abs(got[key] - fd).max() / max(1.0, np.abs(fd).max())
        assert err < 1e-6, (key, err)


def test_wy_stage_pieces_against_the_full_gradient_terms():
    """Cross-check with the full oracle's chunk algebra: when h, dh, v_new and dv are the true chunk
    quantities of a one-chunk problem whose state starts at h, the stage's dv equals beta A^T dV_new, and the
    stage's dq plus the intra-chunk term P K (P = (D V_new^T) (.) M) equals the token-recurrence oracle's dq."""
    import oracle
    from oracle import wy_forward, wy_stage
    rng = np.random.default_rng(5)
    C, K, V, scale = 6, 3, 3, 0.5
    q = rng.standard_normal((C, K)); k = rng.standard_normal((C, K)); v = rng.standard_normal((C, V))
    gr = -np.log1p(np.exp(-rng.standard_normal((C, K))))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(C)))
    S0 = 0.3 * rng.standard_normal((V, K)); dO = rng.standard_normal((C, V)); dht = rng.standard_normal((V, K))
    cu = np.array([0, C])
    f = lambda a: a[:, None, :]
    full = oracle.backward(cu, 1, 1, K, V, True, scale, f(q), f(k), f(v), beta[:, None], f(gr), S0[None, None],
                           f(dO), dht[None, None])
    _, _, parts = wy_forward.chunk_forward(S0, q, k, v, beta, gr, scale, True)
    g = parts["gamma"]
    A = parts["T"]
    v_new = parts["V_new"]
    # dV_new and the state gradient of the one-chunk problem: dS_next = dht, dV_new = P^T-side terms
    Mq = np.einsum("ic,jc,ijc->ij", q, k, np.exp(g[:, None, :] - g[None, :, :])) * np.tril(np.ones((C, C)))
    D = scale * dO
    dv_new = Mq.T @ D + (k * np.exp(g[-1][None, :] - g)) @ dht.T
    st = wy_stage.chunk_grads(q, k, v, v_new, g, beta, A, S0.T, dO, dht.T, dv_new, scale)
    # dq of the full problem = stage's inter-chunk dq + intra-chunk (P K with per-channel decay)
    P = (D @ v_new.T) * np.tril(np.ones((C, C)))
    dq_intra = np.einsum("ij,jc,ijc->ic", P, k, np.exp(g[:, None, :] - g[None, :, :]))
    np.testing.assert_allclose(st["dq"] + dq_intra, full["dq"][:, 0], rtol=1e-9, atol=1e-10)
    np.testing.assert_allclose(st["dv"], beta[:, None] * (A.T @ dv_new), rtol=1e-12, atol=1e-12)


def test_wy_stage_packed_driver_assembles_the_chunks():
    """The packed, varlen driver of the WY stage (wy_stage.wy_stage) equals per-chunk calls of chunk_grads
    placed by hand: two sequences of 23 and 37 tokens with BT = 16 give the chunks [0, 16), [16, 23) of the
    first and [23, 39), [39, 55), [55, 60) of the second, numbered 0..4 for h and dh; the rows of dA beyond a
    chunk's length stay zero."""
    from oracle import wy_stage
    rng = np.random.default_rng(31)
    H, K, V, BT, scale = 2, 4, 3, 16, 0.6
    Tt = 60
    cu = np.array([0, 23, 60])
    q, k = rng.standard_normal((Tt, H, K)), rng.standard_normal((Tt, H, K))
    v, v_new, do, dv = (rng.standard_normal((Tt, H, V)) for _ in range(4))
    g = -np.abs(rng.standard_normal((Tt, H, K)))
    beta = rng.random((Tt, H))
    A = rng.standard_normal((Tt, H, BT))
    h, dh = rng.standard_normal((5, H, K, V)), rng.standard_normal((5, H, K, V))
    got = wy_stage.wy_stage(cu, H, K, V, BT, scale, q, k, v, v_new, g, beta, A, h, do, dh, dv)
    chunks = [(0, 16, 0), (16, 23, 1), (23, 39, 2), (39, 55, 3), (55, 60, 4)]
    want = {key: np.zeros_like(val) for key, val in got.items()}
    for c0, c1, n in chunks:
        C = c1 - c0
        for hh in range(H):
            r = wy_stage.chunk_grads(q[c0:c1, hh], k[c0:c1, hh], v[c0:c1, hh], v_new[c0:c1, hh], g[c0:c1, hh],
                                     beta[c0:c1, hh], A[c0:c1, hh, :C], h[n, hh], do[c0:c1, hh], dh[n, hh],
                                     dv[c0:c1, hh], scale)
            for key in ("dq", "dk", "dv", "db", "dg"):
                want[key][c0:c1, hh] = r[key]
            want["dA"][c0:c1, hh, :C] = r["dA"]
    for key in want:
        np.testing.assert_array_equal(got[key], want[key], err_msg=key)
    # a chunk's dA columns beyond its length are zero (the 7-token and 5-token chunks)
    assert not got["dA"][16:23, :, 7:].any() and not got["dA"][55:60, :, 5:].any()
