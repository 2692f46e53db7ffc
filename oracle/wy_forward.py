"""Independent fp64 chunkwise (WY-form) forward of the gated delta rule.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  It exists to pin the token-recurrence oracle:
both must give the same outputs o and final states, although they share no code and compute in a
different order.  It follows the chunk quantities named on the pages: the chunk-local cumulative gate
("FlashQLA backward explained", section 1, entry convention on g), the strictly-lower beta-weighted,
gate-decayed K K^T whose inverse is the chunk's triangular matrix A [B, T, H, BT] (MindSpeed-Ops
chunk_kda_bwd.md, input table and "implementation principle"), and the per-chunk state h
[B, NT, H, K, V] that the forward saves.

Per chunk with entry state S0 (V x K), chunk-local cumulative gate gamma_r = sum_{i<=r} g_i and
Gamma_r = exp(gamma_r):
    A_kk[i, j] = beta_i exp(gamma_i - gamma_j) (k_i . k_j)          for j < i, else 0
    T          = (I + A_kk)^{-1}                      (numpy.linalg.inv, a library primitive)
    W          = T diag(beta Gamma) K,   U = T diag(beta) V
    V_new      = U - W S0^T
    O          = scale [diag(Gamma) Q S0^T + (M (.) Q K^T) V_new],   M[r, j] = exp(gamma_r - gamma_j) [j <= r]
    S_C        = Gamma_C S0 + V_new^T diag(exp(gamma_C - gamma)) K
Per-channel gate: every exp(gamma_a - gamma_b) factor becomes the K-vector exp(gamma_a[c] - gamma_b[c])
applied inside the K-contraction, and Gamma_C S0 becomes S0 diag(Gamma_C).
"""
from __future__ import annotations

import numpy as np


def chunk_forward(S0, q, k, v, beta, g, scale, per_channel):
    """One chunk.  q, k [C, K]; v [C, V]; beta [C]; g [C] or [C, K]; S0 [V, K].

    Returns (o [C, V], S_C [V, K], parts) where parts holds gamma, T, W, U, V_new.
    """
    C = q.shape[0]
    gam = np.cumsum(g, axis=0)  # [C] or [C, K]
    if per_channel:
        # D[i, j, c] = exp(gamma_i[c] - gamma_j[c])
        D = np.exp(gam[:, None, :] - gam[None, :, :])
        KK = np.einsum("ic,jc,ijc->ij", k, k, D)
        QK = np.einsum("ic,jc,ijc->ij", q, k, D)
        Kg = k * np.exp(gam)                       # K (.) Gamma
        Qg = q * np.exp(gam)
        Kc = k * np.exp(gam[-1][None, :] - gam)    # K (.) exp(gamma_C - gamma)
    else:
        D = np.exp(gam[:, None] - gam[None, :])
        KK = (k @ k.T) * D
        QK = (q @ k.T) * D
        Kg = k * np.exp(gam)[:, None]
        Qg = q * np.exp(gam)[:, None]
        Kc = k * np.exp(gam[-1] - gam)[:, None]
    strict = np.tril(np.ones((C, C)), -1)
    causal = np.tril(np.ones((C, C)), 0)
    A_kk = beta[:, None] * KK * strict
    T = np.linalg.inv(np.eye(C) + A_kk)
    W = T @ (beta[:, None] * Kg)
    U = T @ (beta[:, None] * v)
    V_new = U - W @ S0.T
    o = scale * (Qg @ S0.T + (QK * causal) @ V_new)
    if per_channel:
        S_C = S0 * np.exp(gam[-1])[None, :] + V_new.T @ Kc
    else:
        S_C = np.exp(gam[-1]) * S0 + V_new.T @ Kc
    return o, S_C, dict(gamma=gam, T=T, W=W, U=U, V_new=V_new)


def forward(cu, Hk, Hv, K, V, per_channel, scale, q, k, v, beta, g, h0, BT):
    """Chunkwise forward on packed inputs (same shapes as ``oracle.forward``).

    Returns (o [T, Hv, V], hT [N, Hv, V, K], states [NC, Hv, V, K]) with states the state entering each
    chunk, chunks enumerated sequence-major then chunk ascending.
    """
    cu = np.asarray(cu, dtype=np.int64)
    N = len(cu) - 1
    G = Hv // Hk
    Ttot = int(cu[-1]) if N > 0 else 0
    o = np.zeros((Ttot, Hv, V))
    hT = np.zeros((N, Hv, V, K))
    nc = sum((int(cu[s + 1] - cu[s]) + BT - 1) // BT for s in range(N))
    states = np.zeros((nc, Hv, V, K))
    ci = 0
    for s in range(N):
        bos, eos = int(cu[s]), int(cu[s + 1])
        nchunks = (eos - bos + BT - 1) // BT
        for hv in range(Hv):
            hk = hv // G
            S = np.zeros((V, K)) if h0 is None else np.array(h0[s, hv], dtype=np.float64)
            for c in range(nchunks):
                a, b = bos + c * BT, min(bos + (c + 1) * BT, eos)
                states[ci + c, hv] = S
                oc, S, _ = chunk_forward(S, q[a:b, hk], k[a:b, hk], v[a:b, hv], beta[a:b, hv],
                                         g[a:b, hv], scale, per_channel)
                o[a:b, hv] = oc
            hT[s, hv] = S
        ci += nchunks
    return o, hT, states
