"""fp64 definition of the WY-gradient stage taken alone (row f4 of the build): the operation that
MindSpeed-Ops chunk_kda_bwd.md documents as chunk_kda_bwd_wy_dqkg_fused (signature, input / output tables,
"implementation principle": dq = do @ h^T, dk = v_new @ dh^T, dw = -(dv @ h^T), then the corrections through
g, beta and A, and dA = -A (dA_pre A) in its post-processing).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``); nothing here is used by the product.

Readings of the page (it states the tensors, not every convention):
  * g [.., K] is the chunk-local cumulative log gate (the form the KDA backward passes along; "FlashQLA
    backward explained", section 1 states the same for the scalar gate), so gate factors are
    exp(g_i - g_j) within a chunk and dg is the gradient with respect to that cumulative gate.
  * A [.., BT] is the chunk's triangular matrix T = (I + A_kk)^-1 (row = token, column = chunk position);
    the WY factors are W = A diag(beta) (K (.) exp(g)) and U = A diag(beta) V.
  * h [.., K, V] is the state entering the chunk, dh [.., K, V] the gradient of the state leaving it, v_new
    the chunk's V_new = U - W h, dv (input) the gradient of V_new, do the output gradient.
  * The operation returns the gradients that flow through the chunk's state terms and its WY factors, with
    h, dh, v_new, dv and do held fixed: the terms through Q K^T (the intra-chunk attention) and through
    A_kk (via dA) are left to the later stages, which receive dA.
  * dA is the gradient with respect to A_kk (strictly lower, zero elsewhere): -T^T dT T^T with dT the
    gradient with respect to T = A; the page's -A (dA_pre A) is this product in its own transposition.

With E = exp(g) and Ec = exp(g_C - g) (g_C the chunk's last valid row), per chunk and head the stage is the
gradient of the scalar
    L = scale <(Q (.) E) h, dO>                (inter-chunk output)
      + <K (.) Ec, V_new dh^T>                 (the chunk's contribution to the state it leaves)
      + <W, -dV h^T> + <U, dV>                 (V_new = U - W h)
      + sum_k exp(g_C[k]) sum_v h[k, v] dh[k, v]   (the decay of the entering state)
with respect to q, k, v, beta, g and A_kk (through A = (I + A_kk)^-1).
"""
from __future__ import annotations

import numpy as np


def chunk_loss(q, k, v, v_new, g, beta, A, h, do, dh, dv, scale):
    """The scalar L of the module docstring for one chunk (all arrays fp64, C valid rows)."""
    E = np.exp(g)
    Ec = np.exp(g[-1][None, :] - g)
    W = A @ (beta[:, None] * k * E)
    U = A @ (beta[:, None] * v)
    L = scale * np.sum(((q * E) @ h) * do)
    L += np.sum((k * Ec) * (v_new @ dh.T))
    L += np.sum(W * (-dv @ h.T)) + np.sum(U * dv)
    L += np.sum(np.exp(g[-1]) * np.sum(h * dh, axis=1))
    return L


def chunk_grads(q, k, v, v_new, g, beta, A, h, do, dh, dv, scale):
    """Gradients of :func:`chunk_loss`: dict(dq, dk, dv, db, dg, dA), dA with respect to A_kk."""
    C = q.shape[0]
    E = np.exp(g)
    Ec = np.exp(g[-1][None, :] - g)
    # inter-chunk output: L1 = scale <(Q E) h, dO>
    dq = scale * (do @ h.T) * E
    dg = q * dq
    # chunk contribution to the leaving state: L2 = <K Ec, V_new dh^T>
    dk_sc = (v_new @ dh.T) * Ec
    dk = dk_sc.copy()
    dg = dg - k * dk_sc
    dg_last = np.sum(k * dk_sc, axis=0)
    # WY factors: L3 = <W, dW>, dW = -dV h^T; L4 = <U, dV>
    dW = -dv @ h.T
    kE = k * E
    AtdW = A.T @ dW
    dk_w = beta[:, None] * AtdW * E
    dk = dk + dk_w
    dg = dg + k * dk_w
    AtdU = A.T @ dv
    dv_out = beta[:, None] * AtdU
    db = np.sum(AtdW * kE, axis=1) + np.sum(AtdU * v, axis=1)
    dT = dW @ (beta[:, None] * kE).T + dv @ (beta[:, None] * v).T
    # decay of the entering state: L5 = sum_k exp(g_C) <h, dh>_k
    dg_last = dg_last + np.exp(g[-1]) * np.sum(h * dh, axis=1)
    dg[-1] += dg_last
    # gradient with respect to A_kk, where A = (I + A_kk)^-1: -A^T dT A^T, strictly lower part
    dA = np.tril(-(A.T @ dT @ A.T), -1)
    return dict(dq=dq, dk=dk, dv=dv_out, db=db, dg=dg, dA=dA)


def wy_stage(cu, H, K, V, BT, scale, q, k, v, v_new, g, beta, A, h, do, dh, dv):
    """The stage on packed inputs: cu int [N+1]; q, k [T, H, K]; v, v_new, do, dv [T, H, V]; g [T, H, K];
    beta [T, H]; A [T, H, BT]; h, dh [NT, H, K, V] with chunks numbered sequence-major.  Returns dict of
    dq, dk [T, H, K], dv [T, H, V], db [T, H], dg [T, H, K], dA [T, H, BT] (fp64)."""
    cu = [int(x) for x in cu]
    Tt = cu[-1]
    out = dict(dq=np.zeros((Tt, H, K)), dk=np.zeros((Tt, H, K)), dv=np.zeros((Tt, H, V)),
               db=np.zeros((Tt, H)), dg=np.zeros((Tt, H, K)), dA=np.zeros((Tt, H, BT)))
    n = 0
    for s in range(len(cu) - 1):
        for c0 in range(cu[s], cu[s + 1], BT):
            c1 = min(c0 + BT, cu[s + 1])
            C = c1 - c0
            for hh in range(H):
                gr = chunk_grads(q[c0:c1, hh], k[c0:c1, hh], v[c0:c1, hh], v_new[c0:c1, hh], g[c0:c1, hh],
                                 beta[c0:c1, hh], A[c0:c1, hh, :C], h[n, hh], do[c0:c1, hh], dh[n, hh],
                                 dv[c0:c1, hh], scale)
                for key in ("dq", "dk", "dv", "db", "dg"):
                    out[key][c0:c1, hh] = gr[key]
                out["dA"][c0:c1, hh, :C] = gr["dA"]
            n += 1
    return out
