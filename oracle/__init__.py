"""fp64 CPU oracle for the chunked gated delta rule backward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA product path never calls it, and the two share no code:
the only module both sides use is the seeded input generator, which holds none of the method's
arithmetic.

Contents
  gdr_oracle.c    token-by-token fp64 forward and hand-derived reverse-mode adjoints (C, OpenMP)
  wy_forward.py   an independent fp64 chunkwise (WY-form) forward, used to pin the token forward
  chunk_index.py  plain enumeration of varlen chunk indices
  __init__.py     builds gdr_oracle.c with gcc and wraps it with ctypes (this file)

Parity status: every function here is pinned by ``tests/test_oracle_*.py`` (finite differences,
symbolic gradients, closed forms, invariants, planted mistakes).  The chunk-state export of
``forward(..., BTs=...)`` is pinned by the chunkwise forward.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdr_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libgdr_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile gdr_oracle.c into a shared library with gcc (plain -O2, OpenMP)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            i64p = ctypes.POINTER(ctypes.c_int64)
            ci, cd = ctypes.c_int, ctypes.c_double
            lib.gdr_oracle_fwd.argtypes = [ci, i64p, ci, ci, ci, ci, ci, cd,
                                           dp, dp, dp, dp, dp, dp, dp, dp, ci, dp, ci]
            lib.gdr_oracle_fwd.restype = ci
            lib.gdr_oracle_bwd.argtypes = [ci, i64p, ci, ci, ci, ci, ci, cd,
                                           dp, dp, dp, dp, dp, dp, dp, dp,
                                           dp, dp, dp, dp, dp, dp, ci, ci]
            lib.gdr_oracle_bwd.restype = ci
            lib.gdr_oracle_max_threads.restype = ci
            _lib = lib
    return _lib


def _ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    assert a.dtype == np.float64 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def max_threads() -> int:
    return int(_load().gdr_oracle_max_threads())


def forward(cu, Hk, Hv, K, V, per_channel, scale, q, k, v, beta, g, h0=None, BTs=0, nthreads=0):
    """Token-recurrence forward on packed inputs.

    cu: int64 [N+1] token offsets.  q, k [T, Hk, K]; v [T, Hv, V]; beta [T, Hv];
    g [T, Hv] or [T, Hv, K]; h0 [N, Hv, V, K] or None.
    Returns (o [T, Hv, V], hT [N, Hv, V, K], states [NC, Hv, V, K] or None), where states holds the
    state entering every chunk of BTs tokens (sequence-major, chunk ascending) when BTs > 0.
    """
    lib = _load()
    cu = np.ascontiguousarray(np.asarray(cu, dtype=np.int64))
    N = len(cu) - 1
    T = int(cu[-1]) if N > 0 else 0
    q, k, v, beta, g, h0 = map(_f64, (q, k, v, beta, g, h0))
    o = np.zeros((T, Hv, V))
    hT = np.zeros((N, Hv, V, K))
    states = None
    if BTs > 0:
        nc = int(sum((int(cu[s + 1] - cu[s]) + BTs - 1) // BTs for s in range(N)))
        states = np.zeros((nc, Hv, V, K))
    rc = lib.gdr_oracle_fwd(N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), Hk, Hv, K, V,
                            int(per_channel), float(scale), _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                            _ptr(g), _ptr(h0), _ptr(o), _ptr(hT), int(BTs), _ptr(states), int(nthreads))
    if rc != 0:
        raise ValueError(f"gdr_oracle_fwd rejected its arguments (rc={rc})")
    return o, hT, states


def backward(cu, Hk, Hv, K, V, per_channel, scale, q, k, v, beta, g, h0, dO, dht,
             mutation=0, nthreads=0):
    """Exact fp64 gradients of L = <o, dO> + <S_T, dht> with respect to q, k, v, beta, raw g, h0.

    Shapes as in :func:`forward`; dO [T, Hv, V]; dht [N, Hv, V, K] or None.
    Returns a dict with dq, dk [T, Hk, K]; dv [T, Hv, V]; dbeta [T, Hv]; dg [T, Hv(, K)];
    dh0 [N, Hv, V, K].  ``mutation`` > 0 plants a known mistake (tests only).
    """
    lib = _load()
    cu = np.ascontiguousarray(np.asarray(cu, dtype=np.int64))
    N = len(cu) - 1
    T = int(cu[-1]) if N > 0 else 0
    q, k, v, beta, g, h0, dO, dht = map(_f64, (q, k, v, beta, g, h0, dO, dht))
    out = dict(dq=np.zeros((T, Hk, K)), dk=np.zeros((T, Hk, K)), dv=np.zeros((T, Hv, V)),
               dbeta=np.zeros((T, Hv)),
               dg=np.zeros((T, Hv, K)) if per_channel else np.zeros((T, Hv)),
               dh0=np.zeros((N, Hv, V, K)))
    rc = lib.gdr_oracle_bwd(N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), Hk, Hv, K, V,
                            int(per_channel), float(scale), _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                            _ptr(g), _ptr(h0), _ptr(dO), _ptr(dht), _ptr(out["dq"]), _ptr(out["dk"]),
                            _ptr(out["dv"]), _ptr(out["dbeta"]), _ptr(out["dg"]), _ptr(out["dh0"]),
                            int(mutation), int(nthreads))
    if rc != 0:
        raise ValueError(f"gdr_oracle_bwd rejected its arguments (rc={rc})")
    return out


def loss(cu, Hk, Hv, K, V, per_channel, scale, q, k, v, beta, g, h0, dO, dht):
    """L = sum <o, dO> + sum <S_T, dht> from the token forward (fp64)."""
    o, hT, _ = forward(cu, Hk, Hv, K, V, per_channel, scale, q, k, v, beta, g, h0)
    L = float(np.sum(o * np.asarray(dO, dtype=np.float64)))
    if dht is not None:
        L += float(np.sum(hT * np.asarray(dht, dtype=np.float64)))
    return L


def problem_backward(prob, mutation=0, nthreads=0):
    """Oracle gradients for a :class:`chunked_gated_delta_09_gb300.inputs.Problem` (CPU tensors).

    Upcasts the stored (already rounded) inputs to fp64, runs :func:`backward` on the packed layout and
    returns arrays in the problem's own shapes ([B, T, ...] for dense problems).
    """
    a = prob.packed_f64()
    out = backward(a["cu"], prob.Hk, prob.Hv, prob.K, prob.V, prob.per_channel, prob.scale,
                   a["q"], a["k"], a["v"], a["beta"], a["g"], a["h0"], a["dO"], a["dht"],
                   mutation=mutation, nthreads=nthreads)
    return prob.unpack(out)
