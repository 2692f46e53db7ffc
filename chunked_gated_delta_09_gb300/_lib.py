"""ctypes view of include/gdr_bwd.h (libgdrbwd.so).  Argument marshalling only."""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libgdrbwd.so")

GDR_OK, GDR_ERR_INVALID_ARG, GDR_ERR_UNSUPPORTED, GDR_ERR_CUDA, GDR_ERR_OOM, GDR_ERR_TIMEOUT, GDR_ERR_DEVICE = range(7)
GDR_F32, GDR_BF16, GDR_F16 = 0, 1, 2

# every function the header declares
EXPORTS = ("gdr_bwd_create", "gdr_bwd_workspace_bytes", "gdr_bwd_run", "gdr_bwd_run_profiled",
           "gdr_bwd_launch_count", "gdr_bwd_get_status", "gdr_bwd_run_noalloc", "gdr_bwd_get_status_noalloc",
           "gdr_bwd_destroy",
           "gdr_chunk_indices", "gdr_status_string", "gdr_fwd_run", "gdr_fwd_launch_count", "gdr_wy_bwd_run")
NOALLOC_MAX_WORKSPACE = 64 << 20
NUM_STAGES = 6
STAGE_NAMES = ("k0_chunk_indices", "k1_wy_prep", "k2_fused_gdr_h", "k3_dh_scan", "k4_intra_grad", "k5_dg_reduce")


class GdrBwdDesc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("Hk", ctypes.c_int), ("Hv", ctypes.c_int),
                ("K", ctypes.c_int), ("V", ctypes.c_int), ("BT", ctypes.c_int), ("num_seqs", ctypes.c_int),
                ("gate_per_channel", ctypes.c_int), ("scale", ctypes.c_float),
                ("qkv_dtype", ctypes.c_int), ("beta_dtype", ctypes.c_int), ("dqdk_dtype", ctypes.c_int),
                ("dv_dtype", ctypes.c_int), ("has_h0", ctypes.c_int), ("has_dht", ctypes.c_int)]


class GdrBwdArgs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("q", "k", "v", "beta", "g", "h0", "dO", "dht", "cu_seqlens",
                                                "dq", "dk", "dv", "dbeta", "dg", "dh0")]


class GdrFwdArgs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("q", "k", "v", "beta", "g", "h0", "cu_seqlens", "o", "ht")]


class GdrWyArgs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("q", "k", "v", "v_new", "beta", "A", "dO", "dv", "g", "h", "dh",
                                                "cu_seqlens", "dq", "dk", "dv_out", "db", "dg", "dA")]


class GdrError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Load libgdrbwd.so.  Raises if it has not been built: there is no fallback path."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it with chunked_gated_delta_09_gb300.build.build()")
        lib = ctypes.CDLL(p)
        vp, sz, ci = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        lib.gdr_bwd_create.argtypes = [ctypes.POINTER(GdrBwdDesc), ctypes.POINTER(vp)]
        lib.gdr_bwd_create.restype = ci
        lib.gdr_bwd_workspace_bytes.argtypes = [vp]
        lib.gdr_bwd_workspace_bytes.restype = sz
        lib.gdr_bwd_run.argtypes = [vp, ctypes.POINTER(GdrBwdArgs), vp, sz, vp]
        lib.gdr_bwd_run.restype = ci
        lib.gdr_bwd_run_profiled.argtypes = [vp, ctypes.POINTER(GdrBwdArgs), vp, sz, vp, ctypes.POINTER(vp)]
        lib.gdr_bwd_run_profiled.restype = ci
        lib.gdr_bwd_launch_count.argtypes = [vp]
        lib.gdr_bwd_launch_count.restype = ci
        lib.gdr_bwd_run_noalloc.argtypes = [vp, ctypes.POINTER(GdrBwdArgs), vp]
        lib.gdr_bwd_run_noalloc.restype = ci
        lib.gdr_bwd_get_status.argtypes = [vp, vp, vp]
        lib.gdr_bwd_get_status.restype = ci
        lib.gdr_bwd_get_status_noalloc.argtypes = [vp, vp]
        lib.gdr_bwd_get_status_noalloc.restype = ci
        lib.gdr_bwd_destroy.argtypes = [vp]
        lib.gdr_bwd_destroy.restype = None
        lib.gdr_chunk_indices.argtypes = [vp, ci, ci, ci, vp, vp, vp]
        lib.gdr_chunk_indices.restype = ci
        lib.gdr_fwd_run.argtypes = [vp, ctypes.POINTER(GdrFwdArgs), vp, sz, vp]
        lib.gdr_fwd_run.restype = ci
        lib.gdr_fwd_launch_count.argtypes = [vp]
        lib.gdr_fwd_launch_count.restype = ci
        lib.gdr_wy_bwd_run.argtypes = [vp, ctypes.POINTER(GdrWyArgs), vp, sz, vp]
        lib.gdr_wy_bwd_run.restype = ci
        lib.gdr_status_string.argtypes = [ci]
        lib.gdr_status_string.restype = ctypes.c_char_p
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().gdr_status_string(int(status)).decode()
