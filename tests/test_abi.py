"""The C ABI library builds, loads and exports every symbol include/gdr_bwd.h declares, and its host-side
argument checks reject bad input before anything reaches a GPU.  No compute call is made here."""
import ctypes
import os
import re

import pytest

from chunked_gated_delta_09_gb300 import _lib
from chunked_gated_delta_09_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdr_bwd.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdr_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert names == sorted(_lib.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def _desc(**kw):
    base = dict(B=1, T=256, Hk=2, Hv=4, K=128, V=128, BT=64, num_seqs=0, gate_per_channel=0, scale=0.0,
                qkv_dtype=_lib.GDR_BF16, beta_dtype=_lib.GDR_F32, dqdk_dtype=_lib.GDR_BF16,
                dv_dtype=_lib.GDR_BF16, has_h0=1, has_dht=1)
    base.update(kw)
    return _lib.GdrBwdDesc(**base)


def _create(lib, d):
    h = ctypes.c_void_p()
    st = lib.gdr_bwd_create(ctypes.byref(d), ctypes.byref(h))
    return st, h


BAD = [dict(B=0), dict(T=-1), dict(Hk=0), dict(Hv=3, Hk=2), dict(K=0), dict(K=130), dict(K=12), dict(V=256),
       dict(BT=48), dict(BT=128), dict(num_seqs=-1), dict(num_seqs=2, B=2), dict(gate_per_channel=2),
       dict(qkv_dtype=7), dict(beta_dtype=-1), dict(has_h0=3)]


@pytest.mark.parametrize("bad", BAD, ids=[str(b) for b in BAD])
def test_create_rejects_bad_descriptors(lib, bad):
    st, h = _create(lib, _desc(**bad))
    assert st == _lib.GDR_ERR_INVALID_ARG
    assert not h.value


def test_create_accepts_supported_descriptors_and_sizes_workspace(lib):
    for kw in (dict(), dict(K=32, V=32, BT=16), dict(num_seqs=3, T=1000), dict(gate_per_channel=1),
               dict(T=0), dict(qkv_dtype=_lib.GDR_F32, dqdk_dtype=_lib.GDR_F32, dv_dtype=_lib.GDR_F32)):
        st, h = _create(lib, _desc(**kw))
        assert st == _lib.GDR_OK, kw
        ws = lib.gdr_bwd_workspace_bytes(h)
        assert ws > 0 and ws % 256 == 0
        lib.gdr_bwd_destroy(h)
    assert lib.gdr_bwd_workspace_bytes(None) == 0
    lib.gdr_bwd_destroy(None)


def test_create_rejects_null_pointers(lib):
    h = ctypes.c_void_p()
    assert lib.gdr_bwd_create(None, ctypes.byref(h)) == _lib.GDR_ERR_INVALID_ARG
    d = _desc()
    assert lib.gdr_bwd_create(ctypes.byref(d), None) == _lib.GDR_ERR_INVALID_ARG


def test_run_rejects_bad_arguments_on_the_host(lib):
    st, h = _create(lib, _desc())
    assert st == _lib.GDR_OK
    ws_bytes = lib.gdr_bwd_workspace_bytes(h)
    good = 0x10000
    names = [f[0] for f in _lib.GdrBwdArgs._fields_]

    def args(**over):
        a = {n: good for n in names}
        a["cu_seqlens"] = None
        a.update(over)
        return _lib.GdrBwdArgs(**a)

    def run(a, ws=good, nbytes=ws_bytes):
        return lib.gdr_bwd_run(h, ctypes.byref(a), ws, nbytes, None)

    assert lib.gdr_bwd_run(None, ctypes.byref(args()), good, ws_bytes, None) == _lib.GDR_ERR_INVALID_ARG
    assert lib.gdr_bwd_run(h, None, good, ws_bytes, None) == _lib.GDR_ERR_INVALID_ARG
    for n in ("q", "k", "v", "beta", "g", "dO", "dq", "dk", "dv", "dbeta", "dg", "h0", "dht"):
        assert run(args(**{n: None})) == _lib.GDR_ERR_INVALID_ARG, n
    for n in ("q", "k", "v", "dO", "dq", "dk", "dv"):
        assert run(args(**{n: good + 8})) == _lib.GDR_ERR_INVALID_ARG, n
    for n in ("beta", "g", "dbeta", "dg", "h0", "dht", "dh0"):
        assert run(args(**{n: good + 2})) == _lib.GDR_ERR_INVALID_ARG, n
    assert run(args(), ws=None) == _lib.GDR_ERR_INVALID_ARG
    assert run(args(), ws=good + 16) == _lib.GDR_ERR_INVALID_ARG
    assert run(args(), nbytes=ws_bytes - 1) == _lib.GDR_ERR_INVALID_ARG
    lib.gdr_bwd_destroy(h)
    # varlen without cu_seqlens
    st, h = _create(lib, _desc(num_seqs=2))
    assert run.__call__ and lib.gdr_bwd_run(h, ctypes.byref(args()), good, lib.gdr_bwd_workspace_bytes(h),
                                             None) == _lib.GDR_ERR_INVALID_ARG
    lib.gdr_bwd_destroy(h)


def test_chunk_indices_rejects_bad_arguments(lib):
    p = 0x10000
    assert lib.gdr_chunk_indices(None, 2, 64, 4, p, p, None) == _lib.GDR_ERR_INVALID_ARG
    assert lib.gdr_chunk_indices(p, 0, 64, 4, p, p, None) == _lib.GDR_ERR_INVALID_ARG
    assert lib.gdr_chunk_indices(p, 2, 0, 4, p, p, None) == _lib.GDR_ERR_INVALID_ARG
    assert lib.gdr_chunk_indices(p, 2, 64, -1, p, p, None) == _lib.GDR_ERR_INVALID_ARG
    assert lib.gdr_chunk_indices(p, 2, 64, 4, None, p, None) == _lib.GDR_ERR_INVALID_ARG


def test_status_strings(lib):
    for s in range(7):
        assert lib.gdr_status_string(s)
    assert lib.gdr_status_string(99) == b"unknown status"
