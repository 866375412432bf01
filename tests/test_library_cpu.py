"""Host-side checks of the CUDA library that need no GPU.

The library must load and export every symbol include/linformer_attn.h declares,
and argument errors must come back as status codes before anything touches the
device (no compute call is made here).
"""
import ctypes
import os
import re

import pytest

import rank_linear_complexity_gb300.linformer as lf
from rank_linear_complexity_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def L():
    libbuild.build()
    return lf.lib()


def declared_symbols():
    names = set()
    for h in HEADERS:
        src = open(h).read()
        names.update(re.findall(r"LINFORMER_API\s+[\w\s\*]*?\b(linformer_\w+)\s*\(", src))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_symbols()
    assert "linformer_attn_fwd" in names and "linformer_project_fwd" in names
    assert len(names) >= 11


def test_library_exports_every_declared_symbol(L):
    for name in declared_symbols():
        assert hasattr(L, name), f"{name} declared in include/ but not exported"
    assert set(declared_symbols()) <= set(lf.SYMBOLS) | set(declared_symbols())


def test_status_strings(L):
    for code in range(0, -10, -1):
        assert lf.status_string(code) not in ("", "unknown status")


A = 1 << 20  # a 16-byte aligned fake address: never dereferenced, every call below fails validation


@pytest.mark.parametrize("args,expected", [
    (dict(Q=None), -1),
    (dict(O=None), -1),
    (dict(b=0), -2),
    (dict(k=0), -2),
    (dict(n=-5), -2),
    (dict(d=129), -3),
    (dict(k=1025), -3),
    (dict(share_mode=4), -4),
    (dict(dtype=3), -4),
    (dict(Q=A + 8), -5),
    (dict(E=A + 2), -5),
    (dict(F=None, share_mode=0), -6),
    (dict(F=None, share_mode=2), -6),
    (dict(F=A + 4096, share_mode=1), -6),
    (dict(F=A + 4096, share_mode=3), -6),
])
def test_argument_errors_are_reported_before_launch(L, args, expected):
    a = dict(Q=A, K=A, V=A, E=A, F=A + 4096, pad=None, O=A, b=2, h=3, n=64, d=64, k=32,
             share_mode=0, dtype=1)
    a.update(args)
    st = lf.linformer_attn_fwd(a["Q"], a["K"], a["V"], a["E"], a["F"], a["pad"], a["O"],
                               a["b"], a["h"], a["n"], a["d"], a["k"], a["share_mode"],
                               a["dtype"], stream=0)
    assert st == expected, lf.status_string(st)


def test_project_argument_errors(L):
    st = lf.linformer_project_fwd(A, A, A, None, None, A, A, 1, 1, 8, 64, 8, 0, 1, stream=0)
    assert st == -6
    st = lf.linformer_project_fwd(A, A, A, None, None, None, A, 1, 1, 8, 64, 8, 3, 1, stream=0)
    assert st == -1


def test_path_selection(L):
    # fp32 always runs on the SIMT kernels; invalid arguments give a status.
    assert lf.linformer_select_path(2, 4, 512, 64, 128, 0, 0) == lf.PATH_SIMT
    assert lf.linformer_select_path(1, 1, 512, 100, 128, 0, 1) == lf.PATH_SIMT
    assert lf.linformer_select_path(0, 1, 512, 64, 128, 0, 1) == -2
    assert lf.linformer_select_path(1, 1, 512, 64, 128, 9, 1) == -4


def test_pv_terms_setting(L):
    prev = lf.linformer_set_pv_terms(3)
    assert lf.linformer_set_pv_terms(prev) == 3
    assert lf.linformer_set_pv_terms(2) == prev
    assert lf.linformer_set_pv_terms(prev) == 2
    assert lf.linformer_set_pv_terms(4) == -4


@pytest.mark.parametrize("args,expected", [
    (dict(dO=None), -1),
    (dict(dE=None), -1),
    (dict(dF=None, share_mode=0), -1),          # PER_HEAD has a distinct F: dF required
    (dict(share_mode=1), -6),                   # KV: F is E, so dF must be NULL
    (dict(dtype=1), -3),                        # fp32 only
    (dict(d=129), -3),
    (dict(b=300, h=300), -2),                   # more than 65535 units
    (dict(dQ=A + 8), -5),
    (dict(share_mode=7), -4),
])
def test_backward_argument_errors_are_reported_before_launch(L, args, expected):
    a = dict(Q=A, K=A, V=A, E=A, F=A + 4096, pad=None, dO=A, dQ=A, dK=A, dV=A, dE=A,
             dF=A + 4096, b=2, h=3, n=64, d=64, k=32, share_mode=0, dtype=0)
    a.update(args)
    st = lf.linformer_attn_bwd(a["Q"], a["K"], a["V"], a["E"], a["F"], a["pad"], a["dO"],
                               a["dQ"], a["dK"], a["dV"], a["dE"], a["dF"], a["b"], a["h"],
                               a["n"], a["d"], a["k"], a["share_mode"], a["dtype"], stream=0)
    assert st == expected, lf.status_string(st)


@pytest.mark.parametrize("args,expected", [
    (dict(O=None), -1),
    (dict(V=None), -1),
    (dict(dtype=1), -3),                        # fp32 only
    (dict(d=129), -3),
    (dict(n=0), -2),
    (dict(b=300, h=300), -2),                   # more than 65535 units
    (dict(K=A + 4), -5),
    (dict(pad=A + 2), -5),
    (dict(dtype=9), -4),
])
def test_dense_argument_errors_are_reported_before_launch(L, args, expected):
    a = dict(Q=A, K=A, V=A, pad=None, O=A, b=2, h=3, n=64, d=64, dtype=0)
    a.update(args)
    st = lf.linformer_dense_attn_fwd(a["Q"], a["K"], a["V"], a["pad"], a["O"], a["b"], a["h"],
                                     a["n"], a["d"], a["dtype"], stream=0)
    assert st == expected, lf.status_string(st)
