"""fp64 CPU oracle for the Linformer attention forward: ctypes wrapper.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  The CUDA library never
imports it and it never imports the CUDA library.

The arithmetic lives in ``linformer_oracle.c`` (plain loops, double precision).
This module only compiles it with gcc, converts arrays to float64 and calls it.
Every value is read exactly as stored: bf16 and fp32 inputs widen to float64
without rounding.

Definitions followed (see the C file for the full list):
  * "Linformer(Self-Attention with Linear Complexity) 요약 설명", section Model:
    Kbar = E.K, Vbar = F.V with E, F of shape k x n; output O is n x d.
  * PaperWeekly efficient-Transformer survey, section 2.1: scaled dot product.
  * "Linformer: Self-Attention with Linear Complexity - 中文验证版", section 方法适配:
    headwise, key-value and layerwise sharing.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

PER_HEAD, KV, HEADWISE, LAYERWISE = 0, 1, 2, 3

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "linformer_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liblinformer_oracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library (gcc, OpenMP, no fp contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-shared",
           "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path: str):
    """Load a compiled oracle (the real one, or a test's deliberately broken copy)."""
    lib = ctypes.CDLL(path)
    lib.oracle_project.argtypes = [ctypes.c_int] * 4 + [_dp, _dp, _dp]
    lib.oracle_project.restype = None
    lib.oracle_attend.argtypes = ([ctypes.c_int] * 4 + [_dp, _dp, _dp]
                                  + [ctypes.POINTER(ctypes.c_int64), ctypes.c_int64, _dp, _dp])
    lib.oracle_attend.restype = ctypes.c_int
    lib.oracle_linformer_fwd.argtypes = ([_dp] * 5 + [ctypes.POINTER(ctypes.c_int32)]
                                         + [_dp] * 3 + [ctypes.c_int] * 7)
    lib.oracle_linformer_fwd.restype = ctypes.c_int
    lib.oracle_full_attention.argtypes = [ctypes.c_int, ctypes.c_int, _dp, _dp, _dp, _dp]
    lib.oracle_full_attention.restype = None
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def _f64(a) -> np.ndarray:
    """Exact widening to a C-contiguous float64 array (accepts numpy or torch)."""
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor: bf16 has no numpy dtype, widen via fp32
        import torch
        t = a.detach().to("cpu")
        if t.dtype in (torch.bfloat16, torch.float16):
            t = t.to(torch.float32)
        a = t.numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray):
    return None if a is None else a.ctypes.data_as(_dp)


def project(Ehat, X, L: int | None = None, lib=None) -> np.ndarray:
    """Xbar = Ehat[:, :L] . X[:L]  (Ehat: k x n, X: n x d)."""
    E64, X64 = _f64(Ehat), _f64(X)
    k, n = E64.shape
    n2, d = X64.shape
    assert n == n2
    L = n if L is None else max(0, min(int(L), n))
    out = np.empty((k, d), np.float64)
    (lib or _load()).oracle_project(n, d, k, L, _ptr(E64), _ptr(X64), _ptr(out))
    return out


def attend(Q, Kbar, Vbar, L: int | None = None, rows=None, return_p: bool = False, lib=None):
    """Rows of softmax(Q.Kbar^T/sqrt(d)).Vbar for one unit; rows >= L are zero."""
    Q64, K64, V64 = _f64(Q), _f64(Kbar), _f64(Vbar)
    n, d = Q64.shape
    k = K64.shape[0]
    L = n if L is None else max(0, min(int(L), n))
    rows = np.arange(n, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, np.int64)
    O = np.empty((len(rows), d), np.float64)
    P = np.empty((len(rows), k), np.float64) if return_p else None
    rc = (lib or _load()).oracle_attend(n, d, k, L, _ptr(Q64), _ptr(K64), _ptr(V64),
                               rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                               len(rows), _ptr(O), _ptr(P))
    if rc != 0:
        raise ValueError(f"oracle_attend failed ({rc})")
    return (O, P) if return_p else O


def unit_projections(E, F, share_mode: int, head: int):
    """The (Ehat, Fhat) pair a unit of head `head` uses, as float64 k x n arrays."""
    E64 = _f64(E)
    if share_mode in (PER_HEAD, KV):
        Eh = E64[head]
    else:
        Eh = E64
    if share_mode in (KV, LAYERWISE):
        Fh = Eh
    else:
        F64 = _f64(F)
        Fh = F64[head] if share_mode == PER_HEAD else F64
    return Eh, Fh


def linformer_fwd(Q, K, V, E, F, pad_lengths, share_mode: int, nthreads: int = 0,
                  return_proj: bool = False, lib=None):
    """Whole problem: Q, K, V [b][h][n][d]; returns O [b][h][n][d] (float64).

    Also returns the thread count used, and Kbar / Vbar [b][h][k][d] if asked."""
    Q64, K64, V64 = _f64(Q), _f64(K), _f64(V)
    b, h, n, d = Q64.shape
    E64 = _f64(E)
    k = E64.shape[-2]
    F64 = None if (F is None or share_mode in (KV, LAYERWISE)) else _f64(F)
    if F64 is None:
        F64 = E64  # never read in KV / LAYERWISE modes
    pad = None
    if pad_lengths is not None:
        if hasattr(pad_lengths, "detach"):
            pad_lengths = pad_lengths.detach().cpu().numpy()
        pad = np.ascontiguousarray(pad_lengths, np.int32)
        assert pad.shape == (b,)
    O = np.empty_like(Q64)
    Kb = np.empty((b, h, k, d), np.float64) if return_proj else None
    Vb = np.empty((b, h, k, d), np.float64) if return_proj else None
    used = (lib or _load()).oracle_linformer_fwd(
        _ptr(Q64), _ptr(K64), _ptr(V64), _ptr(E64), _ptr(F64),
        None if pad is None else pad.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
        _ptr(O), _ptr(Kb), _ptr(Vb), b, h, n, d, k, share_mode, nthreads)
    if used < 0:
        raise ValueError(f"oracle_linformer_fwd failed ({used})")
    if return_proj:
        return O, used, Kb, Vb
    return O, used


def full_attention(Q, K, V, lib=None) -> np.ndarray:
    """softmax(Q K^T / sqrt(d)) V over all keys, for small n x d inputs."""
    Q64, K64, V64 = _f64(Q), _f64(K), _f64(V)
    n, d = Q64.shape
    O = np.empty((n, d), np.float64)
    (lib or _load()).oracle_full_attention(n, d, _ptr(Q64), _ptr(K64), _ptr(V64), _ptr(O))
    return O


def unit_rows(Q, K, V, E, F, pad_lengths, share_mode: int, batch: int, head: int, rows):
    """Sampled rows of one unit (for full-size checks the oracle computes row by row).

    Q, K, V may be torch tensors of shape [b][h][n][d] on any device; only the
    selected unit is copied to the host.  Returns (O_rows, Kbar, Vbar)."""
    q, kk, vv = Q[batch, head], K[batch, head], V[batch, head]
    n = q.shape[0]
    L = n
    if pad_lengths is not None:
        pl = pad_lengths
        if hasattr(pl, "detach"):
            pl = pl.detach().cpu().numpy()
        L = max(0, min(int(pl[batch]), n))
    Eh, Fh = unit_projections(E, F, share_mode, head)
    Kb = project(Eh, kk, L)
    Vb = project(Fh, vv, L)
    return attend(q, Kb, Vb, L, rows), Kb, Vb
