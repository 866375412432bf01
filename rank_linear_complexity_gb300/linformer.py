"""Python binding of the C ABI in include/linformer_attn.h (argument marshalling only).

Every function here converts its arguments to pointers and integers and calls
the CUDA library of the same name; all computation runs in the library's
kernels.  Importing this module does not load the library; the first call does,
and raises if the library has not been built (there is no other implementation
to fall back to).
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

PER_HEAD, KV, HEADWISE, LAYERWISE = 0, 1, 2, 3
F32, BF16, BF16_F32OUT = 0, 1, 2
PATH_SIMT, PATH_TENSOR = 0, 1
KERNEL_COUNT = 7

_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i = ctypes.c_int

SYMBOLS = [
    "linformer_attn_fwd", "linformer_project_fwd", "linformer_attn_fwd_host",
    "linformer_select_path", "linformer_status_string", "linformer_debug_read_device_status",
    "linformer_set_pv_terms", "linformer_launch_count", "linformer_profile_enable",
    "linformer_profile_collect", "linformer_kernel_name", "linformer_attn_fwd_noalloc",
    "linformer_window_projection", "linformer_attn_bwd", "linformer_dense_attn_fwd",
    "linformer_pool_peak_bytes", "linformer_debug_wait_probe",
]


class LinformerError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: status {status} ({status_string(status)})")


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """The loaded CUDA library (raises if it was never built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(
                    f"CUDA library not built ({path} missing): run "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(path)
            fwd_args = [_vp] * 5 + [_vp, _vp] + [_i] * 7 + [_vp]
            L.linformer_attn_fwd.argtypes = fwd_args
            L.linformer_attn_fwd.restype = _i
            L.linformer_attn_fwd_host.argtypes = fwd_args
            L.linformer_attn_fwd_host.restype = _i
            L.linformer_attn_fwd_noalloc.argtypes = fwd_args
            L.linformer_attn_fwd_noalloc.restype = _i
            L.linformer_project_fwd.argtypes = [_vp] * 5 + [_vp, _vp] + [_i] * 7 + [_vp]
            L.linformer_project_fwd.restype = _i
            L.linformer_select_path.argtypes = [_i] * 7
            L.linformer_select_path.restype = _i
            L.linformer_status_string.argtypes = [_i]
            L.linformer_status_string.restype = ctypes.c_char_p
            L.linformer_debug_read_device_status.argtypes = [_vp]
            L.linformer_debug_read_device_status.restype = _i
            L.linformer_set_pv_terms.argtypes = [_i]
            L.linformer_set_pv_terms.restype = _i
            L.linformer_launch_count.argtypes = []
            L.linformer_launch_count.restype = ctypes.c_int64
            L.linformer_profile_enable.argtypes = [_i]
            L.linformer_profile_enable.restype = _i
            L.linformer_profile_collect.argtypes = [ctypes.POINTER(ctypes.c_double),
                                                    ctypes.POINTER(ctypes.c_int64)]
            L.linformer_profile_collect.restype = _i
            L.linformer_dense_attn_fwd.argtypes = [_vp] * 5 + [_i] * 5 + [_vp]
            L.linformer_dense_attn_fwd.restype = _i
            L.linformer_debug_wait_probe.argtypes = [_vp]
            L.linformer_debug_wait_probe.restype = _i
            L.linformer_pool_peak_bytes.argtypes = [_i]
            L.linformer_pool_peak_bytes.restype = ctypes.c_int64
            L.linformer_attn_bwd.argtypes = [_vp] * 12 + [_i] * 7 + [_vp]
            L.linformer_attn_bwd.restype = _i
            L.linformer_window_projection.argtypes = [_vp, _vp, _i, _i, _i, _vp]
            L.linformer_window_projection.restype = _i
            L.linformer_kernel_name.argtypes = [_i]
            L.linformer_kernel_name.restype = ctypes.c_char_p
            _lib = L
    return _lib


def _ptr(x):
    """Device/host address of a tensor (or an int address, or None -> NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream_handle(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def linformer_attn_fwd(Q, K, V, E, F, pad_lengths, O, b, h, n, d, k, share_mode, dtype,
                       stream=None) -> int:
    return lib().linformer_attn_fwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(E), _ptr(F),
                                    _ptr(pad_lengths), _ptr(O), b, h, n, d, k, share_mode,
                                    dtype, _stream_handle(stream))


def linformer_project_fwd(K, V, E, F, pad_lengths, Kbar, Vbar, b, h, n, d, k, share_mode,
                          dtype, stream=None) -> int:
    return lib().linformer_project_fwd(_ptr(K), _ptr(V), _ptr(E), _ptr(F), _ptr(pad_lengths),
                                       _ptr(Kbar), _ptr(Vbar), b, h, n, d, k, share_mode,
                                       dtype, _stream_handle(stream))


def linformer_attn_fwd_host(Q, K, V, E, F, pad_lengths, O, b, h, n, d, k, share_mode, dtype,
                            stream=None) -> int:
    return lib().linformer_attn_fwd_host(_ptr(Q), _ptr(K), _ptr(V), _ptr(E), _ptr(F),
                                         _ptr(pad_lengths), _ptr(O), b, h, n, d, k,
                                         share_mode, dtype, _stream_handle(stream))


def linformer_attn_fwd_noalloc(Q, K, V, E, F, pad_lengths, O, b, h, n, d, k, share_mode,
                               dtype, stream=None) -> int:
    """Same as linformer_attn_fwd, with the library's fixed device workspace (no allocation)."""
    return lib().linformer_attn_fwd_noalloc(_ptr(Q), _ptr(K), _ptr(V), _ptr(E), _ptr(F),
                                            _ptr(pad_lengths), _ptr(O), b, h, n, d, k,
                                            share_mode, dtype, _stream_handle(stream))


def linformer_select_path(b, h, n, d, k, share_mode, dtype) -> int:
    return lib().linformer_select_path(b, h, n, d, k, share_mode, dtype)


def status_string(status: int) -> str:
    try:
        return lib().linformer_status_string(status).decode()
    except Exception:  # library unavailable: still give a message
        return "unknown"


def linformer_debug_read_device_status(stream=None) -> int:
    return lib().linformer_debug_read_device_status(_stream_handle(stream))


def linformer_debug_wait_probe(stream=None) -> int:
    return lib().linformer_debug_wait_probe(_stream_handle(stream))


def linformer_set_pv_terms(terms: int) -> int:
    return lib().linformer_set_pv_terms(terms)


def linformer_launch_count() -> int:
    return lib().linformer_launch_count()


def linformer_profile_enable(enable: bool) -> int:
    return lib().linformer_profile_enable(1 if enable else 0)


def linformer_profile_collect():
    """Returns {kernel name: (total ms, launches)} for kernels that ran."""
    ms = (ctypes.c_double * KERNEL_COUNT)()
    cnt = (ctypes.c_int64 * KERNEL_COUNT)()
    st = lib().linformer_profile_collect(ms, cnt)
    if st != 0:
        raise LinformerError(st, "linformer_profile_collect")
    out = {}
    for i in range(KERNEL_COUNT):
        if cnt[i]:
            out[lib().linformer_kernel_name(i).decode()] = (ms[i], cnt[i])
    return out


# --- tensor-level conveniences (still marshalling only) ------------------------------

def _dims(Q, E, share_mode):
    b, h, n, d = Q.shape
    k = E.shape[-2]
    return b, h, n, d, k


def dtype_code(t, out_fp32: bool = False) -> int:
    import torch
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16_F32OUT if out_fp32 else BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def attention(Q, K, V, E, F=None, lengths=None, share_mode: int = PER_HEAD,
              out_fp32: bool = False, out=None, stream=None):
    """O = Linformer attention of device tensors Q, K, V [b][h][n][d] (allocates O)."""
    import torch
    b, h, n, d, k = _dims(Q, E, share_mode)
    code = dtype_code(Q, out_fp32)
    if out is None:
        odt = torch.bfloat16 if code == BF16 else torch.float32
        out = torch.empty((b, h, n, d), dtype=odt, device=Q.device)
    st = linformer_attn_fwd(Q, K, V, E, F, lengths, out, b, h, n, d, k, share_mode, code,
                            stream)
    if st != 0:
        raise LinformerError(st, "linformer_attn_fwd")
    return out


def projection(K, V, E, F=None, lengths=None, share_mode: int = PER_HEAD, stream=None):
    """(Kbar, Vbar) fp32 [b][h][k][d] of device tensors K, V."""
    import torch
    b, h, n, d = K.shape
    k = E.shape[-2]
    Kb = torch.empty((b, h, k, d), dtype=torch.float32, device=K.device)
    Vb = torch.empty_like(Kb)
    st = linformer_project_fwd(K, V, E, F, lengths, Kb, Vb, b, h, n, d, k, share_mode,
                               dtype_code(K), stream)
    if st != 0:
        raise LinformerError(st, "linformer_project_fwd")
    return Kb, Vb


def linformer_window_projection(P, weights, n, k, dtype, stream=None) -> int:
    return lib().linformer_window_projection(_ptr(P), _ptr(weights), n, k, dtype,
                                             _stream_handle(stream))


def window_projection(n: int, k: int, weights=None, dtype=None, device="cuda", stream=None):
    """[k][n] device tensor: mean pooling (weights None) or a convolution with kernel =
    stride = n / k (weights: float32 device tensor of n / k values), to pass as E (and F)."""
    import torch
    dt = torch.bfloat16 if dtype is None else dtype
    P = torch.empty((k, n), dtype=dt, device=device)
    code = F32 if dt == torch.float32 else BF16
    st = linformer_window_projection(P, weights, n, k, code, stream)
    if st != 0:
        raise LinformerError(st, "linformer_window_projection")
    return P


def linformer_attn_bwd(Q, K, V, E, F, pad_lengths, dO, dQ, dK, dV, dE, dF, b, h, n, d, k,
                       share_mode, dtype, stream=None) -> int:
    return lib().linformer_attn_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(E), _ptr(F),
                                    _ptr(pad_lengths), _ptr(dO), _ptr(dQ), _ptr(dK), _ptr(dV),
                                    _ptr(dE), _ptr(dF), b, h, n, d, k, share_mode, dtype,
                                    _stream_handle(stream))


def attention_backward(Q, K, V, E, F, lengths, dO, share_mode: int = PER_HEAD, stream=None):
    """(dQ, dK, dV, dE, dF) of device fp32 tensors; dF is None when F is E (KV, LAYERWISE)."""
    import torch
    b, h, n, d, k = _dims(Q, E, share_mode)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    dE = torch.empty_like(E)
    distinct = share_mode in (PER_HEAD, HEADWISE)
    dF = torch.empty_like(F if F is not None else E) if distinct else None
    st = linformer_attn_bwd(Q, K, V, E, F, lengths, dO, dQ, dK, dV, dE, dF, b, h, n, d, k,
                            share_mode, dtype_code(Q), stream)
    if st != 0:
        raise LinformerError(st, "linformer_attn_bwd")
    return dQ, dK, dV, dE, dF


def linformer_dense_attn_fwd(Q, K, V, pad_lengths, O, b, h, n, d, dtype, stream=None) -> int:
    return lib().linformer_dense_attn_fwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(pad_lengths), _ptr(O),
                                          b, h, n, d, dtype, _stream_handle(stream))


def linformer_pool_peak_bytes(reset: bool = False) -> int:
    return lib().linformer_pool_peak_bytes(1 if reset else 0)


def dense_attention(Q, K, V, lengths=None, out=None, stream=None):
    """O = softmax(Q K^T / sqrt(d)) V of device fp32 tensors [b][h][n][d] (allocates O)."""
    import torch
    b, h, n, d = Q.shape
    if out is None:
        out = torch.empty((b, h, n, d), dtype=torch.float32, device=Q.device)
    st = linformer_dense_attn_fwd(Q, K, V, lengths, out, b, h, n, d, dtype_code(Q), stream)
    if st != 0:
        raise LinformerError(st, "linformer_dense_attn_fwd")
    return out
