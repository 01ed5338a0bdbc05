"""fp64 CPU oracle for the attention backward pass (wraps attention_bwd_ref.c).

TEST INFRASTRUCTURE ONLY: imported by tests/ alone.  Shares no code with the
CUDA library.  Inputs are [B, H, N, d] arrays of float64 or of uint16 bf16
bits (all of one kind); outputs are float64.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import compile_oracle

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention_bwd_ref.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle_attn_bwd.so")
_lock = threading.Lock()
_lib = None


def build() -> str:
    if (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        compile_oracle(_SRC, _LIB_PATH)
    return _LIB_PATH


def _declare(lib):
    i64, vp, ci = ctypes.c_longlong, ctypes.c_void_p, ctypes.c_int
    lib.oracle_attention_bwd.argtypes = [vp, vp, vp, vp, ci, vp, vp, vp, i64, i64, i64, i64, i64, ctypes.c_double,
                                         ci, ci]
    lib.oracle_attention_bwd.restype = ci
    lib.oracle_attention_bwd_dq_rows.argtypes = [vp, vp, vp, vp, ci, vp, i64, vp, i64, i64, i64, i64, i64,
                                                 ctypes.c_double, ci, ci]
    lib.oracle_attention_bwd_dq_rows.restype = ci
    lib.oracle_attention_bwd_dkdv_keys.argtypes = [vp, vp, vp, vp, ci, i64, vp, i64, vp, vp, i64, i64, i64, i64,
                                                   i64, ctypes.c_double, ci, ci]
    lib.oracle_attention_bwd_dkdv_keys.restype = ci
    lib.oracle_attention_bwd_window.argtypes = [vp, vp, vp, vp, ci, vp, vp, vp, i64, i64, i64, i64, i64,
                                                ctypes.c_double, i64, i64, ci]
    lib.oracle_attention_bwd_window.restype = ci
    lib.oracle_attention_bwd_dq_rows_window.argtypes = [vp, vp, vp, vp, ci, vp, i64, vp, i64, i64, i64, i64, i64,
                                                        ctypes.c_double, i64, i64, ci]
    lib.oracle_attention_bwd_dq_rows_window.restype = ci
    lib.oracle_attention_bwd_dkdv_keys_window.argtypes = [vp, vp, vp, vp, ci, i64, vp, i64, vp, vp, i64, i64, i64,
                                                          i64, i64, ctypes.c_double, i64, i64, ci]
    lib.oracle_attention_bwd_dkdv_keys_window.restype = ci
    return lib


def load_library(path: str | None = None):
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
        return _lib


def _prep(arrs):
    out, kinds = [], set()
    for a in arrs:
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            kinds.add(1)
        elif a.dtype == np.float64:
            kinds.add(0)
        else:
            raise TypeError(f"expected float64 or uint16 bf16 bits, got {a.dtype}")
        out.append(a)
    if len(kinds) != 1:
        raise TypeError("q, k, v, dout must share one element kind")
    return out, kinds.pop()


def attention_bwd(q, k, v, dout, scale, causal=False, nthreads=0, lib=None, window=None):
    """(dq [B,H,Nq,d], dk [B,H,Nk,d], dv [B,H,Nk,d]) in float64.

    window=(wl, wr): key j kept for row i iff i + s - wl <= j <= i + s + wr,
    s = Nk - Nq (aligned bottom-right), a negative bound leaving that side
    open; causal is then ignored."""
    lib = lib or load_library()
    (q, k, v, dout), kind = _prep([q, k, v, dout])
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    dq = np.zeros(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    if window is not None:
        rc = lib.oracle_attention_bwd_window(q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data, kind,
                                             dq.ctypes.data, dk.ctypes.data, dv.ctypes.data, B, H, Nq, Nk, d,
                                             float(scale), int(window[0]), int(window[1]), int(nthreads))
    else:
        rc = lib.oracle_attention_bwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data, kind,
                                      dq.ctypes.data, dk.ctypes.data, dv.ctypes.data, B, H, Nq, Nk, d,
                                      float(scale), int(bool(causal)), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_attention_bwd failed ({rc})")
    return dq, dk, dv


def attention_bwd_dq_rows(q, k, v, dout, rows, scale, causal=False, nthreads=0, lib=None, window=None):
    """dQ of selected flat query rows (b*H + h)*Nq + i: [len(rows), d]; window as in attention_bwd."""
    lib = lib or load_library()
    (q, k, v, dout), kind = _prep([q, k, v, dout])
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.zeros((rows.size, d))
    if window is not None:
        rc = lib.oracle_attention_bwd_dq_rows_window(q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data,
                                                     kind, rows.ctypes.data, rows.size, out.ctypes.data, B, H, Nq,
                                                     Nk, d, float(scale), int(window[0]), int(window[1]),
                                                     int(nthreads))
    else:
        rc = lib.oracle_attention_bwd_dq_rows(q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data, kind,
                                              rows.ctypes.data, rows.size, out.ctypes.data, B, H, Nq, Nk, d,
                                              float(scale), int(bool(causal)), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_attention_bwd_dq_rows failed ({rc})")
    return out


def attention_bwd_dkdv_keys(q, k, v, dout, bh, keys, scale, causal=False, nthreads=0, lib=None, window=None):
    """dK and dV rows of selected keys of head bh: ([len(keys), d], [len(keys), d]); window as in attention_bwd."""
    lib = lib or load_library()
    (q, k, v, dout), kind = _prep([q, k, v, dout])
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    keys = np.ascontiguousarray(keys, dtype=np.int64)
    dk = np.zeros((keys.size, d))
    dv = np.zeros((keys.size, d))
    if window is not None:
        rc = lib.oracle_attention_bwd_dkdv_keys_window(q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                                       dout.ctypes.data, kind, int(bh), keys.ctypes.data, keys.size,
                                                       dk.ctypes.data, dv.ctypes.data, B, H, Nq, Nk, d, float(scale),
                                                       int(window[0]), int(window[1]), int(nthreads))
    else:
        rc = lib.oracle_attention_bwd_dkdv_keys(q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data,
                                                kind, int(bh), keys.ctypes.data, keys.size, dk.ctypes.data,
                                                dv.ctypes.data, B, H, Nq, Nk, d, float(scale), int(bool(causal)),
                                                int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_attention_bwd_dkdv_keys failed ({rc})")
    return dk, dv
