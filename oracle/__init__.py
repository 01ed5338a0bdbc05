"""fp64 CPU oracle for the exact-attention forward pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
library never calls it, and it shares no code with the CUDA path.

``attention_fwd`` / ``attention_rows`` wrap ``attention_ref.c`` (plain C,
OpenMP over rows, double precision, S and P rows materialised).  The C file is
compiled with the host's gcc on first use (or by ``build()``) into
``oracle/_build/``.  ``online`` holds the test-only tiled recurrence.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention_ref.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_attn.so")

F64 = 0
BF16 = 1

_lock = threading.Lock()
_lib = None


def compile_oracle(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile an oracle C source into a shared library; returns its path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", *extra_flags, "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, out)
    return out


def build() -> str:
    """(Re)compile the oracle library if the source is newer."""
    if (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        compile_oracle()
    return _LIB_PATH


def _declare(lib):
    i64 = ctypes.c_longlong
    vp = ctypes.c_void_p
    lib.oracle_attention_fwd.argtypes = [vp, vp, vp, ctypes.c_int, vp, vp, i64, i64, i64, i64, i64,
                                         ctypes.c_double, ctypes.c_int, ctypes.c_int]
    lib.oracle_attention_fwd.restype = ctypes.c_int
    lib.oracle_attention_rows.argtypes = [vp, vp, vp, ctypes.c_int, vp, i64, vp, vp, i64, i64, i64,
                                          i64, i64, ctypes.c_double, ctypes.c_int, ctypes.c_int]
    lib.oracle_attention_rows.restype = ctypes.c_int
    lib.oracle_attention_fwd_window.argtypes = [vp, vp, vp, ctypes.c_int, vp, vp, i64, i64, i64, i64, i64,
                                                ctypes.c_double, i64, i64, ctypes.c_int]
    lib.oracle_attention_fwd_window.restype = ctypes.c_int
    lib.oracle_attention_rows_window.argtypes = [vp, vp, vp, ctypes.c_int, vp, i64, vp, vp, i64, i64, i64,
                                                 i64, i64, ctypes.c_double, i64, i64, ctypes.c_int]
    lib.oracle_attention_rows_window.restype = ctypes.c_int
    lib.oracle_threads.argtypes = []
    lib.oracle_threads.restype = ctypes.c_int
    return lib


def load_library(path: str | None = None):
    """Load the oracle library (the default one, or a given build of it)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
        return _lib


def threads() -> int:
    return int(load_library().oracle_threads())


def _prep(x, name):
    a = np.ascontiguousarray(x)
    if a.dtype == np.uint16:
        return a, BF16
    if a.dtype == np.float64:
        return a, F64
    raise TypeError(f"{name}: expected float64 values or uint16 bf16 bits, got {a.dtype}")


def _shapes(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B, H, N, d]")
    B, H, Nq, d = q.shape
    if k.shape[:2] != (B, H) or v.shape != k.shape or k.shape[3] != d:
        raise ValueError(f"shape mismatch q{q.shape} k{k.shape} v{v.shape}")
    return B, H, Nq, k.shape[2], d


def attention_fwd(q, k, v, scale, causal=False, nthreads=0, lib=None, window=None):
    """O [B,H,Nq,d] and LSE [B,H,Nq], both float64, for every query row.

    q, k, v: arrays [B, H, N, d] of float64, or of uint16 holding bf16 bits
    (all three the same kind).  window=(wl, wr): keep key j for row i iff
    i + (Nk - Nq) - wl <= j <= i + (Nk - Nq) + wr, a negative bound meaning
    unbounded (overrides ``causal``).
    """
    lib = lib or load_library()
    q, dq = _prep(q, "q")
    k, dk = _prep(k, "k")
    v, dv = _prep(v, "v")
    if not (dq == dk == dv):
        raise TypeError("q, k, v must share one element kind")
    B, H, Nq, Nk, d = _shapes(q, k, v)
    o = np.zeros((B, H, Nq, d), dtype=np.float64)
    lse = np.zeros((B, H, Nq), dtype=np.float64)
    if window is not None:
        rc = lib.oracle_attention_fwd_window(q.ctypes.data, k.ctypes.data, v.ctypes.data, dq, o.ctypes.data,
                                             lse.ctypes.data, B, H, Nq, Nk, d, float(scale), int(window[0]),
                                             int(window[1]), int(nthreads))
        if rc != 0:
            raise RuntimeError(f"oracle_attention_fwd_window failed ({rc})")
        return o, lse
    rc = lib.oracle_attention_fwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, dq, o.ctypes.data,
                                  lse.ctypes.data, B, H, Nq, Nk, d, float(scale), int(bool(causal)),
                                  int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_attention_fwd failed ({rc})")
    return o, lse


def attention_rows(q, k, v, rows, scale, causal=False, nthreads=0, lib=None, window=None):
    """O and LSE for selected query rows only.

    rows: flat indices (b*H + h)*Nq + i.  Returns o [len(rows), d], lse [len(rows)].
    window as in ``attention_fwd``.
    """
    lib = lib or load_library()
    q, dq = _prep(q, "q")
    k, dk = _prep(k, "k")
    v, dv = _prep(v, "v")
    if not (dq == dk == dv):
        raise TypeError("q, k, v must share one element kind")
    B, H, Nq, Nk, d = _shapes(q, k, v)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    o = np.zeros((rows.size, d), dtype=np.float64)
    lse = np.zeros(rows.size, dtype=np.float64)
    if window is not None:
        rc = lib.oracle_attention_rows_window(q.ctypes.data, k.ctypes.data, v.ctypes.data, dq, rows.ctypes.data,
                                              rows.size, o.ctypes.data, lse.ctypes.data, B, H, Nq, Nk, d,
                                              float(scale), int(window[0]), int(window[1]), int(nthreads))
        if rc != 0:
            raise RuntimeError(f"oracle_attention_rows_window failed ({rc})")
        return o, lse
    rc = lib.oracle_attention_rows(q.ctypes.data, k.ctypes.data, v.ctypes.data, dq,
                                   rows.ctypes.data, rows.size, o.ctypes.data, lse.ctypes.data,
                                   B, H, Nq, Nk, d, float(scale), int(bool(causal)), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_attention_rows failed ({rc})")
    return o, lse
