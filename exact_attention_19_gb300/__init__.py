"""GB300-native fused exact attention (sm_103a): forward, split-KV, sliding
window and backward.

Thin ctypes binding over ``libfa_gb300.so`` (C ABI in ``include/fa.h``):
argument marshalling only, every step of the computation runs in the CUDA
kernels.  PyTorch supplies device memory and streams.

    o, lse = fwd(q, k, v, causal=False)          # torch bf16 [B, H, N, d]
    dq, dk, dv = bwd(q, k, v, o, lse, do, causal=False)
    fa_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, Nq, Nk, d, scale, causal, stream)

There is no fallback: if the library cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os

__all__ = [
    "FaError", "STATUS", "NOALLOC_SCRATCH_BYTES", "library_path", "load",
    "fwd", "bwd",
    "fa_fwd", "fa_fwd_window", "fa_fwd_splitkv", "fa_fwd_splitkv_noalloc", "fa_splitkv_workspace_bytes",
    "fa_splitkv_heuristic", "fa_bwd", "fa_bwd_window", "fa_bwd_workspace_bytes", "fa_probe_exp2", "fa_selftest_wait",
    "fa_fwd_status",
    "fa_strerror", "fa_version",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_lib", "libfa_gb300.so")

STATUS = {
    0: "FA_OK", 1: "FA_ERR_NULL", 2: "FA_ERR_ALIGN", 3: "FA_ERR_SHAPE", 4: "FA_ERR_HEADDIM",
    5: "FA_ERR_CAUSAL_SHAPE", 6: "FA_ERR_LAUNCH", 7: "FA_ERR_DEVICE", 8: "FA_ERR_TIMEOUT",
    9: "FA_ERR_SCALE", 10: "FA_ERR_POINTER", 11: "FA_ERR_WORKSPACE",
}

NOALLOC_SCRATCH_BYTES = 16 << 20  # FA_NOALLOC_SCRATCH_BYTES in include/fa.h

_lib = None


class FaError(RuntimeError):
    def __init__(self, status: int, where: str = "fa_fwd"):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({fa_strerror(status)})")


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load libfa_gb300.so (built by ``build.py`` / ``__graft_entry__.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(f"{_LIB_PATH} is missing: build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i32 = ctypes.c_void_p, ctypes.c_int
        lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, ctypes.c_float, i32, vp]
        lib.fa_fwd.restype = i32
        lib.fa_strerror.argtypes = [i32]
        lib.fa_strerror.restype = ctypes.c_char_p
        lib.fa_version.argtypes = []
        lib.fa_version.restype = i32
        lib.fa_fwd_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint), i32]
        lib.fa_fwd_status.restype = i32
        lib.fa_probe_exp2.argtypes = [i32, ctypes.POINTER(ctypes.c_double), vp]
        lib.fa_probe_exp2.restype = i32
        lib.fa_selftest_wait.argtypes = [i32, ctypes.POINTER(ctypes.c_uint), ctypes.POINTER(ctypes.c_ulonglong), vp]
        lib.fa_selftest_wait.restype = i32
        lib.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, ctypes.c_float, i32, i32, vp,
                                       ctypes.c_size_t, vp]
        lib.fa_fwd_splitkv.restype = i32
        lib.fa_splitkv_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
        lib.fa_splitkv_workspace_bytes.restype = ctypes.c_size_t
        lib.fa_splitkv_heuristic.argtypes = [i32, i32, i32, i32, i32, i32]
        lib.fa_splitkv_heuristic.restype = i32
        lib.fa_fwd_splitkv_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, ctypes.c_float, i32,
                                               i32, vp]
        lib.fa_fwd_splitkv_noalloc.restype = i32
        lib.fa_fwd_window.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, ctypes.c_float, i32, i32, vp]
        lib.fa_fwd_window.restype = i32
        lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, ctypes.c_float, i32, vp,
                               ctypes.c_size_t, vp]
        lib.fa_bwd.restype = i32
        lib.fa_bwd_window.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, ctypes.c_float, i32,
                                      i32, vp, ctypes.c_size_t, vp]
        lib.fa_bwd_window.restype = i32
        lib.fa_bwd_workspace_bytes.argtypes = [i32, i32, i32]
        lib.fa_bwd_workspace_bytes.restype = ctypes.c_size_t
        _lib = lib
    return _lib


def fa_strerror(status: int) -> str:
    return load().fa_strerror(int(status)).decode()


def fa_version() -> int:
    return int(load().fa_version())


def fa_fwd(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, stream) -> int:
    """Raw C-ABI call with integer device pointers and a raw stream handle.

    Returns the status code (0 = FA_OK); does not raise.
    """
    return int(load().fa_fwd(q, k, v, o, lse, int(B), int(H), int(Nq), int(Nk), int(d), float(scale),
                             int(causal), stream))


def fa_fwd_window(q, k, v, o, lse, B, H, Nq, Nk, d, scale, window_left, window_right, stream) -> int:
    """Raw C-ABI sliding-window call (bottom-right aligned, -1 = unbounded); returns the status code."""
    return int(load().fa_fwd_window(q, k, v, o, lse, int(B), int(H), int(Nq), int(Nk), int(d), float(scale),
                                    int(window_left), int(window_right), stream))


def fa_fwd_splitkv(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, n_splits, workspace, workspace_bytes,
                   stream) -> int:
    """Raw C-ABI split-KV call; returns the status code (does not raise)."""
    return int(load().fa_fwd_splitkv(q, k, v, o, lse, int(B), int(H), int(Nq), int(Nk), int(d), float(scale),
                                     int(causal), int(n_splits), workspace, int(workspace_bytes), stream))


def fa_fwd_splitkv_noalloc(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, n_splits, stream) -> int:
    """Raw C-ABI split-KV call that allocates nothing (the library's fixed
    device array holds the slice buffers); returns the status code.

    For callers that cannot allocate device memory themselves.  Calls that
    overlap on the GPU share that array and must be serialised by the caller.
    """
    return int(load().fa_fwd_splitkv_noalloc(q, k, v, o, lse, int(B), int(H), int(Nq), int(Nk), int(d),
                                             float(scale), int(causal), int(n_splits), stream))


def fa_splitkv_workspace_bytes(B, H, Nq, Nk, d, n_splits) -> int:
    return int(load().fa_splitkv_workspace_bytes(int(B), int(H), int(Nq), int(Nk), int(d), int(n_splits)))


def fa_splitkv_heuristic(B, H, Nq, Nk, d, causal) -> int:
    return int(load().fa_splitkv_heuristic(int(B), int(H), int(Nq), int(Nk), int(d), int(causal)))


def fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, Nq, Nk, d, scale, causal, workspace, workspace_bytes,
           stream) -> int:
    """Raw C-ABI backward call; returns the status code (does not raise)."""
    return int(load().fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, int(B), int(H), int(Nq), int(Nk), int(d),
                             float(scale), int(causal), workspace, int(workspace_bytes), stream))


def fa_bwd_window(q, k, v, o, lse, dout, dq, dk, dv, B, H, Nq, Nk, d, scale, window_left, window_right, workspace,
                  workspace_bytes, stream) -> int:
    """Raw C-ABI sliding-window backward call (bottom-right aligned, -1 = unbounded); returns the status code."""
    return int(load().fa_bwd_window(q, k, v, o, lse, dout, dq, dk, dv, int(B), int(H), int(Nq), int(Nk), int(d),
                                    float(scale), int(window_left), int(window_right), workspace,
                                    int(workspace_bytes), stream))


def fa_bwd_workspace_bytes(B, H, Nq) -> int:
    return int(load().fa_bwd_workspace_bytes(int(B), int(H), int(Nq)))


def fa_fwd_status(stream=None, clear: bool = False):
    """(status, raw device status word) after synchronising ``stream``."""
    word = ctypes.c_uint(0)
    st = int(load().fa_fwd_status(stream, ctypes.byref(word), int(bool(clear))))
    return st, int(word.value)


def fa_probe_exp2(method: int = 0, stream=None) -> float:
    """2^x results per SM clock: method 0 ex2.approx (special-function unit), 1 cubic polynomial on the
    FMA pipes.  Synchronises ``stream``."""
    rate = ctypes.c_double(0.0)
    st = int(load().fa_probe_exp2(int(method), ctypes.byref(rate), stream))
    if st != 0:
        raise FaError(st, "fa_probe_exp2")
    return float(rate.value)


def fa_selftest_wait(mode: int, stream=None):
    """Run the bounded-wait self-test (0: time limit, 1: abort flag); returns (status word, wait ns)."""
    word, ns = ctypes.c_uint(0), ctypes.c_ulonglong(0)
    st = int(load().fa_selftest_wait(int(mode), ctypes.byref(word), ctypes.byref(ns), stream))
    if st != 0:
        raise FaError(st, "fa_selftest_wait")
    return int(word.value), int(ns.value)


def _stream_handle(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def fwd(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None, stream=None,
        n_splits: int | None = None, workspace=None, window: tuple | None = None):
    """O = softmax(q k^T * scale) v and the per-row LSE, on the GPU.

    q: [B, H, Nq, d], k, v: [B, H, Nk, d] torch.bfloat16 CUDA tensors,
    contiguous.  ``scale`` defaults to 1/sqrt(d).  ``out`` (bf16 [B,H,Nq,d])
    and ``lse`` (fp32 [B,H,Nq]) may be given to avoid allocation.  Runs on
    ``stream`` (default: the current torch stream), asynchronously.

    ``n_splits``: K/V slices per query tile (split-KV, for shapes with too few
    query tiles to fill the GPU); None asks the library's heuristic, 1 forces
    the single-pass kernel.  ``workspace`` (a CUDA tensor of at least
    ``fa_splitkv_workspace_bytes`` bytes) may be given to avoid allocating it.

    ``window=(left, right)``: sliding-window mask aligned bottom-right (key j
    visible to row i iff i+Nk-Nq-left <= j <= i+Nk-Nq+right, -1 = unbounded);
    replaces ``causal`` and runs the single-pass kernel.
    """
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA torch.bfloat16 tensor")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [B, H, N, d] tensor")
    B, H, Nq, d = q.shape
    if k.shape[:2] != (B, H) or k.shape[3] != d or v.shape != k.shape:
        raise ValueError(f"shape mismatch: q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor shaped like q")
    if lse.shape != (B, H, Nq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, H, Nq] tensor")
    if window is not None:
        st = fa_fwd_window(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, Nq, Nk,
                           d, scale, int(window[0]), int(window[1]), _stream_handle(stream))
        if st != 0:
            raise FaError(st, "fa_fwd_window")
        return out, lse
    if n_splits is None:
        n_splits = fa_splitkv_heuristic(B, H, Nq, Nk, d, int(bool(causal))) if Nq > 0 else 1
    if n_splits > 1:
        need = fa_splitkv_workspace_bytes(B, H, Nq, Nk, d, n_splits)
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        if not workspace.is_cuda or workspace.numel() * workspace.element_size() < need:
            raise ValueError(f"workspace must be a CUDA tensor of at least {need} bytes")
        st = fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, Nq,
                            Nk, d, scale, int(bool(causal)), n_splits, workspace.data_ptr(),
                            workspace.numel() * workspace.element_size(), _stream_handle(stream))
        if st != 0:
            raise FaError(st, "fa_fwd_splitkv")
        return out, lse
    st = fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, Nq, Nk, d,
                scale, int(bool(causal)), _stream_handle(stream))
    if st != 0:
        raise FaError(st)
    return out, lse


def bwd(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None, dq=None, dk=None, dv=None,
        workspace=None, stream=None, window: tuple | None = None):
    """(dq, dk, dv) of attention by recomputation from the forward's ``lse``.

    q, o, dout: [B, H, Nq, d]; k, v: [B, H, Nk, d], CUDA bf16, contiguous;
    lse: fp32 [B, H, Nq] from ``fwd``.  ``workspace`` (CUDA tensor of at least
    ``fa_bwd_workspace_bytes`` bytes) may be given to avoid allocating it.
    ``window=(left, right)``: the sliding-window mask of ``fwd(window=...)``
    (pass the same window to both; ``causal`` is then ignored).
    """
    import torch

    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous CUDA torch.bfloat16 tensor")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if o.shape != q.shape or dout.shape != q.shape or v.shape != k.shape or k.shape[:2] != (B, H) or k.shape[3] != d:
        raise ValueError("shape mismatch")
    if lse.shape != (B, H, Nq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, H, Nq] tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t, like in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        if (not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda or
                not t.is_contiguous() or t.shape != like.shape):
            raise ValueError(f"{name} must be a contiguous CUDA bf16 tensor shaped like {tuple(like.shape)}")
    need = fa_bwd_workspace_bytes(B, H, Nq)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    if window is not None:
        st = fa_bwd_window(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
                           dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Nq, Nk, d, scale, int(window[0]),
                           int(window[1]), workspace.data_ptr(), ws_bytes, _stream_handle(stream))
        if st != 0:
            raise FaError(st, "fa_bwd_window")
        return dq, dk, dv
    st = fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
                dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Nq, Nk, d, scale, int(bool(causal)),
                workspace.data_ptr(), ws_bytes, _stream_handle(stream))
    if st != 0:
        raise FaError(st, "fa_bwd")
    return dq, dk, dv
