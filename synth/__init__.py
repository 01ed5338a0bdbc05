"""Seeded synthetic attention inputs (no attention arithmetic here).

Both the CUDA path's tests/bench and the oracle consume the bf16 bits made
here, so the two sides always see identical inputs.  The generator is
SplitMix64 + Box-Muller, counter-based (see ``synth.c`` for its definition);
``normal_bf16_numpy`` restates it in numpy for the generator's own tests.

Workloads: the shapes the attention pages talk about, with i.i.d. normal
inputs (no dataset exists for them; GPT-2 attention is represented by its
shape only).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libsynth.so")
_lock = threading.Lock()
_lib = None

STREAM_Q, STREAM_K, STREAM_V = 0, 1, 2


def build() -> str:
    if (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                        "-o", tmp, _SRC, "-lm"], check=True, capture_output=True, text=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64 = ctypes.c_uint64
            lib.synth_normal_bf16.argtypes = [u64, u64, u64, u64, ctypes.c_double, ctypes.c_double,
                                              ctypes.c_void_p]
            lib.synth_normal_bf16.restype = None
            lib.synth_bf16_to_f32.argtypes = [ctypes.c_void_p, u64, ctypes.c_void_p]
            lib.synth_bf16_to_f32.restype = None
            lib.synth_stream_state.argtypes = [u64, u64]
            lib.synth_stream_state.restype = u64
            lib.synth_splitmix64_at.argtypes = [u64, u64]
            lib.synth_splitmix64_at.restype = u64
            _lib = lib
        return _lib


def normal_bf16(seed: int, stream: int, shape, sigma: float = 1.0, mean: float = 0.0,
                first: int = 0, out: np.ndarray | None = None) -> np.ndarray:
    """bf16 bits (uint16 array of ``shape``) of mean + sigma * N(0, 1)."""
    count = int(np.prod(shape)) if len(shape) else 1
    if out is None:
        out = np.empty(shape, dtype=np.uint16)
    if out.dtype != np.uint16 or out.size != count or not out.flags.c_contiguous:
        raise ValueError("out must be a contiguous uint16 array of the requested size")
    _load().synth_normal_bf16(seed, stream, first, count, float(mean), float(sigma), out.ctypes.data)
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bits to float32."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bits, round to nearest even (finite inputs)."""
    w = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    w = w + 0x7FFF + ((w >> 16) & 1)
    return ((w >> 16) & 0xFFFF).astype(np.uint16)


def splitmix64_at(state: int, n: int) -> int:
    return int(_load().synth_splitmix64_at(state, n))


def stream_state(seed: int, stream: int) -> int:
    return int(_load().synth_stream_state(seed, stream))


# numpy restatement of the same generator (used to test the C one) ----------
_M64 = (1 << 64) - 1
_GAMMA = 0x9E3779B97F4A7C15


def _mix_np(z):
    z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def normal_bf16_numpy(seed: int, stream: int, count: int, sigma: float = 1.0, mean: float = 0.0,
                      first: int = 0) -> np.ndarray:
    with np.errstate(over="ignore"):
        x = _mix_np(np.array([(seed * _GAMMA + stream + 1) & _M64], dtype=np.uint64))[0]
        e = np.arange(first, first + count, dtype=np.uint64)
        p = e >> np.uint64(1)
        g = np.uint64(_GAMMA)
        z1 = _mix_np(x + (np.uint64(2) * p + np.uint64(1)) * g)
        z2 = _mix_np(x + (np.uint64(2) * p + np.uint64(2)) * g)
    u1 = ((z1 >> np.uint64(11)).astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)
    u2 = ((z2 >> np.uint64(11)).astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)
    r = np.sqrt(-2.0 * np.log(u1))
    t = 2.0 * math.pi * u2
    z = np.where((e & np.uint64(1)) == 1, r * np.sin(t), r * np.cos(t))
    return f32_to_bf16_bits((mean + sigma * z).astype(np.float32))


# workloads ------------------------------------------------------------------
@dataclass(frozen=True)
class Workload:
    """One attention problem: shapes, mask, input distribution, seed."""

    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    causal: bool
    sigma_q: float = 1.0
    sigma_k: float = 1.0
    sigma_v: float = 1.0
    seed: int = 1000
    window: tuple | None = None  # (left, right) sliding-window bounds, -1 = open; None: no window

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def flops(self) -> float:
        """4*B*H*Nq*Nk*d, halved under a causal mask (the counting convention)."""
        f = 4.0 * self.B * self.H * self.Nq * self.Nk * self.d
        return f / 2.0 if self.causal else f

    @property
    def algorithmic_bytes(self) -> int:
        """Compulsory HBM bytes: read Q, K, V (bf16), write O (bf16) and LSE (fp32)."""
        bh = self.B * self.H
        return bh * (2 * self.d * (2 * self.Nq + 2 * self.Nk) + 4 * self.Nq)

    def q_shape(self):
        return (self.B, self.H, self.Nq, self.d)

    def kv_shape(self):
        return (self.B, self.H, self.Nk, self.d)

    def make(self):
        """(q, k, v) as bf16 bits, uint16 numpy arrays [B,H,N,d]."""
        q = normal_bf16(self.seed, STREAM_Q, self.q_shape(), self.sigma_q)
        k = normal_bf16(self.seed, STREAM_K, self.kv_shape(), self.sigma_k)
        v = normal_bf16(self.seed, STREAM_V, self.kv_shape(), self.sigma_v)
        return q, k, v

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


WORKLOADS = {
    # the small single-head case
    "single_head_256_d64": Workload("single_head_256_d64", 1, 1, 256, 256, 64, False, seed=1000),
    # the pages' memory-budget example: one head, N = 4096, d = 64
    "single_head_4096_d64": Workload("single_head_4096_d64", 1, 1, 4096, 4096, 64, False, seed=1001),
    # GPT-2-small-shaped attention: 8 x 12 heads, N = 1024, d = 64, causal
    "gpt2_small_causal_1024_d64": Workload("gpt2_small_causal_1024_d64", 8, 12, 1024, 1024, 64, True,
                                           seed=1002),
    # long context: 4 x 32 heads, N = 8192, d = 128, non-causal and causal
    "long_8192_d128": Workload("long_8192_d128", 4, 32, 8192, 8192, 128, False, seed=1003),
    "long_8192_d128_causal": Workload("long_8192_d128_causal", 4, 32, 8192, 8192, 128, True,
                                      seed=1003),
    # stress: 16 heads, N = 32000, Q ~ N(0, 4^2), causal
    "stress_32000_d128_causal": Workload("stress_32000_d128_causal", 1, 16, 32000, 32000, 128, True,
                                         sigma_q=4.0, seed=1004),
    # not one of the pages' shapes: the long-context shape at d = 64, to measure
    # whether the exponential unit or the tensor pipe binds at the smaller head
    "long_8192_d64": Workload("long_8192_d64", 4, 32, 8192, 8192, 64, False, seed=1005),
}
