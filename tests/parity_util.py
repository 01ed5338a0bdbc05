"""Helpers shared by the GPU parity tests: upload bf16 bits, run the CUDA path
through the C ABI binding, compare with the fp64 oracle.

Tolerances (the stated bar, with the readings noted):
  O:   |O_gpu - O_ref| <= min(1e-2 * max(1, |O_ref|), 1e-2 + u(O_ref) / 2)
       elementwise, u(x) the spacing of bf16 numbers at x (2^(floor(log2 |x|) - 7)).
       O is returned in bf16, 8 significant bits, as the operation specifies;
       rounding a value to bf16 moves it by up to u/2, between 2^-9 and 2^-8
       of its magnitude, and the bf16 P of the P.V product moves the value
       before that rounding by up to about 2^-8 of the spread of the V rows
       it mixes.  The bar reads "max |dO| <= 1e-2" as an error of at most
       1e-2 before the final rounding to bf16, plus that rounding: absolute
       1e-2 below |O| = 1 (no looser than before anywhere), and 1e-2 + u/2
       above (0.0178 on [2, 4), 0.0256 on [4, 8), against the 0.02-0.08 of a
       relative 1e-2 * |O| there).
  LSE: |LSE_gpu - LSE_ref| <= 1e-3 * max(1, |LSE_ref|).
"""
from __future__ import annotations

import numpy as np

O_TOL = 1e-2
LSE_TOL = 1e-3


def to_device(bits, device="cuda"):
    import torch

    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def run_gpu(q, k, v, scale, causal, n_splits=None):
    """q, k, v: uint16 bf16 bits [B,H,N,d].  Returns (o float64 numpy, lse float64 numpy).

    n_splits: None lets the library choose (split-KV for small grids), 1 forces
    the single-pass kernel, > 1 forces that many K/V slices.
    """
    import torch

    import exact_attention_19_gb300 as fa

    tq, tk, tv = to_device(q), to_device(k), to_device(v)
    o, lse = fa.fwd(tq, tk, tv, causal=causal, scale=scale, n_splits=n_splits)
    torch.cuda.synchronize()
    st, word = fa.fa_fwd_status(None, clear=True)
    assert st == 0, f"kernel wait timed out, status word {word:#x}"
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def o_tol(o_ref):
    """Elementwise O bar: min(1e-2 * max(1, |O_ref|), 1e-2 + half the bf16 spacing at O_ref)."""
    mag = np.abs(o_ref)
    with np.errstate(divide="ignore"):
        expo = np.floor(np.log2(np.where(mag > 0, mag, 1.0)))
    half_ulp = np.where(mag > 0, np.exp2(expo - 8.0), 0.0)
    return np.minimum(O_TOL * np.maximum(1.0, mag), O_TOL + half_ulp)


def o_err(o_gpu, o_ref):
    """Largest |O_gpu - O_ref| / (o_tol(O_ref) / 1e-2): <= 1e-2 passes."""
    if not o_ref.size:
        return 0.0
    return float(np.max(np.abs(o_gpu - o_ref) / (o_tol(o_ref) / O_TOL)))


def lse_err(l_gpu, l_ref):
    return float(np.max(np.abs(l_gpu - l_ref) / np.maximum(1.0, np.abs(l_ref)))) if l_ref.size else 0.0


def assert_close(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite O"
    assert np.all(np.isfinite(lse_gpu)), f"{what}: non-finite LSE"
    eo, el = o_err(o_gpu, o_ref), lse_err(lse_gpu, lse_ref)
    assert eo <= O_TOL, f"{what}: O error {eo:.3e} (max abs {np.max(np.abs(o_gpu - o_ref)):.3e})"
    assert el <= LSE_TOL, f"{what}: LSE error {el:.3e}"
    return eo, el


def sample_rows(B, H, Nq, n, seed):
    """Flat row indices: first and last rows of the first and last heads,
    the tile boundaries around row 128/256 of one head, plus n random rows."""
    rng = np.random.default_rng(seed)
    BH = B * H
    picks = set()
    for bh in {0, BH - 1, BH // 2}:
        for i in (0, 1, 2, 127, 128, 129, 255, 256, Nq // 2, Nq - 3, Nq - 2, Nq - 1):
            if 0 <= i < Nq:
                picks.add(bh * Nq + i)
    picks.update(int(x) for x in rng.integers(0, BH * Nq, size=n))
    return np.array(sorted(picks), dtype=np.int64)
