"""Backward pass (fa_bwd) against the fp64 backward oracle (GB300 only).

The GPU forward's own O and LSE feed the GPU backward (as a user would call
it); the oracle recomputes everything in double precision from the same
bf16 Q, K, V, dO.  Tolerance, element by element:

    |d_gpu - d_ref| <= atol_r + rtol * |d_ref|,  rtol = 1e-2,  atol_r = 1e-2 * M_r

with M_r the size of the sums that define row r of dQ (key r of dK, dV),
taken over the magnitudes of their terms (tests/grad_scale.py).  P and
dS = P (dP - D) are rounded to bf16 before their products, D comes from the
forward's bf16 O and the gradients are returned in bf16, each rounding
relative (2^-9) to what it rounds, so an entry's error scales with the size
of its terms, not with the entry, which cancels to near zero in some rows
(a query that sees one key has dQ = 0).  A row whose M_r is zero (no kept
key) must come out exactly zero.
"""
import numpy as np
import pytest

import synth
from oracle import backward
from grad_scale import dkdv_key_scales, dq_row_scales, row_scales
from parity_util import to_device

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_19_gb300 as fa
    from exact_attention_19_gb300 import build

    build.build()
    fa.load()
    backward.build()
    yield


def _gpu_grads(q, k, v, do, scale, causal):
    import torch

    import exact_attention_19_gb300 as fa

    tq, tk, tv, tdo = (to_device(x) for x in (q, k, v, do))
    o, lse = fa.fwd(tq, tk, tv, causal=causal, scale=scale, n_splits=1)
    dq, dk, dv = fa.bwd(tq, tk, tv, o, lse, tdo, causal=causal, scale=scale)
    torch.cuda.synchronize()
    st, word = fa.fa_fwd_status(None, clear=True)
    assert st == 0, f"kernel wait timed out, status word {word:#x}"
    return tuple(t.float().cpu().numpy().astype(np.float64) for t in (dq, dk, dv))


def _err(a, ref, m_row):
    """Largest |a - ref| / (M_r + |ref|) over all entries, M_r broadcast along the last
    axis (a row); <= TOL passes.  Where M_r + |ref| is zero the entry must be exactly zero."""
    mag = np.abs(ref)
    denom = np.asarray(m_row)[..., None] + mag
    diff = np.abs(a - ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(denom > 0, diff / np.where(denom > 0, denom, 1.0), np.where(diff > 0, np.inf, 0.0))
    return float(np.max(ratio)) if ratio.size else 0.0


def _check(w: synth.Workload, what=""):
    q, k, v = w.make()
    do = synth.normal_bf16(w.seed + 7, 3, w.q_shape())
    got = _gpu_grads(q, k, v, do, w.scale, w.causal)
    ref = backward.attention_bwd(q, k, v, do, w.scale, w.causal)
    scales = row_scales(q, k, v, do, w.scale, w.causal)
    errs = [_err(g, r, m) for g, r, m in zip(got, ref, scales)]
    for name, g, e in zip(("dq", "dk", "dv"), got, errs):
        assert np.all(np.isfinite(g)), f"{what} {name} not finite"
        assert e <= TOL, f"{what} {name} error {e:.3e} of the row-scaled bar"
    return errs


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n", [1, 63, 128, 129, 300, 1000])
def test_bwd_square(n, d, causal):
    _check(synth.Workload(f"bwd{n}", 1, 2, n, n, d, causal, seed=800 + n), f"n={n} d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("nq,nk", [(100, 300), (513, 64), (256, 1000), (1, 700), (700, 1), (129, 1)])
def test_bwd_rectangular(nq, nk, d):
    _check(synth.Workload("bwd_rect", 2, 1, nq, nk, d, False, seed=810 + nq), f"{nq}x{nk} d={d}")


def test_bwd_multi_head_and_wide_logits():
    _check(synth.Workload("bwd_bh", 2, 3, 257, 257, 128, True, sigma_q=3.0, seed=820))
    _check(synth.Workload("bwd_bh", 3, 2, 200, 200, 64, False, sigma_q=3.0, seed=821))


# hundreds of short heads with a ragged second tile: grids of ~1000 small CTAs in
# both backward kernels (and the single-tile forward for causal d = 64)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_many_short_heads(d, causal):
    _check(synth.Workload("bwd_many", 8, 64, 130, 130, d, causal, seed=840 + d + causal),
           f"many heads d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("shape", [(333, 333, True), (333, 200, False), (77, 461, False)])
def test_bwd_outputs_not_written_outside(d, shape):
    """dQ, dK, dV embedded in larger guard-filled buffers: the guards stay
    untouched and every gradient inside is finite.  The gradients go out
    through tiled tensor stores of whole 128-row tiles; every head's last
    tile here is ragged, so the stores must drop the rows past Nq (dQ) or Nk
    (dK, dV) of each head."""
    import torch

    import exact_attention_19_gb300 as fa

    nq, nk, causal = shape
    B, H = 2, 3
    w = synth.Workload("bwd_guard", B, H, nq, nk, d, causal, seed=12)
    q, k, v = w.make()
    do = synth.normal_bf16(w.seed + 7, 3, w.q_shape())
    tq, tk, tv, tdo = (to_device(x) for x in (q, k, v, do))
    o, lse = fa.fwd(tq, tk, tv, causal=causal, scale=w.scale, n_splits=1)
    pad = 4096

    def guarded(n_rows):
        big = torch.full((B * H * n_rows * d + 2 * pad,), 7.0, dtype=torch.bfloat16, device="cuda")
        return big, big[pad:pad + B * H * n_rows * d].view(B, H, n_rows, d)

    (bq, dq), (bk, dk), (bv, dv) = guarded(nq), guarded(nk), guarded(nk)
    fa.bwd(tq, tk, tv, o, lse, tdo, causal=causal, scale=w.scale, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    for big, t in ((bq, dq), (bk, dk), (bv, dv)):
        assert torch.all(big[:pad] == 7.0) and torch.all(big[pad + t.numel():] == 7.0)
        assert torch.isfinite(t).all()
    ref = backward.attention_bwd(q, k, v, do, w.scale, causal)
    scales = row_scales(q, k, v, do, w.scale, causal)
    got = tuple(t.float().cpu().numpy().astype(np.float64) for t in (dq, dk, dv))
    for name, g, r, m in zip(("dq", "dk", "dv"), got, ref, scales):
        assert _err(g, r, m) <= TOL, f"{name} error {_err(g, r, m):.3e} of the row-scaled bar"


# --- sliding window (fa_bwd_window) ------------------------------------------
# (B, H, Nq, Nk, window): a band, a symmetric window, the causal mask aligned
# bottom-right for Nq != Nk, Nq > Nk with rows (whole query tiles) that keep no
# key, Nq < Nk with key tiles no row keeps, the diagonal alone, an open window
# (no mask) and a one-tile-wide band over ragged tiles
WINDOW_CASES = [
    (1, 2, 1000, 1000, (100, 0)),
    (1, 2, 1000, 1000, (64, 64)),
    (2, 1, 300, 1000, (-1, 0)),
    (1, 2, 640, 200, (0, 1)),
    (1, 2, 200, 640, (0, 0)),
    (1, 1, 461, 77, (5, 5)),
    (1, 2, 333, 333, (0, 0)),
    (1, 1, 257, 129, (-1, -1)),
    (2, 2, 129, 1000, (127, 1)),
]


def _window_grads(q, k, v, do, scale, window, guard=0):
    import torch

    import exact_attention_19_gb300 as fa

    tq, tk, tv, tdo = (to_device(x) for x in (q, k, v, do))
    o, lse = fa.fwd(tq, tk, tv, scale=scale, window=window)
    bufs, outs = [], []
    for like in (tq, tk, tv):
        big = torch.full((like.numel() + 2 * guard,), 7.0, dtype=torch.bfloat16, device="cuda")
        bufs.append(big)
        outs.append(big[guard:guard + like.numel()].view(like.shape))
    fa.bwd(tq, tk, tv, o, lse, tdo, scale=scale, window=window, dq=outs[0], dk=outs[1], dv=outs[2])
    torch.cuda.synchronize()
    st, word = fa.fa_fwd_status(None, clear=True)
    assert st == 0, f"kernel wait timed out, status word {word:#x}"
    for big, t in zip(bufs, outs):
        assert torch.all(big[:guard] == 7.0) and torch.all(big[guard + t.numel():] == 7.0)
    return tuple(t.float().cpu().numpy().astype(np.float64) for t in outs)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("case", WINDOW_CASES, ids=[f"{c[2]}x{c[3]}_w{c[4][0]}_{c[4][1]}" for c in WINDOW_CASES])
def test_bwd_window(d, case):
    B, H, nq, nk, window = case
    w = synth.Workload("bwd_window", B, H, nq, nk, d, False, seed=31 + nq + nk)
    q, k, v = w.make()
    do = synth.normal_bf16(w.seed + 7, 3, w.q_shape())
    got = _window_grads(q, k, v, do, w.scale, window, guard=2048)
    ref = backward.attention_bwd(q, k, v, do, w.scale, window=window)
    scales = row_scales(q, k, v, do, w.scale, window=window)
    for name, g, r, m in zip(("dq", "dk", "dv"), got, ref, scales):
        assert np.all(np.isfinite(g)), f"{name} not finite"
        assert _err(g, r, m) <= TOL, f"{name} error {_err(g, r, m):.3e} of the row-scaled bar"
    # rows that keep no key and keys no row keeps (keep-matrix by enumeration)
    # have gradients of exactly zero
    wl, wr = window
    off = np.arange(nk)[None, :] - (np.arange(nq)[:, None] + nk - nq)
    keep = ((wl < 0) | (off >= -wl)) & ((wr < 0) | (off <= wr))
    dead_rows, dead_keys = ~keep.any(axis=1), ~keep.any(axis=0)
    assert np.all(got[0][:, :, dead_rows] == 0.0)
    assert np.all(got[1][:, :, dead_keys] == 0.0) and np.all(got[2][:, :, dead_keys] == 0.0)
    if window == (0, 1) or window == (0, 0) and nq != nk:
        assert dead_rows.any() or dead_keys.any()  # the empty-tile paths are exercised


def test_bwd_window_bottom_right_causal_matches_causal():
    """(-1, 0) with Nq == Nk is the causal mask: same gradients as fa_bwd(causal)."""
    w = synth.Workload("bwd_wc", 2, 2, 700, 700, 128, True, seed=37)
    q, k, v = w.make()
    do = synth.normal_bf16(w.seed + 7, 3, w.q_shape())
    got_w = _window_grads(q, k, v, do, w.scale, (-1, 0))
    got_c = _gpu_grads(q, k, v, do, w.scale, True)
    for a, b in zip(got_w, got_c):
        assert np.array_equal(a, b)


def test_bwd_window_errors():
    import torch

    import exact_attention_19_gb300 as fa

    q = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, 1, 128), dtype=torch.float32, device="cuda")
    ws = torch.empty(fa.fa_bwd_workspace_bytes(1, 1, 128), dtype=torch.uint8, device="cuda")
    args = [q.data_ptr()] * 3 + [q.data_ptr(), lse.data_ptr(), q.data_ptr()]
    outs = [torch.empty_like(q).data_ptr() for _ in range(3)]
    st = fa.fa_bwd_window(*args, *outs, 1, 1, 128, 128, 64, 0.125, -2, 0, ws.data_ptr(), ws.numel(), None)
    assert st == 3  # FA_ERR_SHAPE: a bound below -1
    st = fa.fa_bwd_window(*args, *outs, 1, 1, 128, 128, 64, 0.125, 4, 4, ws.data_ptr(), 16, None)
    assert st == 11  # FA_ERR_WORKSPACE


def test_bwd_deterministic():
    w = synth.Workload("bwd_det", 1, 3, 700, 700, 128, True, seed=830)
    q, k, v = w.make()
    do = synth.normal_bf16(831, 3, w.q_shape())
    a = _gpu_grads(q, k, v, do, w.scale, True)
    b = _gpu_grads(q, k, v, do, w.scale, True)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))


def test_bwd_workspace_errors():
    import torch

    import exact_attention_19_gb300 as fa

    t = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, 1, 128), dtype=torch.float32, device="cuda")
    need = fa.fa_bwd_workspace_bytes(1, 1, 128)
    assert need == 2 * 128 * 4
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    args = [t.data_ptr()] * 4 + [lse.data_ptr(), t.data_ptr()] + [torch.empty_like(t).data_ptr() for _ in range(3)]
    assert fa.fa_bwd(*args, 1, 1, 128, 128, 64, 0.125, 0, ws.data_ptr(), need - 16, None) == 11
    assert fa.fa_bwd(*args, 1, 1, 128, 128, 64, 0.125, 1, ws.data_ptr(), need, None) == 0
    assert fa.fa_bwd(*args, 1, 1, 0, 128, 64, 0.125, 0, ws.data_ptr(), need, None) == 3
    torch.cuda.synchronize()


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_full_size_sampled(causal):
    """B=4 H=32 N=8192 d=128: sampled dQ rows over all heads, sampled dK/dV keys of one head."""
    from parity_util import sample_rows

    w = synth.WORKLOADS["long_8192_d128_causal" if causal else "long_8192_d128"]
    q, k, v = w.make()
    do = synth.normal_bf16(w.seed + 7, 3, w.q_shape())
    dq, dk, dv = _gpu_grads(q, k, v, do, w.scale, causal)
    rows = sample_rows(w.B, w.H, w.Nq, 120, seed=840)
    dq_ref = backward.attention_bwd_dq_rows(q, k, v, do, rows, w.scale, causal)
    assert _err(dq.reshape(-1, w.d)[rows], dq_ref, dq_row_scales(q, k, v, do, rows, w.scale, causal)) <= TOL
    bh = 37
    keys = np.array([0, 1, 127, 128, 4000, 8190, 8191])
    dk_ref, dv_ref = backward.attention_bwd_dkdv_keys(q, k, v, do, bh, keys, w.scale, causal)
    mk, mv = dkdv_key_scales(q, k, v, do, bh, keys, w.scale, causal)
    assert _err(dk.reshape(-1, w.Nk, w.d)[bh][keys], dk_ref, mk) <= TOL
    assert _err(dv.reshape(-1, w.Nk, w.d)[bh][keys], dv_ref, mv) <= TOL


def test_bwd_stress_sampled_dq():
    """1 x 16 heads, N = 32000, Q ~ N(0, 4^2), causal: 250 K/V tiles per query tile wrap both rings
    many times; sampled dQ rows against the oracle (the oracle's dK/dV of a head costs a full
    N^2 d recomputation here, so dK and dV are checked for finiteness only)."""
    from parity_util import sample_rows

    w = synth.WORKLOADS["stress_32000_d128_causal"]
    q, k, v = w.make()
    do = synth.normal_bf16(w.seed + 7, 3, w.q_shape())
    dq, dk, dv = _gpu_grads(q, k, v, do, w.scale, True)
    rows = sample_rows(w.B, w.H, w.Nq, 48, seed=850)
    dq_ref = backward.attention_bwd_dq_rows(q, k, v, do, rows, w.scale, True)
    assert _err(dq.reshape(-1, w.d)[rows], dq_ref, dq_row_scales(q, k, v, do, rows, w.scale, True)) <= TOL
    assert np.all(np.isfinite(dk)) and np.all(np.isfinite(dv))


def test_bwd_binding_rejects_bad_gradient_buffers():
    import torch

    import exact_attention_19_gb300 as fa

    t = torch.zeros((1, 2, 130, 64), dtype=torch.bfloat16, device="cuda")
    o, lse = fa.fwd(t, t, t)
    with pytest.raises(ValueError):
        fa.bwd(t, t, t, o, lse, t, dq=torch.empty((1, 2, 129, 64), dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(ValueError):
        fa.bwd(t, t, t, o, lse, t, dk=torch.empty((1, 2, 130, 64), dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
