"""CPU checks of the parity bars' helpers: the forward O bar (parity_util.o_tol)
and the backward row scales (grad_scale), neither of which is an expected
value; the expected values come from the oracles."""
import numpy as np
import pytest

import synth
from grad_scale import dkdv_key_scales, dq_row_scales, keep_matrix, row_scales
from parity_util import o_tol


def test_o_tol_values():
    # absolute 1e-2 below |O| = 1; 1e-2 + half the bf16 spacing above it (capped by 1e-2 * |O|)
    x = np.array([0.0, 0.5, -0.99, 1.0, 1.5, 3.0, -3.0, 6.0, 100.0])
    want = np.array([1e-2, 1e-2, 1e-2, 1e-2, min(1.5e-2, 1e-2 + 2 ** -8), 1e-2 + 2 ** -7, 1e-2 + 2 ** -7,
                     1e-2 + 2 ** -6, 1e-2 + 2 ** -2])
    assert np.allclose(o_tol(x), want, rtol=0, atol=1e-15)


def test_o_tol_half_spacing_is_the_bf16_spacing():
    """u/2 in the bar is half the distance from a bf16 number to its upper neighbour."""
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(2000) * np.exp2(rng.integers(-6, 8, 2000))).astype(np.float32)
    bits = synth.f32_to_bf16_bits(x)
    xb = synth.bf16_to_f32(bits).astype(np.float64)
    up = synth.bf16_to_f32((bits & 0x8000) | ((bits & 0x7FFF) + 1)).astype(np.float64)
    half_spacing = np.abs(up - xb) / 2
    # o_tol - 1e-2 is u/2 wherever the 1e-2 * |O| cap does not bind (|O| >= 1.4)
    sel = np.abs(xb) >= 1.4
    assert np.allclose(o_tol(xb[sel]) - 1e-2, half_spacing[sel], rtol=1e-12, atol=0)


def _case(seed, nq=70, nk=90, d=16, window=None, causal=False):
    w = synth.Workload("gs", 2, 2, nq, nk, d, causal, seed=seed)
    q, k, v = w.make()
    do = synth.normal_bf16(seed + 7, 3, w.q_shape())
    return w, q, k, v, do


@pytest.mark.parametrize("causal,window", [(False, None), (True, None), (False, (10, 0)), (False, (0, 3))])
def test_row_scale_bounds_the_gradient(causal, window):
    """Triangle inequality: every gradient entry is at most the magnitude sum M_rc <= M_r."""
    from oracle import backward

    backward.build()
    n = 80 if causal else None
    w, q, k, v, do = _case(5, nq=n or 70, nk=n or 90, causal=causal, window=window)
    refs = backward.attention_bwd(q, k, v, do, w.scale, causal, window=window)
    scales = row_scales(q, k, v, do, w.scale, causal, window)
    for ref, m in zip(refs, scales):
        assert np.all(np.max(np.abs(ref), axis=-1) <= m * (1 + 1e-12))
        assert np.all(m >= 0)


def test_row_scale_zero_exactly_where_nothing_is_kept():
    w, q, k, v, do = _case(6, nq=40, nk=200, window=(0, 0))
    mq, mk, mv = row_scales(q, k, v, do, w.scale, window=(0, 0))
    keep = keep_matrix(40, 200, window=(0, 0))
    assert np.array_equal(mq[0, 0] == 0, ~keep.any(axis=1))
    assert np.array_equal(mk[0, 0] == 0, ~keep.any(axis=0))
    assert np.array_equal(mv[0, 0] == 0, ~keep.any(axis=0))


def test_row_scale_does_not_vanish_where_the_gradient_cancels():
    """One key per query: dQ is exactly zero, its terms are not."""
    w, q, k, v, do = _case(7, nq=50, nk=1)
    mq, _, _ = row_scales(q, k, v, do, w.scale)
    assert np.all(mq > 0)


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_scales_match_whole_heads(causal):
    w, q, k, v, do = _case(8, nq=300, nk=300, causal=causal)
    mq, mk, mv = row_scales(q, k, v, do, w.scale, causal)
    rows = np.array([0, 1, 129, 299, 300, 777, 1199])
    assert np.allclose(dq_row_scales(q, k, v, do, rows, w.scale, causal), mq.reshape(-1)[rows], rtol=1e-12)
    keys = np.array([0, 5, 128, 299])
    bh = 3
    sk, sv = dkdv_key_scales(q, k, v, do, bh, keys, w.scale, causal, chunk=64)
    assert np.allclose(sk, mk.reshape(-1, 300)[bh][keys], rtol=1e-12)
    assert np.allclose(sv, mv.reshape(-1, 300)[bh][keys], rtol=1e-12)
