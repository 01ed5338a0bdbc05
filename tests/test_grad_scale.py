"""CPU checks of the backward parity bar's row scales (grad_scale), which are
not expected values; the expected values come from the backward oracle."""
import numpy as np
import pytest

import synth
from grad_scale import dkdv_key_scales, dq_row_scales, keep_matrix, row_scales


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
