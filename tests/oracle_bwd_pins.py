"""Pins of the fp64 backward oracle: finite differences of the (pinned)
forward oracle, torch float64 autograd, closed forms and invariants.

Every pin takes a backward-oracle library handle (the real build, or a build
of a copy with one planted mistake)."""
from __future__ import annotations

import math

import numpy as np

import oracle
from oracle import backward


def _rng(seed):
    return np.random.default_rng(seed)


def _heads(*arrs):
    return [np.asarray(a, dtype=np.float64)[None, None] for a in arrs]


def pin_finite_differences(lib):
    """Central differences of L = sum(dO * O(q, k, v)), O from the forward oracle."""
    rng = _rng(41)
    h = 1e-6
    for (nq, nk, d, causal) in [(4, 4, 3, False), (5, 5, 2, True), (3, 6, 2, False), (1, 3, 1, False)]:
        q = rng.normal(size=(nq, d))
        k = rng.normal(size=(nk, d))
        v = rng.normal(size=(nk, d))
        do = rng.normal(size=(nq, d))
        scale = 0.7
        dq, dk, dv = backward.attention_bwd(*_heads(q, k, v, do), scale=scale, causal=causal, lib=lib)

        def loss(qq, kk, vv):
            o, _ = oracle.attention_fwd(*_heads(qq, kk, vv), scale=scale, causal=causal)
            return float(np.sum(o[0, 0] * do))

        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp = x.copy(); xp[idx] += h
                xm = x.copy(); xm[idx] -= h
                args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
                args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
                num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
            err = np.max(np.abs(num - g[0, 0]))
            assert err < 1e-7, (name, nq, nk, d, causal, err)


def pin_torch_autograd(lib):
    """Small shapes: torch float64 autograd of softmax(q k^T s) v gives the same gradients to 1e-12."""
    import torch

    gen = torch.Generator().manual_seed(3)
    for (B, H, nq, nk, d, causal) in [(1, 2, 6, 6, 4, True), (2, 1, 5, 9, 3, False), (1, 1, 17, 17, 8, True)]:
        q = torch.randn(B, H, nq, d, generator=gen, dtype=torch.float64, requires_grad=True)
        k = torch.randn(B, H, nk, d, generator=gen, dtype=torch.float64, requires_grad=True)
        v = torch.randn(B, H, nk, d, generator=gen, dtype=torch.float64, requires_grad=True)
        do = torch.randn(B, H, nq, d, generator=gen, dtype=torch.float64)
        s = (q @ k.transpose(-2, -1)) * 0.45
        if causal:
            s = s.masked_fill(torch.ones(nq, nk, dtype=torch.bool).triu(1), float("-inf"))
        o = torch.softmax(s, dim=-1) @ v
        o.backward(do)
        dq, dk, dv = backward.attention_bwd(q.detach().numpy(), k.detach().numpy(), v.detach().numpy(), do.numpy(),
                                            scale=0.45, causal=causal, lib=lib)
        for a, b in ((dq, q.grad), (dk, k.grad), (dv, v.grad)):
            assert np.max(np.abs(a - b.numpy())) < 1e-12


def pin_closed_forms(lib):
    rng = _rng(43)
    n, d = 7, 3
    q = rng.normal(size=(n, d))
    do = rng.normal(size=(n, d))
    # one key: P = 1 everywhere, so dV_0 = sum of dO rows and dQ = dK = 0
    k1 = rng.normal(size=(1, d))
    v1 = rng.normal(size=(1, d))
    dq, dk, dv = backward.attention_bwd(*_heads(q, k1, v1, do), scale=1.3, lib=lib)
    assert np.max(np.abs(dv[0, 0, 0] - do.sum(axis=0))) < 1e-13
    assert np.max(np.abs(dq)) < 1e-14 and np.max(np.abs(dk)) < 1e-14
    # all value rows equal: O is that row whatever P is, so dQ = dK = 0 and dV = P^T dO
    k = rng.normal(size=(n, d))
    vc = np.tile(rng.normal(size=(1, d)), (n, 1))
    for causal in (False, True):
        dq, dk, dv = backward.attention_bwd(*_heads(q, k, vc, do), scale=0.9, causal=causal, lib=lib)
        assert np.max(np.abs(dq)) < 1e-13 and np.max(np.abs(dk)) < 1e-13
        # and the dV columns add up to the dO columns (each P row sums to 1)
        assert np.max(np.abs(dv[0, 0].sum(axis=0) - do.sum(axis=0))) < 1e-12


def pin_invariants(lib):
    rng = _rng(44)
    B, H, nq, nk, d = 2, 2, 9, 11, 4
    q = rng.normal(size=(B, H, nq, d))
    k = rng.normal(size=(B, H, nk, d))
    v = rng.normal(size=(B, H, nk, d))
    do = rng.normal(size=(B, H, nq, d))
    dq, dk, dv = backward.attention_bwd(q, k, v, do, scale=0.6, lib=lib)
    # each dS row sums to 0 (softmax Jacobian), hence dK summed over keys is 0
    assert np.max(np.abs(dk.sum(axis=2))) < 1e-12
    # adding one vector u to every key shifts each row's logits by a constant:
    # P, dS, dV and dQ are unchanged (dQ because each dS row sums to 0)
    u = rng.normal(size=(1, 1, 1, d))
    dq2, dk2, dv2 = backward.attention_bwd(q, k + u, v, do, scale=0.6, lib=lib)
    assert np.max(np.abs(dq2 - dq)) < 1e-12 and np.max(np.abs(dv2 - dv)) < 1e-12
    assert np.max(np.abs(dk2 - dk)) < 1e-12
    # per-head independence and the selected-row / selected-key entry points
    for b in range(B):
        for hh in range(H):
            g1 = backward.attention_bwd(q[b, hh][None, None], k[b, hh][None, None], v[b, hh][None, None],
                                        do[b, hh][None, None], scale=0.6, lib=lib)
            for x, y in zip(g1, (dq, dk, dv)):
                assert np.max(np.abs(x[0, 0] - y[b, hh])) < 1e-13
    rows = np.array([0, 5, 17, B * H * nq - 1])
    dqr = backward.attention_bwd_dq_rows(q, k, v, do, rows, scale=0.6, lib=lib)
    assert np.max(np.abs(dqr - dq.reshape(-1, d)[rows])) < 1e-13
    keys = np.array([0, 3, nk - 1])
    dkr, dvr = backward.attention_bwd_dkdv_keys(q, k, v, do, 3, keys, scale=0.6, lib=lib)
    assert np.max(np.abs(dkr - dk[1, 1][keys])) < 1e-13 and np.max(np.abs(dvr - dv[1, 1][keys])) < 1e-13


def pin_causal_structure(lib):
    """Under the causal mask query i never touches key j > i: the last key's dK and dV
    come from the last query alone, and the first query's dQ involves key 0 only."""
    rng = _rng(45)
    n, d = 8, 3
    q, k, v, do = (rng.normal(size=(n, d)) for _ in range(4))
    dq, dk, dv = backward.attention_bwd(*_heads(q, k, v, do), scale=0.8, causal=True, lib=lib)
    # row 0 sees only key 0: P = 1, dS = 0 -> dQ_0 = 0
    assert np.max(np.abs(dq[0, 0, 0])) < 1e-14
    # key n-1 is seen by row n-1 only
    o, lse = oracle.attention_fwd(*_heads(q, k, v), scale=0.8, causal=True)
    p_last = math.exp(0.8 * float(q[-1] @ k[-1]) - lse[0, 0, -1])
    assert np.max(np.abs(dv[0, 0, -1] - p_last * do[-1])) < 1e-13
    # selected keys agree with the full computation under the mask too
    dkr, dvr = backward.attention_bwd_dkdv_keys(*_heads(q, k, v, do), 0, np.arange(n), scale=0.8, causal=True,
                                                lib=lib)
    assert np.max(np.abs(dkr - dk[0, 0])) < 1e-13 and np.max(np.abs(dvr - dv[0, 0])) < 1e-13


BWD_PINS = [pin_finite_differences, pin_torch_autograd, pin_closed_forms, pin_invariants, pin_causal_structure]


def _window_keep(nq, nk, wl, wr):
    """Keep-matrix of a bottom-right window, by enumeration of every (row, key)."""
    keep = np.zeros((nq, nk), dtype=bool)
    for i in range(nq):
        for j in range(nk):
            d_ij = j - (i + nk - nq)  # key offset from the row's diagonal
            keep[i, j] = (wl < 0 or d_ij >= -wl) and (wr < 0 or d_ij <= wr)
    return keep


WINDOW_CASES = [(5, 5, 2, (1, 0)), (4, 7, 2, (2, 1)), (6, 3, 2, (0, 1)), (5, 5, 2, (-1, 1)), (3, 6, 1, (-1, 0)),
                (6, 4, 2, (1, -1)), (7, 2, 3, (0, 0))]


def pin_window_finite_differences(lib):
    """Windowed gradients against central differences of L = sum(dO * O), O from the
    (separately pinned) windowed forward oracle; includes Nq > Nk windows whose
    first rows keep no key (their O is 0 whatever the inputs, so every gradient
    through them is 0)."""
    rng = _rng(46)
    h = 1e-6
    for (nq, nk, d, win) in WINDOW_CASES:
        q = rng.normal(size=(nq, d))
        k = rng.normal(size=(nk, d))
        v = rng.normal(size=(nk, d))
        do = rng.normal(size=(nq, d))
        scale = 0.8
        dq, dk, dv = backward.attention_bwd(*_heads(q, k, v, do), scale=scale, window=win, lib=lib)

        def loss(qq, kk, vv):
            o, _ = oracle.attention_fwd(*_heads(qq, kk, vv), scale=scale, window=win)
            return float(np.sum(o[0, 0] * do))

        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp = x.copy(); xp[idx] += h
                xm = x.copy(); xm[idx] -= h
                args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
                args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
                num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
            err = np.max(np.abs(num - g[0, 0]))
            assert err < 1e-7, (name, nq, nk, d, win, err)


def pin_window_autograd(lib):
    """torch float64 autograd through a masked softmax whose keep-matrix is built by
    enumerating every (row, key) pair; rows that keep no key are left out of the
    softmax (O = 0 there)."""
    import torch

    gen = torch.Generator().manual_seed(4)
    for (B, H, nq, nk, d, win) in [(1, 2, 9, 9, 4, (3, 0)), (2, 1, 6, 11, 3, (2, 2)), (1, 1, 12, 5, 5, (1, 1)),
                                   (1, 1, 17, 17, 8, (-1, 0)), (1, 2, 8, 13, 4, (-1, 0))]:
        keep = torch.from_numpy(_window_keep(nq, nk, *win))
        q = torch.randn(B, H, nq, d, generator=gen, dtype=torch.float64, requires_grad=True)
        k = torch.randn(B, H, nk, d, generator=gen, dtype=torch.float64, requires_grad=True)
        v = torch.randn(B, H, nk, d, generator=gen, dtype=torch.float64, requires_grad=True)
        do = torch.randn(B, H, nq, d, generator=gen, dtype=torch.float64)
        s = ((q @ k.transpose(-2, -1)) * 0.5).masked_fill(~keep, float("-inf"))
        live = keep.any(dim=1)
        p = torch.softmax(s[..., live, :], dim=-1)
        o = torch.zeros(B, H, nq, d, dtype=torch.float64)
        o[..., live, :] = p @ v
        o.backward(do)
        dq, dk, dv = backward.attention_bwd(q.detach().numpy(), k.detach().numpy(), v.detach().numpy(), do.numpy(),
                                            scale=0.5, window=win, lib=lib)
        for a, b in ((dq, q.grad), (dk, k.grad), (dv, v.grad)):
            assert np.max(np.abs(a - b.numpy())) < 1e-12, win


def pin_window_reductions(lib):
    """A window wider than the keys is no mask; (-1, 0) with Nq = Nk is the causal
    mask; the selected-row and selected-key entry points agree with the full
    windowed computation."""
    rng = _rng(47)
    B, H, n, d = 1, 2, 10, 3
    q, k, v, do = (rng.normal(size=(B, H, n, d)) for _ in range(4))
    full = backward.attention_bwd(q, k, v, do, scale=0.7, lib=lib)
    wide = backward.attention_bwd(q, k, v, do, scale=0.7, window=(n, n), lib=lib)
    causal = backward.attention_bwd(q, k, v, do, scale=0.7, causal=True, lib=lib)
    bottom = backward.attention_bwd(q, k, v, do, scale=0.7, window=(-1, 0), lib=lib)
    for a, b in zip(full, wide):
        assert np.array_equal(a, b)
    for a, b in zip(causal, bottom):
        assert np.array_equal(a, b)
    nq, nk = 9, 5
    q = rng.normal(size=(B, H, nq, d))
    do = rng.normal(size=(B, H, nq, d))
    k = rng.normal(size=(B, H, nk, d))
    v = rng.normal(size=(B, H, nk, d))
    win = (1, 0)
    dq, dk, dv = backward.attention_bwd(q, k, v, do, scale=0.7, window=win, lib=lib)
    # rows 0 .. nq - nk - 2 keep no key: their dQ is exactly 0
    assert np.all(dq[:, :, : nq - nk - 1] == 0.0)
    rows = np.array([0, 3, 4, 8, nq + 5, 2 * nq - 1])
    dqr = backward.attention_bwd_dq_rows(q, k, v, do, rows, scale=0.7, window=win, lib=lib)
    assert np.max(np.abs(dqr - dq.reshape(-1, d)[rows])) < 1e-13
    keys = np.arange(nk)
    dkr, dvr = backward.attention_bwd_dkdv_keys(q, k, v, do, 1, keys, scale=0.7, window=win, lib=lib)
    assert np.max(np.abs(dkr - dk[0, 1])) < 1e-13 and np.max(np.abs(dvr - dv[0, 1])) < 1e-13


BWD_PINS += [pin_window_finite_differences, pin_window_autograd, pin_window_reductions]
