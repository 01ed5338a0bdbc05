"""Pins of the fp64 oracle to values fixed by the pages and by mathematics.

Every pin takes an oracle library handle (the normal build, or a build of a
deliberately broken copy of the C source) and raises AssertionError when the
oracle disagrees.  ``test_oracle.py`` runs them against the real oracle;
``test_oracle_mutants.py`` checks that each planted mistake trips one.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle
from oracle.online import RowTrace, online_row, tiled_attention

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def _one_head(q, k, v):
    """[N, d] arrays -> [1, 1, N, d]."""
    return _f64(q)[None, None], _f64(k)[None, None], _f64(v)[None, None]


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------------------
# printed worked examples
# ---------------------------------------------------------------------------
def pin_worked_row(lib):
    """lumenova section 03: scores [1,2,0,3], values, tile 2 -> [0.795176, 2.200684].

    The row is encoded as attention with d = 2, scale = 1: q = [1, 0] and
    k_j = [s_j, 0], so that q.k_j = s_j exactly.
    """
    g = golden("worked_row_tile2.json")
    s = g["scores"]
    q = [[1.0, 0.0]]
    k = [[x, 0.0] for x in s]
    o, lse = oracle.attention_fwd(*_one_head(q, k, g["values"]), scale=1.0, lib=lib)
    half = 0.5 * 10.0 ** (-g["printed_decimals"])
    assert np.max(np.abs(o[0, 0, 0] - g["result"])) <= half + 1e-12, o[0, 0, 0]
    assert abs(lse[0, 0, 0] - g["lse_closed_form"]["value"]) < 1e-13, lse[0, 0, 0]


def pin_worked_row_tiled_state(lib):
    """Same row by the tiled recurrence: state after block 1 and the final row."""
    g = golden("worked_row_tile2.json")
    tr = RowTrace()
    o, lse = online_row(g["scores"], g["values"], g["tile"], trace=tr)
    half = 0.5 * 10.0 ** (-g["printed_decimals"])
    b1 = g["after_block_1"]
    assert tr.m[0] == b1["m"]
    assert abs(tr.l[0] - b1["l"]) <= half
    assert np.max(np.abs(np.array(tr.acc[0]) - b1["acc"])) <= half
    assert np.max(np.abs(np.array(o) - g["result"])) <= half
    # the page's own check: tiled equals one-shot within 1e-12
    q = [[1.0, 0.0]]
    k = [[x, 0.0] for x in g["scores"]]
    o_ref, lse_ref = oracle.attention_fwd(*_one_head(q, k, g["values"]), scale=1.0, lib=lib)
    assert np.max(np.abs(np.array(o) - o_ref[0, 0, 0])) < g["page_tolerance_vs_one_shot"]
    assert abs(lse - lse_ref[0, 0, 0]) < 1e-12


def pin_softmax_vectors(lib):
    """jianzhnie A.4: softmax of two printed vectors, the second near 1000.

    Attention with q = e_0, k_j = x_j e_0, V = identity and scale 1 returns
    softmax(x) as its output row.
    """
    g = golden("softmax_vectors.json")
    tol = 0.5 * 10.0 ** (-g["printed_decimals"]) + 1e-12
    for case in g["cases"]:
        x = case["x"]
        n = len(x)
        q = np.zeros((1, n))
        q[0, 0] = 1.0
        k = np.zeros((n, n))
        k[:, 0] = x
        o, lse = oracle.attention_fwd(*_one_head(q, k, np.eye(n)), scale=1.0, lib=lib)
        assert np.all(np.isfinite(o)), o
        assert np.max(np.abs(o[0, 0, 0] - case["softmax"])) <= tol, (o[0, 0, 0], case["softmax"])


def pin_single_row_attention(lib):
    """jianzhnie A.5: one query row, K 4x3, V 4x2 (padded to d = 3 with zeros)."""
    g = golden("single_row_attention.json")
    V = np.zeros((4, 3))
    V[:, :2] = g["V"]
    o, lse = oracle.attention_fwd(*_one_head([g["q"]], g["K"], V), scale=1.0, lib=lib)
    tol = 0.5 * 10.0 ** (-g["printed_decimals"]) + 1e-12
    assert np.max(np.abs(o[0, 0, 0, :2] - g["result"])) <= tol, o[0, 0, 0]
    assert o[0, 0, 0, 2] == 0.0
    assert abs(lse[0, 0, 0] - g["lse_closed_form"]["value"]) < 1e-13


def pin_alpha_update(lib):
    """llm-infra-atlas section 2: m = 3, l = 10, new block max 5 -> alpha ~ 0.135, l -> 1.35 + rowsum.

    Built as a row whose first block is ten scores of 3 (so m = 3 and l = 10)
    and whose second block is the single score 5.
    """
    g = golden("alpha_update.json")
    scores = [3.0] * 10 + [5.0]
    values = [[1.0]] * 11
    tr = RowTrace()
    o, lse = online_row(scores, values, tile=10, trace=tr)
    assert tr.m[0] == g["m_old"] and abs(tr.l[0] - g["l_old"]) < 1e-12
    assert tr.m[1] == g["block_max"]
    assert round(tr.alpha[1], g["alpha_decimals"]) == g["alpha"]
    l_scaled = tr.l[1] - 1.0  # the new block's row sum is exp(5 - 5) = 1
    assert round(l_scaled, g["l_scaled_decimals"]) == g["l_scaled"]
    assert all(a <= 1.0 for a in tr.alpha)
    # and the one-shot oracle agrees with the recurrence on this row
    q = [[1.0]]
    k = [[s] for s in scores]
    o_ref, lse_ref = oracle.attention_fwd(*_one_head(q, k, values), scale=1.0, lib=lib)
    assert abs(lse - lse_ref[0, 0, 0]) < 1e-12


# ---------------------------------------------------------------------------
# tiled recurrence == one-shot definition
# ---------------------------------------------------------------------------
def pin_tiled_equals_one_shot(lib):
    """Tiled online recurrence (all tile sizes, plain and conditional rescale) == oracle to 1e-12."""
    rng = _rng(11)
    for (n, d, causal, sq) in [(1, 3, False, 1.0), (5, 3, True, 1.0), (63, 16, False, 4.0),
                               (130, 64, True, 4.0), (257, 8, False, 1.0)]:
        q = rng.normal(0.0, sq, (n, d))
        k = rng.normal(0.0, 1.0, (n, d))
        v = rng.normal(0.0, 1.0, (n, d))
        scale = 1.0 / math.sqrt(d)
        o_ref, lse_ref = oracle.attention_fwd(*_one_head(q, k, v), scale=scale, causal=causal, lib=lib)
        for tile in (1, 2, 3, 64, 128):
            for tau in (None, 8.0):
                o, lse, _ = tiled_attention(q, k, v, scale, causal, tile, tau)
                assert np.max(np.abs(o - o_ref[0, 0])) < 1e-12, (n, d, tile, tau)
                assert np.max(np.abs(lse - lse_ref[0, 0])) < 1e-12, (n, d, tile, tau)


def pin_lazy_rescale_is_lazy(lib):
    """With tau = 8 (base 2) the recurrence rescales less often, and still matches."""
    rng = _rng(5)
    n, d = 512, 32
    q = rng.normal(0.0, 4.0, (n, d))
    k = rng.normal(0.0, 1.0, (n, d))
    v = rng.normal(0.0, 1.0, (n, d))
    scale = 1.0 / math.sqrt(d)
    o_ref, lse_ref = oracle.attention_fwd(*_one_head(q, k, v), scale=scale, lib=lib)
    o0, l0, moves_eager = tiled_attention(q, k, v, scale, False, 16, None)
    o1, l1, moves_lazy = tiled_attention(q, k, v, scale, False, 16, 8.0)
    assert moves_lazy < moves_eager
    assert np.max(np.abs(o1 - o_ref[0, 0])) < 1e-12 and np.max(np.abs(l1 - lse_ref[0, 0])) < 1e-12


# ---------------------------------------------------------------------------
# invariants and closed forms
# ---------------------------------------------------------------------------
def pin_normalisation(lib):
    """sum_j exp(s_j - LSE) = 1 for every row (P rows sum to 1), with s from a library matmul."""
    rng = _rng(3)
    for causal in (False, True):
        n, d = 40, 8
        q = rng.normal(0.0, 3.0, (n, d))
        k = rng.normal(0.0, 1.0, (n, d))
        v = rng.normal(0.0, 1.0, (n, d))
        scale = 0.37
        _, lse = oracle.attention_fwd(*_one_head(q, k, v), scale=scale, causal=causal, lib=lib)
        s = (q @ k.T) * scale
        for i in range(n):
            keys = range(i + 1) if causal else range(n)
            tot = sum(math.exp(s[i, j] - lse[0, 0, i]) for j in keys)
            assert abs(tot - 1.0) < 1e-12, (causal, i, tot)


def pin_closed_forms(lib):
    rng = _rng(7)
    # Nk = 1: O = V[0] and LSE = scale * q.k_0
    q = np.array([[1.0, 2.0, -1.0]])
    k = np.array([[0.5, -1.0, 2.0]])
    v = np.array([[3.0, -4.0, 0.25]])
    o, lse = oracle.attention_fwd(*_one_head(q, k, v), scale=0.5, lib=lib)
    assert np.array_equal(o[0, 0, 0], v[0])
    assert lse[0, 0, 0] == 0.5 * (0.5 - 2.0 - 2.0)
    # K = 0: uniform weights. O = mean of visible V rows, LSE = ln(count)
    n, d = 9, 4
    q = rng.normal(size=(n, d))
    v = rng.normal(size=(n, d))
    for causal in (False, True):
        o, lse = oracle.attention_fwd(*_one_head(q, np.zeros((n, d)), v), scale=0.3, causal=causal,
                                      lib=lib)
        for i in range(n):
            cnt = i + 1 if causal else n
            assert np.max(np.abs(o[0, 0, i] - v[:cnt].mean(axis=0))) < 1e-14
            assert abs(lse[0, 0, i] - math.log(cnt)) < 1e-14
    # V = 1: O = 1 everywhere
    k = rng.normal(size=(n, d))
    o, _ = oracle.attention_fwd(*_one_head(q, k, np.ones((n, d))), scale=1.0, causal=True, lib=lib)
    assert np.max(np.abs(o - 1.0)) < 1e-14


def pin_shift_invariance(lib):
    """Adding c to every logit of a row leaves O unchanged and moves LSE by c.

    Realised with one extra dimension: q gets a column of 1, k a column of
    c / scale (jianzhnie section 4.3: softmax is shift invariant).
    """
    rng = _rng(9)
    n, d = 17, 6
    q = rng.normal(size=(n, d))
    k = rng.normal(size=(n, d))
    v = rng.normal(size=(n, d))
    scale, c = 0.25, 700.0
    qa = np.concatenate([q, np.ones((n, 1))], axis=1)
    ka0 = np.concatenate([k, np.zeros((n, 1))], axis=1)
    ka1 = np.concatenate([k, np.full((n, 1), c / scale)], axis=1)
    va = np.concatenate([v, np.zeros((n, 1))], axis=1)
    for causal in (False, True):
        o0, l0 = oracle.attention_fwd(*_one_head(qa, ka0, va), scale=scale, causal=causal, lib=lib)
        o1, l1 = oracle.attention_fwd(*_one_head(qa, ka1, va), scale=scale, causal=causal, lib=lib)
        assert np.max(np.abs(o0 - o1)) < 1e-12
        assert np.max(np.abs((l1 - l0) - c)) < 1e-9


def pin_permutation_invariance(lib):
    """Non-causal: permuting the K and V rows together leaves O and LSE unchanged."""
    rng = _rng(13)
    n, d = 23, 5
    q = rng.normal(size=(n, d))
    k = rng.normal(size=(n, d))
    v = rng.normal(size=(n, d))
    perm = rng.permutation(n)
    o0, l0 = oracle.attention_fwd(*_one_head(q, k, v), scale=0.5, lib=lib)
    o1, l1 = oracle.attention_fwd(*_one_head(q, k[perm], v[perm]), scale=0.5, lib=lib)
    assert np.max(np.abs(o0 - o1)) < 1e-13 and np.max(np.abs(l0 - l1)) < 1e-13


def pin_batch_head_layout(lib):
    """[B, H, N, d] indexing: every (b, h) equals the same head computed alone."""
    rng = _rng(17)
    B, H, Nq, Nk, d = 2, 3, 7, 11, 4
    q = rng.normal(size=(B, H, Nq, d))
    k = rng.normal(size=(B, H, Nk, d))
    v = rng.normal(size=(B, H, Nk, d))
    o, lse = oracle.attention_fwd(q, k, v, scale=0.7, lib=lib)
    for b in range(B):
        for h in range(H):
            oh, lh = oracle.attention_fwd(q[b, h][None, None], k[b, h][None, None],
                                          v[b, h][None, None], scale=0.7, lib=lib)
            assert np.array_equal(o[b, h], oh[0, 0]) and np.array_equal(lse[b, h], lh[0, 0])
    rows = np.array([0, 5, 13, 40, B * H * Nq - 1])
    orow, lrow = oracle.attention_rows(q, k, v, rows, scale=0.7, lib=lib)
    assert np.array_equal(orow, o.reshape(-1, d)[rows]) and np.array_equal(lrow, lse.reshape(-1)[rows])


# ---------------------------------------------------------------------------
# library special cases and brute force
# ---------------------------------------------------------------------------
def pin_torch_softmax(lib):
    """Tiny shapes: torch.softmax in float64 then @ V gives the same O to 1e-12."""
    import torch

    g = torch.Generator().manual_seed(0)
    for (n, m, d, causal) in [(4, 4, 3, False), (6, 6, 5, True), (3, 9, 2, False)]:
        q = torch.randn(n, d, generator=g, dtype=torch.float64)
        k = torch.randn(m, d, generator=g, dtype=torch.float64)
        v = torch.randn(m, d, generator=g, dtype=torch.float64)
        s = (q @ k.T) * 0.8
        if causal:
            s = s.masked_fill(torch.ones(n, m, dtype=torch.bool).triu(1), float("-inf"))
        ref = torch.softmax(s, dim=-1) @ v
        lse_ref = torch.logsumexp(s, dim=-1)
        o, lse = oracle.attention_fwd(*_one_head(q.numpy(), k.numpy(), v.numpy()), scale=0.8,
                                      causal=causal, lib=lib)
        assert np.max(np.abs(o[0, 0] - ref.numpy())) < 1e-12
        assert np.max(np.abs(lse[0, 0] - lse_ref.numpy())) < 1e-12


def pin_sim_cases(lib):
    """datawhalechina step 5: three seeded cases vs a float32 softmax reference, bound 1e-5."""
    import torch

    g = golden("sim_cases.json")
    for case in g["cases"]:
        torch.manual_seed(case["seed"])
        n, d = case["seq_len"], case["dim"]
        q = torch.randn(n, d)
        k = torch.randn(n, d)
        v = torch.randn(n, d)
        scale = 1.0 / math.sqrt(d)
        ref = torch.softmax((q @ k.transpose(-2, -1)) * scale, dim=-1) @ v
        o, _ = oracle.attention_fwd(*_one_head(q.double().numpy(), k.double().numpy(),
                                               v.double().numpy()), scale=scale, lib=lib)
        assert np.max(np.abs(o[0, 0] - ref.double().numpy())) < g["max_abs_error"], case
        # the tiled recurrence with the page's block size reaches the same
        o_t, _, _ = tiled_attention(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                    scale, False, case["block_size"])
        assert np.max(np.abs(o_t - o[0, 0])) < 1e-12


def _brute(q, k, v, scale, causal):
    """Direct double loop, plain exp / sum without max subtraction (small logits only)."""
    n, d = len(q), len(q[0])
    m = len(k)
    o = [[0.0] * d for _ in range(n)]
    lse = [0.0] * n
    for i in range(n):
        keys = [j for j in range(m) if (not causal) or j <= i]
        w = []
        for j in keys:
            s = 0.0
            for c in range(d):
                s += q[i][c] * k[j][c]
            w.append(math.exp(scale * s))
        z = sum(w)
        for c in range(d):
            o[i][c] = sum(wj * v[j][c] for wj, j in zip(w, keys)) / z
        lse[i] = math.log(z)
    return o, lse


def pin_brute_force(lib):
    rng = _rng(21)
    for n in range(1, 9):
        for d in (1, 2, 4):
            for causal in (False, True):
                q = rng.normal(size=(n, d))
                k = rng.normal(size=(n, d))
                v = rng.normal(size=(n, d))
                ob, lb = _brute(q.tolist(), k.tolist(), v.tolist(), 0.9, causal)
                o, lse = oracle.attention_fwd(*_one_head(q, k, v), scale=0.9, causal=causal, lib=lib)
                assert np.max(np.abs(o[0, 0] - np.array(ob))) < 1e-12, (n, d, causal)
                assert np.max(np.abs(lse[0, 0] - np.array(lb))) < 1e-12, (n, d, causal)
    # rectangular, non-causal
    q = rng.normal(size=(3, 2))
    k = rng.normal(size=(7, 2))
    v = rng.normal(size=(7, 2))
    ob, lb = _brute(q.tolist(), k.tolist(), v.tolist(), 1.3, False)
    o, lse = oracle.attention_fwd(*_one_head(q, k, v), scale=1.3, lib=lib)
    assert np.max(np.abs(o[0, 0] - np.array(ob))) < 1e-12


def pin_bf16_inputs(lib):
    """bf16-bit inputs are widened exactly: same result as the float64 of the same values."""
    import synth

    q = synth.normal_bf16(1, 0, (1, 2, 33, 8))
    k = synth.normal_bf16(1, 1, (1, 2, 40, 8))
    v = synth.normal_bf16(1, 2, (1, 2, 40, 8))
    wide = [synth.bf16_to_f32(x).astype(np.float64) for x in (q, k, v)]
    o0, l0 = oracle.attention_fwd(q, k, v, scale=0.35, lib=lib)
    o1, l1 = oracle.attention_fwd(*wide, scale=0.35, lib=lib)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


PINS = [
    pin_worked_row, pin_worked_row_tiled_state, pin_softmax_vectors, pin_single_row_attention,
    pin_alpha_update, pin_tiled_equals_one_shot, pin_lazy_rescale_is_lazy, pin_normalisation,
    pin_closed_forms, pin_shift_invariance, pin_permutation_invariance, pin_batch_head_layout,
    pin_torch_softmax, pin_sim_cases, pin_brute_force, pin_bf16_inputs,
]


# ---------------------------------------------------------------------------
# window masks (bottom-right aligned sliding window; causal = (-1, 0))
# ---------------------------------------------------------------------------
def _brute_window(q, k, v, scale, wl, wr):
    """Direct loop: key j kept for row i iff i+s-wl <= j <= i+s+wr, s = Nk - Nq."""
    nq, nk, d = len(q), len(k), len(q[0])
    s = nk - nq
    o = [[0.0] * d for _ in range(nq)]
    lse = [0.0] * nq
    for i in range(nq):
        keys = [j for j in range(nk) if (wl < 0 or j >= i + s - wl) and (wr < 0 or j <= i + s + wr)]
        if not keys:
            lse[i] = -math.inf
            continue
        w = [math.exp(scale * sum(q[i][c] * k[j][c] for c in range(d))) for j in keys]
        z = sum(w)
        for c in range(d):
            o[i][c] = sum(wj * v[j][c] for wj, j in zip(w, keys)) / z
        lse[i] = math.log(z)
    return o, lse


def pin_window_brute_force(lib):
    rng = _rng(31)
    for (nq, nk) in [(5, 5), (3, 8), (8, 3), (1, 6), (7, 1)]:
        for (wl, wr) in [(-1, 0), (0, 0), (2, 1), (1, -1), (-1, -1), (0, 3), (4, 0)]:
            q = rng.normal(size=(nq, 3))
            k = rng.normal(size=(nk, 3))
            v = rng.normal(size=(nk, 3))
            ob, lb = _brute_window(q.tolist(), k.tolist(), v.tolist(), 0.8, wl, wr)
            o, lse = oracle.attention_fwd(*_one_head(q, k, v), scale=0.8, window=(wl, wr), lib=lib)
            lb = np.array(lb)
            fin = np.isfinite(lb)
            assert np.array_equal(np.isfinite(lse[0, 0]), fin), (nq, nk, wl, wr)
            assert np.max(np.abs(lse[0, 0][fin] - lb[fin]), initial=0.0) < 1e-12, (nq, nk, wl, wr)
            assert np.max(np.abs(o[0, 0] - np.array(ob))) < 1e-12, (nq, nk, wl, wr)
            # rows without a visible key: O = 0 exactly
            assert np.all(o[0, 0][~fin] == 0.0)


def pin_window_special_cases(lib):
    rng = _rng(32)
    n, d = 20, 4
    q = rng.normal(size=(n, d))
    k = rng.normal(size=(n, d))
    v = rng.normal(size=(n, d))
    # unbounded on both sides = no mask; (-1, 0) with Nq = Nk = causal
    o0, l0 = oracle.attention_fwd(*_one_head(q, k, v), scale=0.5, lib=lib)
    o1, l1 = oracle.attention_fwd(*_one_head(q, k, v), scale=0.5, window=(-1, -1), lib=lib)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
    o0, l0 = oracle.attention_fwd(*_one_head(q, k, v), scale=0.5, causal=True, lib=lib)
    o1, l1 = oracle.attention_fwd(*_one_head(q, k, v), scale=0.5, window=(-1, 0), lib=lib)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
    # K = 0 under a window: uniform weights over the visible keys
    nq, nk, wl, wr = 6, 10, 2, 1
    qz = rng.normal(size=(nq, d))
    vz = rng.normal(size=(nk, d))
    o, lse = oracle.attention_fwd(*_one_head(qz, np.zeros((nk, d)), vz), scale=1.0, window=(wl, wr), lib=lib)
    for i in range(nq):
        lo = max(0, i + (nk - nq) - wl)
        hi = min(nk - 1, i + (nk - nq) + wr)
        assert abs(lse[0, 0, i] - math.log(hi - lo + 1)) < 1e-14
        assert np.max(np.abs(o[0, 0, i] - vz[lo:hi + 1].mean(axis=0))) < 1e-14
    # selected-rows entry agrees with the all-rows entry
    rows = np.array([0, 3, 5])
    orow, lrow = oracle.attention_rows(*_one_head(qz, np.zeros((nk, d)), vz), rows, scale=1.0, window=(wl, wr),
                                       lib=lib)
    assert np.array_equal(orow, o.reshape(-1, d)[rows]) and np.array_equal(lrow, lse.reshape(-1)[rows])


PINS += [pin_window_brute_force, pin_window_special_cases]
