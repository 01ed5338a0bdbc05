"""Per-row size of the sums that define each backward gradient entry, for the
backward parity bar (test infrastructure; no expected value comes from here,
the expected gradients are the fp64 backward oracle's).

With P = softmax(scale * Q K^T) under the mask, dP = dO V^T and
D_i = sum_c dO_ic O_ic, the gradients are sums of products
(page "llm-infra-atlas / FlashAttention 01", section 5):

    dV_jc = sum_i P_ij dO_ic
    dQ_ic = scale * sum_j P_ij (dP_ij - D_i) K_jc
    dK_jc = scale * sum_i P_ij (dP_ij - D_i) Q_ic

The CUDA path rounds P and dS = P (dP - D) to bf16 before their products,
takes D from the forward's bf16 O, and returns the gradients in bf16; each
rounding is relative to the term it rounds.  The error of an entry is
therefore bounded by a small multiple of 2^-9 times the same sum taken over
the magnitudes of its terms, with |D_i| replaced by E_i = sum_c |dO_ic O_ic|
(the size of the terms D is summed from):

    M^dV_jc = sum_i P_ij |dO_ic|
    M^dQ_ic = scale * sum_j P_ij (|dP_ij| + E_i) |K_jc|
    M^dK_jc = scale * sum_i P_ij (|dP_ij| + E_i) |Q_ic|

An entry can be far smaller than its M (its terms cancel, e.g. a query that
sees one key has dQ = 0 exactly), so the bar's absolute part is set per row
of dQ, per key of dK and dV: M_r = max_c M_rc.  This module computes M_r in
fp64 with numpy, for whole heads or for selected rows and keys.
"""
from __future__ import annotations

import numpy as np

import synth


def _f64(x):
    return synth.bf16_to_f32(x).astype(np.float64) if x.dtype == np.uint16 else np.asarray(x, dtype=np.float64)


def keep_matrix(nq, nk, causal=False, window=None, rows=None):
    """Boolean [len(rows) or nq, nk]: key j is kept for query row i.  Causal is
    top-left (j <= i, Nq == Nk); a window (wl, wr) is bottom-right:
    i + (nk - nq) - wl <= j <= i + (nk - nq) + wr, a negative bound open."""
    i = np.arange(nq) if rows is None else np.asarray(rows)
    j = np.arange(nk)
    if window is not None:
        wl, wr = window
        off = j[None, :] - (i[:, None] + nk - nq)
        return ((wl < 0) | (off >= -wl)) & ((wr < 0) | (off <= wr))
    if causal:
        return j[None, :] <= i[:, None]
    return np.ones((i.size, nk), dtype=bool)


def _softmax_rows(s, keep):
    s = np.where(keep, s, -np.inf)
    m = np.max(s, axis=1, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    p = np.where(keep, np.exp(s - m), 0.0)
    tot = np.sum(p, axis=1, keepdims=True)
    return p / np.where(tot > 0, tot, 1.0)


def _head_terms(qh, kh, vh, doh, scale, keep):
    p = _softmax_rows(scale * (qh @ kh.T), keep)
    o = p @ vh
    e = np.sum(np.abs(doh * o), axis=1)
    t = p * (np.abs(doh @ vh.T) + e[:, None])
    return p, t


def row_scales(q, k, v, do, scale, causal=False, window=None):
    """M_r for every row: (dQ [B,H,Nq], dK [B,H,Nk], dV [B,H,Nk]).  Whole heads at once (small shapes)."""
    q, k, v, do = (_f64(x) for x in (q, k, v, do))
    B, H, nq, _ = q.shape
    nk = k.shape[2]
    keep = keep_matrix(nq, nk, causal, window)
    mq, mk, mv = np.zeros((B, H, nq)), np.zeros((B, H, nk)), np.zeros((B, H, nk))
    for b in range(B):
        for h in range(H):
            p, t = _head_terms(q[b, h], k[b, h], v[b, h], do[b, h], scale, keep)
            mq[b, h] = np.max(scale * (t @ np.abs(k[b, h])), axis=1)
            mk[b, h] = np.max(scale * (t.T @ np.abs(q[b, h])), axis=1)
            mv[b, h] = np.max(p.T @ np.abs(do[b, h]), axis=1)
    return mq, mk, mv


def dq_row_scales(q, k, v, do, rows, scale, causal=False):
    """M_r of dQ for selected flat rows (b*H + h)*Nq + i, one row at a time (any size)."""
    q, k, v, do = (_f64(x) for x in (q, k, v, do))
    B, H, nq, d = q.shape
    nk = k.shape[2]
    out = np.zeros(len(rows))
    for n, r in enumerate(rows):
        bh, i = divmod(int(r), nq)
        b, h = divmod(bh, H)
        keep = keep_matrix(nq, nk, causal, rows=[i])
        p, t = _head_terms(q[b, h, i:i + 1], k[b, h], v[b, h], do[b, h, i:i + 1], scale, keep)
        out[n] = np.max(scale * (t @ np.abs(k[b, h])))
    return out


def dkdv_key_scales(q, k, v, do, bh, keys, scale, causal=False, chunk=512):
    """M_r of dK and dV for selected keys of head bh, summed over all query rows in chunks."""
    q, k, v, do = (_f64(x) for x in (q, k, v, do))
    B, H, nq, d = q.shape
    nk = k.shape[2]
    b, h = divmod(int(bh), H)
    keys = np.asarray(keys)
    mk, mv = np.zeros((keys.size, d)), np.zeros((keys.size, d))
    for i0 in range(0, nq, chunk):
        rows = np.arange(i0, min(nq, i0 + chunk))
        keep = keep_matrix(nq, nk, causal, rows=rows)
        p, t = _head_terms(q[b, h, rows], k[b, h], v[b, h], do[b, h, rows], scale, keep)
        mk += scale * (t[:, keys].T @ np.abs(q[b, h, rows]))
        mv += p[:, keys].T @ np.abs(do[b, h, rows])
    return np.max(mk, axis=1), np.max(mv, axis=1)
