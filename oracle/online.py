"""Test-only CPU restatement of the tiled online-softmax recurrence.

TEST INFRASTRUCTURE ONLY: imported by tests/ alone.  It is the second, tiled
form of the oracle's arithmetic, used to check that the block-by-block
recurrence reaches the one-shot definition (``oracle.attention_fwd``) and to
expose the per-block state (m, l, unnormalised O) that the pages print.

Sources, stated in my own words:

* page "llm-infra-atlas / 01 IO awareness & online softmax", section 2: a row
  is consumed one block of columns at a time.  The state is the running
  maximum m, the running denominator l and the running numerator O, the
  latter two both relative to the current m.  A new block S_j first raises
  m to m_new = max(m, rowmax S_j); the old l and O are carried over to the new
  reference by the factor alpha = exp(m - m_new) (<= 1); the block adds
  rowsum(exp(S_j - m_new)) to l and exp(S_j - m_new) V_j to O.  After the
  last block O / l is the attention row, and m + ln(l) its log-sum-exp
  (section 3 and section 5 of the same page).
* page "pinghaoyang FlashAttention 1-4 guide", FA4 section, conditional
  softmax rescaling: the reference value m_bar used for the exponentials only
  moves when the candidate maximum exceeds it by more than tau; otherwise the
  block is exponentiated against the old m_bar and O, l are not rescaled.
  The final division by the true normaliser makes the result exact for any
  tau.  tau is given in base-2 units (the page's tau = log2(256) = 8); the
  test in natural units is m_new - m_bar > tau * ln 2.
* page "lumenova research-attention", section 03: the worked single row
  (scores [1, 2, 0, 3], tile 2) whose per-block state this module reports.

Masked scores are -inf.  A row whose every score so far is -inf keeps
m = -inf; its exponentials are taken against 0 instead, which gives 0 and no
NaN (the "Check_inf" guard of the FA2 mainloop on the infra-atlas page).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

LN2 = math.log(2.0)


@dataclass
class RowTrace:
    """Per-block state of one row: after block b, m[b], l[b], acc[b]."""

    m: list = field(default_factory=list)
    l: list = field(default_factory=list)
    acc: list = field(default_factory=list)
    alpha: list = field(default_factory=list)
    rescaled: list = field(default_factory=list)


def online_row(scores, values, tile, tau_log2=None, trace: RowTrace | None = None):
    """One attention row by the tiled online recurrence.

    scores: length-n sequence of (already scaled) logits; values: n x dv.
    tile: number of columns per block (>= 1; the last block may be short).
    tau_log2: None for the plain rule (rescale on every max increase), or the
    conditional-rescaling threshold in base-2 units.
    Returns (o_row as list of float, lse as float).
    """
    if tile < 1:
        raise ValueError("tile must be >= 1")
    n = len(scores)
    dv = len(values[0]) if n else 0
    m = -math.inf  # reference maximum (m_bar under conditional rescaling)
    l = 0.0
    acc = [0.0] * dv
    for start in range(0, n, tile):
        block = [float(s) for s in scores[start:start + tile]]
        cand = max(m, max(block))
        if tau_log2 is None:
            move = cand > m
        else:
            move = (m == -math.inf and cand > m) or (cand - m > tau_log2 * LN2)
        if move:
            alpha = math.exp(m - cand) if m != -math.inf else 0.0
            l = alpha * l
            acc = [alpha * a for a in acc]
            m = cand
        else:
            alpha = 1.0
        ref = m if m != -math.inf else 0.0
        weights = [math.exp(s - ref) for s in block]
        l = l + sum(weights)
        for c in range(dv):
            acc[c] = acc[c] + sum(w * float(values[start + j][c]) for j, w in enumerate(weights))
        if trace is not None:
            trace.m.append(m)
            trace.l.append(l)
            trace.acc.append(list(acc))
            trace.alpha.append(alpha)
            trace.rescaled.append(bool(move))
    if l == 0.0:
        return [0.0] * dv, -math.inf
    return [a / l for a in acc], m + math.log(l)


def tiled_attention(q, k, v, scale, causal, tile, tau_log2=None):
    """Whole-head attention by the tiled recurrence, rows updated together.

    q: [Nq, d], k, v: [Nk, d] float64 arrays.  The query rows form one block
    (all rows at once, vectors of state), the keys are consumed ``tile`` at a
    time in ascending order, as in the FA2-order loop of the infra-atlas
    page, section 3.  Causal keeps key j for row i iff j <= i.
    Returns (o [Nq, d], lse [Nq], n_rescales) with n_rescales the number of
    (row, block) pairs whose reference maximum moved.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    nq, nk = q.shape[0], k.shape[0]
    m = np.full(nq, -np.inf)
    l = np.zeros(nq)
    acc = np.zeros((nq, v.shape[1]))
    rows = np.arange(nq)[:, None]
    moves = 0
    for start in range(0, nk, tile):
        stop = min(start + tile, nk)
        s = (q @ k[start:stop].T) * scale
        if causal:
            cols = np.arange(start, stop)[None, :]
            s = np.where(cols > rows, -np.inf, s)
        cand = np.maximum(m, s.max(axis=1))
        if tau_log2 is None:
            move = cand > m
        else:
            move = ((m == -np.inf) & (cand > m)) | (cand - m > tau_log2 * LN2)
        with np.errstate(invalid="ignore"):
            alpha = np.where(m == -np.inf, 0.0, np.exp(m - cand))
        alpha = np.where(move, alpha, 1.0)
        l = alpha * l
        acc = alpha[:, None] * acc
        m = np.where(move, cand, m)
        moves += int(move.sum())
        ref = np.where(m == -np.inf, 0.0, m)
        p = np.exp(s - ref[:, None])
        l = l + p.sum(axis=1)
        acc = acc + p @ v[start:stop]
    with np.errstate(divide="ignore", invalid="ignore"):
        o = np.where(l[:, None] > 0, acc / l[:, None], 0.0)
        lse = np.where(l > 0, m + np.log(l), -np.inf)
    return o, lse, moves
