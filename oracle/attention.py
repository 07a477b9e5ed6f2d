"""Oracle: masked attention forward and KV-split merge in fp64 (TEST INFRASTRUCTURE).

What is computed (plain definition; the pages' formulas were lost in text
extraction, so the textbook form they describe in prose is written out):

  A(i)      = { j : some mask slice contains (i, j) and its predicate holds }
  O[i, h]   = sum_{j in A(i)} softmax_j(scale * q_{i,h} . k_{j,g}) v_{j,g}
  lse[h, i] = ln sum_{j in A(i)} exp(scale * q_{i,h} . k_{j,g}),   g = h // (H / H_k)

A row with A(i) empty gets O = 0 and lse = -inf.  The max-shift used to
evaluate the softmax is the "m" of the mergeable summary (m, l, o) on the
UltraAttn page, section 3.2 (m aligns the numeric range, l is the local
normaliser, o the equally scaled value sum).

Slice predicates (local coordinates a = i - q_start, b = j - k_start,
L_q = q_end - q_start, L_k = k_end - k_start).  The pages name the mask kinds
of a flexible mask (MagiAttention v1.1.0 page, flexible-mask bullet; the
Full/Causal/Empty block kinds of the UltraAttn page, section 3) but never
define them; the reading taken here is:
  full        : every (a, b) in the rectangle
  causal      : b <= a + (L_k - L_q)      (bottom-right aligned; b <= a if square)
  inv-causal  : b >= a                    (top-left aligned)
  bi-causal   : both of the above
A Causal block of a block grid is the causal slice of that square block.

Parity: pinned (tests/test_oracle_attention.py): hand-worked two-key softmax,
uniform scores -> mean / prefix mean of V, merge-of-split == whole, -inf
partial is the identity of the merge, brute force against a second
independent per-element evaluator on S <= 64 for all four slice kinds.
"""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor
from typing import Callable, Iterable, Optional, Sequence

import numpy as np

FULL, CAUSAL, INV_CAUSAL, BI_CAUSAL = 0, 1, 2, 3


def mask_rows(slices: np.ndarray, rows: Sequence[int], sk: int) -> np.ndarray:
    """Dense boolean mask rows ``M[r, j] = (rows[r], j) in A`` from a slice list.

    Every slice is evaluated element by element over its own rectangle with
    the predicate of its kind (module docstring); slices are OR-ed.
    """
    rows = np.asarray(rows, dtype=np.int64)
    M = np.zeros((rows.size, sk), dtype=bool)
    for qs, qe, ks, ke, t in np.asarray(slices, dtype=np.int64).reshape(-1, 5):
        if qe <= qs or ke <= ks:
            continue
        sel = (rows >= qs) & (rows < qe)
        if not sel.any():
            continue
        a = (rows[sel] - qs)[:, None]
        b = np.arange(ke - ks, dtype=np.int64)[None, :]
        lq, lk = qe - qs, ke - ks
        if t == FULL:
            p = np.ones((a.shape[0], b.shape[1]), dtype=bool)
        elif t == CAUSAL:
            p = b <= a + (lk - lq)
        elif t == INV_CAUSAL:
            p = b >= a
        elif t == BI_CAUSAL:
            p = (b <= a + (lk - lq)) & (b >= a)
        else:
            raise ValueError(f"unknown slice type {t}")
        M[np.nonzero(sel)[0][:, None], np.arange(ks, ke)[None, :]] |= p
    return M


def mask_rows_grid(grid: np.ndarray, block: int, rows: Sequence[int], sk: int) -> np.ndarray:
    """Dense mask rows from a Full(1)/Causal(2)/Empty(0) block grid.

    A Full block admits all of its pairs, a Causal block the pairs with
    local key index <= local query index, an Empty block none (UltraAttn page,
    section 3: Full = all positions valid, Causal = part valid, Empty = all
    masked).
    """
    rows = np.asarray(rows, dtype=np.int64)
    M = np.zeros((rows.size, sk), dtype=bool)
    j = np.arange(sk, dtype=np.int64)
    bj = j // block
    jl = j % block
    for r, i in enumerate(rows):
        kinds = grid[i // block][bj]
        il = i % block
        M[r] = (kinds == 1) | ((kinds == 2) & (jl <= il))
    return M


def _attend_rows(qh: np.ndarray, kg: np.ndarray, vg: np.ndarray, M: np.ndarray, scale: float):
    """Softmax attention of query rows ``qh`` [r, d] over keys with mask M [r, S_k]."""
    r = qh.shape[0]
    d = vg.shape[1]
    O = np.zeros((r, d), dtype=np.float64)
    lse = np.full(r, -np.inf, dtype=np.float64)
    cols = np.nonzero(M.any(axis=0))[0]
    if cols.size == 0:
        return O, lse
    # Keys outside [lo, hi) are masked for every row of this block: their
    # exp() would be exactly 0, so they are left out of the arithmetic.
    lo, hi = int(cols[0]), int(cols[-1]) + 1
    Mw = M[:, lo:hi]
    s = (qh @ kg[lo:hi].T) * scale
    s = np.where(Mw, s, -np.inf)
    m = s.max(axis=1)
    live = np.isfinite(m)
    if not live.any():
        return O, lse
    e = np.exp(s[live] - m[live][:, None])
    l = e.sum(axis=1)
    O[live] = (e @ vg[lo:hi]) / l[:, None]
    lse[live] = m[live] + np.log(l)
    return O, lse


def oracle_attention(q, k, v, scale: float, mask: Callable[[np.ndarray], np.ndarray],
                     rows: Optional[Sequence[Sequence[int]]] = None,
                     heads: Optional[Iterable[int]] = None, row_block: int = 128,
                     threads: int = 1):
    """Forward of masked attention in fp64.

    q: [S_q, H, d]; k, v: [S_k, H_k, d] (any real dtype; computed in fp64).
    mask(rows) -> bool [len(rows), S_k] (``mask_rows`` / ``mask_rows_grid``).
    rows: None = every row for every head; else one sorted row list per head
    (indexed by head).  Returns ``{h: (rows, O [r, d], lse [r])}``.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    S_q, H, d = q.shape
    Hk = k.shape[1]
    if H % Hk:
        raise ValueError("H must be a multiple of H_k")
    group = H // Hk
    heads = list(range(H)) if heads is None else list(heads)

    def one_head(h):
        rr = np.arange(S_q) if rows is None else np.asarray(rows[h], dtype=np.int64)
        g = h // group
        kg = np.ascontiguousarray(k[:, g, :])
        vg = np.ascontiguousarray(v[:, g, :])
        O = np.zeros((rr.size, d))
        lse = np.full(rr.size, -np.inf)
        for b0 in range(0, rr.size, row_block):
            rb = rr[b0:b0 + row_block]
            M = mask(rb)
            O[b0:b0 + rb.size], lse[b0:b0 + rb.size] = _attend_rows(q[rb, h, :], kg, vg, M, scale)
        return h, (rr, O, lse)

    if threads > 1:
        with ThreadPoolExecutor(threads) as ex:
            out = dict(ex.map(one_head, heads))
    else:
        out = dict(one_head(h) for h in heads)
    return out


def oracle_merge(o_parts: Sequence[np.ndarray], lse_parts: Sequence[np.ndarray]):
    """Exact merge of KV-split partials (UltraAttn page, section 3.2).

    Each partial i is carried as (O_i normalised, lse_i), i.e. the summary
    (m = lse_i, l = 1, o = O_i).  The merge takes the global maximum m of the
    partials' m, rescales every summary to it and adds:
        l = sum_i exp(m_i - m) l_i,   o = sum_i exp(m_i - m) o_i,
    giving O = o / l and lse = m + ln l.  Partials with lse = -inf carry no
    keys and drop out; if all do, O = 0 and lse = -inf.

    o_parts: [S, H, d] each; lse_parts: [H, S] each.  Returns (O, lse).
    """
    O_in = [np.asarray(o, dtype=np.float64) for o in o_parts]
    L_in = [np.asarray(x, dtype=np.float64) for x in lse_parts]
    m = np.max(np.stack(L_in), axis=0)                       # [H, S]
    live = np.isfinite(m)
    ms = np.where(live, m, 0.0)
    l = np.zeros_like(m)
    o = np.zeros_like(O_in[0])
    for Oi, Li in zip(O_in, L_in):
        w = np.where(np.isfinite(Li), np.exp(Li - ms), 0.0)  # [H, S]
        l += w
        o += w.T[:, :, None] * Oi
    lt = l.T[:, :, None]
    O = np.where(live.T[:, :, None], o / np.where(lt > 0, lt, 1.0), 0.0)
    lse = np.where(live, ms + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return O, lse
