"""Oracle: gradients of masked attention (TEST INFRASTRUCTURE).

Plain definition of the backward pass of O = softmax(scale * Q K^T + mask) V,
in fp64, with the dense mask materialised by ``attention.mask_rows``:

  P      = softmax over the valid keys of each row (0 on masked keys; a row
           with no valid key has P = 0 and O = 0)
  dV_g   = sum_{h in group g} P_h^T dO_h
  dP_h   = dO_h V_g^T
  D_h    = rowsum(dO_h * O_h)            (= rowsum(P_h * dP_h))
  dS_h   = P_h * (dP_h - D_h)            (gradient through the softmax)
  dQ_h   = scale * dS_h K_g
  dK_g   = scale * sum_{h in group g} dS_h^T Q_h

with g = h // (H / H_k).  The pages list the backward pass as work to come
after the forward (the MagiAttention page reports forward and backward
kernels; the FlashAttention-4 page describes a rebuilt backward pipeline);
the formulas above are the textbook chain rule through softmax.

Parity: pinned (tests/test_oracle_backward.py) by central finite differences
of ``oracle_attention`` on small problems for all four slice kinds and
grouped heads, and by the identity rowsum(dO * O) == rowsum(P * dP).
``oracle_attention_backward_sampled`` (gradients at chosen keys and rows of
problems too large for dense score matrices) is pinned by equality with the
dense form at every sampled position, and by exact zeros where no valid pair
reaches.
"""
from __future__ import annotations

import numpy as np


def oracle_attention_backward(q, k, v, dout, scale: float, mask):
    """Returns (dQ [S_q,H,d], dK [S_k,H_k,d], dV [S_k,H_k,d], D [H,S_q]) in fp64.

    mask(rows) -> bool [len(rows), S_k] as for ``oracle_attention``.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(dout, dtype=np.float64)
    S_q, H, d = q.shape
    S_k, Hk, _ = k.shape
    grp = H // Hk
    M = mask(np.arange(S_q))
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    D = np.zeros((H, S_q))
    for h in range(H):
        g = h // grp
        s = scale * (q[:, h, :] @ k[:, g, :].T)
        s = np.where(M, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        live = np.isfinite(m[:, 0])
        e = np.zeros_like(s)
        e[live] = np.exp(s[live] - m[live])
        l = e.sum(axis=1, keepdims=True)
        p = np.where(l > 0, e / np.where(l > 0, l, 1.0), 0.0)
        o = p @ v[:, g, :]
        dp = do[:, h, :] @ v[:, g, :].T
        D[h] = (do[:, h, :] * o).sum(axis=1)
        ds = p * (dp - D[h][:, None])
        dq[:, h, :] = scale * (ds @ k[:, g, :])
        dk[:, g, :] += scale * (ds.T @ q[:, h, :])
        dv[:, g, :] += p.T @ do[:, h, :]
    return dq, dk, dv, D


def oracle_attention_backward_sampled(q, k, v, dout, scale: float, mask, fwd,
                                      keys=None, rows=None, row_block: int = 1024):
    """Gradients at chosen positions only, in fp64, for problems whose dense
    score matrices do not fit: dK and dV at chosen keys, dQ at chosen rows.

    The definitions are those of ``oracle_attention_backward``; the softmax
    probabilities are rebuilt from the forward oracle's row LSE instead of a
    row-wise max and sum, which is the same number written differently:

      P[i, j]  = exp(scale q_i . k_j - lse_i) on valid (i, j), else 0
      D_i      = rowsum(dO_i * O_i)
      dS[i, j] = P[i, j] (dO_i . v_j - D_i)
      dV_j     = sum_{h in group g} sum_i P[i, j] dO_i
      dK_j     = scale sum_{h in group g} sum_i dS[i, j] q_i
      dQ_i     = scale sum_j dS[i, j] k_j

    fwd:  {h: (rows, O_h [S_q, d], lse_h [S_q])} from ``oracle_attention`` on
          every row (rows=None) of every head used: all heads of each group in
          ``keys`` and the heads in ``rows``.
    keys: {g: key indices} -> dK[g], dV[g] [len, d]; every key column is
          visited over all query rows, ``row_block`` rows of the mask at a time.
    rows: {h: row indices} -> dQ[h] [len, d].
    Returns (dk, dv, dq) dicts keyed like ``keys`` / ``rows``.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(dout, dtype=np.float64)
    S_q, H, d = q.shape
    Hk = k.shape[1]
    grp = H // Hk
    keys = {} if keys is None else {g: np.asarray(j, dtype=np.int64) for g, j in keys.items()}
    rows = {} if rows is None else {h: np.asarray(r, dtype=np.int64) for h, r in rows.items()}

    def stats(h):
        _, O, lse = fwd[h]
        D = (do[:, h, :] * O).sum(axis=1)
        # rows with no valid key (lse = -inf) get P = 0: an infinite lse
        # makes every exp(s - lse) exactly 0
        lse_p = np.where(np.isfinite(lse), lse, np.inf)
        return D, lse_p

    st = {h: stats(h) for h in set(rows) | {h for g in keys for h in range(g * grp, (g + 1) * grp)}}

    dq = {}
    for h, R in rows.items():
        g = h // grp
        D, lse_p = st[h]
        M = mask(R)
        s = scale * (q[R, h, :] @ k[:, g, :].T)
        P = np.where(M, np.exp(s - lse_p[R][:, None]), 0.0)
        dS = P * (do[R, h, :] @ v[:, g, :].T - D[R][:, None])
        dq[h] = scale * (dS @ k[:, g, :])

    dk = {g: np.zeros((J.size, d)) for g, J in keys.items()}
    dv = {g: np.zeros((J.size, d)) for g, J in keys.items()}
    if keys:
        for b0 in range(0, S_q, row_block):
            rb = np.arange(b0, min(S_q, b0 + row_block))
            Mb = mask(rb)
            for g, J in keys.items():
                Mj = Mb[:, J]
                if not Mj.any():
                    continue
                for h in range(g * grp, (g + 1) * grp):
                    D, lse_p = st[h]
                    s = scale * (q[rb, h, :] @ k[J, g, :].T)
                    P = np.where(Mj, np.exp(s - lse_p[rb][:, None]), 0.0)
                    dS = P * (do[rb, h, :] @ v[J, g, :].T - D[rb][:, None])
                    dv[g] += P.T @ do[rb, h, :]
                    dk[g] += scale * (dS.T @ q[rb, h, :])
    return dk, dv, dq
