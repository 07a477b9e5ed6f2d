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
