"""Pins of the backward oracle (CPU only): central finite differences of the
forward oracle, and the softmax identity rowsum(dO * O) == rowsum(P * dP)."""
import numpy as np
import pytest

from oracle import mask_rows, oracle_attention
from oracle.backward import oracle_attention_backward
from block_sparse_attention_slice_gb300 import workloads as W


def _forward(q, k, v, scale, sl):
    S_k = k.shape[0]
    res = oracle_attention(q, k, v, scale, lambda r: mask_rows(sl, r, S_k))
    return np.stack([res[h][1] for h in range(q.shape[1])], axis=1)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_gradients_match_central_differences(seed):
    rng = np.random.default_rng(seed)
    S_q, S_k, H, Hk, d = 10, 12, 2, 1, 3
    sl = W.random_slices(S_q, S_k, 4, seed=seed + 30, unit=1, max_len=8)
    assert len(sl) >= 2
    q = rng.standard_normal((S_q, H, d)); k = rng.standard_normal((S_k, Hk, d)); v = rng.standard_normal((S_k, Hk, d))
    G = rng.standard_normal((S_q, H, d))           # dO: the loss is sum(O * G)
    scale = 0.7
    dq, dk, dv, _ = oracle_attention_backward(q, k, v, G, scale, lambda r: mask_rows(sl, r, S_k))
    eps = 1e-6
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = x.copy(); xp[idx] += eps
            xm = x.copy(); xm[idx] -= eps
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            fp = (_forward(args["q"], args["k"], args["v"], scale, sl) * G).sum()
            args[name] = xm
            fm = (_forward(args["q"], args["k"], args["v"], scale, sl) * G).sum()
            num[idx] = (fp - fm) / (2 * eps)
        np.testing.assert_allclose(grad, num, atol=1e-7, rtol=1e-6, err_msg=name)


def test_delta_identity_and_empty_rows():
    rng = np.random.default_rng(4)
    S, H, d = 16, 1, 4
    sl = np.array([[4, 12, 0, 8, 1]], np.int32)       # rows 0-3 and 12-15 see no key
    q = rng.standard_normal((S, H, d)); k = rng.standard_normal((S, H, d)); v = rng.standard_normal((S, H, d))
    G = rng.standard_normal((S, H, d))
    m = lambda r: mask_rows(sl, r, S)
    dq, dk, dv, D = oracle_attention_backward(q, k, v, G, 0.5, m)
    assert np.all(dq[:4] == 0) and np.all(dq[12:] == 0)
    O = _forward(q, k, v, 0.5, sl)
    np.testing.assert_allclose(D[0], (G[:, 0] * O[:, 0]).sum(axis=1), atol=1e-14)
    # keys 8..15 are valid for no row -> no gradient reaches them
    assert np.all(dk[8:] == 0) and np.all(dv[8:] == 0)
    assert np.any(dk[:8] != 0) and np.any(dv[:8] != 0)


@pytest.mark.parametrize("seed", [0, 1])
def test_sampled_gradients_equal_the_dense_ones(seed):
    # The sampled form (P rebuilt from the forward oracle's LSE, keys visited
    # column by column over row blocks) must reproduce the dense backward --
    # itself pinned by finite differences above -- at every sampled position:
    # all four slice kinds, grouped heads, rows and keys that no pair reaches.
    from oracle.backward import oracle_attention_backward_sampled
    rng = np.random.default_rng(seed + 7)
    S_q, S_k, H, Hk, d = 90, 110, 4, 2, 8
    sl = W.random_slices(S_q, S_k, 12, seed=seed + 60, unit=1, max_len=40)
    m = lambda r: mask_rows(sl, r, S_k)
    q = rng.standard_normal((S_q, H, d)); k = rng.standard_normal((S_k, Hk, d))
    v = rng.standard_normal((S_k, Hk, d)); G = rng.standard_normal((S_q, H, d))
    scale = 0.4
    dq, dk, dv, _ = oracle_attention_backward(q, k, v, G, scale, m)
    fwd = oracle_attention(q, k, v, scale, m)
    keys = {g: np.sort(rng.choice(S_k, 30, replace=False)) for g in range(Hk)}
    rows = {h: np.sort(rng.choice(S_q, 25, replace=False)) for h in range(H)}
    sk, sv, sq = oracle_attention_backward_sampled(q, k, v, G, scale, m, fwd, keys, rows, row_block=16)
    for g, J in keys.items():
        np.testing.assert_allclose(sk[g], dk[J, g, :], atol=1e-12, rtol=1e-10)
        np.testing.assert_allclose(sv[g], dv[J, g, :], atol=1e-12, rtol=1e-10)
    for h, R in rows.items():
        np.testing.assert_allclose(sq[h], dq[R, h, :], atol=1e-12, rtol=1e-10)
    # positions that no valid pair reaches come out exactly zero
    M = m(np.arange(S_q))
    dead_k = np.nonzero(~M.any(axis=0))[0]
    dead_q = np.nonzero(~M.any(axis=1))[0]
    assert dead_k.size and dead_q.size
    sk2, sv2, sq2 = oracle_attention_backward_sampled(q, k, v, G, scale, m, fwd,
                                                      {0: dead_k}, {0: dead_q})
    assert np.all(sk2[0] == 0) and np.all(sv2[0] == 0) and np.all(sq2[0] == 0)
