"""Pins of the attention and merge oracle (CPU only).

Each test ties the oracle to something other than itself: a hand-worked
softmax, closed forms for uniform scores, the merge invariant stated on the
UltraAttn page (section 3.2: per-KV-shard summaries merged by a global max
and rescaling give the full softmax), textbook reductions of the mask kinds,
and a second per-element evaluator written independently in pure Python.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import (BI_CAUSAL, CAUSAL, FULL, INV_CAUSAL, mask_rows, mask_rows_grid,
                    oracle_attention, oracle_merge, oracle_slices_from_grid)
from block_sparse_attention_slice_gb300.workloads import random_slices


def _run(q, k, v, scale, slices, rows=None):
    S_k = k.shape[0]
    res = oracle_attention(q, k, v, scale, lambda r: mask_rows(slices, r, S_k), rows=rows)
    H = q.shape[1]
    O = np.stack([res[h][1] for h in range(H)], axis=1)
    lse = np.stack([res[h][2] for h in range(H)], axis=0)
    return O, lse


def test_handworked_two_key_softmax():
    # scores {0, ln 3} -> weights {1/4, 3/4}, lse = ln 4
    q = np.zeros((1, 1, 4)); q[0, 0, 0] = 1.0
    k = np.zeros((2, 1, 4)); k[1, 0, 0] = math.log(3.0)
    v = np.array([[[1.0, 2, 3, 4]], [[5.0, 6, 7, 8]]])
    O, lse = _run(q, k, v, 1.0, np.array([[0, 1, 0, 2, FULL]]))
    np.testing.assert_allclose(O[0, 0], [4.0, 5.0, 6.0, 7.0], rtol=0, atol=1e-15)
    assert abs(lse[0, 0] - math.log(4.0)) < 1e-15


def test_scale_enters_scores():
    q = np.zeros((1, 1, 2)); q[0, 0, 0] = 2.0
    k = np.zeros((2, 1, 2)); k[1, 0, 0] = math.log(3.0)
    v = np.array([[[0.0, 1.0]], [[1.0, 0.0]]])
    O, lse = _run(q, k, v, 0.5, np.array([[0, 1, 0, 2, FULL]]))
    np.testing.assert_allclose(O[0, 0], [0.75, 0.25], atol=1e-15)
    assert abs(lse[0, 0] - math.log(4.0)) < 1e-15


@pytest.mark.parametrize("kind", [FULL, CAUSAL, INV_CAUSAL, BI_CAUSAL])
def test_uniform_scores_closed_forms(kind):
    # q = 0: every valid key scores 0, so O is the plain mean of V over A(i)
    # and lse = ln |A(i)|.  Square slice of side n starting at offset 5.
    rng = np.random.default_rng(7)
    n, off, S = 20, 5, 32
    q = np.zeros((S, 1, 8))
    k = rng.standard_normal((S, 1, 8))
    v = rng.standard_normal((S, 1, 8))
    O, lse = _run(q, k, v, 0.3, np.array([[off, off + n, off, off + n, kind]]))
    for i in range(S):
        if not off <= i < off + n:
            assert np.all(O[i, 0] == 0) and lse[0, i] == -np.inf
            continue
        a = i - off
        if kind == FULL:
            keys = range(off, off + n)
        elif kind == CAUSAL:
            keys = range(off, off + a + 1)          # prefix mean
        elif kind == INV_CAUSAL:
            keys = range(off + a, off + n)          # suffix mean
        else:
            keys = [off + a]                        # the diagonal only
        keys = list(keys)
        np.testing.assert_allclose(O[i, 0], v[keys, 0].mean(axis=0), atol=1e-13)
        assert abs(lse[0, i] - math.log(len(keys))) < 1e-13


def test_causal_non_square_is_bottom_right_aligned():
    # L_q = 4, L_k = 8: row a sees local keys b <= a + 4, i.e. a + 5 keys.
    rng = np.random.default_rng(3)
    q = np.zeros((4, 1, 4)); k = rng.standard_normal((8, 1, 4)); v = rng.standard_normal((8, 1, 4))
    O, lse = _run(q, k, v, 1.0, np.array([[0, 4, 0, 8, CAUSAL]]))
    for a in range(4):
        np.testing.assert_allclose(O[a, 0], v[:a + 5, 0].mean(axis=0), atol=1e-14)
        assert abs(lse[0, a] - math.log(a + 5)) < 1e-14
    # L_q = 8, L_k = 4: the first four rows see nothing.
    q = np.zeros((8, 1, 4)); k = rng.standard_normal((4, 1, 4)); v = rng.standard_normal((4, 1, 4))
    O, lse = _run(q, k, v, 1.0, np.array([[0, 8, 0, 4, CAUSAL]]))
    assert np.all(lse[0, :4] == -np.inf) and np.all(O[:4] == 0)
    for a in range(4, 8):
        assert abs(lse[0, a] - math.log(a - 3)) < 1e-14


def test_square_kinds_reduce_to_triangles():
    n = 9
    r = np.arange(n)
    assert np.array_equal(mask_rows(np.array([[0, n, 0, n, CAUSAL]]), r, n), np.tril(np.ones((n, n), bool)))
    assert np.array_equal(mask_rows(np.array([[0, n, 0, n, INV_CAUSAL]]), r, n), np.triu(np.ones((n, n), bool)))
    assert np.array_equal(mask_rows(np.array([[0, n, 0, n, BI_CAUSAL]]), r, n), np.eye(n, dtype=bool))
    assert np.array_equal(mask_rows(np.array([[0, n, 0, n, FULL]]), r, n), np.ones((n, n), bool))


def _brute_force(q, k, v, scale, slices):
    """Independent per-element evaluator: membership tested in global
    coordinates (causal = distance to the bottom-right corner, inv-causal =
    distance to the top-left corner), softmax without a max shift, sums by
    math.fsum."""
    S_q, H, d = q.shape
    S_k, Hk, _ = k.shape
    grp = H // Hk

    def valid(i, j):
        for qs, qe, ks, ke, t in slices:
            if not (qs <= i < qe and ks <= j < ke):
                continue
            br = (ke - j) >= (qe - i)
            tl = (j - ks) >= (i - qs)
            if t == FULL or (t == CAUSAL and br) or (t == INV_CAUSAL and tl) or (t == BI_CAUSAL and br and tl):
                return True
        return False

    O = np.zeros((S_q, H, d)); lse = np.full((H, S_q), -np.inf)
    for h in range(H):
        g = h // grp
        for i in range(S_q):
            js = [j for j in range(S_k) if valid(i, j)]
            if not js:
                continue
            w = [math.exp(scale * math.fsum(float(q[i, h, c]) * float(k[j, g, c]) for c in range(d))) for j in js]
            den = math.fsum(w)
            for c in range(d):
                O[i, h, c] = math.fsum(wj * float(v[j, g, c]) for wj, j in zip(w, js)) / den
            lse[h, i] = math.log(den)
    return O, lse


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_brute_force_small(seed):
    rng = np.random.default_rng(seed)
    S_q, S_k, H, Hk, d = 40, 48, 4, 2, 8
    slices = random_slices(S_q, S_k, 6, seed=seed + 10, unit=1, max_len=24)
    assert set(slices[:, 4]) <= {0, 1, 2, 3}
    q = rng.standard_normal((S_q, H, d)); k = rng.standard_normal((S_k, Hk, d)); v = rng.standard_normal((S_k, Hk, d))
    O, lse = _run(q, k, v, 0.35, slices)
    Ob, lb = _brute_force(q, k, v, 0.35, slices.tolist())
    assert np.array_equal(np.isneginf(lse), np.isneginf(lb))
    fin = np.isfinite(lb)
    np.testing.assert_allclose(lse[fin], lb[fin], rtol=0, atol=1e-12)
    np.testing.assert_allclose(O, Ob, rtol=0, atol=1e-12)


def test_all_kinds_present_in_brute_force_fuzz():
    kinds = set()
    for seed in (10, 11, 12):
        kinds |= set(random_slices(40, 48, 6, seed=seed, unit=1, max_len=24)[:, 4].tolist())
    assert kinds == {0, 1, 2, 3}


@pytest.mark.parametrize("cuts", [[24], [7, 30], [1, 2, 40]])
def test_merge_of_kv_split_equals_whole(cuts):
    rng = np.random.default_rng(5)
    S, H, Hk, d = 48, 2, 1, 16
    slices = random_slices(S, S, 5, seed=3, unit=4)
    q = rng.standard_normal((S, H, d)); k = rng.standard_normal((S, Hk, d)); v = rng.standard_normal((S, Hk, d))
    O, lse = _run(q, k, v, 0.25, slices)
    edges = [0] + cuts + [S]
    parts_o, parts_l = [], []
    for a, b in zip(edges[:-1], edges[1:]):
        cols = np.zeros(S, bool); cols[a:b] = True
        res = oracle_attention(q, k, v, 0.25, lambda r: mask_rows(slices, r, S) & cols[None, :])
        parts_o.append(np.stack([res[h][1] for h in range(H)], axis=1))
        parts_l.append(np.stack([res[h][2] for h in range(H)], axis=0))
    Om, lm = oracle_merge(parts_o, parts_l)
    assert np.array_equal(np.isneginf(lm), np.isneginf(lse))
    fin = np.isfinite(lse)
    np.testing.assert_allclose(lm[fin], lse[fin], atol=1e-12)
    np.testing.assert_allclose(Om, O, atol=1e-12)
    # the naive combination (average of the per-shard softmax outputs) is not
    # the answer: each shard normalised with its own denominator
    live = [p for p, l in zip(parts_o, parts_l)]
    naive = sum(live) / len(live)
    assert np.max(np.abs(naive - O)) > 1e-3


def test_merge_identity_and_empty():
    rng = np.random.default_rng(9)
    O1 = rng.standard_normal((6, 2, 4)); l1 = rng.standard_normal((2, 6))
    O0 = rng.standard_normal((6, 2, 4)); l0 = np.full((2, 6), -np.inf)
    Om, lm = oracle_merge([O1, O0], [l1, l0])
    np.testing.assert_array_equal(Om, O1)
    np.testing.assert_array_equal(lm, l1)
    Oe, le = oracle_merge([O0, O0], [l0, l0])
    assert np.all(Oe == 0) and np.all(le == -np.inf)


def test_merge_two_summaries_closed_form():
    # two one-key shards with scores 0 and ln 3: weights 1/4 and 3/4
    O1 = np.array([[[1.0, 0.0]]]); O2 = np.array([[[0.0, 1.0]]])
    Om, lm = oracle_merge([O1, O2], [np.array([[0.0]]), np.array([[math.log(3.0)]])])
    np.testing.assert_allclose(Om[0, 0], [0.25, 0.75], atol=1e-15)
    assert abs(lm[0, 0] - math.log(4.0)) < 1e-15


def test_grid_mask_equals_slice_mask():
    rng = np.random.default_rng(2)
    for _ in range(3):
        g = rng.integers(0, 3, size=(6, 6)).astype(np.uint8)
        sl = oracle_slices_from_grid(g, 8)
        r = np.arange(48)
        assert np.array_equal(mask_rows_grid(g, 8, r, 48), mask_rows(sl, r, 48))


def test_empty_rows_are_zero_and_neg_inf():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((16, 1, 4)); k = rng.standard_normal((16, 1, 4)); v = rng.standard_normal((16, 1, 4))
    O, lse = _run(q, k, v, 1.0, np.array([[4, 8, 0, 16, FULL]]))
    for i in range(16):
        if 4 <= i < 8:
            assert np.isfinite(lse[0, i])
        else:
            assert lse[0, i] == -np.inf and np.all(O[i] == 0)
