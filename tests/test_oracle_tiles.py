"""Pins of the tile-metadata oracle (CPU only).

Ties ``oracle_tiles`` to the worked examples printed on the UltraAttn page
(the partition-degree table of section 4.1 and the 7-of-16-blocks pattern of
section 1, both under ``tests/golden/``), to closed-form valid-pair counts of
the workloads, and to a dense element-by-element count.
"""
import numpy as np
import pytest

from conftest import read_golden
from oracle import CAUSAL, FULL, mask_rows, oracle_slices_from_grid, oracle_tiles, oracle_tiles_dense
from block_sparse_attention_slice_gb300 import workloads as W

KEYS = ["row_ptr", "col_idx", "kind", "pairs", "ref_ptr", "ref_idx", "sched"]


def _same(a, b):
    for key in KEYS:
        assert a[key].dtype == b[key].dtype, key
        assert np.array_equal(a[key], b[key]), key
    assert a["total_pairs"] == b["total_pairs"]


@pytest.mark.parametrize("seed,tq,tk", [(0, 8, 8), (1, 16, 8), (2, 24, 40), (3, 64, 32), (4, 7, 13)])
def test_interval_count_equals_dense_count(seed, tq, tk):
    S_q, S_k = 160, 176
    sl = W.random_slices(S_q, S_k, 9, seed=seed, unit=1, max_len=90)
    a = oracle_tiles(sl, S_q, S_k, tq, tk)
    b = oracle_tiles_dense(sl, S_q, S_k, tq, tk)
    _same(a, b)
    assert a["total_pairs"] == int(mask_rows(sl, np.arange(S_q), S_k).sum())


def test_partition_degree_table():
    # Causal grid of P x P blocks: Full below the diagonal, Causal on it.
    rows = read_golden("ultraattn_partition_degree_table.txt")
    T, N = 16, 4
    for P, Wt, WN, ceil_WN, imb in rows:
        P = int(P)
        t = oracle_tiles(np.array([[0, P * T, 0, P * T, CAUSAL]]), P * T, P * T, T, T)
        n_full = int((t["kind"] == 1).sum()); n_masked = int((t["kind"] == 2).sum())
        assert n_full == P * (P - 1) // 2 and n_masked == P
        w = n_full * 1.0 + n_masked * 0.5
        assert w == float(Wt)
        assert w / N == float(WN)
        assert int(np.ceil(w / N)) == int(ceil_WN)
        assert round((np.ceil(w / N) - w / N) / (w / N), 2) == float(imb)


def test_intro_pattern_seven_blocks():
    rows = read_golden("ultraattn_intro_pattern.txt")
    grid = np.array([[int(c) for c in r[0]] for r in rows[1:5]], dtype=np.uint8)
    n_valid = int(rows[5][1])
    sl = oracle_slices_from_grid(grid, 32)
    t = oracle_tiles(sl, 128, 128, 32, 32)
    assert len(t["col_idx"]) == n_valid == 7
    assert np.array_equal(np.diff(t["row_ptr"]), [1, 2, 2, 2])


def test_tiny_causal_counts():
    w = W.tiny_causal()
    t = oracle_tiles(w.slices, 512, 512, 128, 128)
    assert (t["kind"] == 1).sum() == 6 and (t["kind"] == 2).sum() == 4
    assert t["total_pairs"] == 512 * 513 // 2
    t2 = oracle_tiles(w.slices, 512, 512, 256, 128)
    # 256-row query tiles: k-tiles 2b and 2b+1 of query tile b are both masked
    assert np.array_equal(t2["row_ptr"], [0, 2, 6])
    assert np.array_equal(t2["kind"], [2, 2, 1, 1, 2, 2])


def test_varlen_total_pairs_closed_form():
    w = W.varlen_causal()
    docs = W.varlen_doc_lengths()
    assert docs == [2208, 2346, 3219, 3919, 636, 1028, 3028]
    t = oracle_tiles(w.slices, w.S, w.S, 256, 128)
    assert t["total_pairs"] == sum(L * (L + 1) // 2 for L in docs) == 23372975


def test_strided_grid_counts():
    w = W.block_sparse_strided()
    sl = oracle_slices_from_grid(w.grid, w.block)
    assert len(sl) == 4858 + 256
    t = oracle_tiles(sl, w.S, w.S, 128, 128)
    assert (t["kind"] == 1).sum() == 4858 and (t["kind"] == 2).sum() == 256
    assert t["total_pairs"] == 4858 * 128 * 128 + 256 * 128 * 129 // 2 == 81707008
    # every masked tile is one causal diagonal block: exactly one reference
    assert np.all(np.diff(t["ref_ptr"])[t["kind"] == 2] == 1)


def test_video_slices_disjoint_and_base_pairs():
    sl = W.video_slices()
    assert len(sl) == 16 + 15 + 14 + 32
    r = sl.astype(np.int64)
    for i in range(len(r)):
        for j in range(i + 1, len(r)):
            a, b = r[i], r[j]
            assert not (a[0] < b[1] and b[0] < a[1] and a[2] < b[3] and b[2] < a[3])
    base = 16 * 4096 * 4096 + 15 * 4096 * 4096 + 14 * 4096 * 4097 // 2
    assert base == 637562880
    t = oracle_tiles(sl[:45], 65536, 65536, 256, 128)
    assert t["total_pairs"] == base


def test_gqa_causal_counts_and_split():
    S = 131072
    t = oracle_tiles(np.array([[0, S, 0, S, CAUSAL]]), S, S, 256, 128)
    assert t["total_pairs"] == S * (S + 1) // 2 == 8590000128
    nnz = np.diff(t["row_ptr"])
    assert np.array_equal(nnz, 2 * (np.arange(S // 256) + 1))
    # longest-processing-time order: the last query tile first
    assert t["sched"][0] == S // 256 - 1 and t["sched"][-1] == 0
    w = W.gqa_causal_kv_split()
    tot = 0
    for sl in w.kv_splits:
        tot += oracle_tiles(sl, S, S, 256, 128)["total_pairs"]
    assert tot == t["total_pairs"]


def test_sched_is_lpt_with_index_ties():
    sl = W.random_slices(256, 256, 12, seed=5, unit=8, max_len=12)
    t = oracle_tiles(sl, 256, 256, 32, 32)
    nnz = np.diff(t["row_ptr"])
    s = t["sched"]
    assert sorted(s.tolist()) == list(range(len(nnz)))
    for a, b in zip(s[:-1], s[1:]):
        assert nnz[a] > nnz[b] or (nnz[a] == nnz[b] and a < b)


def test_ragged_tiles_never_full():
    t = oracle_tiles(np.array([[0, 100, 0, 100, FULL]]), 100, 100, 32, 32)
    k = t["kind"].reshape(4, 4)
    assert np.all(k[:3, :3] == 1) and np.all(k[3, :] == 2) and np.all(k[:, 3] == 2)
