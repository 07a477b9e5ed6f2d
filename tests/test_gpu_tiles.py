"""attn_build_tiles on the GPU vs the oracle: bit-exact metadata."""
import numpy as np
import pytest

import oracle
from block_sparse_attention_slice_gb300 import attn_build_tiles, attn_slices_from_block_grid
from block_sparse_attention_slice_gb300 import workloads as W

pytestmark = pytest.mark.gpu
KEYS = ["row_ptr", "col_idx", "kind", "pairs", "ref_ptr", "ref_idx", "sched"]


def _check(slices, sq, sk, tq, tk):
    got = attn_build_tiles(slices, sq, sk, tq, tk).to_host()
    ref = oracle.oracle_tiles(slices, sq, sk, tq, tk)
    for key in KEYS:
        assert got[key].dtype == ref[key].dtype, key
        assert np.array_equal(got[key], ref[key]), key
    assert got["total_pairs"] == ref["total_pairs"]
    return got


@pytest.mark.parametrize("seed,sq,sk,tq,tk", [
    (0, 160, 176, 8, 8), (1, 1000, 1100, 256, 128), (2, 777, 513, 64, 32),
    (3, 2048, 2048, 128, 128), (4, 4096, 3000, 256, 128), (5, 300, 300, 7, 13),
    (6, 5000, 5000, 1024, 1024), (7, 64, 4096, 256, 128)])
def test_fuzzed_slices_bit_exact(seed, sq, sk, tq, tk):
    sl = W.random_slices(sq, sk, 24, seed=seed, unit=1, max_len=max(8, min(sq, sk) // 3))
    _check(sl, sq, sk, tq, tk)


def test_empty_and_degenerate_slice_lists():
    _check(np.zeros((0, 5), np.int32), 1000, 1000, 256, 128)
    _check(np.array([[5, 5, 0, 10, 0], [0, 10, 7, 7, 1]], np.int32), 300, 300, 256, 128)
    _check(np.array([[0, 1, 0, 1, 1]], np.int32), 1, 1, 256, 128)


@pytest.mark.parametrize("make,tq", [(W.tiny_causal, 128), (W.tiny_causal, 256),
                                     (W.varlen_causal, 256), (W.video_gen, 256)])
def test_workload_metadata(make, tq):
    w = make()
    _check(w.slices, w.S, w.S, tq, 128)
    for sl in w.kv_splits:
        _check(sl, w.S, w.S, tq, 128)


def test_block_grid_metadata():
    w = W.block_sparse_strided()
    sl = attn_slices_from_block_grid(w.grid, w.block, w.block)
    assert np.array_equal(sl, oracle.oracle_slices_from_grid(w.grid, w.block))
    got = _check(sl, w.S, w.S, 128, 128)
    assert (got["kind"] == 1).sum() == 4858 and (got["kind"] == 2).sum() == 256
    _check(sl, w.S, w.S, 256, 128)


@pytest.mark.slow
def test_long_causal_and_kv_split_metadata():
    w = W.gqa_causal_kv_split()
    _check(w.slices, w.S, w.S, 256, 128)
    for sl in w.kv_splits:
        _check(sl, w.S, w.S, 256, 128)


def test_rebuild_is_identical():
    sl = W.random_slices(3000, 3000, 40, seed=11, unit=16)
    a = attn_build_tiles(sl, 3000, 3000, 256, 128).to_host()
    b = attn_build_tiles(sl, 3000, 3000, 256, 128).to_host()
    for key in KEYS:
        assert np.array_equal(a[key], b[key])


@pytest.mark.parametrize("seed,sq,sk,tq,tk", [
    (11, 1000, 1100, 256, 128), (12, 3000, 2500, 64, 64), (13, 160, 176, 8, 8)])
def test_single_and_two_launch_builds_agree(seed, sq, sk, tq, tk, monkeypatch):
    # the build runs as one cooperative launch when every query tile's CTA
    # fits on the GPU at once, else as two launches; both must give the
    # oracle's metadata bit for bit
    sl = W.random_slices(sq, sk, 24, seed=seed, unit=1, max_len=max(8, min(sq, sk) // 3))
    ref = oracle.oracle_tiles(sl, sq, sk, tq, tk)
    monkeypatch.delenv("ATTN_BUILD_TWO_LAUNCH", raising=False)
    one = attn_build_tiles(sl, sq, sk, tq, tk).to_host()
    monkeypatch.setenv("ATTN_BUILD_TWO_LAUNCH", "1")
    two = attn_build_tiles(sl, sq, sk, tq, tk).to_host()
    for key in KEYS:
        assert np.array_equal(one[key], ref[key]), key
        assert np.array_equal(two[key], ref[key]), key
    assert one["total_pairs"] == two["total_pairs"] == ref["total_pairs"]
