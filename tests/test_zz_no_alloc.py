"""attn_build_tiles_noalloc, the metadata build that allocates nothing.

Some callers cannot give the library extra device memory when they build a
mask -- a server whose device memory is carved up by its own pool when it
starts, or a plugin that is handed only its input and output buffers.  For
them the build keeps its scratch counters in a fixed array inside the
library.  These tests call that entry point through the C ABI twice in a row
and require metadata identical, bit for bit, to the regular attn_build_tiles
that takes a caller workspace.  The file runs last so that a run stopping at
its first failure has run every other test first; it also passes on its own.
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_slice_gb300 import binding as B
from block_sparse_attention_slice_gb300 import workloads as W

pytestmark = pytest.mark.gpu
KEYS = ["row_ptr", "col_idx", "kind", "pairs", "ref_ptr", "ref_idx", "sched"]


def _same(a, b):
    for key in KEYS:
        assert a[key].dtype == b[key].dtype, key
        assert np.array_equal(a[key], b[key]), key
    assert a["total_pairs"] == b["total_pairs"]


def _noalloc(slices, sq, sk, tq, tk):
    nbytes = B.attn_tiles_workspace_bytes(slices, sq, sk, tq, tk)
    out = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    return B.attn_build_tiles_noalloc(slices, sq, sk, out, tq, tk).to_host()


# "1": count and fill as two launches, which hand the counters over through
# the library's array; "0": one cooperative launch where every query tile's
# CTA fits at once (the variable is read on every call)
@pytest.mark.parametrize("two_launch", ["0", "1"])
def test_two_calls_in_a_row_match_the_workspace_build(two_launch, monkeypatch):
    monkeypatch.setenv("ATTN_BUILD_TWO_LAUNCH", two_launch)
    cases = [(W.video_slices(), 65536, 65536, 256, 128),
             (W.random_slices(3000, 2500, 40, seed=21, unit=1, max_len=600), 3000, 2500, 64, 32)]
    for sl, sq, sk, tq, tk in cases:
        ref = B.attn_build_tiles(sl, sq, sk, tq, tk).to_host()
        _same(ref, oracle.oracle_tiles(sl, sq, sk, tq, tk))
        first = _noalloc(sl, sq, sk, tq, tk)
        second = _noalloc(sl, sq, sk, tq, tk)
        _same(first, ref)
        _same(second, ref)


@pytest.mark.parametrize("two_launch", ["0", "1"])
def test_previous_contents_do_not_leak_into_a_smaller_build(two_launch, monkeypatch):
    monkeypatch.setenv("ATTN_BUILD_TWO_LAUNCH", two_launch)
    big = W.random_slices(8192, 8192, 60, seed=5, unit=16, max_len=64)
    small = np.array([[0, 700, 0, 700, 1], [700, 900, 0, 300, 3]], np.int32)
    _noalloc(big, 8192, 8192, 128, 128)
    got = _noalloc(small, 900, 900, 256, 128)
    _same(got, oracle.oracle_tiles(small, 900, 900, 256, 128))


def test_rejects_more_query_tiles_than_the_array_holds():
    sq = 16385
    sl = np.array([[0, sq, 0, 8, 0]], np.int32)
    out = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.AttnError) as e:
        B.attn_build_tiles_noalloc(sl, sq, 8, out, 1, 8)
    assert e.value.code == B.ATTN_ERR_CAPACITY
