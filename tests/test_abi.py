"""The C-ABI library (CPU only): it loads, exports every entry point that
include/attn_slice.h declares, and its host-only logic (block grid -> slices,
workspace sizing, argument checks done before any CUDA call) behaves."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from block_sparse_attention_slice_gb300 import binding as B
from block_sparse_attention_slice_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from block_sparse_attention_slice_gb300 import _build
    _build.build()
    return B.load()


def _declared():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^(?:const\s+)?[a-z_0-9]+\s*\*?\s*(attn_[a-z_0-9]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 10, names
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(B.EXPORTS) == names


def test_block_grid_to_slices_matches_oracle(lib):
    w = W.block_sparse_strided()
    got = B.attn_slices_from_block_grid(w.grid, 128, 128)
    assert np.array_equal(got, oracle.oracle_slices_from_grid(w.grid, 128))
    g = np.array([[2, 0], [1, 2]], np.uint8)
    assert np.array_equal(B.attn_slices_from_block_grid(g, 64, 64),
                          [[0, 64, 0, 64, 1], [64, 128, 0, 64, 0], [64, 128, 64, 128, 1]])
    with pytest.raises(B.AttnError):
        B.attn_slices_from_block_grid(g, 64, 32)          # causal block must be square
    with pytest.raises(B.AttnError):
        B.attn_slices_from_block_grid(np.array([[3]], np.uint8), 64, 64)


def test_workspace_bound_and_argument_checks(lib):
    sl = np.array([[0, 512, 0, 512, 1]], np.int32)
    n = B.attn_tiles_workspace_bytes(sl, 512, 512, 256, 128)
    assert n > 0 and n % 256 == 0
    with pytest.raises(B.AttnError) as e:
        B.attn_tiles_workspace_bytes(np.array([[0, 513, 0, 10, 0]], np.int32), 512, 512, 256, 128)
    assert e.value.code == B.ATTN_ERR_INVALID_ARG
    with pytest.raises(B.AttnError) as e:
        B.attn_tiles_workspace_bytes(np.array([[0, 5, 0, 10, 7]], np.int32), 512, 512, 256, 128)
    assert e.value.code == B.ATTN_ERR_INVALID_ARG
    with pytest.raises(B.AttnError) as e:
        B.attn_tiles_workspace_bytes(sl, 512, 512, 2048, 128)
    assert e.value.code == B.ATTN_ERR_UNSUPPORTED
    # overlap is found on the host, before anything touches the device
    arr, cnt = B._slice_array(np.array([[0, 100, 0, 100, 0], [99, 150, 99, 150, 1]], np.int32))
    st = B.AttnTiles()
    rc = lib.attn_build_tiles(arr, cnt, 512, 512, 256, 128, ctypes.c_void_p(256), 1 << 20,
                              ctypes.byref(st), None)
    assert rc == B.ATTN_ERR_OVERLAP
    assert lib.attn_strerror(B.ATTN_ERR_TIMEOUT).decode().startswith("a bounded")
    # exponential mode: only periods 0, 4 and 8 exist (host-side setting)
    for bad in (-1, 1, 2, 3, 16):
        assert lib.attn_set_exp2_poly(bad) == B.ATTN_ERR_INVALID_ARG
    for good in (4, 8, 0):
        assert lib.attn_set_exp2_poly(good) == B.ATTN_OK


def _brute_overlap(sl):
    r = [x for x in sl.tolist() if x[1] > x[0] and x[3] > x[2]]
    for i in range(len(r)):
        for j in range(i + 1, len(r)):
            a, b = r[i], r[j]
            if a[0] < b[1] and b[0] < a[1] and a[2] < b[3] and b[2] < a[3]:
                return True
    return False


@pytest.mark.parametrize("seed", range(6))
def test_planted_overlaps_are_found_before_any_device_work(lib, seed):
    # a disjoint random list plus one slice overlapping a random member; the
    # host check must reject it before anything reaches the device
    rng = np.random.default_rng(seed)
    base = W.random_slices(4096, 4096, 60, seed=seed, unit=16, max_len=40)
    assert not _brute_overlap(base)
    victim = base[rng.integers(len(base))]
    qs = int(rng.integers(victim[0], victim[1])); ks = int(rng.integers(victim[2], victim[3]))
    extra = np.array([[qs, min(4096, qs + 5), ks, min(4096, ks + 7), int(rng.integers(4))]], np.int32)
    sl = np.concatenate([base, extra])[rng.permutation(len(base) + 1)]
    assert _brute_overlap(sl)
    arr, cnt = B._slice_array(sl)
    st = B.AttnTiles()
    rc = lib.attn_build_tiles(arr, cnt, 4096, 4096, 256, 128, ctypes.c_void_p(256), 1 << 30,
                              ctypes.byref(st), None)
    assert rc == B.ATTN_ERR_OVERLAP
