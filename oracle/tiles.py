"""Oracle: tile metadata of a slice mask (TEST INFRASTRUCTURE).

The attention matrix is cut into tiles of ``tq`` query rows by ``tk`` key
columns -- the two-dimensional blocks of the UltraAttn page, section 3.3.
For every tile the oracle counts the valid (query, key) pairs exactly and
classifies it (UltraAttn page, section 3: a block is Full when every position
is valid, Causal -- here "Masked" -- when only some are, Empty when none):

  count == 0          -> Empty: no entry (its compute and transfer are skipped)
  count == tq * tk    -> FULL (kind 1): no element needs a mask
  otherwise           -> MASKED (kind 2): elements are masked per row

(tiles cut by the end of the sequence are never FULL: they have fewer than
tq*tk positions.)  The non-Empty tiles of each query-tile row are stored in
compressed sparse rows, as the MagiAttention v1.1.0 page describes for the
mask metadata of long sequences ("CSR compression" bullet):

  row_ptr [nq+1]  int32   entries of query tile t are row_ptr[t] .. row_ptr[t+1]-1
  col_idx [nnz]   int32   key-tile index, ascending within a row
  kind    [nnz]   uint8   1 FULL, 2 MASKED
  pairs   [nnz]   int32   valid pairs in the tile
  ref_ptr [nnz+1] int32   entry e references ref_idx[ref_ptr[e] .. ref_ptr[e+1]-1]
  ref_idx [nref]  int32   ids of the slices with >0 valid pairs in a MASKED
                          tile, ascending (FULL tiles reference none)
  sched   [nq]    int32   query tiles by descending entry count, ties by
                          ascending index (longest-processing-time order)
  total_pairs     int64   sum of pairs

Two independent counters are given: ``oracle_tiles_dense`` enumerates the
dense mask of ``attention.mask_rows`` element by element (the plain
definition, small sizes), ``oracle_tiles`` sums per-row key intervals (any
size).  Parity: pinned (tests/test_oracle_tiles.py): the two agree on fuzzed
slice lists; a single causal slice of P*T tokens gives P(P-1)/2 FULL and P
MASKED tiles whose Full=1 / Causal=0.5 weights reproduce the W column of the
partition-degree table on the UltraAttn page (section 4.1); the first-column
plus diagonal pattern of the UltraAttn introduction has 7 of 16 blocks.
"""
from __future__ import annotations

from typing import Dict, List, Tuple

import numpy as np

from .attention import BI_CAUSAL, CAUSAL, FULL, INV_CAUSAL, mask_rows

KIND_FULL, KIND_MASKED = 1, 2


def slice_row_interval(sl, i):
    """Valid global key interval [lo, hi) of slice ``sl`` for query rows ``i``.

    For a fixed row the predicate of each kind (see ``attention``) bounds the
    local key index b from below and/or above, so the valid keys are one
    interval: full [0, L_k); causal [0, a + L_k - L_q + 1); inv-causal [a, L_k);
    bi-causal the intersection; all clipped to [0, L_k).  Works on arrays.
    """
    qs, qe, ks, ke, t = (int(x) for x in sl)
    a = np.asarray(i, dtype=np.int64) - qs
    lq, lk = qe - qs, ke - ks
    lo = np.zeros_like(a)
    hi = np.full_like(a, lk)
    if t in (CAUSAL, BI_CAUSAL):
        hi = np.minimum(hi, a + (lk - lq) + 1)
    if t in (INV_CAUSAL, BI_CAUSAL):
        lo = np.maximum(lo, a)
    if t not in (FULL, CAUSAL, INV_CAUSAL, BI_CAUSAL):
        raise ValueError(f"unknown slice type {t}")
    hi = np.maximum(hi, lo)
    return ks + lo, ks + hi


def _assemble(nq: int, tq: int, tk: int, counts: Dict[Tuple[int, int], int],
              contrib: Dict[Tuple[int, int], List[int]]):
    full_area = tq * tk
    rows: List[List[int]] = [[] for _ in range(nq)]
    for (qt, kt), c in counts.items():
        if c > 0:
            rows[qt].append(kt)
    row_ptr = [0]
    col_idx, kind, pairs, ref_ptr, ref_idx = [], [], [], [0], []
    for qt in range(nq):
        for kt in sorted(rows[qt]):
            c = counts[(qt, kt)]
            col_idx.append(kt)
            pairs.append(c)
            if c == full_area:
                kind.append(KIND_FULL)
            else:
                kind.append(KIND_MASKED)
                ref_idx.extend(sorted(contrib[(qt, kt)]))
            ref_ptr.append(len(ref_idx))
        row_ptr.append(len(col_idx))
    nnz_q = np.diff(np.asarray(row_ptr))
    sched = sorted(range(nq), key=lambda t: (-int(nnz_q[t]), t))
    return {
        "row_ptr": np.asarray(row_ptr, dtype=np.int32),
        "col_idx": np.asarray(col_idx, dtype=np.int32),
        "kind": np.asarray(kind, dtype=np.uint8),
        "pairs": np.asarray(pairs, dtype=np.int32),
        "ref_ptr": np.asarray(ref_ptr, dtype=np.int32),
        "ref_idx": np.asarray(ref_idx, dtype=np.int32),
        "sched": np.asarray(sched, dtype=np.int32),
        "total_pairs": int(sum(pairs)),
    }


def oracle_tiles(slices: np.ndarray, sq: int, sk: int, tq: int, tk: int):
    """Tile metadata by summing each row's valid key interval over key tiles."""
    nq = -(-sq // tq)
    counts: Dict[Tuple[int, int], int] = {}
    contrib: Dict[Tuple[int, int], List[int]] = {}
    for sid, sl in enumerate(np.asarray(slices, dtype=np.int64).reshape(-1, 5)):
        qs, qe, ks, ke, _ = (int(x) for x in sl)
        if qe <= qs or ke <= ks:
            continue
        rows = np.arange(qs, qe, dtype=np.int64)
        lo, hi = slice_row_interval(sl, rows)
        qt_of_row = rows // tq
        for kt in range(ks // tk, (ke - 1) // tk + 1):
            c0, c1 = kt * tk, (kt + 1) * tk
            ov = np.clip(np.minimum(hi, c1) - np.maximum(lo, c0), 0, None)
            per_qt = np.bincount(qt_of_row - qt_of_row[0], weights=ov).astype(np.int64)
            for off in np.nonzero(per_qt)[0]:
                key = (int(qt_of_row[0] + off), kt)
                counts[key] = counts.get(key, 0) + int(per_qt[off])
                contrib.setdefault(key, []).append(sid)
    return _assemble(nq, tq, tk, counts, contrib)


def oracle_tiles_dense(slices: np.ndarray, sq: int, sk: int, tq: int, tk: int):
    """Tile metadata by enumerating every element of every slice's dense mask."""
    nq = -(-sq // tq)
    nk = -(-sk // tk)
    counts: Dict[Tuple[int, int], int] = {}
    contrib: Dict[Tuple[int, int], List[int]] = {}
    all_rows = np.arange(sq)
    for sid, sl in enumerate(np.asarray(slices, dtype=np.int64).reshape(-1, 5)):
        M = mask_rows(sl[None, :], all_rows, sk)
        for qt in range(nq):
            for kt in range(nk):
                c = int(M[qt * tq:(qt + 1) * tq, kt * tk:(kt + 1) * tk].sum())
                if c:
                    counts[(qt, kt)] = counts.get((qt, kt), 0) + c
                    contrib.setdefault((qt, kt), []).append(sid)
    return _assemble(nq, tq, tk, counts, contrib)


def oracle_slices_from_grid(grid: np.ndarray, block: int) -> np.ndarray:
    """Slice list of a Full(1)/Causal(2)/Empty(0) block grid: one slice per
    non-Empty block in row-major block order, Full -> full slice of the block,
    Causal -> causal slice of the (square) block."""
    rows = []
    nbq, nbk = grid.shape
    for bi in range(nbq):
        for bj in range(nbk):
            g = int(grid[bi, bj])
            if g == 0:
                continue
            rows.append((bi * block, (bi + 1) * block, bj * block, (bj + 1) * block,
                         FULL if g == 1 else CAUSAL))
    return np.asarray(rows, dtype=np.int32).reshape(-1, 5)
