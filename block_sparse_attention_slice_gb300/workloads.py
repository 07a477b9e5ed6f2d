"""Seeded synthetic workloads for masked-attention forward.

This module only *draws inputs*: query/key/value tensors and the mask
description (a slice list or a Full/Causal/Empty block grid).  It holds none
of the method's arithmetic -- no softmax, no tile classification, no
grid-to-slice conversion -- so both the CUDA path and the CPU oracle can take
their inputs from here without sharing any code of the method.

Mask slices are ``int32[n, 5]`` rows ``(q_start, q_end, k_start, k_end,
type)`` with half-open ranges and ``type`` in {0 full, 1 causal,
2 inv-causal, 3 bi-causal}: the slice form of a flexible mask described on
the MagiAttention v1.1.0 page ("Blackwell adaptation", flexible-mask bullet).
A block grid is ``uint8[nbq, nbk]`` with 0 Empty, 1 Full, 2 Causal, the block
taxonomy of the UltraAttn page (section 3, two-dimensional attention work).

The five workloads follow the problem statement of the build: tiny causal,
packed varlen causal documents, block-sparse strided, a video-generation
style slice list and a long GQA causal problem with an 8-way KV split.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

FULL, CAUSAL, INV_CAUSAL, BI_CAUSAL = 0, 1, 2, 3
GRID_EMPTY, GRID_FULL, GRID_CAUSAL = 0, 1, 2


@dataclass
class Workload:
    name: str
    S: int                      # sequence length (self-attention: S_q = S_k = S)
    H: int                      # query heads
    Hk: int                     # key/value heads
    d: int                      # head dim
    scale: float
    seed: int                   # seed of the q, k, v draw
    slices: Optional[np.ndarray] = None     # int32 [n, 5]
    grid: Optional[np.ndarray] = None       # uint8 [nbq, nbk]
    block: int = 0                          # block size of ``grid``
    kv_splits: List[np.ndarray] = field(default_factory=list)  # slice list per KV partial
    sample_rows: bool = False               # parity / baseline on sampled rows
    note: str = ""


def draw_qkv(S: int, H: int, Hk: int, d: int, seed: int):
    """Q [S,H,d], K/V [S,Hk,d] as torch bf16 on the CPU.

    numpy ``default_rng(seed).standard_normal(dtype=float32)`` is drawn in
    the order q, k, v and rounded to bf16 (round-to-nearest-even) by torch.
    """
    import torch
    rng = np.random.default_rng(seed)
    out = []
    for shape in ((S, H, d), (S, Hk, d), (S, Hk, d)):
        x = rng.standard_normal(size=shape, dtype=np.float32)
        out.append(torch.from_numpy(x).to(torch.bfloat16))
    return tuple(out)


def _sl(rows):
    return np.asarray(rows, dtype=np.int32).reshape(-1, 5)


def tiny_causal() -> Workload:
    """B=1, H=1, S=512, d=64, one causal slice, seed 0; plus the same problem
    with the keys split at 256 into two partials (recombined by the merge)."""
    S = 512
    part_a = _sl([(0, 256, 0, 256, CAUSAL), (256, 512, 0, 256, FULL)])
    part_b = _sl([(256, 512, 256, 512, CAUSAL)])
    return Workload("tiny_causal_s512_h1_d64", S, 1, 1, 64, 1.0 / 8.0, 0,
                    slices=_sl([(0, S, 0, S, CAUSAL)]), kv_splits=[part_a, part_b])


def varlen_doc_lengths(total: int = 16384, seed: int = 1, lo: int = 512, hi: int = 4096):
    rng = np.random.default_rng(seed)
    docs, s = [], 0
    while s < total:
        L = int(rng.integers(lo, hi + 1))
        docs.append(L)
        s += L
    docs[-1] -= s - total
    return docs


def varlen_causal() -> Workload:
    """Packed documents, total 16384 tokens, lengths uniform in [512, 4096]
    (seed 1, last one truncated), H=16, d=128, one causal slice per document
    on the block diagonal."""
    docs = varlen_doc_lengths()
    rows, o = [], 0
    for L in docs:
        rows.append((o, o + L, o, o + L, CAUSAL))
        o += L
    return Workload("varlen_causal_s16384_h16_d128", 16384, 16, 16, 128,
                    1.0 / np.sqrt(128.0), 0, slices=_sl(rows),
                    note="docs=" + ",".join(map(str, docs)))


def strided_grid(S: int = 32768, block: int = 128, band: int = 4, stride: int = 8) -> np.ndarray:
    """Block grid: global-sink column 0, a causal band of ``band`` blocks on the
    diagonal (diagonal Causal, the rest Full) and every ``stride``-th column
    below the diagonal (Full); everything else Empty."""
    nb = S // block
    g = np.zeros((nb, nb), dtype=np.uint8)
    for r in range(nb):
        g[r, 0] = GRID_FULL
        for c in range(max(0, r - band + 1), r + 1):
            g[r, c] = GRID_FULL
        g[r, 0:r:stride] = GRID_FULL
        g[r, r] = GRID_CAUSAL
    return g


def block_sparse_strided() -> Workload:
    """S=32768, H=16, d=128, 128x128 block grid (sink + band 4 + every 8th)."""
    return Workload("block_sparse_strided_s32768_h16_d128", 32768, 16, 16, 128,
                    1.0 / np.sqrt(128.0), 0, grid=strided_grid(), block=128,
                    sample_rows=True)


def video_slices(S: int = 65536, chunk: int = 4096, n_extra: int = 32, seed: int = 4,
                 unit: int = 256) -> np.ndarray:
    """Video-generation style slice list: chunk 0 is a prefix every chunk
    attends Full, chunk i attends Full to itself and Causal to chunk i-1, plus
    ``n_extra`` random disjoint slices (ranges in ``unit`` tokens, type uniform
    over the four kinds) placed where no other slice lies."""
    nc = S // chunk
    rows = []
    for i in range(nc):
        rows.append((i * chunk, (i + 1) * chunk, 0, chunk, FULL))
    for i in range(1, nc):
        rows.append((i * chunk, (i + 1) * chunk, i * chunk, (i + 1) * chunk, FULL))
    for i in range(2, nc):
        rows.append((i * chunk, (i + 1) * chunk, (i - 1) * chunk, i * chunk, CAUSAL))
    rng = np.random.default_rng(seed)
    nu = S // unit
    extras = []
    while len(extras) < n_extra:
        qs = int(rng.integers(0, nu)); ks = int(rng.integers(0, nu))
        lq = int(rng.integers(1, 17)); lk = int(rng.integers(1, 17))
        typ = int(rng.integers(0, 4))
        q0, q1 = qs * unit, min(S, (qs + lq) * unit)
        k0, k1 = ks * unit, min(S, (ks + lk) * unit)
        clash = False
        for (a0, a1, b0, b1, _) in rows + extras:
            if q0 < a1 and a0 < q1 and k0 < b1 and b0 < k1:
                clash = True
                break
        if not clash:
            extras.append((q0, q1, k0, k1, typ))
    return _sl(rows + extras)


def video_gen() -> Workload:
    """S=65536 as 16 chunks of 4096, H=16, d=128 (prefix + self + previous
    chunk causal + 32 random extra slices)."""
    return Workload("video_slices_s65536_h16_d128", 65536, 16, 16, 128,
                    1.0 / np.sqrt(128.0), 0, slices=video_slices(), sample_rows=True)


def gqa_causal_kv_split(S: int = 131072, H: int = 32, Hk: int = 8, n_split: int = 8) -> Workload:
    """S=131072, 32 query heads / 8 KV heads, d=128, one causal slice; and the
    same problem with keys split into ``n_split`` contiguous chunks."""
    c = S // n_split
    splits = []
    for i in range(n_split):
        rows = [(i * c, (i + 1) * c, i * c, (i + 1) * c, CAUSAL)]
        if (i + 1) * c < S:
            rows.append(((i + 1) * c, S, i * c, (i + 1) * c, FULL))
        splits.append(_sl(rows))
    return Workload("gqa_causal_s131072_h32_hk8_d128", S, H, Hk, 128,
                    1.0 / np.sqrt(128.0), 0, slices=_sl([(0, S, 0, S, CAUSAL)]),
                    kv_splits=splits, sample_rows=True)


def gqa_causal_32k() -> Workload:
    """The long GQA causal problem at a quarter of its length: S=32768,
    32 query heads / 8 KV heads, d=128, one causal slice, no KV split.  Its
    inputs (470 MB) exceed L2, so it stands in for the S=131072 forward where
    a profiler capture of the full size would hold too much device memory."""
    w = gqa_causal_kv_split(S=32768)
    return Workload("gqa_causal_s32768_h32_hk8_d128", w.S, w.H, w.Hk, w.d, w.scale, w.seed,
                    slices=w.slices, sample_rows=True)


ALL = {
    "tiny_causal": tiny_causal,
    "varlen_causal": varlen_causal,
    "block_sparse_strided": block_sparse_strided,
    "video_gen": video_gen,
    "gqa_causal": gqa_causal_kv_split,
    "gqa_causal_32k": gqa_causal_32k,
}


def sample_rows(S: int, h: int, n: int = 4096, extra=()) -> np.ndarray:
    """Sorted query rows checked for head ``h``: ``default_rng(100+h)`` draws
    ``n`` distinct rows, plus the listed boundary rows."""
    rng = np.random.default_rng(100 + h)
    r = rng.choice(S, size=min(n, S), replace=False)
    r = np.concatenate([r, np.asarray([x for x in extra if 0 <= x < S], dtype=np.int64)])
    return np.unique(r.astype(np.int64))


def random_slices(S_q: int, S_k: int, n: int, seed: int, unit: int = 1,
                  max_len: Optional[int] = None) -> np.ndarray:
    """Up to ``n`` random disjoint slices of random type on an S_q x S_k
    grid (rectangle corners on multiples of ``unit``); used for fuzzing."""
    rng = np.random.default_rng(seed)
    nq, nk = max(1, S_q // unit), max(1, S_k // unit)
    ml = max_len or max(nq, nk)
    rows = []
    tries = 0
    while len(rows) < n and tries < 50 * n + 100:
        tries += 1
        qs = int(rng.integers(0, nq)); ks = int(rng.integers(0, nk))
        lq = int(rng.integers(1, ml + 1)); lk = int(rng.integers(1, ml + 1))
        typ = int(rng.integers(0, 4))
        q0, q1 = qs * unit, min(S_q, (qs + lq) * unit)
        k0, k1 = ks * unit, min(S_k, (ks + lk) * unit)
        if q1 <= q0 or k1 <= k0:
            continue
        if any(q0 < a1 and a0 < q1 and k0 < b1 and b0 < k1 for (a0, a1, b0, b1, _) in rows):
            continue
        rows.append((q0, q1, k0, k1, typ))
    return _sl(rows)
