"""attn_bwd on the GPU vs the fp64 backward oracle on identical seeded inputs.

The kernels round P and dS to bf16 (unit roundoff 2^-9) before the MMAs
that consume them and accumulate in f32, and D = rowsum(dO * O) uses the
forward's own O; the bound below (2 % of each gradient's largest magnitude
elementwise, 0.5 % in relative L2 norm) is a few times that rounding, and far
below what a wrong mask, index or missing term produces.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle.backward import oracle_attention_backward
from block_sparse_attention_slice_gb300 import attn_build_tiles, attn_bwd, attn_fwd
from block_sparse_attention_slice_gb300 import workloads as W
from parity import f64

pytestmark = pytest.mark.gpu


def _check(name, got, ref):
    g = got.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(g)), name
    mx = float(np.abs(ref).max())
    err = float(np.abs(g - ref).max())
    l2 = float(np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30))
    assert err <= 2e-2 * mx + 1e-6, f"{name}: max err {err} vs max |ref| {mx}"
    assert l2 <= 5e-3, f"{name}: relative L2 error {l2}"
    return err / max(mx, 1e-30), l2


def _run(sl, sq, sk, H, Hk, d, seed, scale=None):
    rng = np.random.default_rng(seed)
    mk = lambda *sh: torch.from_numpy(rng.standard_normal(sh, dtype=np.float32)).to(torch.bfloat16)
    q, k, v, do = mk(sq, H, d), mk(sk, Hk, d), mk(sk, Hk, d), mk(sq, H, d)
    scale = scale or 1.0 / math.sqrt(d)
    tiles = attn_build_tiles(sl, sq, sk)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    out, lse = attn_fwd(qd, kd, vd, tiles, scale, out_dtype=torch.float32)
    dq, dk, dv = attn_bwd(qd, kd, vd, out, dod, lse, tiles, scale)
    rq, rk, rv, _ = oracle_attention_backward(f64(q), f64(k), f64(v), f64(do), scale,
                                              lambda r: oracle.mask_rows(sl, r, sk))
    return [_check("dq", dq, rq), _check("dk", dk, rk), _check("dv", dv, rv)]


@pytest.mark.parametrize("seed,sq,sk,H,Hk,d", [
    (0, 512, 512, 2, 1, 128), (1, 1000, 1100, 4, 2, 64), (2, 700, 1300, 2, 2, 128),
    (3, 1300, 600, 3, 1, 64), (4, 1536, 1536, 2, 2, 128), (5, 129, 257, 1, 1, 128),
    # S_q = 640: the last query tile's second half starts exactly at S_q
    (6, 640, 700, 2, 1, 128)])
def test_fuzzed_slices_all_kinds(seed, sq, sk, H, Hk, d):
    sl = W.random_slices(sq, sk, 30, seed=seed + 100, unit=1, max_len=max(16, min(sq, sk) // 2))
    _run(sl, sq, sk, H, Hk, d, seed)


def test_causal_gqa():
    S = 2048
    _run(np.array([[0, S, 0, S, 1]], np.int32), S, S, 4, 1, 128, 11)


def test_varlen_documents_short():
    docs = [300, 700, 128, 900]
    rows, o = [], 0
    for L in docs:
        rows.append((o, o + L, o, o + L, 1))
        o += L
    _run(np.array(rows, np.int32), o, o, 2, 2, 128, 12)


def test_block_grid_pattern():
    g = W.strided_grid(S=2048, block=128)
    from block_sparse_attention_slice_gb300 import attn_slices_from_block_grid
    sl = attn_slices_from_block_grid(g, 128, 128)
    _run(sl, 2048, 2048, 2, 1, 128, 13)


def test_keys_without_queries_get_zero_gradient():
    # keys [1024, 1536) are attended by no query
    sl = np.array([[0, 512, 0, 1024, 1], [512, 1024, 1536, 2048, 0]], np.int32)
    rng = np.random.default_rng(14)
    mk = lambda *sh: torch.from_numpy(rng.standard_normal(sh, dtype=np.float32)).to(torch.bfloat16).cuda()
    q, k, v, do = mk(1024, 2, 128), mk(2048, 2, 128), mk(2048, 2, 128), mk(1024, 2, 128)
    tiles = attn_build_tiles(sl, 1024, 2048)
    out, lse = attn_fwd(q, k, v, tiles, 0.09, out_dtype=torch.float32)
    dq, dk, dv = attn_bwd(q, k, v, out, do, lse, tiles, 0.09)
    assert torch.all(dk[1024:1536] == 0) and torch.all(dv[1024:1536] == 0)
    assert torch.any(dk[:1024] != 0) and torch.any(dv[1536:] != 0)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["varlen_causal", "block_sparse_strided"])
def test_workload_scale_sampled(name):
    # The backward at the size ``bench.py --pass bwd`` times, in the same
    # launch configuration: the transposed per-key-tile lists and the long
    # dK/dV walks of the packed documents (S = 16384) and of the block-sparse
    # grid (S = 32768, whose sink column 0 is reached by every query).  dK and
    # dV are compared at 512 seeded keys (plus key 0 and tile edges) of four
    # KV heads, dQ at 512 seeded rows of the same heads, against the sampled
    # form of the backward oracle.
    from oracle.backward import oracle_attention_backward_sampled
    from block_sparse_attention_slice_gb300 import attn_slices_from_block_grid
    from parity import THREADS, mask_fn
    w = W.ALL[name]()
    sl = attn_slices_from_block_grid(w.grid, w.block, w.block) if w.grid is not None else w.slices
    q, k, v = W.draw_qkv(w.S, w.H, w.Hk, w.d, w.seed)
    rng = np.random.default_rng(w.seed + 1)
    do = torch.from_numpy(rng.standard_normal((w.S, w.H, w.d), dtype=np.float32)).to(torch.bfloat16)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    tiles = attn_build_tiles(sl, w.S, w.S)
    out, lse = attn_fwd(qd, kd, vd, tiles, w.scale, out_dtype=torch.float32)
    dq, dk, dv = attn_bwd(qd, kd, vd, out, dod, lse, tiles, w.scale)
    torch.cuda.synchronize()
    heads = [0, 5, 10, 15]
    assert w.H == w.Hk            # one query head per KV head: heads double as groups
    mask = mask_fn(w)
    fwd = oracle.oracle_attention(f64(q), f64(k), f64(v), w.scale, mask, heads=heads,
                                  threads=min(THREADS, len(heads)))
    pick = np.random.default_rng(321)
    edges = [0, 1, 127, 128, w.S // 2, w.S - 1]
    keys = {g: np.unique(np.concatenate([pick.choice(w.S, 512, replace=False), edges]))
            for g in heads}
    rows = {h: np.unique(np.concatenate([pick.choice(w.S, 512, replace=False), edges]))
            for h in heads}
    sk, sv, sq = oracle_attention_backward_sampled(f64(q), f64(k), f64(v), f64(do), w.scale, mask,
                                                   fwd, keys, rows)
    dkc, dvc, dqc = dk.cpu(), dv.cpu(), dq.cpu()
    for g in heads:
        J = torch.as_tensor(keys[g])
        _check(f"dk head {g}", dkc[J, g], sk[g])
        _check(f"dv head {g}", dvc[J, g], sv[g])
        R = torch.as_tensor(rows[g])
        _check(f"dq head {g}", dqc[R, g], sq[g])
