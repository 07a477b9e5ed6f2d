"""attn_fwd / attn_merge on the GPU vs the fp64 oracle on identical seeded inputs.

Workloads: the five problem configurations (tiny causal with a 2-way KV
split, packed varlen causal documents, a block-sparse strided grid, a
video-generation slice list, a long GQA causal problem with an 8-way KV
split), plus fuzzed slice lists over all four slice kinds with ragged sizes,
both head dims, grouped heads, closed-form uniform-score cases and an
Empty-tile poisoning check and a head-dim-64 problem with many work items
per CTA.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_slice_gb300 import (attn_build_tiles, attn_fwd, attn_last_device_error, attn_merge,
                                                attn_slices_from_block_grid)
from block_sparse_attention_slice_gb300 import workloads as W
from parity import SAMPLE_ROWS, compare, f64, mask_fn, rows_per_head, run_oracle

pytestmark = pytest.mark.gpu


def _qkv(w):
    q, k, v = W.draw_qkv(w.S, w.H, w.Hk, w.d, w.seed)
    return q, k, v, q.cuda(), k.cuda(), v.cuda()


def _slices(w):
    if w.grid is not None:
        return attn_slices_from_block_grid(w.grid, w.block, w.block)
    return w.slices


def _fwd_checked(qd, kd, vd, tiles, scale):
    """Forward with f32 output (compared with the oracle) and with bf16
    output, which must be the round-to-nearest-even of the f32 result bit for
    bit: bf16 itself cannot resolve 1e-2 once |O| >= 4 (half an ulp there is
    2^-6), so the numeric tolerance applies to the computed O."""
    out, lse = attn_fwd(qd, kd, vd, tiles, scale, out_dtype=torch.float32)
    ob, lb = attn_fwd(qd, kd, vd, tiles, scale)
    assert torch.equal(ob.view(torch.int16), out.to(torch.bfloat16).view(torch.int16))
    assert torch.equal(lb.view(torch.int32), lse.view(torch.int32))
    return out, lse


def _split_and_merge(w, qd, kd, vd):
    parts = []
    for sl in w.kv_splits:
        t = attn_build_tiles(sl, w.S, w.S)
        parts.append(attn_fwd(qd, kd, vd, t, w.scale, out_dtype=torch.float32))
    return parts, attn_merge([p[0] for p in parts], [p[1] for p in parts], out_dtype=torch.float32)


def test_tiny_causal_and_kv_split():
    w = W.tiny_causal()
    q, k, v, qd, kd, vd = _qkv(w)
    ref = run_oracle(q, k, v, w.scale, mask_fn(w))
    out, lse = _fwd_checked(qd, kd, vd, attn_build_tiles(w.slices, w.S, w.S), w.scale)
    compare(out, lse, ref)
    parts, (mo, ml) = _split_and_merge(w, qd, kd, vd)
    compare(mo, ml, ref)
    # each partial against the oracle of its own slice list
    for sl, (po, pl) in zip(w.kv_splits, parts):
        compare(po, pl, run_oracle(q, k, v, w.scale, mask_fn(w, sl)))


def test_varlen_causal_all_rows():
    w = W.varlen_causal()
    q, k, v, qd, kd, vd = _qkv(w)
    out, lse = _fwd_checked(qd, kd, vd, attn_build_tiles(w.slices, w.S, w.S), w.scale)
    compare(out, lse, run_oracle(q, k, v, w.scale, mask_fn(w)))


def test_block_sparse_strided_sampled():
    w = W.block_sparse_strided()
    q, k, v, qd, kd, vd = _qkv(w)
    out, lse = _fwd_checked(qd, kd, vd, attn_build_tiles(_slices(w), w.S, w.S), w.scale)
    rows = rows_per_head(w, extra=(0, 127, 128, 255, 256, w.S - 1))
    compare(out, lse, run_oracle(q, k, v, w.scale, mask_fn(w), rows=rows))


def test_video_slice_list_sampled():
    w = W.video_gen()
    q, k, v, qd, kd, vd = _qkv(w)
    out, lse = _fwd_checked(qd, kd, vd, attn_build_tiles(w.slices, w.S, w.S), w.scale)
    extra = [0, 4095, 4096, 8191, w.S - 1] + [int(x) for s in w.slices for x in (s[0], s[1] - 1)]
    rows = rows_per_head(w, extra=extra)
    compare(out, lse, run_oracle(q, k, v, w.scale, mask_fn(w), rows=rows))


@pytest.mark.slow
def test_long_gqa_causal_whole_and_kv_split_sampled():
    # the bench's headline problem in its own launch configuration: the whole
    # forward with both output types (bf16 must be the RNE of f32 bit for
    # bit), and the 8-way KV split merged to f32 and to bf16
    w = W.gqa_causal_kv_split()
    q, k, v, qd, kd, vd = _qkv(w)
    out, lse = _fwd_checked(qd, kd, vd, attn_build_tiles(w.slices, w.S, w.S), w.scale)
    extra = [0, 127, 128, w.S - 1] + [c * (w.S // 8) + o for c in range(8) for o in (-1, 0)]
    rows = rows_per_head(w, extra=extra)
    ref = run_oracle(q, k, v, w.scale, mask_fn(w), rows=rows)
    compare(out, lse, ref)
    del out, lse
    parts, (mo, ml) = _split_and_merge(w, qd, kd, vd)
    mb, lb = attn_merge([p[0] for p in parts], [p[1] for p in parts])
    del parts
    assert torch.equal(mb.view(torch.int16), mo.to(torch.bfloat16).view(torch.int16))
    assert torch.equal(lb.view(torch.int32), ml.view(torch.int32))
    compare(mo, ml, ref)


def test_d64_varlen_many_items_per_cta():
    # head dim 64 on the packed-document workload with 4 query heads per KV
    # head: 1024 work items, so every CTA runs several items back to back
    # with row lengths from 2 to 16 key tiles
    import dataclasses
    w = dataclasses.replace(W.varlen_causal(), name="varlen_causal_s16384_h16_hk4_d64",
                            Hk=4, d=64, scale=0.125)
    q, k, v, qd, kd, vd = _qkv(w)
    out, lse = _fwd_checked(qd, kd, vd, attn_build_tiles(w.slices, w.S, w.S), w.scale)
    extra = [0, 127, 128, 255, 256, w.S - 1] + [int(x) for s in w.slices for x in (s[0], s[1] - 1)]
    rows = rows_per_head(w, n=512, extra=extra)
    compare(out, lse, run_oracle(q, k, v, w.scale, mask_fn(w), rows=rows))


@pytest.mark.parametrize("seed,sq,sk,H,Hk,d", [
    (0, 512, 512, 2, 1, 128), (1, 1000, 1100, 4, 2, 64), (2, 700, 1300, 2, 2, 128),
    (3, 1300, 600, 3, 1, 64), (4, 2304, 2304, 2, 2, 128), (5, 129, 257, 1, 1, 128)])
def test_fuzzed_slices_all_kinds(seed, sq, sk, H, Hk, d):
    rng = np.random.default_rng(seed)
    sl = W.random_slices(sq, sk, 30, seed=seed + 100, unit=1, max_len=max(16, min(sq, sk) // 2))
    assert len(sl) > 5
    q = torch.from_numpy(rng.standard_normal((sq, H, d), dtype=np.float32)).to(torch.bfloat16)
    k = torch.from_numpy(rng.standard_normal((sk, Hk, d), dtype=np.float32)).to(torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((sk, Hk, d), dtype=np.float32)).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    tiles = attn_build_tiles(sl, sq, sk)
    out, lse = _fwd_checked(q.cuda(), k.cuda(), v.cuda(), tiles, scale)
    ref = oracle.oracle_attention(f64(q), f64(k), f64(v), scale,
                                  lambda r: oracle.mask_rows(sl, r, sk))
    compare(out, lse, ref)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("kind", [0, 1, 2, 3])
def test_uniform_scores_give_means(kind, d):
    # q = 0: every score is 0, so P = 1 exactly and O is the mean of V over
    # the valid keys (closed form), lse = ln(count).
    S = 640
    rng = np.random.default_rng(kind)
    q = torch.zeros((S, 1, d), dtype=torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((S, 1, d), dtype=np.float32)).to(torch.bfloat16)
    k = torch.from_numpy(rng.standard_normal((S, 1, d), dtype=np.float32)).to(torch.bfloat16)
    sl = np.array([[40, 600, 40, 600, kind]], np.int32)
    out, lse = attn_fwd(q.cuda(), k.cuda(), v.cuda(), attn_build_tiles(sl, S, S), 0.125,
                        out_dtype=torch.float32)
    o, l, vv = out.cpu().numpy()[:, 0], lse.cpu().numpy()[0], f64(v)[:, 0]
    for i in range(S):
        if not 40 <= i < 600:
            assert l[i] == -np.inf and np.all(o[i] == 0)
            continue
        a = i - 40
        keys = {0: range(40, 600), 1: range(40, 41 + a), 2: range(40 + a, 600), 3: [40 + a]}[kind]
        keys = list(keys)
        assert abs(l[i] - math.log(len(keys))) < 1e-4
        assert np.abs(o[i] - vv[keys].mean(axis=0)).max() < 1e-4


def test_empty_tiles_never_read():
    # Key tiles [1024, 1536) are Empty for every query tile: poisoning their
    # K and V with NaN / huge values must leave the output bit-identical.
    sq, sk, H, d = 1024, 2048, 2, 128
    rng = np.random.default_rng(3)
    sl = np.array([[0, 512, 0, 1024, 1], [512, 1024, 0, 700, 0], [512, 1024, 1536, 2048, 2],
                   [0, 300, 1600, 1900, 3]], np.int32)
    q = torch.from_numpy(rng.standard_normal((sq, H, d), dtype=np.float32)).to(torch.bfloat16).cuda()
    k = torch.from_numpy(rng.standard_normal((sk, H, d), dtype=np.float32)).to(torch.bfloat16).cuda()
    v = torch.from_numpy(rng.standard_normal((sk, H, d), dtype=np.float32)).to(torch.bfloat16).cuda()
    tiles = attn_build_tiles(sl, sq, sk)
    assert not np.isin(tiles.to_host()["col_idx"], [8, 9, 10, 11]).any()
    o1, l1 = attn_fwd(q, k, v, tiles, 0.09)
    k2, v2 = k.clone(), v.clone()
    k2[1024:1536] = float("nan")
    v2[1024:1536] = 65504.0
    v2[1024:1100] = float("nan")
    o2, l2 = attn_fwd(q, k2, v2, tiles, 0.09)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))


@pytest.mark.parametrize("d", [64, 128])
def test_mostly_empty_query_tiles(d):
    # 28 of 32 query tiles have no key tile: with 48 heads that is 192
    # non-empty and 1344 empty work items, the empty ones last in the LPT
    # order, so CTAs run several items and meet runs of empty items right
    # after their last non-empty one; those rows must come out as O = 0,
    # lse = -inf.
    sq, sk, H, Hk = 8192, 2048, 48, 16
    rng = np.random.default_rng(11)
    sl = np.array([[0, 256, 0, 2048, 0], [7936, 8192, 0, 1024, 1], [3000, 3100, 500, 700, 3]],
                  np.int32)
    q = torch.from_numpy(rng.standard_normal((sq, H, d), dtype=np.float32)).to(torch.bfloat16)
    k = torch.from_numpy(rng.standard_normal((sk, Hk, d), dtype=np.float32)).to(torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((sk, Hk, d), dtype=np.float32)).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    out, lse = _fwd_checked(q.cuda(), k.cuda(), v.cuda(), attn_build_tiles(sl, sq, sk), scale)
    rows = [np.concatenate([np.arange(0, 300), np.arange(2990, 3110), np.arange(7900, 8192),
                            np.arange(5000, 5010)])] * H
    ref = oracle.oracle_attention(f64(q), f64(k), f64(v), scale,
                                  lambda r: oracle.mask_rows(sl, r, sk), rows=rows)
    compare(out, lse, ref)
    empty = torch.ones(sq, dtype=torch.bool)
    for a, b, *_ in sl:
        empty[a:b] = False
    assert torch.all(out.cpu()[empty] == 0)
    assert torch.all(torch.isneginf(lse.cpu()[:, empty]))


def test_repeat_runs_bit_identical():
    w = W.tiny_causal()
    q, k, v, qd, kd, vd = _qkv(w)
    t = attn_build_tiles(w.slices, w.S, w.S)
    a = attn_fwd(qd, kd, vd, t, w.scale)
    b = attn_fwd(qd, kd, vd, t, w.scale)
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1], b[1])


def test_concurrent_streams_share_the_library_rings():
    # forwards and metadata builds of two different problems enqueued on two
    # streams at once, several times: each launch takes its own work counter
    # and grid-barrier slot from the library's rings, so the results must be
    # bit-identical to the same calls made one at a time
    rng = np.random.default_rng(31)
    probs = []
    for S, H, Hk, sl in ((4096, 8, 2, np.array([[0, 4096, 0, 4096, 1]], np.int32)),
                         (3000, 4, 4, W.random_slices(3000, 3000, 20, seed=77, unit=1, max_len=900))):
        mk = lambda h: torch.from_numpy(rng.standard_normal((S, h, 128), dtype=np.float32)).to(torch.bfloat16).cuda()
        probs.append((S, sl, mk(H), mk(Hk), mk(Hk)))
    ref = []
    for S, sl, q, k, v in probs:
        t = attn_build_tiles(sl, S, S)
        ref.append(attn_fwd(q, k, v, t, 0.088))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for _ in range(4):
        outs, keep = [], []
        for (S, sl, q, k, v), st in zip(probs, streams):
            with torch.cuda.stream(st):
                keep.append(attn_build_tiles(sl, S, S))
                outs.append(attn_fwd(q, k, v, keep[-1], 0.088))
        torch.cuda.synchronize()
        for (o, l), (ro, rl) in zip(outs, ref):
            assert torch.equal(o.view(torch.int16), ro.view(torch.int16))
            assert torch.equal(l.view(torch.int32), rl.view(torch.int32))
    assert attn_last_device_error() == 0


def test_forward_and_merge_replayed_from_a_cuda_graph():
    # a serving loop captures attn_fwd (two KV-split partials) and attn_merge
    # once and replays them; the replays must equal the eager calls bit for
    # bit (each replay reuses the work counter the capture took, one replay
    # at a time, as the header requires)
    w = W.tiny_causal()
    q, k, v, qd, kd, vd = _qkv(w)
    tiles = [attn_build_tiles(sl, w.S, w.S) for sl in w.kv_splits]
    parts = [attn_fwd(qd, kd, vd, t, w.scale, out_dtype=torch.float32) for t in tiles]   # eager (and warm-up)
    ref_o, ref_l = attn_merge([p[0] for p in parts], [p[1] for p in parts])
    torch.cuda.synchronize()
    outs = [(torch.empty_like(p[0]), torch.empty_like(p[1])) for p in parts]
    mo, ml = torch.empty_like(ref_o), torch.empty_like(ref_l)
    g = torch.cuda.CUDAGraph()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        with torch.cuda.graph(g, stream=st):
            for t, (o, l) in zip(tiles, outs):
                attn_fwd(qd, kd, vd, t, w.scale, out=o, lse=l)
            attn_merge([o for o, _ in outs], [l for _, l in outs], out=mo, lse=ml)
    for _ in range(3):
        mo.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(mo.view(torch.int16), ref_o.view(torch.int16))
        assert torch.equal(ml.view(torch.int32), ref_l.view(torch.int32))
    assert attn_last_device_error() == 0
