"""The CTA-pair forward (metadata of 512-row query tiles, head dim 128)
against the fp64 oracle on the same seeded inputs as the single-CTA kernel.

Two CTAs of a cluster share each M = 256 tcgen05 MMA (FlashAttention-4 page,
2-CTA MMA): each holds 128 rows of both MMA tiles of a work item and loads
half of every K and V tile.  Same tolerances as the single-CTA kernel, and
the bf16 output is the round-to-nearest-even of the f32 output bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_slice_gb300 import (AttnError, attn_build_tiles, attn_fwd,
                                                attn_slices_from_block_grid)
from block_sparse_attention_slice_gb300 import binding as B
from block_sparse_attention_slice_gb300 import workloads as W
from parity import compare, f64, mask_fn, rows_per_head, run_oracle

pytestmark = pytest.mark.gpu
TQ = 512


def _qkv(w):
    q, k, v = W.draw_qkv(w.S, w.H, w.Hk, w.d, w.seed)
    return q, k, v, q.cuda(), k.cuda(), v.cuda()


def _fwd_checked(qd, kd, vd, tiles, scale):
    out, lse = attn_fwd(qd, kd, vd, tiles, scale, out_dtype=torch.float32)
    ob, lb = attn_fwd(qd, kd, vd, tiles, scale)
    torch.cuda.synchronize()
    assert B.attn_last_device_error() == 0
    assert torch.equal(ob.view(torch.int16), out.to(torch.bfloat16).view(torch.int16))
    assert torch.equal(lb.view(torch.int32), lse.view(torch.int32))
    return out, lse


def test_small_causal_and_ragged_tail():
    # 3 query tiles of 512 (the last one ragged), 2 heads over 1 KV head
    S = 1300
    rng = np.random.default_rng(41)
    mk = lambda h: torch.from_numpy(rng.standard_normal((S, h, 128), dtype=np.float32)).to(torch.bfloat16)
    q, k, v = mk(2), mk(1), mk(1)
    sl = np.array([[0, S, 0, S, 1]], np.int32)
    out, lse = _fwd_checked(q.cuda(), k.cuda(), v.cuda(), attn_build_tiles(sl, S, S, TQ, 128), 0.088)
    compare(out, lse, oracle.oracle_attention(f64(q), f64(k), f64(v), 0.088,
                                              lambda r: oracle.mask_rows(sl, r, S)))


def test_varlen_causal_all_rows():
    w = W.varlen_causal()
    q, k, v, qd, kd, vd = _qkv(w)
    out, lse = _fwd_checked(qd, kd, vd, attn_build_tiles(w.slices, w.S, w.S, TQ, 128), w.scale)
    compare(out, lse, run_oracle(q, k, v, w.scale, mask_fn(w)))


def test_block_sparse_strided_sampled():
    w = W.block_sparse_strided()
    q, k, v, qd, kd, vd = _qkv(w)
    sl = attn_slices_from_block_grid(w.grid, w.block, w.block)
    out, lse = _fwd_checked(qd, kd, vd, attn_build_tiles(sl, w.S, w.S, TQ, 128), w.scale)
    rows = rows_per_head(w, n=1024, extra=(0, 127, 128, 255, 256, 511, 512, w.S - 1))
    compare(out, lse, run_oracle(q, k, v, w.scale, mask_fn(w), rows=rows))


def test_video_slice_list_sampled():
    w = W.video_gen()
    q, k, v, qd, kd, vd = _qkv(w)
    out, lse = _fwd_checked(qd, kd, vd, attn_build_tiles(w.slices, w.S, w.S, TQ, 128), w.scale)
    extra = [0, 4095, 4096, 8191, w.S - 1] + [int(x) for s in w.slices for x in (s[0], s[1] - 1)]
    compare(out, lse, run_oracle(q, k, v, w.scale, mask_fn(w), rows=rows_per_head(w, n=1024, extra=extra)))


def test_gqa_causal_quarter_length_sampled():
    w = W.gqa_causal_32k()
    q, k, v, qd, kd, vd = _qkv(w)
    out, lse = _fwd_checked(qd, kd, vd, attn_build_tiles(w.slices, w.S, w.S, TQ, 128), w.scale)
    rows = rows_per_head(w, n=512, extra=(0, 255, 256, 511, 512, w.S - 1))
    compare(out, lse, run_oracle(q, k, v, w.scale, mask_fn(w), rows=rows))


@pytest.mark.parametrize("seed,sq,sk,H,Hk", [
    (0, 512, 512, 2, 1), (2, 700, 1300, 2, 2), (4, 2304, 2304, 2, 2), (5, 129, 257, 1, 1),
    (6, 3000, 1700, 4, 2)])
def test_fuzzed_slices_all_kinds(seed, sq, sk, H, Hk):
    rng = np.random.default_rng(seed)
    sl = W.random_slices(sq, sk, 30, seed=seed + 100, unit=1, max_len=max(16, min(sq, sk) // 2))
    q = torch.from_numpy(rng.standard_normal((sq, H, 128), dtype=np.float32)).to(torch.bfloat16)
    k = torch.from_numpy(rng.standard_normal((sk, Hk, 128), dtype=np.float32)).to(torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((sk, Hk, 128), dtype=np.float32)).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(128)
    out, lse = _fwd_checked(q.cuda(), k.cuda(), v.cuda(), attn_build_tiles(sl, sq, sk, TQ, 128), scale)
    compare(out, lse, oracle.oracle_attention(f64(q), f64(k), f64(v), scale,
                                              lambda r: oracle.mask_rows(sl, r, sk)))


@pytest.mark.parametrize("kind", [0, 1, 2, 3])
def test_uniform_scores_give_means(kind):
    S = 1152
    rng = np.random.default_rng(kind)
    q = torch.zeros((S, 1, 128), dtype=torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((S, 1, 128), dtype=np.float32)).to(torch.bfloat16)
    k = torch.from_numpy(rng.standard_normal((S, 1, 128), dtype=np.float32)).to(torch.bfloat16)
    sl = np.array([[40, 1100, 40, 1100, kind]], np.int32)
    out, lse = attn_fwd(q.cuda(), k.cuda(), v.cuda(), attn_build_tiles(sl, S, S, TQ, 128), 0.125,
                        out_dtype=torch.float32)
    o, l, vv = out.cpu().numpy()[:, 0], lse.cpu().numpy()[0], f64(v)[:, 0]
    for i in range(S):
        if not 40 <= i < 1100:
            assert l[i] == -np.inf and np.all(o[i] == 0)
            continue
        a = i - 40
        keys = list({0: range(40, 1100), 1: range(40, 41 + a), 2: range(40 + a, 1100),
                     3: [40 + a]}[kind])
        assert abs(l[i] - math.log(len(keys))) < 1e-4
        assert np.abs(o[i] - vv[keys].mean(axis=0)).max() < 1e-4


def test_mostly_empty_query_tiles():
    sq, sk, H, Hk = 8192, 2048, 48, 16
    rng = np.random.default_rng(11)
    sl = np.array([[0, 256, 0, 2048, 0], [7936, 8192, 0, 1024, 1], [3000, 3100, 500, 700, 3]],
                  np.int32)
    q = torch.from_numpy(rng.standard_normal((sq, H, 128), dtype=np.float32)).to(torch.bfloat16)
    k = torch.from_numpy(rng.standard_normal((sk, Hk, 128), dtype=np.float32)).to(torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((sk, Hk, 128), dtype=np.float32)).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(128)
    out, lse = _fwd_checked(q.cuda(), k.cuda(), v.cuda(), attn_build_tiles(sl, sq, sk, TQ, 128), scale)
    rows = [np.concatenate([np.arange(0, 300), np.arange(2990, 3110), np.arange(7900, 8192)])] * H
    compare(out, lse, oracle.oracle_attention(f64(q), f64(k), f64(v), scale,
                                              lambda r: oracle.mask_rows(sl, r, sk), rows=rows))
    empty = torch.ones(sq, dtype=torch.bool)
    for a, b, *_ in sl:
        empty[a:b] = False
    assert torch.all(out.cpu()[empty] == 0)
    assert torch.all(torch.isneginf(lse.cpu()[:, empty]))


def test_same_result_as_the_single_cta_kernel_up_to_rounding():
    # both kernels compute the same softmax; the pair kernel only changes
    # which CTA holds which rows and operand halves, so the f32 outputs agree
    # to a few f32 roundings
    w = W.varlen_causal()
    q, k, v, qd, kd, vd = _qkv(w)
    o1, l1 = attn_fwd(qd, kd, vd, attn_build_tiles(w.slices, w.S, w.S), w.scale, out_dtype=torch.float32)
    o2, l2 = attn_fwd(qd, kd, vd, attn_build_tiles(w.slices, w.S, w.S, TQ, 128), w.scale,
                      out_dtype=torch.float32)
    assert float((o1 - o2).abs().max()) < 2e-2
    assert float((l1 - l2).abs().max()) < 1e-3


def test_pair_tiles_need_head_dim_128():
    S = 1024
    q = torch.zeros((S, 1, 64), dtype=torch.bfloat16, device="cuda")
    t = attn_build_tiles(np.array([[0, S, 0, S, 1]], np.int32), S, S, TQ, 128)
    with pytest.raises(AttnError) as e:
        attn_fwd(q, q, q, t, 0.125)
    assert e.value.code == B.ATTN_ERR_UNSUPPORTED


def test_kv_split_partials_merged():
    # the pair kernel writing f32 partials of a 4-way KV split of the
    # quarter-length GQA causal problem, merged by attn_merge, against the
    # oracle of the whole problem (the chunk-c partial: the causal diagonal
    # block of chunk c and the full block of every later row against it)
    from block_sparse_attention_slice_gb300 import attn_merge
    w = W.gqa_causal_32k()
    q, k, v, qd, kd, vd = _qkv(w)
    c = w.S // 4
    parts = []
    for i in range(4):
        rows = [(i * c, (i + 1) * c, i * c, (i + 1) * c, W.CAUSAL)]
        if (i + 1) * c < w.S:
            rows.append(((i + 1) * c, w.S, i * c, (i + 1) * c, W.FULL))
        t = attn_build_tiles(np.asarray(rows, np.int32), w.S, w.S, TQ, 128)
        parts.append(attn_fwd(qd, kd, vd, t, w.scale, out_dtype=torch.float32))
    mo, ml = attn_merge([x[0] for x in parts], [x[1] for x in parts], out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert B.attn_last_device_error() == 0
    rows = rows_per_head(w, n=256, extra=[0, 511, 512, w.S - 1] + [i * c + o for i in range(4) for o in (-1, 0)])
    compare(mo, ml, run_oracle(q, k, v, w.scale, mask_fn(w), rows=rows))


def test_pair_abort_path_ends_with_timeout(monkeypatch):
    # the pair's abort path, driven like the single-CTA kernel's: with
    # ATTN_TEST_STALL_FWD=1 both CTAs of every pair leave their second K/V
    # load unissued, so rank 0's bounded wait for that slot runs out; both
    # CTAs leave their waits, rank 0 waits for its loads and MMAs, rank 1
    # gives its loads a bounded time to land, and the pair meets at its
    # closing cluster barrier before freeing tensor memory.  Afterwards the
    # forward is bit-identical to a run made before.
    from block_sparse_attention_slice_gb300 import attn_set_wait_limit_ns
    S, H, Hk = 8192, 4, 2
    rng = np.random.default_rng(8)
    mk = lambda h: torch.from_numpy(rng.standard_normal((S, h, 128), dtype=np.float32)).to(torch.bfloat16).cuda()
    q, k, v = mk(H), mk(Hk), mk(Hk)
    t = attn_build_tiles(np.array([[0, S, 0, S, 1]], np.int32), S, S, TQ, 128)
    ref_o, ref_l = attn_fwd(q, k, v, t, 0.088)
    torch.cuda.synchronize()
    assert B.attn_last_device_error() == 0
    attn_set_wait_limit_ns(50_000_000)
    monkeypatch.setenv("ATTN_TEST_STALL_FWD", "1")
    try:
        attn_fwd(q, k, v, t, 0.088)
        rc = B.attn_last_device_error()
    finally:
        monkeypatch.delenv("ATTN_TEST_STALL_FWD")
        attn_set_wait_limit_ns(4_000_000_000)
    assert rc == B.ATTN_ERR_TIMEOUT
    o2, l2 = attn_fwd(q, k, v, t, 0.088)
    torch.cuda.synchronize()
    assert B.attn_last_device_error() == 0
    assert torch.equal(o2.view(torch.int16), ref_o.view(torch.int16))
    assert torch.equal(l2.view(torch.int32), ref_l.view(torch.int32))
