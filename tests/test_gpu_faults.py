"""Failure paths that fault no GPU: host-side argument rejection before any
launch, and a bounded device wait that runs out and reports a status."""
import numpy as np
import pytest
import torch

from block_sparse_attention_slice_gb300 import (AttnError, attn_build_tiles, attn_fwd,
                                                attn_last_device_error, attn_selftest_wait_timeout,
                                                attn_set_wait_limit_ns)
from block_sparse_attention_slice_gb300 import binding as B

pytestmark = pytest.mark.gpu


def _qkv(S=512, H=2, Hk=2, d=128):
    g = torch.Generator().manual_seed(0)
    mk = lambda h: torch.randn((S, h, d), generator=g).to(torch.bfloat16).cuda()
    return mk(H), mk(Hk), mk(Hk)


def test_rejects_bad_arguments_on_host():
    q, k, v = _qkv()
    t = attn_build_tiles(np.array([[0, 512, 0, 512, 1]], np.int32), 512, 512)
    with pytest.raises(AttnError) as e:
        attn_fwd(q[:, :, :96].contiguous(), k[:, :, :96].contiguous(), v[:, :, :96].contiguous(), t, 0.1)
    assert e.value.code == B.ATTN_ERR_UNSUPPORTED
    with pytest.raises(AttnError) as e:
        attn_fwd(q, k, v, t, -1.0)
    assert e.value.code == B.ATTN_ERR_INVALID_ARG
    q3 = torch.zeros((512, 3, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(AttnError) as e:
        attn_fwd(q3, k, v, t, 0.1)
    assert e.value.code == B.ATTN_ERR_INVALID_ARG          # 3 % 2 != 0
    t128 = attn_build_tiles(np.array([[0, 512, 0, 512, 1]], np.int32), 512, 512, 128, 128)
    with pytest.raises(AttnError) as e:
        attn_fwd(q, k, v, t128, 0.1)
    assert e.value.code == B.ATTN_ERR_UNSUPPORTED
    # misaligned q (2-byte offset)
    buf = torch.zeros(512 * 2 * 128 + 8, dtype=torch.bfloat16, device="cuda")
    qm = buf[1:1 + 512 * 2 * 128].view(512, 2, 128)
    with pytest.raises(AttnError) as e:
        attn_fwd(qm, k, v, t, 0.1)
    assert e.value.code == B.ATTN_ERR_UNSUPPORTED
    with pytest.raises(AttnError) as e:
        attn_build_tiles(np.array([[0, 100, 0, 100, 0], [50, 150, 50, 150, 1]], np.int32), 512, 512)
    assert e.value.code == B.ATTN_ERR_OVERLAP
    with pytest.raises(AttnError) as e:
        attn_build_tiles(np.array([[0, 600, 0, 100, 0]], np.int32), 512, 512)
    assert e.value.code == B.ATTN_ERR_INVALID_ARG
    assert attn_last_device_error() == 0


def test_bounded_wait_times_out_and_reports():
    attn_set_wait_limit_ns(20_000_000)     # 20 ms
    try:
        attn_selftest_wait_timeout()
        assert attn_last_device_error() == B.ATTN_ERR_TIMEOUT
        assert attn_last_device_error() == 0    # the status was cleared
    finally:
        attn_set_wait_limit_ns(4_000_000_000)
    # the context is still usable afterwards
    q, k, v = _qkv()
    t = attn_build_tiles(np.array([[0, 512, 0, 512, 1]], np.int32), 512, 512)
    out, lse = attn_fwd(q, k, v, t, 0.1)
    torch.cuda.synchronize()
    assert attn_last_device_error() == 0
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("seed", range(4))
def test_overlap_check_agrees_with_brute_force(seed):
    from block_sparse_attention_slice_gb300 import workloads as W
    rng = np.random.default_rng(seed + 50)
    for trial in range(6):
        sl = W.random_slices(2048, 2048, 40, seed=seed * 10 + trial, unit=8, max_len=30)
        if trial % 2:
            v = sl[rng.integers(len(sl))]
            q0 = min(2039, int(rng.integers(max(0, v[0] - 8), v[1])))
            k0 = min(2039, int(rng.integers(max(0, v[2] - 8), v[3])))
            sl = np.concatenate([sl, np.array([[q0, q0 + 9, k0, k0 + 9, 0]], np.int32)])
        rows = [x for x in sl.tolist() if x[1] > x[0] and x[3] > x[2]]
        expect = any(a[0] < b[1] and b[0] < a[1] and a[2] < b[3] and b[2] < a[3]
                     for i, a in enumerate(rows) for b in rows[i + 1:])
        if expect:
            with pytest.raises(AttnError) as e:
                attn_build_tiles(sl, 2048, 2048)
            assert e.value.code == B.ATTN_ERR_OVERLAP
        else:
            attn_build_tiles(sl, 2048, 2048).to_host()


def _status_word(tiles):
    """The metadata's totals[0..3] as an int64 view into its device workspace."""
    return tiles._view(tiles.struct.totals, 4, torch.int64)


def test_metadata_with_a_failed_status_is_refused():
    # Metadata whose build did not finish with ATTN_OK -- made here on the
    # host by writing CAPACITY into the status word of good metadata -- is
    # not read by the forward or the backward: the forward leaves its outputs
    # untouched, both report the status, and the same metadata with its
    # status put back gives the original result bit for bit.
    S, H, d = 1024, 2, 128
    q, k, v = _qkv(S, H, H, d)
    t = attn_build_tiles(np.array([[0, S, 0, S, 1]], np.int32), S, S)
    ref_o, ref_l = attn_fwd(q, k, v, t, 0.1)
    torch.cuda.synchronize()
    assert attn_last_device_error() == 0
    st = _status_word(t)
    st[3] = B.ATTN_ERR_CAPACITY
    out = torch.full_like(ref_o, 7.0)
    lse = torch.full_like(ref_l, 7.0)
    attn_fwd(q, k, v, t, 0.1, out=out, lse=lse)
    assert attn_last_device_error() == B.ATTN_ERR_CAPACITY
    assert torch.all(out == 7.0) and torch.all(lse == 7.0)
    do = torch.ones_like(q)
    B.attn_bwd(q, k, v, ref_o, do, ref_l, t, 0.1)
    assert attn_last_device_error() == B.ATTN_ERR_CAPACITY
    assert attn_last_device_error() == 0          # cleared by the read
    st[3] = 0
    o2, l2 = attn_fwd(q, k, v, t, 0.1)
    torch.cuda.synchronize()
    assert attn_last_device_error() == 0
    assert torch.equal(o2.view(torch.int16), ref_o.view(torch.int16))
    assert torch.equal(l2.view(torch.int32), ref_l.view(torch.int32))


def test_short_wait_limit_times_out_the_build_barrier():
    # With a 1 us bound, the grid barrier of a cooperative build whose 512
    # query tiles finish counting microseconds apart runs out (the barrier
    # polls the global timer directly).  Every CTA then follows one "abort"
    # decision: every list is left empty, the totals are zero and the status
    # is TIMEOUT, which the forward refuses without writing its outputs.
    # With the normal bound the same build gives the causal mask's
    # closed-form totals.
    d, L = 128, 131072
    big = np.array([[0, L, 0, L, 1]], np.int32)
    qb, kb, vb = _qkv(L, 1, 1, d)
    build_rc, refused = [], []
    attn_set_wait_limit_ns(1000)
    try:
        for _ in range(3):
            tb = attn_build_tiles(big, L, L)
            rc = attn_last_device_error()
            build_rc.append((rc, tb.totals()))
            if rc == B.ATTN_ERR_TIMEOUT:
                o = torch.full((L, 1, d), 3.0, dtype=torch.bfloat16, device="cuda")
                attn_fwd(qb, kb, vb, tb, 0.088, out=o)
                refused.append((attn_last_device_error(), bool(torch.all(o == 3.0))))
    finally:
        attn_set_wait_limit_ns(4_000_000_000)
    assert B.ATTN_ERR_TIMEOUT in [rc for rc, _ in build_rc], build_rc
    for rc, tot in build_rc:
        assert rc in (0, B.ATTN_ERR_TIMEOUT)
        assert tot == ([0, 0, 0, B.ATTN_ERR_TIMEOUT] if rc else [tot[0], tot[1], tot[2], 0])
    assert refused and all(r == (B.ATTN_ERR_TIMEOUT, True) for r in refused), refused
    # query tile i (256 rows) meets key tiles 0 .. 2i+1 (128 keys), the last
    # two MASKED, each referencing the one slice
    tb = attn_build_tiles(big, L, L)
    assert tb.totals() == [sum(2 * i + 2 for i in range(L // 256)), 2 * (L // 256),
                           L * (L + 1) // 2, 0]
    assert attn_last_device_error() == 0


def test_forward_wait_that_never_completes_aborts_cleanly(monkeypatch):
    # The forward's own abort path, driven by a barrier that nothing
    # completes: with ATTN_TEST_STALL_FWD=1 every CTA leaves its second K/V
    # load unissued, so the MMA lane's bounded wait for that ring slot runs
    # out (50 ms here).  The CTA then raises its abort flag, the producer
    # lets its issued loads land, the MMA lane waits for its issued MMAs, the
    # softmax warps leave their waits, tensor memory is freed and the last
    # CTA resets the work counter; the launch reports TIMEOUT.  Afterwards,
    # without the switch and with the normal bound, the forward on the same
    # inputs is bit-identical to a run made before the test.
    S, H, Hk, d = 8192, 4, 2, 128
    q, k, v = _qkv(S, H, Hk, d)
    t = attn_build_tiles(np.array([[0, S, 0, S, 1]], np.int32), S, S)
    ref_o, ref_l = attn_fwd(q, k, v, t, 0.088)
    torch.cuda.synchronize()
    assert attn_last_device_error() == 0
    attn_set_wait_limit_ns(50_000_000)
    monkeypatch.setenv("ATTN_TEST_STALL_FWD", "1")
    try:
        attn_fwd(q, k, v, t, 0.088)
        rc = attn_last_device_error()
    finally:
        monkeypatch.delenv("ATTN_TEST_STALL_FWD")
        attn_set_wait_limit_ns(4_000_000_000)
    assert rc == B.ATTN_ERR_TIMEOUT
    for _ in range(2):
        o2, l2 = attn_fwd(q, k, v, t, 0.088)
        torch.cuda.synchronize()
        assert attn_last_device_error() == 0
        assert torch.equal(o2.view(torch.int16), ref_o.view(torch.int16))
        assert torch.equal(l2.view(torch.int32), ref_l.view(torch.int32))
