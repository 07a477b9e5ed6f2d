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
