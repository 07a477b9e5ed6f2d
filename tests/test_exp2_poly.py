"""The FMA-pipe exp2 of the forward kernel (opt-in, attn_set_exp2_poly).

CPU: the kernel's coefficients are the ones exp2_poly_fit.py produces, and a
step-by-step float32 emulation of the kernel's evaluation (range reduction by
the 1.5 * 2^23 rounding trick, cubic in Horner form, exponent-field add)
stays within its stated bound of exp2 over the arguments the softmax feeds
it, is exact at integers, and stays a positive normal number at the clamp.
GPU (gpu marker): the forward with the polynomial enabled matches the fp64
oracle within the same tolerances as the default path.
"""
import importlib.util
import math
import pathlib
import re

import numpy as np
import pytest

CSRC = pathlib.Path(__file__).resolve().parents[1] / "block_sparse_attention_slice_gb300" / "csrc"


def _fit_module():
    spec = importlib.util.spec_from_file_location("exp2_poly_fit", CSRC / "exp2_poly_fit.py")
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _kernel_coeffs():
    src = (CSRC / "ptx.cuh").read_text()
    m = re.search(r"c3 = ([0-9.e+-]+)f, c2 = ([0-9.e+-]+)f,\s*c1 = ([0-9.e+-]+)f", src)
    assert m, "coefficients not found in ptx.cuh"
    c3, c2, c1 = (np.float32(float(x)) for x in m.groups())
    return np.array([1.0, c1, c2, c3], dtype=np.float32)


def _emulate(a):
    """Float32 emulation of exp2_poly2, one step per kernel instruction."""
    c = _kernel_coeffs()
    f32 = np.float32
    x = np.maximum(a.astype(f32), f32(-125.0))
    t = (x + f32(12582912.0)).astype(f32)
    n = (t + f32(-12582912.0)).astype(f32)
    f = (n * f32(-1.0) + x).astype(f32)
    q = (c[3] * f + c[2]).astype(f32)
    q = (q * f + c[1]).astype(f32)
    q = (q * f + c[0]).astype(f32)
    bits = (t.view(np.uint32).astype(np.uint64) * 8388608 + q.view(np.uint32)) & 0xFFFFFFFF
    return bits.astype(np.uint32).view(np.float32)


def test_kernel_coefficients_are_the_fit():
    fit = _fit_module().fit()
    np.testing.assert_array_equal(_kernel_coeffs(), fit.astype(np.float32))


def test_relative_error_bound_and_exact_integers():
    a = np.linspace(-60.0, 8.0, 2_000_001).astype(np.float32)
    got = _emulate(a).astype(np.float64)
    rel = np.abs(got / np.exp2(a.astype(np.float64)) - 1.0)
    assert rel.max() < 1.2e-4, rel.max()
    ints = np.arange(-120, 9, dtype=np.float32)
    np.testing.assert_array_equal(_emulate(ints), np.exp2(ints.astype(np.float64)).astype(np.float32))


def test_clamp_keeps_a_tiny_positive_normal():
    out = _emulate(np.array([-125.0, -300.0, -1e30], dtype=np.float32))
    assert np.all(out > 0) and np.all(out < 1e-37)
    assert np.all(out >= np.finfo(np.float32).tiny)


@pytest.mark.gpu
@pytest.mark.parametrize("period", [4, 8])
def test_forward_parity_with_polynomial(period):
    import torch
    import oracle
    from block_sparse_attention_slice_gb300 import attn_build_tiles, attn_fwd, attn_set_exp2_poly
    from block_sparse_attention_slice_gb300 import workloads as W
    from parity import compare, run_oracle

    cases = [(1536, 1536, 4, 2, 128, np.array([[0, 1536, 0, 1536, 1]], np.int32)),
             (1000, 1300, 2, 1, 64, W.random_slices(1000, 1300, 20, seed=period, unit=1, max_len=500))]
    try:
        attn_set_exp2_poly(period)
        for sq, sk, H, Hk, d, sl in cases:
            rng = np.random.default_rng(period + d)
            mk = lambda *sh: torch.from_numpy(rng.standard_normal(sh, dtype=np.float32)).to(torch.bfloat16)
            q, k, v = mk(sq, H, d), mk(sk, Hk, d), mk(sk, Hk, d)
            scale = 1.0 / math.sqrt(d)
            tiles = attn_build_tiles(sl, sq, sk)
            out, lse = attn_fwd(q.cuda(), k.cuda(), v.cuda(), tiles, scale, out_dtype=torch.float32)
            ref = run_oracle(q, k, v, scale, lambda r: oracle.mask_rows(sl, r, sk))
            compare(out, lse, ref)
    finally:
        attn_set_exp2_poly(0)
