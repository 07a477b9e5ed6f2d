"""Helpers shared by the parity tests: run the oracle on the same seeded
inputs the CUDA path gets, and compare element by element.

Tolerances (bf16 inputs, fp32 accumulation): |O - O_ref| <= 1e-2 and
|lse - lse_ref| <= 1e-3 absolute; rows with no valid key must give
lse = -inf exactly on both sides.
"""
import os

import numpy as np

import oracle

TOL_O = 1e-2
TOL_LSE = 1e-3
THREADS = max(1, len(os.sched_getaffinity(0)))
# rows per head checked on the sampled (large) workloads
SAMPLE_ROWS = int(os.environ.get("ATTN_PARITY_ROWS", "4096"))


def f64(t):
    """bf16 / f32 torch tensor -> float64 numpy (exact)."""
    return t.detach().float().cpu().numpy().astype(np.float64)


def mask_fn(workload, slices=None):
    if slices is None and workload.grid is not None:
        return lambda r: oracle.mask_rows_grid(workload.grid, workload.block, r, workload.S)
    sl = workload.slices if slices is None else slices
    return lambda r: oracle.mask_rows(sl, r, workload.S)


def rows_per_head(workload, n=None, extra=()):
    from block_sparse_attention_slice_gb300.workloads import sample_rows
    n = SAMPLE_ROWS if n is None else n
    return [sample_rows(workload.S, h, n, extra) for h in range(workload.H)]


def run_oracle(q, k, v, scale, mask, rows=None):
    return oracle.oracle_attention(f64(q), f64(k), f64(v), scale, mask, rows=rows,
                                   threads=THREADS)


def compare(out, lse, ref, tol_o=TOL_O, tol_l=TOL_LSE, rel_o=0.0):
    """out [S,H,d] / lse [H,S] (torch, any device) vs the oracle dict.
    Asserts |O - O_ref| <= tol_o + rel_o |O_ref| and |lse - lse_ref| <= tol_l;
    returns (max excess-free |dO|, max |dlse|)."""
    import torch
    worst_o = worst_l = 0.0
    for h, (rows, O_ref, L_ref) in ref.items():
        idx = torch.as_tensor(rows, dtype=torch.long, device=out.device)
        o = out.index_select(0, idx)[:, h].float().cpu().numpy().astype(np.float64)
        l = lse[h].index_select(0, idx).cpu().numpy().astype(np.float64)
        ninf_ref, ninf = np.isneginf(L_ref), np.isneginf(l)
        assert np.array_equal(ninf, ninf_ref), f"head {h}: -inf rows differ"
        assert np.all(np.isfinite(o)), f"head {h}: non-finite output"
        fin = ~ninf_ref
        if fin.any():
            worst_l = max(worst_l, float(np.abs(l[fin] - L_ref[fin]).max()))
        worst_o = max(worst_o, float((np.abs(o - O_ref) - rel_o * np.abs(O_ref)).max()))
    assert worst_o <= tol_o, f"max |O - O_ref| (less {rel_o} |O_ref|) = {worst_o}"
    assert worst_l <= tol_l, f"max |lse - lse_ref| = {worst_l}"
    return worst_o, worst_l
