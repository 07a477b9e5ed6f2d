"""attn_merge on the GPU vs the oracle's merge (UltraAttn page, section 3.2)."""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_attention_slice_gb300 import attn_merge
from parity import compare

pytestmark = pytest.mark.gpu


def _parts(n, S, H, d, seed, dtype, empty_frac=0.2):
    rng = np.random.default_rng(seed)
    O = [rng.standard_normal((S, H, d)).astype(np.float32) for _ in range(n)]
    L = [(rng.standard_normal((H, S)) * 4).astype(np.float32) for _ in range(n)]
    for i in range(n):
        L[i][rng.random((H, S)) < empty_frac] = -np.inf
    # some rows empty in every partial
    for i in range(n):
        L[i][:, :3] = -np.inf
    Ot = [torch.from_numpy(o).to(dtype).cuda() for o in O]
    Lt = [torch.from_numpy(x).cuda() for x in L]
    O64 = [o.float().cpu().numpy().astype(np.float64) for o in Ot]
    return Ot, Lt, O64, [x.astype(np.float64) for x in L]


@pytest.mark.parametrize("n,S,H,d,pdt,odt", [
    (2, 512, 1, 64, torch.float32, torch.bfloat16), (8, 1000, 4, 128, torch.float32, torch.bfloat16),
    (3, 777, 2, 128, torch.bfloat16, torch.float32), (16, 64, 3, 64, torch.bfloat16, torch.bfloat16),
    (1, 100, 2, 128, torch.float32, torch.float32), (5, 300, 2, 64, torch.float32, torch.float32)])
def test_merge_matches_oracle(n, S, H, d, pdt, odt):
    Ot, Lt, O64, L64 = _parts(n, S, H, d, seed=n * 7 + d, dtype=pdt)
    out, lse = attn_merge(Ot, Lt, out_dtype=odt)
    Or, Lr = oracle.oracle_merge(O64, L64)
    ref = {h: (np.arange(S), Or[:, h, :], Lr[h]) for h in range(H)}
    # bf16 output: round-to-nearest-even keeps 8 significant bits, so the
    # bound is relative (2^-8 |O|); f32 output: fp32 accumulation only
    if odt == torch.bfloat16:
        compare(out, lse, ref, tol_o=1e-6, tol_l=1e-5, rel_o=2.0 ** -8)
    else:
        compare(out, lse, ref, tol_o=1e-5, tol_l=1e-5)
    assert torch.all(out[:3] == 0) and torch.all(torch.isneginf(lse[:, :3]))
