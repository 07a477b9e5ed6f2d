"""CPU oracle for flexibly masked attention forward -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU
baseline and ``--impl reference`` legs) may import anything here.  The
library (``block_sparse_attention_slice_gb300``) never imports it and shares
no code with it: the oracle is the plain, slow, obviously correct statement
of what the CUDA path computes, written from the pages:

* ``attention``  -- O = softmax(scale*Q K^T + mask) V and the per-row
  natural-log LSE, with the dense mask materialised element by element from
  the slice list or block grid (fp64 arithmetic on the bf16 input values);
* ``merge``      -- the exact combination of KV-split partial summaries
  (UltraAttn page, section 3.2, "split along KV: partial results must be
  merged");
* ``tiles``      -- the per-tile valid-pair counts, Full/Masked/Empty
  classification and CSR lists that the metadata builder must reproduce bit
  for bit.

Parity status of every function is recorded in its docstring; every one is
pinned by ``tests/test_oracle_*.py`` against closed forms, worked examples
printed on the pages (``tests/golden/``), invariants or brute force.
"""
from .attention import (FULL, CAUSAL, INV_CAUSAL, BI_CAUSAL, mask_rows,
                        mask_rows_grid, oracle_attention, oracle_merge)
from .tiles import (oracle_slices_from_grid, oracle_tiles, oracle_tiles_dense,
                    slice_row_interval)

__all__ = ["FULL", "CAUSAL", "INV_CAUSAL", "BI_CAUSAL", "mask_rows", "mask_rows_grid",
           "oracle_attention", "oracle_merge", "oracle_tiles", "oracle_tiles_dense",
           "slice_row_interval", "oracle_slices_from_grid"]
