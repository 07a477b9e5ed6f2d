"""GB300 (sm_103a) masked-attention forward behind a small C ABI.

    tiles      = attn_build_tiles(slices, S_q, S_k)        # slice list -> CSR tile metadata
    out, lse   = attn_fwd(q, k, v, tiles, scale)           # softmax(scale QK^T + mask) V, row LSE
    out, lse   = attn_merge([o_1, o_2, ...], [lse_1, ...]) # exact KV-split merge

All three run as hand-written CUDA kernels in ``libattn_slice.so`` (see
``include/attn_slice.h``); this package only marshals arguments.
"""
from .binding import (ATTN_DTYPE_BF16, ATTN_DTYPE_F32, ATTN_FWD_TILE_K, ATTN_FWD_TILE_Q,
                      AttnError, Tiles, attn_build_tiles, attn_bwd, attn_fwd, attn_last_device_error,
                      attn_merge, attn_selftest_wait_timeout, attn_set_exp2_poly,
                      attn_set_wait_limit_ns, attn_slices_from_block_grid,
                      attn_tiles_workspace_bytes, load)

__all__ = ["attn_build_tiles", "attn_fwd", "attn_bwd", "attn_merge", "attn_slices_from_block_grid",
           "attn_tiles_workspace_bytes", "attn_last_device_error", "attn_set_wait_limit_ns",
           "attn_set_exp2_poly",
           "attn_selftest_wait_timeout", "Tiles", "AttnError", "load",
           "ATTN_DTYPE_BF16", "ATTN_DTYPE_F32", "ATTN_FWD_TILE_Q", "ATTN_FWD_TILE_K"]
