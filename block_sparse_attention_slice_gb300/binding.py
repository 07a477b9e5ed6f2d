"""Thin Python binding of the C ABI in ``include/attn_slice.h``.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libattn_slice.so``.  PyTorch provides device memory and streams.
There is no fallback: if the library is missing or no GPU is present, the
calls raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libattn_slice.so")

ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_OVERLAP, ATTN_ERR_UNSUPPORTED, ATTN_ERR_CAPACITY, \
    ATTN_ERR_CUDA, ATTN_ERR_TIMEOUT = range(7)
ATTN_DTYPE_BF16, ATTN_DTYPE_F32 = 0, 1
ATTN_FWD_TILE_Q, ATTN_FWD_TILE_K = 256, 128
ATTN_MERGE_MAX_PARTS = 16

# every entry point declared in include/attn_slice.h
EXPORTS = ["attn_tiles_workspace_bytes", "attn_build_tiles", "attn_build_tiles_noalloc",
           "attn_tiles_totals",
           "attn_slices_from_block_grid", "attn_fwd", "attn_merge", "attn_bwd_workspace_bytes",
           "attn_bwd", "attn_last_device_error",
           "attn_set_wait_limit_ns", "attn_set_exp2_poly", "attn_selftest_wait_timeout",
           "attn_strerror"]


class AttnSlice(ctypes.Structure):
    _fields_ = [("q_start", ctypes.c_int32), ("q_end", ctypes.c_int32),
                ("k_start", ctypes.c_int32), ("k_end", ctypes.c_int32), ("type", ctypes.c_int32)]


class AttnTiles(ctypes.Structure):
    _fields_ = [("sq", ctypes.c_int32), ("sk", ctypes.c_int32), ("tile_q", ctypes.c_int32),
                ("tile_k", ctypes.c_int32), ("n_qtiles", ctypes.c_int32),
                ("n_ktiles", ctypes.c_int32), ("n_slices", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("cap_entries", ctypes.c_int64),
                ("cap_refs", ctypes.c_int64),
                ("row_ptr", ctypes.c_void_p), ("col_idx", ctypes.c_void_p),
                ("pairs", ctypes.c_void_p), ("ref_ptr", ctypes.c_void_p),
                ("ref_idx", ctypes.c_void_p), ("sched", ctypes.c_void_p),
                ("kind", ctypes.c_void_p), ("totals", ctypes.c_void_p),
                ("slices", ctypes.c_void_p), ("scratch", ctypes.c_void_p)]


class AttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {strerror(code)} (code {code})")
        self.code = code


_lib = None


def load(path: Optional[str] = None):
    """Loads the shared library (built by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA library not built: {p} is missing (run __graft_entry__.build())")
    lib = ctypes.CDLL(p)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    lib.attn_tiles_workspace_bytes.argtypes = [vp, i32, i32, i32, i32, i32, ctypes.POINTER(sz)]
    lib.attn_build_tiles.argtypes = [vp, i32, i32, i32, i32, i32, vp, sz, ctypes.POINTER(AttnTiles), vp]
    lib.attn_build_tiles_noalloc.argtypes = [vp, i32, i32, i32, i32, i32, vp, sz,
                                             ctypes.POINTER(AttnTiles), vp]
    lib.attn_tiles_totals.argtypes = [ctypes.POINTER(AttnTiles), ctypes.POINTER(ctypes.c_int64), vp]
    lib.attn_slices_from_block_grid.argtypes = [vp, i32, i32, i32, i32, vp, i32, ctypes.POINTER(ctypes.c_int)]
    lib.attn_fwd.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, ctypes.c_float,
                             ctypes.POINTER(AttnTiles), vp, i32, vp, vp]
    lib.attn_merge.argtypes = [vp, vp, i32, i32, i32, i32, i32, vp, i32, vp, vp]
    lib.attn_bwd_workspace_bytes.argtypes = [ctypes.POINTER(AttnTiles), i32, ctypes.POINTER(sz)]
    lib.attn_bwd.argtypes = [vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, ctypes.c_float,
                             ctypes.POINTER(AttnTiles), vp, vp, vp, i32, vp, sz, vp]
    lib.attn_last_device_error.argtypes = [vp]
    lib.attn_set_wait_limit_ns.argtypes = [i64]
    lib.attn_set_exp2_poly.argtypes = [i32]
    lib.attn_selftest_wait_timeout.argtypes = [vp]
    lib.attn_strerror.argtypes = [i32]
    lib.attn_strerror.restype = ctypes.c_char_p
    for name in EXPORTS:
        if name != "attn_strerror":
            getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    if os.environ.get("ATTN_WAIT_LIMIT_NS"):
        attn_set_wait_limit_ns(int(os.environ["ATTN_WAIT_LIMIT_NS"]))
    return lib


def strerror(code: int) -> str:
    try:
        return load().attn_strerror(code).decode()
    except Exception:
        return f"status {code}"


def _check(code: int, where: str):
    if code != ATTN_OK:
        raise AttnError(code, where)


def _stream_ptr(stream) -> ctypes.c_void_p:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _slice_array(slices) -> ctypes.Array:
    a = np.ascontiguousarray(np.asarray(slices, dtype=np.int32).reshape(-1, 5))
    arr = (AttnSlice * max(1, len(a)))()
    ctypes.memmove(arr, a.ctypes.data, a.nbytes)
    return arr, len(a)


def host_slices(slices):
    """Slice list as a contiguous int32 [n, 5] host array plus its count.

    attn_build_tiles copies the slices into an input image of its own before
    it returns, so the caller may reuse or free the array right away."""
    a = np.ascontiguousarray(np.asarray(slices, dtype=np.int32).reshape(-1, 5))
    return (a if len(a) else np.zeros((1, 5), np.int32)), len(a)


class Tiles:
    """Tile metadata on the device: the ``attn_tiles_t`` struct and the torch
    workspace tensor its pointers point into (kept alive here)."""

    def __init__(self, struct: AttnTiles, ws, n_slices: int):
        self.struct = struct
        self.ws = ws
        self.n_slices = n_slices

    @property
    def n_qtiles(self):
        return self.struct.n_qtiles

    def totals(self, stream=None):
        t = (ctypes.c_int64 * 4)()
        _check(load().attn_tiles_totals(ctypes.byref(self.struct), t, _stream_ptr(stream)), "attn_tiles_totals")
        return [int(x) for x in t]

    def _view(self, ptr: int, count: int, dtype):
        import torch
        off = ptr - self.ws.data_ptr()
        nbytes = count * torch.empty(0, dtype=dtype).element_size()
        return self.ws[off:off + nbytes].view(dtype)

    def to_host(self, stream=None):
        """Downloads the metadata arrays (same keys as the oracle's)."""
        import torch
        nnz, nref, total, status = self.totals(stream)
        if status != ATTN_OK:
            raise AttnError(status, "attn_build_tiles (device)")
        s = self.struct
        out = {
            "row_ptr": self._view(s.row_ptr, s.n_qtiles + 1, torch.int32),
            "col_idx": self._view(s.col_idx, nnz, torch.int32),
            "kind": self._view(s.kind, nnz, torch.uint8),
            "pairs": self._view(s.pairs, nnz, torch.int32),
            "ref_ptr": self._view(s.ref_ptr, nnz + 1, torch.int32),
            "ref_idx": self._view(s.ref_idx, nref, torch.int32),
            "sched": self._view(s.sched, s.n_qtiles, torch.int32),
        }
        res = {k: v.cpu().numpy().copy() for k, v in out.items()}
        res["total_pairs"] = total
        return res


def attn_tiles_workspace_bytes(slices, sq: int, sk: int, tile_q: int, tile_k: int) -> int:
    arr, n = _slice_array(slices)
    out = ctypes.c_size_t(0)
    _check(load().attn_tiles_workspace_bytes(arr, n, sq, sk, tile_q, tile_k, ctypes.byref(out)),
           "attn_tiles_workspace_bytes")
    return int(out.value)


def attn_build_tiles(slices, sq: int, sk: int, tile_q: int = ATTN_FWD_TILE_Q,
                     tile_k: int = ATTN_FWD_TILE_K, ws=None, stream=None, device=None,
                     prepared=None) -> Tiles:
    """Slice list (``int32[n, 5]``) -> device tile metadata.

    ``prepared`` may pass the ``host_slices(slices)`` pair to skip the
    conversion on repeated builds; ``ws`` a device workspace to reuse."""
    import torch
    arr, n = prepared if prepared is not None else host_slices(slices)
    if ws is None:
        nbytes = ctypes.c_size_t(0)
        _check(load().attn_tiles_workspace_bytes(arr.ctypes.data, n, sq, sk, tile_q, tile_k,
                                                 ctypes.byref(nbytes)),
               "attn_tiles_workspace_bytes")
        ws = torch.empty(int(nbytes.value), dtype=torch.uint8, device=device or "cuda")
    st = AttnTiles()
    _check(load().attn_build_tiles(arr.ctypes.data, n, sq, sk, tile_q, tile_k,
                                   ctypes.c_void_p(ws.data_ptr()), ws.numel(), ctypes.byref(st),
                                   _stream_ptr(stream)),
           "attn_build_tiles")
    return Tiles(st, ws, n)


def attn_build_tiles_noalloc(slices, sq: int, sk: int, out, tile_q: int = ATTN_FWD_TILE_Q,
                             tile_k: int = ATTN_FWD_TILE_K, stream=None) -> Tiles:
    """Like ``attn_build_tiles``, but the library's fixed device array holds
    the build's scratch counters: nothing is allocated, ``out`` (a uint8 CUDA
    tensor of at least ``attn_tiles_workspace_bytes`` bytes) receives the
    metadata.  Calls that overlap on the GPU share that array and race."""
    arr, n = host_slices(slices)
    st = AttnTiles()
    _check(load().attn_build_tiles_noalloc(arr.ctypes.data, n, sq, sk, tile_q, tile_k,
                                           ctypes.c_void_p(out.data_ptr()), out.numel(),
                                           ctypes.byref(st), _stream_ptr(stream)),
           "attn_build_tiles_noalloc")
    return Tiles(st, out, n)


def attn_slices_from_block_grid(grid, block_q: int, block_k: int) -> np.ndarray:
    """Full(1)/Causal(2)/Empty(0) block grid -> slice list (host)."""
    g = np.ascontiguousarray(np.asarray(grid, dtype=np.uint8))
    nbq, nbk = g.shape
    n = ctypes.c_int(0)
    lib = load()
    rc = lib.attn_slices_from_block_grid(g.ctypes.data, nbq, nbk, block_q, block_k, None, 0, ctypes.byref(n))
    if rc not in (ATTN_OK, ATTN_ERR_CAPACITY):
        _check(rc, "attn_slices_from_block_grid")
    out = np.zeros((max(1, n.value), 5), dtype=np.int32)
    _check(lib.attn_slices_from_block_grid(g.ctypes.data, nbq, nbk, block_q, block_k, out.ctypes.data,
                                           n.value, ctypes.byref(n)), "attn_slices_from_block_grid")
    return out[:n.value]


def attn_fwd(q, k, v, tiles: Tiles, scale: float, out=None, lse=None, out_dtype=None, stream=None):
    """O, lse = masked attention forward (q [S_q,H,d], k/v [S_k,H_k,d] bf16 CUDA)."""
    import torch
    sq, hq, d = q.shape
    sk, hk, _ = k.shape
    for x in (q, k, v):
        if x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous():
            raise ValueError("q, k, v must be contiguous bf16 CUDA tensors")
    if out is None:
        out = torch.empty((sq, hq, d), dtype=out_dtype or torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((hq, sq), dtype=torch.float32, device=q.device)
    code = ATTN_DTYPE_F32 if out.dtype == torch.float32 else ATTN_DTYPE_BF16
    _check(load().attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), sq, sk, hq, hk, d, float(scale),
                           ctypes.byref(tiles.struct), out.data_ptr(), code, lse.data_ptr(),
                           _stream_ptr(stream)), "attn_fwd")
    return out, lse


def attn_merge(o_parts: Sequence, lse_parts: Sequence, out=None, lse=None, out_dtype=None, stream=None):
    """Exact merge of KV-split partials (each O_i [S,H,d], lse_i [H,S])."""
    import torch
    n = len(o_parts)
    S, H, d = o_parts[0].shape
    if out is None:
        out = torch.empty((S, H, d), dtype=out_dtype or torch.bfloat16, device=o_parts[0].device)
    if lse is None:
        lse = torch.empty((H, S), dtype=torch.float32, device=o_parts[0].device)
    optr = (ctypes.c_void_p * n)(*[o.data_ptr() for o in o_parts])
    lptr = (ctypes.c_void_p * n)(*[x.data_ptr() for x in lse_parts])
    pd = ATTN_DTYPE_F32 if o_parts[0].dtype == torch.float32 else ATTN_DTYPE_BF16
    od = ATTN_DTYPE_F32 if out.dtype == torch.float32 else ATTN_DTYPE_BF16
    _check(load().attn_merge(optr, lptr, n, pd, S, H, d, out.data_ptr(), od, lse.data_ptr(),
                             _stream_ptr(stream)), "attn_merge")
    return out, lse


def attn_bwd(q, k, v, out, dout, lse, tiles: Tiles, scale: float, grad_dtype=None, ws=None,
             stream=None):
    """dQ, dK, dV of the masked attention forward (dout bf16 like q)."""
    import torch
    sq, hq, d = q.shape
    sk, hk, _ = k.shape
    for x in (q, k, v, dout):
        if x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous():
            raise ValueError("q, k, v, dout must be contiguous bf16 CUDA tensors")
    gd = grad_dtype or torch.float32
    dq = torch.empty((sq, hq, d), dtype=gd, device=q.device)
    dk = torch.empty((sk, hk, d), dtype=gd, device=q.device)
    dv = torch.empty((sk, hk, d), dtype=gd, device=q.device)
    nb = ctypes.c_size_t(0)
    _check(load().attn_bwd_workspace_bytes(ctypes.byref(tiles.struct), hq, ctypes.byref(nb)),
           "attn_bwd_workspace_bytes")
    if ws is None or ws.numel() < nb.value:
        ws = torch.empty(int(nb.value), dtype=torch.uint8, device=q.device)
    od = ATTN_DTYPE_F32 if out.dtype == torch.float32 else ATTN_DTYPE_BF16
    gc = ATTN_DTYPE_F32 if gd == torch.float32 else ATTN_DTYPE_BF16
    _check(load().attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), od, dout.data_ptr(),
                           lse.data_ptr(), sq, sk, hq, hk, d, float(scale), ctypes.byref(tiles.struct),
                           dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), gc, ctypes.c_void_p(ws.data_ptr()),
                           ws.numel(), _stream_ptr(stream)), "attn_bwd")
    return dq, dk, dv


def attn_last_device_error(stream=None) -> int:
    return int(load().attn_last_device_error(_stream_ptr(stream)))


def attn_set_wait_limit_ns(ns: int):
    _check(load().attn_set_wait_limit_ns(int(ns)), "attn_set_wait_limit_ns")


def attn_set_exp2_poly(period: int):
    """0: all exponentials on the special-function unit (default); 4 or 8:
    every 4th / 8th pair of a FULL tile's exponentials on the FMA-pipe
    polynomial.  Applies to later attn_fwd calls of this process."""
    _check(load().attn_set_exp2_poly(int(period)), "attn_set_exp2_poly")


def attn_selftest_wait_timeout(stream=None):
    _check(load().attn_selftest_wait_timeout(_stream_ptr(stream)), "attn_selftest_wait_timeout")
