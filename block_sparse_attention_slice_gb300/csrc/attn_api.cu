// C ABI of the library: argument checks on the host, workspace layout of the
// tile metadata, and dispatch to the kernels of the other translation units.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#include "attn_internal.h"

namespace attn {
namespace host {

constexpr size_t kAlign = 256;
size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

int check_slices(const attn_slice_t *s, int n, int sq, int sk) {
  if (n < 0 || (n > 0 && !s)) return ATTN_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    const attn_slice_t &x = s[i];
    if (x.q_start < 0 || x.q_start > x.q_end || x.q_end > sq) return ATTN_ERR_INVALID_ARG;
    if (x.k_start < 0 || x.k_start > x.k_end || x.k_end > sk) return ATTN_ERR_INVALID_ARG;
    if (x.type < ATTN_MASK_FULL || x.type > ATTN_MASK_BI_CAUSAL) return ATTN_ERR_INVALID_ARG;
  }
  return ATTN_OK;
}

// Rectangles of non-empty slices must be pairwise disjoint.  Sorted by
// (q_start, k_start), a slice can only meet the following ones that start
// before it ends in q; within a run of equal q_start, once a k_start reaches
// its k_end the rest of the run is past it too, so the scan skips to the
// next run.  Lists that come sorted (block grids, most slice lists) skip the
// sort, and a grid is checked in linear time.
int check_overlap(const attn_slice_t *s, int n) {
  // order of the non-empty slices by (q_start, k_start): their own order when
  // it already is sorted, else a sorted index list (per-thread buffers, kept
  // across calls)
  static thread_local std::vector<int> idx, run_end;
  auto empty = [&](int i) { return s[i].q_end <= s[i].q_start || s[i].k_end <= s[i].k_start; };
  auto before = [&](int a, int b) {
    return s[a].q_start != s[b].q_start ? s[a].q_start < s[b].q_start : s[a].k_start < s[b].k_start;
  };
  idx.clear();
  bool sorted = true;
  int last = -1;
  for (int i = 0; i < n; ++i) {
    if (empty(i)) continue;
    if (last >= 0 && before(i, last)) sorted = false;
    idx.push_back(i);
    last = i;
  }
  if (!sorted) std::sort(idx.begin(), idx.end(), before);
  const int m = static_cast<int>(idx.size());
  run_end.resize(m);
  for (int u = m; u-- > 0;)
    run_end[u] = (u + 1 < m && s[idx[u + 1]].q_start == s[idx[u]].q_start) ? run_end[u + 1] : u + 1;
  for (int u = 0; u < m; ++u) {
    const attn_slice_t &a = s[idx[u]];
    int v = u + 1;
    while (v < m && s[idx[v]].q_start < a.q_end) {
      const attn_slice_t &b = s[idx[v]];
      if (b.q_start == a.q_start && b.k_start >= a.k_end) {
        v = run_end[v];
        continue;
      }
      if (a.k_start < b.k_end && b.k_start < a.k_end) return ATTN_ERR_OVERLAP;
      ++v;
    }
  }
  return ATTN_OK;
}

// x / d for x >= 0, by a shift when d is a power of two
struct TileDiv {
  int d, sh = -1;
  explicit TileDiv(int d_) : d(d_) {
    if (d_ > 0 && (d_ & (d_ - 1)) == 0)
      for (sh = 0; (1 << sh) < d_; ++sh) {
      }
  }
  int operator()(int x) const { return sh >= 0 ? x >> sh : x / d; }
};

int shape_ok(int sq, int sk, int tq, int tk, int *nq, int *nk) {
  if (sq < 1 || sk < 1 || tq < 1 || tk < 1) return ATTN_ERR_INVALID_ARG;
  if (tq > 1024 || tk > 1024) return ATTN_ERR_UNSUPPORTED;
  *nq = (sq + tq - 1) / tq;
  *nk = (sk + tk - 1) / tk;
  if (*nk > 8192) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(*nq) * *nk >= (int64_t(1) << 31)) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

WsLayout layout(const attn_slice_t *s, int n, int nq, int nk, int tq, int tk) {
  WsLayout L{};
  int64_t touched = 0, touched_q = 0;
  const TileDiv dq(tq), dk(tk);
  for (int i = 0; i < n; ++i) {
    if (s[i].q_end <= s[i].q_start || s[i].k_end <= s[i].k_start) continue;
    const int64_t a = dq(s[i].q_end - 1) - dq(s[i].q_start) + 1;
    const int64_t b = dk(s[i].k_end - 1) - dk(s[i].k_start) + 1;
    touched += a * b;
    touched_q += a;
  }
  L.cap_e = std::min<int64_t>(touched, static_cast<int64_t>(nq) * nk);
  L.cap_r = touched;
  L.n_qb = touched_q;
  // input region: packed back to back (one image), 4-byte aligned parts
  L.slices = 0;
  L.qb_ptr = sizeof(attn_slice_t) * n;
  L.qb_idx = L.qb_ptr + sizeof(int32_t) * (nq + 1);
  L.input_bytes = L.qb_idx + sizeof(int32_t) * touched_q;
  size_t o = up(L.input_bytes);
  auto put = [&](size_t bytes) {
    const size_t at = o;
    o = up(o + std::max<size_t>(bytes, 1));
    return at;
  };
  L.row_ptr = put(sizeof(int32_t) * (nq + 1));
  L.sched = put(sizeof(int32_t) * nq);
  L.nnz_q = put(sizeof(int32_t) * nq);
  L.nref_q = put(sizeof(int32_t) * nq);
  L.ref_base_q = put(sizeof(int32_t) * nq);
  L.pairs_q = put(sizeof(int64_t) * nq);
  L.totals = put(sizeof(int64_t) * 4);
  L.col_idx = put(sizeof(int32_t) * L.cap_e);
  L.pairs = put(sizeof(int32_t) * L.cap_e);
  L.ref_ptr = put(sizeof(int32_t) * (L.cap_e + 1));
  L.kind = put(L.cap_e);
  L.ref_idx = put(sizeof(int32_t) * L.cap_r);
  L.total = o;
  return L;
}

void stage_inputs(const attn_slice_t *s, int n, int nq, int tq, const WsLayout &L,
                  std::vector<uint8_t> *img) {
  // every byte is written below: the slices and the bucket ids fully, the
  // bucket pointers after zeroing, so the buffer is not cleared first
  img->resize(L.input_bytes);
  if (n > 0) std::memcpy(img->data() + L.slices, s, sizeof(attn_slice_t) * n);
  int32_t *ptr = reinterpret_cast<int32_t *>(img->data() + L.qb_ptr);
  int32_t *idx = reinterpret_cast<int32_t *>(img->data() + L.qb_idx);
  std::memset(ptr, 0, sizeof(int32_t) * (nq + 1));
  const TileDiv dq(tq);
  for (int i = 0; i < n; ++i) {
    if (s[i].q_end <= s[i].q_start || s[i].k_end <= s[i].k_start) continue;
    for (int q = dq(s[i].q_start), q1 = dq(s[i].q_end - 1); q <= q1; ++q) ++ptr[q + 1];
  }
  for (int q = 0; q < nq; ++q) ptr[q + 1] += ptr[q];
  static thread_local std::vector<int32_t> fill;
  fill.assign(ptr, ptr + nq);
  for (int i = 0; i < n; ++i) {          // ascending ids within every bucket
    if (s[i].q_end <= s[i].q_start || s[i].k_end <= s[i].k_start) continue;
    for (int q = dq(s[i].q_start), q1 = dq(s[i].q_end - 1); q <= q1; ++q) idx[fill[q]++] = i;
  }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace host
}  // namespace attn

using namespace attn::host;

extern "C" {

int attn_tiles_workspace_bytes(const attn_slice_t *h_slices, int n_slices, int sq, int sk,
                               int tile_q, int tile_k, size_t *bytes) {
  if (!bytes) return ATTN_ERR_INVALID_ARG;
  int nq, nk, rc;
  if ((rc = shape_ok(sq, sk, tile_q, tile_k, &nq, &nk)) != ATTN_OK) return rc;
  if ((rc = check_slices(h_slices, n_slices, sq, sk)) != ATTN_OK) return rc;
  *bytes = layout(h_slices, n_slices, nq, nk, tile_q, tile_k).total;
  return ATTN_OK;
}

int attn_build_tiles(const attn_slice_t *h_slices, int n_slices, int sq, int sk, int tile_q,
                     int tile_k, void *d_ws, size_t ws_bytes, attn_tiles_t *tiles,
                     attn_stream_t stream) {
  if (!tiles || !d_ws) return ATTN_ERR_INVALID_ARG;
  int nq, nk, rc;
  if ((rc = shape_ok(sq, sk, tile_q, tile_k, &nq, &nk)) != ATTN_OK) return rc;
  if ((rc = check_slices(h_slices, n_slices, sq, sk)) != ATTN_OK) return rc;
  if ((rc = check_overlap(h_slices, n_slices)) != ATTN_OK) return rc;
  if (static_cast<int64_t>(tile_q) * tile_k >= (int64_t(1) << 31)) return ATTN_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(d_ws) & (kAlign - 1)) != 0) return ATTN_ERR_UNSUPPORTED;
  const WsLayout L = layout(h_slices, n_slices, nq, nk, tile_q, tile_k);
  if (ws_bytes < L.total) return ATTN_ERR_CAPACITY;
  uint8_t *ws = static_cast<uint8_t *>(d_ws);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  attn_tiles_t t;
  std::memset(&t, 0, sizeof(t));
  t.sq = sq;
  t.sk = sk;
  t.tile_q = tile_q;
  t.tile_k = tile_k;
  t.n_qtiles = nq;
  t.n_ktiles = nk;
  t.n_slices = n_slices;
  t.cap_entries = L.cap_e;
  t.cap_refs = L.cap_r;
  t.row_ptr = reinterpret_cast<int32_t *>(ws + L.row_ptr);
  t.col_idx = reinterpret_cast<int32_t *>(ws + L.col_idx);
  t.pairs = reinterpret_cast<int32_t *>(ws + L.pairs);
  t.ref_ptr = reinterpret_cast<int32_t *>(ws + L.ref_ptr);
  t.ref_idx = reinterpret_cast<int32_t *>(ws + L.ref_idx);
  t.sched = reinterpret_cast<int32_t *>(ws + L.sched);
  t.kind = ws + L.kind;
  t.totals = reinterpret_cast<int64_t *>(ws + L.totals);
  t.slices = reinterpret_cast<attn_slice_t *>(ws + L.slices);
  t.scratch = reinterpret_cast<int32_t *>(ws + L.nnz_q);

  static thread_local std::vector<uint8_t> img;   // kept across calls
  stage_inputs(h_slices, n_slices, nq, tile_q, L, &img);
  attn::BuildLaunch b;
  b.slices = t.slices;
  b.qb_ptr = reinterpret_cast<const int32_t *>(ws + L.qb_ptr);
  b.qb_idx = reinterpret_cast<const int32_t *>(ws + L.qb_idx);
  b.n_slices = n_slices;
  b.sq = sq;
  b.sk = sk;
  b.tq = tile_q;
  b.tk = tile_k;
  b.nq = nq;
  b.nk = nk;
  b.nnz_q = reinterpret_cast<int32_t *>(ws + L.nnz_q);
  b.nref_q = reinterpret_cast<int32_t *>(ws + L.nref_q);
  b.ref_base_q = reinterpret_cast<int32_t *>(ws + L.ref_base_q);
  b.pairs_q = reinterpret_cast<int64_t *>(ws + L.pairs_q);
  b.off_qb_ptr = static_cast<uint32_t>(L.qb_ptr);
  b.off_qb_idx = static_cast<uint32_t>(L.qb_idx);
  b.wait_ns = attn::wait_limit_ns();
  b.row_ptr = t.row_ptr;
  b.col_idx = t.col_idx;
  b.pairs = t.pairs;
  b.ref_ptr = t.ref_ptr;
  b.ref_idx = t.ref_idx;
  b.sched = t.sched;
  b.kind = t.kind;
  b.totals = t.totals;
  b.cap_entries = L.cap_e;
  b.cap_refs = L.cap_r;
  if ((rc = attn::build_tiles_launch(b, img.data(), img.size(), ws, s)) != ATTN_OK) return rc;
  *tiles = t;
  return ATTN_OK;
}

int attn_tiles_totals(const attn_tiles_t *tiles, int64_t h_totals[4], attn_stream_t stream) {
  if (!tiles || !h_totals || !tiles->totals) return ATTN_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(h_totals, tiles->totals, 4 * sizeof(int64_t), cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

int attn_slices_from_block_grid(const uint8_t *h_grid, int nbq, int nbk, int block_q, int block_k,
                                attn_slice_t *h_out, int capacity, int *n_out) {
  if (!h_grid || !n_out || nbq < 0 || nbk < 0 || block_q < 1 || block_k < 1)
    return ATTN_ERR_INVALID_ARG;
  if (static_cast<int64_t>(nbq) * block_q >= (int64_t(1) << 31) ||
      static_cast<int64_t>(nbk) * block_k >= (int64_t(1) << 31))
    return ATTN_ERR_INVALID_ARG;
  int n = 0;
  for (int bi = 0; bi < nbq; ++bi)
    for (int bj = 0; bj < nbk; ++bj) {
      const uint8_t g = h_grid[static_cast<size_t>(bi) * nbk + bj];
      if (g == ATTN_GRID_EMPTY) continue;
      if (g != ATTN_GRID_FULL && g != ATTN_GRID_CAUSAL) return ATTN_ERR_INVALID_ARG;
      if (g == ATTN_GRID_CAUSAL && block_q != block_k) return ATTN_ERR_INVALID_ARG;
      if (n < capacity && h_out)
        h_out[n] = attn_slice_t{bi * block_q, (bi + 1) * block_q, bj * block_k, (bj + 1) * block_k,
                                g == ATTN_GRID_FULL ? ATTN_MASK_FULL : ATTN_MASK_CAUSAL};
      ++n;
    }
  *n_out = n;
  return n > capacity ? ATTN_ERR_CAPACITY : ATTN_OK;
}

int attn_fwd(const void *q, const void *k, const void *v, int sq, int sk, int hq, int hk, int d,
             float scale, const attn_tiles_t *tiles, void *out, int out_dtype, float *lse,
             attn_stream_t stream) {
  if (!q || !k || !v || !tiles || !out || !lse) return ATTN_ERR_INVALID_ARG;
  if (sq < 1 || sk < 1 || hq < 1 || hk < 1 || hq % hk != 0) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (out_dtype != ATTN_DTYPE_BF16 && out_dtype != ATTN_DTYPE_F32) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (tiles->sq != sq || tiles->sk != sk || !tiles->row_ptr) return ATTN_ERR_INVALID_ARG;
  if (tiles->tile_k != ATTN_FWD_TILE_K ||
      !(tiles->tile_q == ATTN_FWD_TILE_Q || (tiles->tile_q == ATTN_FWD_PAIR_TILE_Q && d == 128)))
    return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return ATTN_ERR_UNSUPPORTED;
  // q, k, v (read through TMA while O is written) must not overlap out
  const char *ob = static_cast<const char *>(out);
  const size_t obytes = static_cast<size_t>(sq) * hq * d * (out_dtype == ATTN_DTYPE_F32 ? 4 : 2);
  const size_t qbytes = static_cast<size_t>(sq) * hq * d * 2;
  const size_t kvbytes = static_cast<size_t>(sk) * hk * d * 2;
  auto meets_out = [&](const void *x, size_t n) {
    const char *xb = static_cast<const char *>(x);
    return xb < ob + obytes && ob < xb + n;
  };
  if (meets_out(q, qbytes) || meets_out(k, kvbytes) || meets_out(v, kvbytes))
    return ATTN_ERR_INVALID_ARG;
  return attn::fwd_launch(q, k, v, sq, sk, hq, hk, d, scale, tiles, out, out_dtype, lse,
                          reinterpret_cast<cudaStream_t>(stream));
}

int attn_bwd_workspace_bytes(const attn_tiles_t *tiles, int hq, size_t *bytes) {
  if (!tiles || !bytes || hq < 1 || !tiles->row_ptr) return ATTN_ERR_INVALID_ARG;
  *bytes = attn::bwd_workspace_bytes(tiles->sq, hq, tiles->n_ktiles, tiles->cap_entries);
  return ATTN_OK;
}

int attn_bwd(const void *q, const void *k, const void *v, const void *out, int out_dtype,
             const void *dout, const float *lse, int sq, int sk, int hq, int hk, int d, float scale,
             const attn_tiles_t *tiles, void *dq, void *dk, void *dv, int grad_dtype, void *d_ws,
             size_t ws_bytes, attn_stream_t stream) {
  if (!q || !k || !v || !out || !dout || !lse || !tiles || !dq || !dk || !dv || !d_ws)
    return ATTN_ERR_INVALID_ARG;
  if (sq < 1 || sk < 1 || hq < 1 || hk < 1 || hq % hk != 0) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if ((out_dtype != ATTN_DTYPE_BF16 && out_dtype != ATTN_DTYPE_F32) ||
      (grad_dtype != ATTN_DTYPE_BF16 && grad_dtype != ATTN_DTYPE_F32))
    return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (tiles->sq != sq || tiles->sk != sk || !tiles->row_ptr) return ATTN_ERR_INVALID_ARG;
  if (tiles->tile_q != ATTN_FWD_TILE_Q || tiles->tile_k != ATTN_FWD_TILE_K) return ATTN_ERR_UNSUPPORTED;
  const void *ptrs[] = {q, k, v, out, dout, dq, dk, dv, d_ws};
  for (const void *ptr : ptrs)
    if (!aligned16(ptr)) return ATTN_ERR_UNSUPPORTED;
  if (ws_bytes < attn::bwd_workspace_bytes(sq, hq, tiles->n_ktiles, tiles->cap_entries))
    return ATTN_ERR_CAPACITY;
  return attn::bwd_launch(q, k, v, out, out_dtype, dout, lse, sq, sk, hq, hk, d, scale, tiles, dq, dk,
                          dv, grad_dtype, d_ws, reinterpret_cast<cudaStream_t>(stream));
}

int attn_merge(const void *const *h_o_parts, const float *const *h_lse_parts, int n_parts,
               int part_dtype, int s_len, int h, int d, void *out, int out_dtype, float *lse,
               attn_stream_t stream) {
  if (!h_o_parts || !h_lse_parts || !out || !lse) return ATTN_ERR_INVALID_ARG;
  if (n_parts < 1 || n_parts > ATTN_MERGE_MAX_PARTS || s_len < 0 || h < 1)
    return ATTN_ERR_INVALID_ARG;
  if ((part_dtype != ATTN_DTYPE_BF16 && part_dtype != ATTN_DTYPE_F32) ||
      (out_dtype != ATTN_DTYPE_BF16 && out_dtype != ATTN_DTYPE_F32))
    return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(out)) return ATTN_ERR_UNSUPPORTED;
  for (int i = 0; i < n_parts; ++i) {
    if (!h_o_parts[i] || !h_lse_parts[i]) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(h_o_parts[i])) return ATTN_ERR_UNSUPPORTED;
    if (h_o_parts[i] == out || static_cast<const void *>(h_lse_parts[i]) == lse)
      return ATTN_ERR_INVALID_ARG;
  }
  return attn::merge_launch(h_o_parts, h_lse_parts, n_parts, part_dtype, s_len, h, d, out,
                            out_dtype, lse, reinterpret_cast<cudaStream_t>(stream));
}

int attn_last_device_error(attn_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  unsigned int st[3] = {0, 0, 0};
  if (attn::build_status_take(&st[0]) != ATTN_OK || attn::fwd_status_take(&st[1]) != ATTN_OK ||
      attn::bwd_status_take(&st[2]) != ATTN_OK)
    return ATTN_ERR_CUDA;
  for (unsigned int x : st)
    if (x) return static_cast<int>(x);
  return ATTN_OK;
}

int attn_set_wait_limit_ns(int64_t ns) {
  if (ns < 1000) return ATTN_ERR_INVALID_ARG;
  attn::fwd_set_wait_ns(static_cast<unsigned long long>(ns));
  return ATTN_OK;
}

int attn_set_exp2_poly(int period) {
  if (period != 0 && period != 4 && period != 8) return ATTN_ERR_INVALID_ARG;
  attn::fwd_set_exp2_poly(period);
  return ATTN_OK;
}

int attn_selftest_wait_timeout(attn_stream_t stream) {
  return attn::selftest_timeout_launch(reinterpret_cast<cudaStream_t>(stream));
}

const char *attn_strerror(int code) {
  switch (code) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_OVERLAP: return "mask slices overlap";
    case ATTN_ERR_UNSUPPORTED: return "unsupported shape, head dim or alignment";
    case ATTN_ERR_CAPACITY: return "workspace or output capacity too small";
    case ATTN_ERR_CUDA: return "CUDA runtime error";
    case ATTN_ERR_TIMEOUT: return "a bounded device wait ran out";
    default: return "unknown status";
  }
}

}  // extern "C"
