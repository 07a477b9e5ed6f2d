// attn_build_tiles_noalloc: the tile-metadata build with its scratch
// counters in a fixed device array owned by this library, for callers that
// cannot hand out or allocate extra device memory when they build a mask.
//
// attn_build_tiles keeps four per-query-tile counters (entries, references,
// reference base, valid pairs) in the caller's workspace.  Here they live in
// g_tiles_scratch below, a file-scope device array of kMaxQTiles entries that
// every device loading this library holds until the process exits.  The
// caller still provides the slice list and the buffer that receives the
// metadata.  The kernels are the same as those of attn_build_tiles.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kMaxQTiles = ATTN_NOALLOC_MAX_QTILES;
constexpr int kMaxDevices = 64;

// nnz_q int32 | nref_q int32 | ref_base_q int32 | pairs_q int64, kMaxQTiles each.
static __device__ __align__(256) unsigned char g_tiles_scratch[kMaxQTiles * 20];

std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_tiles_scratch on the current device.  In host code the
// symbol's name is only a host-side stand-in, so the real address is asked
// for once per device (with that device current) and kept.
int scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_tiles_scratch) != cudaSuccess || !p) return ATTN_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return ATTN_OK;
}

}  // namespace
}  // namespace attn

using namespace attn::host;

extern "C" int attn_build_tiles_noalloc(const attn_slice_t *h_slices, int n_slices, int sq, int sk,
                                        int tile_q, int tile_k, void *d_out, size_t out_bytes,
                                        attn_tiles_t *tiles, attn_stream_t stream) {
  if (!tiles || !d_out) return ATTN_ERR_INVALID_ARG;
  int nq, nk, rc;
  if ((rc = shape_ok(sq, sk, tile_q, tile_k, &nq, &nk)) != ATTN_OK) return rc;
  if (nq > attn::kMaxQTiles) return ATTN_ERR_CAPACITY;
  if ((rc = check_slices(h_slices, n_slices, sq, sk)) != ATTN_OK) return rc;
  if ((rc = check_overlap(h_slices, n_slices)) != ATTN_OK) return rc;
  if (static_cast<int64_t>(tile_q) * tile_k >= (int64_t(1) << 31)) return ATTN_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(d_out) & 255u) != 0) return ATTN_ERR_UNSUPPORTED;
  const WsLayout L = layout(h_slices, n_slices, nq, nk, tile_q, tile_k);
  if (out_bytes < L.total) return ATTN_ERR_CAPACITY;
  void *scratch = nullptr;
  if ((rc = attn::scratch_address(&scratch)) != ATTN_OK) return rc;
  uint8_t *ws = static_cast<uint8_t *>(d_out);
  uint8_t *sc = static_cast<uint8_t *>(scratch);
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
  t.scratch = reinterpret_cast<int32_t *>(sc);

  static thread_local std::vector<uint8_t> img;   // kept across calls
  stage_inputs(h_slices, n_slices, nq, tile_q, L, &img);
  // The counters are written (not accumulated) by the count kernel before
  // the fill kernel reads them, so the previous call's contents in
  // the shared array need no clearing.
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
  b.nnz_q = reinterpret_cast<int32_t *>(sc);
  b.nref_q = reinterpret_cast<int32_t *>(sc + 4 * static_cast<size_t>(attn::kMaxQTiles));
  b.ref_base_q = reinterpret_cast<int32_t *>(sc + 8 * static_cast<size_t>(attn::kMaxQTiles));
  b.pairs_q = reinterpret_cast<int64_t *>(sc + 12 * static_cast<size_t>(attn::kMaxQTiles));
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
