// Declarations shared by the translation units of the library (host side).
#pragma once
#include <cuda_runtime.h>

#include <cstdint>
#include <vector>

#include "../../include/attn_slice.h"

namespace attn {

// Host-side checks and workspace layout of the tile metadata (attn_api.cu).
namespace host {
struct WsLayout {
  // input region: slices | qb_ptr | qb_idx, then the outputs
  size_t slices, qb_ptr, qb_idx, input_bytes;
  size_t row_ptr, sched, nnz_q, nref_q, ref_base_q, pairs_q, totals, col_idx, pairs, ref_ptr,
      kind, ref_idx, total;
  int64_t cap_e, cap_r, n_qb;
};
int check_slices(const attn_slice_t *s, int n, int sq, int sk);
int check_overlap(const attn_slice_t *s, int n);
int shape_ok(int sq, int sk, int tq, int tk, int *nq, int *nk);
WsLayout layout(const attn_slice_t *s, int n, int nq, int nk, int tq, int tk);
// Host image of the input region: the slices, then per query tile the ids of
// the non-empty slices whose rows meet it (CSR, ascending ids).
void stage_inputs(const attn_slice_t *s, int n, int nq, int tq, const WsLayout &L,
                  std::vector<uint8_t> *img);
}  // namespace host

struct BuildLaunch {
  const attn_slice_t *slices;
  const int32_t *qb_ptr, *qb_idx;   // slices meeting each query tile, ascending ids
  int n_slices, sq, sk, tq, tk, nq, nk;
  int32_t *nnz_q, *nref_q, *ref_base_q;
  int64_t *pairs_q;
  int32_t *row_ptr, *col_idx, *pairs, *ref_ptr, *ref_idx, *sched;
  uint8_t *kind;
  int64_t *totals;
  int64_t cap_entries, cap_refs;
  uint32_t off_qb_ptr, off_qb_idx;  // byte offsets of qb_ptr / qb_idx in the input image
  int32_t *grid_bar, *grid_dep, *grid_state;   // set by build_tiles_launch
  unsigned long long wait_ns;       // bound of the single-launch build's grid barrier
};

// Uploads the input region's host image `img` (slices at offset 0, then
// qb_ptr, qb_idx) to the start of the workspace `ws` and builds.  Small
// images ride in the launch's parameters instead (no copy); the build then
// writes the slices into the workspace itself.
int build_tiles_launch(BuildLaunch b, const uint8_t *img, size_t img_bytes, void *ws, cudaStream_t s);
// Reads and clears the first failure status of single-launch builds on the
// current device (0 when none).
int build_status_take(unsigned int *status);

int fwd_launch(const void *q, const void *k, const void *v, int sq, int sk, int hq, int hk, int d,
               float scale, const attn_tiles_t *tiles, void *out, int out_dtype, float *lse,
               cudaStream_t stream);
int fwd_status_take(unsigned int *status);
void fwd_set_wait_ns(unsigned long long ns);
void fwd_set_exp2_poly(int period);
unsigned long long wait_limit_ns();
int selftest_timeout_launch(cudaStream_t s);

size_t bwd_workspace_bytes(int sq, int hq, int n_ktiles, int64_t cap_entries);
int bwd_launch(const void *q, const void *k, const void *v, const void *out, int out_dtype,
               const void *dout, const float *lse, int sq, int sk, int hq, int hk, int d, float scale,
               const attn_tiles_t *tiles, void *dq, void *dk, void *dv, int grad_dtype, void *d_ws,
               cudaStream_t stream);
int bwd_status_take(unsigned int *status);

int merge_launch(const void *const *o_parts, const float *const *lse_parts, int n_parts,
                 int part_dtype, int s_len, int h, int d, void *out, int out_dtype, float *lse,
                 cudaStream_t s);

}  // namespace attn
