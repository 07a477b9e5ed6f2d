// Slice list -> tile metadata, on the GPU, without materialising the mask
// (MagiAttention v1.1.0 page: block-sparse mask generation operator, CSR
// compression of the metadata).  Integer work only, so the output is exact
// and identical run to run.
//
// For query tile qt (rows [r0, r1)) and key tile kt the number of valid
// pairs contributed by slice s is the sum over the tile's rows of the
// length of (row interval of s) ∩ (columns of kt); the row interval follows
// from the slice kind (full / causal / inv-causal / bi-causal).  Slices are
// disjoint, so the tile count is the sum over slices.  A tile is
//   Empty   (count 0)          -> no entry
//   FULL    (count == tq * tk) -> no per-element mask needed
//   MASKED  (otherwise)        -> references the slices with pairs in it
// (UltraAttn page, section 3: Full / Causal / Empty blocks).
//
// Three launches on one stream:
//   count  one CTA per query tile: per-key-tile counts in shared memory ->
//          entries, references and pairs of the query tile
//   scan   one CTA: exclusive scans -> row pointers, reference bases, totals
//   fill   one CTA per query tile: recount, compact the entries in ascending
//          key-tile order, write the ascending slice references, and place
//          the query tile at its rank of the longest-processing-time order
#include <cuda_runtime.h>

#include <cstdint>

#include "attn_internal.h"

namespace attn {

constexpr int BT = 256;   // threads of the count / fill CTAs

__device__ __forceinline__ void row_interval(const attn_slice_t &s, int i, int &lo, int &hi) {
  const int a = i - s.q_start, lq = s.q_end - s.q_start, lk = s.k_end - s.k_start;
  int l = 0, h = lk;
  if (s.type == ATTN_MASK_CAUSAL || s.type == ATTN_MASK_BI_CAUSAL) h = min(h, a + (lk - lq) + 1);
  if (s.type == ATTN_MASK_INV_CAUSAL || s.type == ATTN_MASK_BI_CAUSAL) l = max(l, a);
  if (h < l) h = l;
  lo = s.k_start + l;
  hi = s.k_start + h;
}

// Valid pairs of slice s inside rows [r0, r1) x columns [c0, c1).
__device__ __forceinline__ int pairs_in(const attn_slice_t &s, int r0, int r1, int c0, int c1) {
  const int a = max(r0, s.q_start), b = min(r1, s.q_end);
  int c = 0;
  for (int i = a; i < b; ++i) {
    int lo, hi;
    row_interval(s, i, lo, hi);
    c += max(0, min(hi, c1) - max(lo, c0));
  }
  return c;
}

__device__ __forceinline__ bool hits_rows(const attn_slice_t &s, int r0, int r1) {
  return s.q_end > s.q_start && s.k_end > s.k_start && s.q_start < r1 && r0 < s.q_end;
}

// Block-wide exclusive scan of one int per thread (BT threads); returns the
// prefix and writes the block total to *total.
__device__ int block_excl_scan(int v, int *sh, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < BT / 32 ? sh[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < BT / 32) sh[lane] = w;
  }
  __syncthreads();
  const int before = (warp > 0 ? sh[warp - 1] : 0) + x - v;
  *total = sh[BT / 32 - 1];
  __syncthreads();
  return before;
}

// Collects, in ascending order, the ids of the slices that touch rows
// [r0, r1) into `list` (at most BT per call, starting from slice `from`).
__device__ int gather_hits(const BuildLaunch &b, int from, int r0, int r1, int *list, int *sh) {
  const int s = from + threadIdx.x;
  const int hit = (s < b.n_slices && hits_rows(b.slices[s], r0, r1)) ? 1 : 0;
  int total;
  const int pos = block_excl_scan(hit, sh, &total);
  if (hit) list[pos] = s;
  __syncthreads();
  return total;
}

// Per-key-tile valid-pair counts (cnt) and numbers of contributing slices
// (nref) of query tile qt, accumulated in shared memory.
__device__ void count_tile_row(const BuildLaunch &b, int qt, int *cnt, int *nref, int *list,
                               int *sh) {
  const int r0 = qt * b.tq, r1 = min(r0 + b.tq, b.sq);
  for (int t = threadIdx.x; t < b.nk; t += BT) {
    cnt[t] = 0;
    nref[t] = 0;
  }
  __syncthreads();
  for (int from = 0; from < b.n_slices; from += BT) {
    const int m = gather_hits(b, from, r0, r1, list, sh);
    for (int u = 0; u < m; ++u) {
      const attn_slice_t s = b.slices[list[u]];
      const int kt0 = s.k_start / b.tk, kt1 = (s.k_end - 1) / b.tk;
      for (int kt = kt0 + threadIdx.x; kt <= kt1; kt += BT) {
        const int c = pairs_in(s, r0, r1, kt * b.tk, min((kt + 1) * b.tk, b.sk));
        if (c > 0) {
          atomicAdd(&cnt[kt], c);
          atomicAdd(&nref[kt], 1);
        }
      }
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(BT) count_kernel(const BuildLaunch b) {
  extern __shared__ int shm[];
  int *cnt = shm, *nref = shm + b.nk, *list = shm + 2 * b.nk, *sh = list + BT;
  const int qt = blockIdx.x;
  count_tile_row(b, qt, cnt, nref, list, sh);
  const int full = b.tq * b.tk;
  int e = 0, r = 0;
  long long pr = 0;
  for (int t = threadIdx.x; t < b.nk; t += BT) {
    const int c = cnt[t];
    if (c > 0) {
      ++e;
      pr += c;
      if (c != full) r += nref[t];
    }
  }
  int te, tr;
  block_excl_scan(e, sh, &te);
  block_excl_scan(r, sh, &tr);
  // 64-bit pair total: warp shuffles then one shared atomic per warp
  __shared__ unsigned long long psum;
  if (threadIdx.x == 0) psum = 0;
  __syncthreads();
  for (int o = 16; o > 0; o >>= 1) pr += __shfl_down_sync(0xffffffffu, pr, o);
  if ((threadIdx.x & 31) == 0) atomicAdd(&psum, static_cast<unsigned long long>(pr));
  __syncthreads();
  if (threadIdx.x == 0) {
    b.nnz_q[qt] = te;
    b.nref_q[qt] = tr;
    b.pairs_q[qt] = static_cast<int64_t>(psum);
  }
}

// One CTA of 1024 threads: exclusive scans over the query tiles.
__global__ void __launch_bounds__(1024) scan_kernel(const BuildLaunch b) {
  __shared__ long long sh_e[1024], sh_r[1024], sh_p[1024];
  const int per = (b.nq + 1023) / 1024;
  const int i0 = threadIdx.x * per, i1 = min(i0 + per, b.nq);
  long long e = 0, r = 0, pr = 0;
  for (int i = i0; i < i1; ++i) {
    e += b.nnz_q[i];
    r += b.nref_q[i];
    pr += b.pairs_q[i];
  }
  sh_e[threadIdx.x] = e;
  sh_r[threadIdx.x] = r;
  sh_p[threadIdx.x] = pr;
  __syncthreads();
  // inclusive Hillis-Steele scan over the 1024 partial sums
  for (int o = 1; o < 1024; o <<= 1) {
    long long ve = 0, vr = 0, vp = 0;
    if (threadIdx.x >= o) {
      ve = sh_e[threadIdx.x - o];
      vr = sh_r[threadIdx.x - o];
      vp = sh_p[threadIdx.x - o];
    }
    __syncthreads();
    sh_e[threadIdx.x] += ve;
    sh_r[threadIdx.x] += vr;
    sh_p[threadIdx.x] += vp;
    __syncthreads();
  }
  long long be = threadIdx.x ? sh_e[threadIdx.x - 1] : 0;
  long long br = threadIdx.x ? sh_r[threadIdx.x - 1] : 0;
  for (int i = i0; i < i1; ++i) {
    b.row_ptr[i] = static_cast<int32_t>(be);
    b.ref_base_q[i] = static_cast<int32_t>(br);
    be += b.nnz_q[i];
    br += b.nref_q[i];
  }
  if (threadIdx.x == 1023) {
    const long long nnz = sh_e[1023], nref = sh_r[1023];
    b.row_ptr[b.nq] = static_cast<int32_t>(nnz);
    b.totals[0] = nnz;
    b.totals[1] = nref;
    b.totals[2] = sh_p[1023];
    const bool over = nnz > b.cap_entries || nref > b.cap_refs;
    b.totals[3] = over ? ATTN_ERR_CAPACITY : ATTN_OK;
    if (!over) b.ref_ptr[nnz] = static_cast<int32_t>(nref);
  }
}

__global__ void __launch_bounds__(BT) fill_kernel(const BuildLaunch b) {
  extern __shared__ int shm[];
  int *cnt = shm, *nref = shm + b.nk, *rpos = shm + 2 * b.nk, *list = shm + 3 * b.nk,
      *sh = list + BT;
  const int qt = blockIdx.x;

  // longest-processing-time rank of this query tile: tiles with more entries
  // first, ties broken by the lower index
  {
    const int w = b.nnz_q[qt];
    int rank = 0;
    for (int j = threadIdx.x; j < b.nq; j += BT) {
      const int wj = b.nnz_q[j];
      rank += (wj > w || (wj == w && j < qt)) ? 1 : 0;
    }
    int tot;
    block_excl_scan(rank, sh, &tot);
    if (threadIdx.x == 0) b.sched[tot] = qt;
  }
  if (b.totals[3] != ATTN_OK) return;   // capacity exceeded: leave the lists unwritten

  count_tile_row(b, qt, cnt, nref, list, sh);
  const int full = b.tq * b.tk;
  // entries of this query tile in ascending key-tile order: each thread owns
  // a contiguous run of key tiles so a single scan orders them
  const int per = (b.nk + BT - 1) / BT;
  const int t0 = threadIdx.x * per, t1 = min(t0 + per, b.nk);
  int e = 0, r = 0;
  for (int t = t0; t < t1; ++t)
    if (cnt[t] > 0) {
      ++e;
      if (cnt[t] != full) r += nref[t];
    }
  int te, tr;
  int ebase = block_excl_scan(e, sh, &te) + b.row_ptr[qt];
  int rbase = block_excl_scan(r, sh, &tr) + b.ref_base_q[qt];
  for (int t = t0; t < t1; ++t) {
    const int c = cnt[t];
    if (c <= 0) continue;
    const bool masked = c != full;
    b.col_idx[ebase] = t;
    b.pairs[ebase] = c;
    b.kind[ebase] = masked ? ATTN_TILE_MASKED : ATTN_TILE_FULL;
    b.ref_ptr[ebase] = rbase;
    rpos[t] = rbase;
    ++ebase;
    if (masked) rbase += nref[t];
  }
  __syncthreads();
  // slice references of MASKED tiles, ascending slice id: slices are visited
  // in ascending order and each key tile is written by one thread per slice
  const int r0 = qt * b.tq, r1 = min(r0 + b.tq, b.sq);
  for (int from = 0; from < b.n_slices; from += BT) {
    const int m = gather_hits(b, from, r0, r1, list, sh);
    for (int u = 0; u < m; ++u) {
      const int sid = list[u];
      const attn_slice_t s = b.slices[sid];
      const int kt0 = s.k_start / b.tk, kt1 = (s.k_end - 1) / b.tk;
      for (int kt = kt0 + threadIdx.x; kt <= kt1; kt += BT) {
        if (cnt[kt] <= 0 || cnt[kt] == full) continue;
        if (pairs_in(s, r0, r1, kt * b.tk, min((kt + 1) * b.tk, b.sk)) > 0)
          b.ref_idx[rpos[kt]++] = sid;
      }
      __syncthreads();
    }
  }
}

int build_tiles_launch(const BuildLaunch &b, cudaStream_t s) {
  const size_t sm_count = (2 * static_cast<size_t>(b.nk) + BT + 64) * sizeof(int);
  const size_t sm_fill = (3 * static_cast<size_t>(b.nk) + BT + 64) * sizeof(int);
  static int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    if (cudaFuncSetAttribute(count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             200 * 1024) != cudaSuccess ||
        cudaFuncSetAttribute(fill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             200 * 1024) != cudaSuccess)
      return ATTN_ERR_CUDA;
    configured_dev = dev;
  }
  if (b.nq > 0) {
    count_kernel<<<b.nq, BT, sm_count, s>>>(b);
    scan_kernel<<<1, 1024, 0, s>>>(b);
    fill_kernel<<<b.nq, BT, sm_fill, s>>>(b);
  }
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn
