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
// One cooperative launch (both phases, a grid-wide barrier between them)
// when every query tile's CTA fits on the GPU at once, else two launches on
// one stream:
//   count  one CTA per query tile: per-key-tile counts in shared memory ->
//          entries, references and pairs of the query tile; the slices
//          visited are the query tile's bucket (built on the host with the
//          argument checks: ids of the slices meeting its rows, ascending)
//   fill   one CTA per query tile: its offsets (sums over the preceding
//          query tiles), recount, compact the entries in ascending key-tile
//          order, write the ascending slice references (one warp per masked
//          key tile), and place the query tile at its rank of the
//          longest-processing-time order; CTA 0 also writes the totals
// For every slice kind the row interval's ends never decrease with the row,
// so the first row's start and the last row's end bound the key tiles a
// slice can touch inside a query tile, and decide in O(1) the tiles it
// covers or misses entirely; only tiles cut by an interval end are counted
// row by row, lane-parallel.  Warps take one slice each when a query tile
// has many, or split one slice's key tiles when it has few.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {

constexpr int BT = 256;   // threads of the count / fill CTAs

// Where a build reads its inputs: the workspace, or the launch's parameters.
struct Inputs {
  const attn_slice_t *slices;
  const int32_t *qb_ptr, *qb_idx;
};

__device__ __forceinline__ void row_interval(const attn_slice_t &s, int i, int &lo, int &hi) {
  const int a = i - s.q_start, lq = s.q_end - s.q_start, lk = s.k_end - s.k_start;
  int l = 0, h = lk;
  if (s.type == ATTN_MASK_CAUSAL || s.type == ATTN_MASK_BI_CAUSAL) h = min(h, a + (lk - lq) + 1);
  if (s.type == ATTN_MASK_INV_CAUSAL || s.type == ATTN_MASK_BI_CAUSAL) l = max(l, a);
  if (h < l) h = l;
  lo = s.k_start + l;
  hi = s.k_start + h;
}

// Valid pairs of slice s inside rows [r0, r1) x columns [c0, c1), summed by
// the 32 lanes of a warp over interleaved rows; every lane gets the total.
__device__ __forceinline__ int warp_pairs_in(const attn_slice_t &s, int r0, int r1, int c0, int c1,
                                             int lane) {
  const int a = max(r0, s.q_start), b = min(r1, s.q_end);
  int c = 0;
  for (int i = a + lane; i < b; i += 32) {
    int lo, hi;
    row_interval(s, i, lo, hi);
    c += max(0, min(hi, c1) - max(lo, c0));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  return c;
}

// Same count, exact in O(1) when every row of the slice inside [r0, r1)
// covers [c0, c1) or misses it: the row interval's ends never decrease with
// the row, so the first and last rows bound all of them.  Only tiles cut by
// an interval end fall back to the row loop.
__device__ __forceinline__ int warp_pairs_fast(const attn_slice_t &s, int r0, int r1, int c0,
                                               int c1, int lane) {
  const int a = max(r0, s.q_start), b = min(r1, s.q_end);
  if (a >= b) return 0;
  int lo_a, hi_a, lo_b, hi_b;
  row_interval(s, a, lo_a, hi_a);
  row_interval(s, b - 1, lo_b, hi_b);
  if (hi_b <= c0 || lo_a >= c1) return 0;
  if (lo_b <= c0 && hi_a >= c1) return (b - a) * (c1 - c0);
  return warp_pairs_in(s, r0, r1, c0, c1, lane);
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

// A query tile's bucket is staged in shared memory kChunk slices at a time
// (one load per thread, all in flight together).
constexpr int kChunk = BT;
constexpr int kCutList = 1024;
__shared__ attn_slice_t s_stage[kChunk];   // staged slices
__shared__ int s_stage_id[kChunk];          // their ids (reference pass)
__shared__ int s_stage_off[kChunk];         // their first work item (count pass)
__shared__ int s_stage_kt0[kChunk];         // their first key tile (count pass)

// Key tiles [*kt0, *kt1] that slice s can touch within rows [r0, r1); empty
// when *kt1 < *kt0.
__device__ __forceinline__ void slice_ktiles(const attn_slice_t &s, int r0, int r1, int tk, int *kt0,
                                             int *kt1) {
  const int a = max(r0, s.q_start), e = min(r1, s.q_end);
  *kt0 = 1;
  *kt1 = 0;
  if (a >= e) return;
  int lo_a, hi_a, lo_e, hi_e;
  row_interval(s, a, lo_a, hi_a);
  row_interval(s, e - 1, lo_e, hi_e);
  if (hi_e <= lo_a) return;
  *kt0 = lo_a / tk;
  *kt1 = (hi_e - 1) / tk;
}

// Per-key-tile valid-pair counts (cnt) and numbers of contributing slices
// (nref) of query tile qt, in shared memory; the slices are those of the
// query tile's bucket.  Per staged chunk, every (slice, key tile it can
// touch) pair is one work item, spread over the threads by a block scan.
// A tile that every row's interval covers counts rows x width at once, a
// tile no row reaches is skipped, and a tile cut by an interval end goes to
// a shared list, whose tiles the warps then count row by row,
// lane-parallel (a full list makes the thread count the tile itself).
__device__ void count_tile_row(const BuildLaunch &b, const Inputs in, int qt, int *cnt, int *nref, int *sh) {
  const int r0 = qt * b.tq, r1 = min(r0 + b.tq, b.sq);
  const int tid = static_cast<int>(threadIdx.x), warp = tid >> 5, lane = tid & 31;
  __shared__ int cut_n;
  __shared__ int2 cut[kCutList];   // (staged slice, key tile)
  for (int t = tid; t < b.nk; t += BT) {
    cnt[t] = 0;
    nref[t] = 0;
  }
  const int u0 = in.qb_ptr[qt], u1 = in.qb_ptr[qt + 1];
  for (int base = u0; base < u1; base += kChunk) {
    const int m = min(kChunk, u1 - base);
    int ntiles = 0;
    if (tid < m) {
      const attn_slice_t s = in.slices[in.qb_idx[base + tid]];
      int kt0, kt1;
      slice_ktiles(s, r0, r1, b.tk, &kt0, &kt1);
      s_stage[tid] = s;
      s_stage_kt0[tid] = kt0;
      ntiles = max(0, kt1 - kt0 + 1);
    }
    if (tid == 0) cut_n = 0;
    int total;
    const int off = block_excl_scan(ntiles, sh, &total);   // synchronises the block
    if (tid < m) s_stage_off[tid] = off;
    __syncthreads();
    for (int wi = tid; wi < total; wi += BT) {
      // the item's slice: the last staged one whose first item is <= wi
      int lo = 0, hi = m - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_stage_off[mid] <= wi) lo = mid;
        else hi = mid - 1;
      }
      const attn_slice_t &s = s_stage[lo];
      const int kt = s_stage_kt0[lo] + (wi - s_stage_off[lo]);
      const int c0 = kt * b.tk, c1 = min(c0 + b.tk, b.sk);
      const int a = max(r0, s.q_start), e = min(r1, s.q_end);
      int lo_a, hi_a, lo_e, hi_e;
      row_interval(s, a, lo_a, hi_a);
      row_interval(s, e - 1, lo_e, hi_e);
      if (hi_e <= c0 || lo_a >= c1) continue;
      if (lo_e <= c0 && hi_a >= c1) {
        atomicAdd(&cnt[kt], (e - a) * (c1 - c0));
        atomicAdd(&nref[kt], 1);
        continue;
      }
      const int k = atomicAdd(&cut_n, 1);
      if (k < kCutList) {
        cut[k] = make_int2(lo, kt);
      } else {
        int c = 0;
        for (int i = a; i < e; ++i) {
          int l, h;
          row_interval(s, i, l, h);
          c += max(0, min(h, c1) - max(l, c0));
        }
        if (c > 0) {
          atomicAdd(&cnt[kt], c);
          atomicAdd(&nref[kt], 1);
        }
      }
    }
    __syncthreads();
    const int n_cut = min(cut_n, kCutList);
    for (int k = warp; k < n_cut; k += BT / 32) {
      const int2 item = cut[k];
      const int kt = item.y;
      const int c = warp_pairs_in(s_stage[item.x], r0, r1, kt * b.tk, min((kt + 1) * b.tk, b.sk), lane);
      if (c > 0 && lane == 0) {
        atomicAdd(&cnt[kt], c);
        atomicAdd(&nref[kt], 1);
      }
    }
    __syncthreads();
  }
  __syncthreads();
}

// Count phase of query tile qt: per-key-tile counts (cnt, nref, kept in
// shared memory) -> the tile's entries, references and pairs.
__device__ void count_phase(const BuildLaunch &b, const Inputs in, int qt, int *cnt, int *nref, int *sh) {
  count_tile_row(b, in, qt, cnt, nref, sh);
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

// Fill phase of query tile qt: offsets (sums over the preceding query
// tiles), the longest-processing-time rank, then the tile's entries in
// ascending key-tile order and its slice references.  `recount` recomputes
// cnt / nref (two-launch path); the single-launch path still has them.
// The per-tile counters of other CTAs are read through L2 (__ldcg).
__device__ void fill_phase(const BuildLaunch &b, const Inputs in, int qt, int *cnt, int *nref, int *rpos,
                           int *sh, bool recount) {
  const int w = __ldcg(b.nnz_q + qt);

  // offsets of this query tile (sums over the preceding ones), and the
  // longest-processing-time rank: tiles with more entries first, ties broken
  // by the lower index
  long long e_before = 0, r_before = 0, e_all = 0, r_all = 0, p_all = 0;
  int rank = 0;
  for (int j = threadIdx.x; j < b.nq; j += BT) {
    const int wj = __ldcg(b.nnz_q + j), rj = __ldcg(b.nref_q + j);
    rank += (wj > w || (wj == w && j < qt)) ? 1 : 0;
    if (j < qt) {
      e_before += wj;
      r_before += rj;
    }
    if (qt == 0) {
      e_all += wj;
      r_all += rj;
      p_all += __ldcg(reinterpret_cast<const long long *>(b.pairs_q) + j);
    }
  }
  __shared__ long long red[6][BT / 32];
  {
    long long v[6] = {e_before, r_before, e_all, r_all, p_all, rank};
#pragma unroll
    for (int k = 0; k < 6; ++k)
      for (int o = 16; o > 0; o >>= 1) v[k] += __shfl_xor_sync(0xffffffffu, v[k], o);
    if ((threadIdx.x & 31) == 0)
#pragma unroll
      for (int k = 0; k < 6; ++k) red[k][threadIdx.x >> 5] = v[k];
  }
  __syncthreads();
  long long tot[6] = {0, 0, 0, 0, 0, 0};
#pragma unroll
  for (int k = 0; k < 6; ++k)
    for (int u = 0; u < BT / 32; ++u) tot[k] += red[k][u];
  const long long row_start = tot[0], ref_start = tot[1];
  if (threadIdx.x == 0) {
    b.sched[tot[5]] = qt;
    b.row_ptr[qt] = static_cast<int32_t>(row_start);
    if (qt == 0) {
      const bool over = tot[2] > b.cap_entries || tot[3] > b.cap_refs;
      b.row_ptr[b.nq] = static_cast<int32_t>(tot[2]);
      b.totals[0] = tot[2];
      b.totals[1] = tot[3];
      b.totals[2] = tot[4];
      b.totals[3] = over ? ATTN_ERR_CAPACITY : ATTN_OK;
      if (!over) b.ref_ptr[tot[2]] = static_cast<int32_t>(tot[3]);
    }
  }
  // capacity exceeded: leave this tile's lists unwritten (the status says so)
  if (row_start + w > b.cap_entries || ref_start + __ldcg(b.nref_q + qt) > b.cap_refs) return;

  if (recount) count_tile_row(b, in, qt, cnt, nref, sh);
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
  int ebase = block_excl_scan(e, sh, &te) + static_cast<int>(row_start);
  int rbase = block_excl_scan(r, sh, &tr) + static_cast<int>(ref_start);
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
  // slice references of MASKED tiles: the threads list them (nref is free
  // now), then one warp per listed tile walks the bucket in ascending slice
  // id, so each tile's references come out ordered
  __shared__ int n_masked;
  if (threadIdx.x == 0) n_masked = 0;
  __syncthreads();
  int *mlist = nref;
  for (int t = t0; t < t1; ++t)
    if (cnt[t] > 0 && cnt[t] != full) mlist[atomicAdd(&n_masked, 1)] = t;
  __syncthreads();
  const int r0 = qt * b.tq, r1 = min(r0 + b.tq, b.sq);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u0 = in.qb_ptr[qt], u1 = in.qb_ptr[qt + 1];
  for (int base = u0; base < u1; base += kChunk) {
    const int m = min(kChunk, u1 - base);
    if (static_cast<int>(threadIdx.x) < m) {
      const int sid = in.qb_idx[base + threadIdx.x];
      s_stage_id[threadIdx.x] = sid;
      s_stage[threadIdx.x] = in.slices[sid];
    }
    __syncthreads();
    for (int k = warp; k < n_masked; k += BT / 32) {
      const int kt = mlist[k];
      int pos = rpos[kt];
      const int c0 = kt * b.tk, c1 = min((kt + 1) * b.tk, b.sk);
      for (int i = 0; i < m; ++i) {
        const attn_slice_t &s = s_stage[i];
        if (s.k_end <= c0 || s.k_start >= c1) continue;
        if (warp_pairs_fast(s, r0, r1, c0, c1, lane) > 0) {
          if (lane == 0) b.ref_idx[pos] = s_stage_id[i];
          ++pos;
        }
      }
      __syncwarp();
      if (lane == 0) rpos[kt] = pos;   // the next chunk continues from here
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(BT) count_kernel(const BuildLaunch b) {
  extern __shared__ int shm[];
  count_phase(b, Inputs{b.slices, b.qb_ptr, b.qb_idx}, blockIdx.x, shm, shm + b.nk, shm + 2 * b.nk);
}

__global__ void __launch_bounds__(BT) fill_kernel(const BuildLaunch b) {
  extern __shared__ int shm[];
  fill_phase(b, Inputs{b.slices, b.qb_ptr, b.qb_idx}, blockIdx.x, shm, shm + b.nk, shm + 2 * b.nk,
             shm + 3 * b.nk, true);
}

// Input images of up to kParamImage bytes travel in the single-launch
// build's parameters.
constexpr int kParamImage = 2048;
template <int N>
struct BuildImage {
  int32_t w[N / 4];
};

// Grid barriers of single-launch builds: one (arrived, departed, decision)
// triple of words per launch from a ring (host side, round robin); all start
// at 0 (static device memory) and the launch's last CTA to depart puts them
// back to 0, so no launch needs them cleared first.
constexpr int kBarSlots = 1024;
__device__ int g_build_bar[3 * kBarSlots];
constexpr int kBarGo = 1, kBarAbort = 2;   // decision word: 0 while undecided

// First failure status of a single-launch build on this device (its bounded
// grid barrier ran out); read and cleared by attn_last_device_error().
__device__ unsigned int g_build_status;

// Both phases in one cooperative launch (every CTA resident): the counts
// stay in shared memory across a grid-wide barrier, so nothing is
// recounted and one launch is saved.  The barrier's wait is bounded.  The
// barrier ends with one decision that every CTA follows: "go", set by the
// last CTA to arrive, or "abort", set by a CTA whose wait ran out first
// (only the first of the two compare-and-swaps on the decision word takes).
// On abort no CTA fills; each writes an empty list for its query tile and
// CTA 0 writes zero totals with ATTN_ERR_TIMEOUT as the status, so the
// metadata stays valid (every list empty) and the kernels that read it see
// the status and refuse it.  PARAM: the inputs are read from `img` (the
// launch's parameters), and CTA 0 also writes the slices into the workspace
// for the kernels that follow.

template <bool PARAM>
__global__ void __launch_bounds__(BT) build_kernel(const BuildLaunch b,
                                                   const __grid_constant__ BuildImage<kParamImage> img) {
  extern __shared__ int shm[];
  int *cnt = shm, *nref = shm + b.nk, *rpos = shm + 2 * b.nk, *sh = shm + 3 * b.nk;
  const int qt = blockIdx.x;
  Inputs in{b.slices, b.qb_ptr, b.qb_idx};
  if (PARAM) {
    const uint8_t *base = reinterpret_cast<const uint8_t *>(img.w);
    in.slices = reinterpret_cast<const attn_slice_t *>(base);
    in.qb_ptr = reinterpret_cast<const int32_t *>(base + b.off_qb_ptr);
    in.qb_idx = reinterpret_cast<const int32_t *>(base + b.off_qb_idx);
    if (qt == 0) {
      int32_t *dst = reinterpret_cast<int32_t *>(const_cast<attn_slice_t *>(b.slices));
      const int words = static_cast<int>(sizeof(attn_slice_t) / 4) * b.n_slices;
      for (int i = threadIdx.x; i < words; i += BT) dst[i] = img.w[i];
    }
  }
  count_phase(b, in, qt, cnt, nref, sh);
  __shared__ int go;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();                   // this tile's counters before the arrival
    if (atomicAdd(b.grid_bar, 1) == static_cast<int>(gridDim.x) - 1) {
      __threadfence();                 // every arrival (and its counters) before "go"
      atomicCAS(b.grid_state, 0, kBarGo);
    }
    const unsigned long long deadline = globaltimer_ns() + b.wait_ns;
    int st;
    while ((st = *reinterpret_cast<volatile int *>(b.grid_state)) == 0) {
      if (globaltimer_ns() > deadline) {
        const int prev = atomicCAS(b.grid_state, 0, kBarAbort);
        st = prev == 0 ? kBarAbort : prev;
        break;
      }
    }
    __threadfence();
    go = st == kBarGo;
    // the last CTA out (every CTA has read the decision) resets the slot
    if (atomicAdd(b.grid_dep, 1) == static_cast<int>(gridDim.x) - 1) {
      atomicExch(b.grid_bar, 0);
      atomicExch(b.grid_state, 0);
      atomicExch(b.grid_dep, 0);
    }
  }
  __syncthreads();
  if (!go) {
    if (threadIdx.x == 0) {
      b.row_ptr[qt] = 0;
      b.sched[qt] = qt;
      if (qt == 0) {
        b.row_ptr[b.nq] = 0;
        b.ref_ptr[0] = 0;
        b.totals[0] = 0;
        b.totals[1] = 0;
        b.totals[2] = 0;
        b.totals[3] = ATTN_ERR_TIMEOUT;
        atomicCAS(&g_build_status, 0u, static_cast<unsigned>(ATTN_ERR_TIMEOUT));
      }
    }
    return;
  }
  fill_phase(b, in, qt, cnt, nref, rpos, sh, false);
}

int build_tiles_launch(BuildLaunch b, const uint8_t *img, size_t img_bytes, void *ws, cudaStream_t s) {
  const size_t sm_count = (2 * static_cast<size_t>(b.nk) + 64) * sizeof(int);
  const size_t sm_fill = (3 * static_cast<size_t>(b.nk) + 64) * sizeof(int);
  constexpr int kMaxDev = 64;
  static int coresident[kMaxDev][2] = {};   // CTAs of build_kernel<PARAM> that fit at once
  static size_t coresident_smem[kMaxDev] = {};
  static int *bar_base[kMaxDev] = {};
  int fit[2] = {0, 0};   // this call's copy of coresident[dev], taken under the lock
  static std::atomic<unsigned> bar_seq{0};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return ATTN_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lock(mu);
    static bool configured[kMaxDev] = {};
    if (!configured[dev]) {
      void *ptr = nullptr;
      if (cudaFuncSetAttribute(count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               200 * 1024) != cudaSuccess ||
          cudaFuncSetAttribute(fill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               200 * 1024) != cudaSuccess ||
          cudaFuncSetAttribute(build_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               200 * 1024) != cudaSuccess ||
          cudaFuncSetAttribute(build_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               200 * 1024) != cudaSuccess ||
          cudaGetSymbolAddress(&ptr, g_build_bar) != cudaSuccess)
        return ATTN_ERR_CUDA;
      bar_base[dev] = static_cast<int *>(ptr);
      configured[dev] = true;
    }
    // one launch when every query tile's CTA can be resident at once
    if (coresident_smem[dev] != sm_fill) {
      int per_sm[2] = {0, 0}, sms = 0, coop = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm[0], build_kernel<false>, BT, sm_fill) !=
              cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm[1], build_kernel<true>, BT, sm_fill) !=
              cudaSuccess ||
          cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess)
        return ATTN_ERR_CUDA;
      coresident[dev][0] = coop ? per_sm[0] * sms : 0;
      coresident[dev][1] = coop ? per_sm[1] * sms : 0;
      coresident_smem[dev] = sm_fill;
    }
    fit[0] = coresident[dev][0];
    fit[1] = coresident[dev][1];
  }
  // ATTN_BUILD_TWO_LAUNCH=1 in the environment selects the two-launch path
  // (used by the tests to check that all paths give the same metadata)
  const char *two = std::getenv("ATTN_BUILD_TWO_LAUNCH");
  const bool force_two = two && two[0] == '1';
  const bool param = img_bytes <= static_cast<size_t>(kParamImage) && !force_two &&
                     b.nq <= fit[1];
  if (b.nq <= 0 || !param) {
    if (img_bytes > 0 && cudaMemcpyAsync(ws, img, img_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
      return ATTN_ERR_CUDA;
    if (b.nq <= 0) return ATTN_OK;
  }
  BuildImage<kParamImage> im;
  if (param) {
    std::memset(&im, 0, sizeof(im));
    std::memcpy(im.w, img, img_bytes);
  }
  if (param || (!force_two && b.nq <= fit[0])) {
    const unsigned slot = bar_seq.fetch_add(1) % kBarSlots;
    b.grid_bar = bar_base[dev] + slot;
    b.grid_dep = bar_base[dev] + kBarSlots + slot;
    b.grid_state = bar_base[dev] + 2 * kBarSlots + slot;
    void *args[] = {&b, &im};
    const void *fn = param ? reinterpret_cast<const void *>(build_kernel<true>)
                           : reinterpret_cast<const void *>(build_kernel<false>);
    if (cudaLaunchCooperativeKernel(fn, dim3(b.nq), dim3(BT), args, sm_fill, s) != cudaSuccess)
      return ATTN_ERR_CUDA;
    return ATTN_OK;
  }
  count_kernel<<<b.nq, BT, sm_count, s>>>(b);
  fill_kernel<<<b.nq, BT, sm_fill, s>>>(b);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int build_status_take(unsigned int *status) {
  unsigned int zero = 0;
  if (cudaMemcpyFromSymbol(status, g_build_status, sizeof(unsigned int)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (*status && cudaMemcpyToSymbol(g_build_status, &zero, sizeof(unsigned int)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

}  // namespace attn
