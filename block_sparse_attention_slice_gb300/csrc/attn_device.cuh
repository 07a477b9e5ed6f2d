// Pieces shared by the forward and backward attention kernels: bounded
// warp-wide waits, tensor-memory loads, the per-row (and per-key) valid
// intervals of a mask slice and their 128-bit tile masks, and the host-side
// TMA descriptor and SM-count helpers.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/attn_slice.h"
#include "ptx.cuh"

namespace attn {

// ------------------------------------------------------------------ device

__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity, volatile int *abort,
                                         uint64_t limit) {
  bool ok = mbar_wait_bounded(bar, parity, abort, limit);
  return __all_sync(0xffffffffu, ok);
}

// wait_all with a cluster-scope acquire (barriers the other CTA of a pair
// completes).
__device__ __forceinline__ bool wait_all_cl(uint32_t bar, uint32_t parity, volatile int *abort,
                                            uint64_t limit) {
  bool ok = mbar_wait_bounded_cl(bar, parity, abort, limit);
  return __all_sync(0xffffffffu, ok);
}

// Waits for in-flight asynchronous work before tensor memory and shared
// memory are released on the failure path; bounded independently of *abort.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t dl = globaltimer_ns() + limit_ns;
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() > dl) break;
  }
}

__device__ __forceinline__ void tmem_ld32_wait(uint32_t taddr, uint32_t (&r)[32]) {
  tmem_ld32(taddr, r);
  tmem_wait_ld();
#pragma unroll
  for (int k = 0; k < 32; ++k) asm volatile("" : "+r"(r[k]));
}

__device__ __forceinline__ uint32_t bits_below(int x) {   // bits [0, x) set, 0 <= x <= 32
  return x >= 32 ? 0xffffffffu : ((1u << x) - 1u);
}

// Valid key interval [lo, hi) of slice `s` for query row i (global indices);
// empty (lo == hi) when row i is outside the slice.
__device__ __forceinline__ void slice_interval(const attn_slice_t &s, int i, int &lo, int &hi) {
  if (i < s.q_start || i >= s.q_end) {
    lo = hi = 0;
    return;
  }
  const int a = i - s.q_start, lq = s.q_end - s.q_start, lk = s.k_end - s.k_start;
  int l = 0, h = lk;
  if (s.type == ATTN_MASK_CAUSAL || s.type == ATTN_MASK_BI_CAUSAL) h = min(h, a + (lk - lq) + 1);
  if (s.type == ATTN_MASK_INV_CAUSAL || s.type == ATTN_MASK_BI_CAUSAL) l = max(l, a);
  if (h < l) h = l;
  lo = s.k_start + l;
  hi = s.k_start + h;
}

// Valid query interval [lo, hi) of slice `s` for key j (global indices): the
// same predicates solved for the row, local a against local b = j - k_start:
// causal b <= a + (L_k - L_q)  <=>  a >= b - (L_k - L_q);  inv-causal a <= b.
__device__ __forceinline__ void slice_col_interval(const attn_slice_t &s, int j, int &lo, int &hi) {
  if (j < s.k_start || j >= s.k_end) {
    lo = hi = 0;
    return;
  }
  const int b = j - s.k_start, lq = s.q_end - s.q_start, lk = s.k_end - s.k_start;
  int l = 0, h = lq;
  if (s.type == ATTN_MASK_CAUSAL || s.type == ATTN_MASK_BI_CAUSAL) l = max(l, b - (lk - lq));
  if (s.type == ATTN_MASK_INV_CAUSAL || s.type == ATTN_MASK_BI_CAUSAL) h = min(h, b + 1);
  if (h < l) h = l;
  lo = s.q_start + l;
  hi = s.q_start + h;
}

// ORs the columns [lo, hi) (global) falling in tile [c0, c0+128) into the
// 128-bit mask w (bit k of w[k/32] = column c0 + k).
__device__ __forceinline__ void or_span(int lo, int hi, int c0, uint32_t (&w)[4]) {
  lo = min(max(lo - c0, 0), 128);
  hi = min(max(hi - c0, 0), 128);
  if (hi <= lo) return;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int a = min(max(lo - 32 * c, 0), 32), b = min(max(hi - 32 * c, 0), 32);
    w[c] |= bits_below(b) & ~bits_below(a);
  }
}

// ORs the valid keys of slice `s` for query `row` inside key tile [c0, c0+128).
__device__ __forceinline__ void add_mask(const attn_slice_t &s, int row, int c0, uint32_t (&w)[4]) {
  int lo, hi;
  slice_interval(s, row, lo, hi);
  or_span(lo, hi, c0, w);
}

// ORs the valid queries of slice `s` for key `key` inside query tile [r0, r0+128).
__device__ __forceinline__ void add_col_mask(const attn_slice_t &s, int key, int r0, uint32_t (&w)[4]) {
  int lo, hi;
  slice_col_interval(s, key, lo, hi);
  or_span(lo, hi, r0, w);
}

// ------------------------------------------------------------------ host

inline PFN_cuTensorMapEncodeTiled_v12000 tma_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 2-D bf16 map over a [rows, cols] row-major matrix, boxes of 64 columns x
// box_rows rows with the 128-byte swizzle the MMA descriptors expect.
inline int make_tma_2d(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows,
                       uint32_t box_rows = 128) {
  auto enc = tma_encode_fn();
  if (!enc) return ATTN_ERR_CUDA;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// 2-D f32 map over a [rows, cols] row-major matrix, 32 x 128 boxes (128-byte
// rows), no swizzle: used to store rows of zeros from shared memory.
inline int make_tma_2d_f32(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows) {
  auto enc = tma_encode_fn();
  if (!enc) return ATTN_ERR_CUDA;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 4};
  cuuint32_t box[2] = {32, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// Number of SMs of the current device (cached per device), or -1.
inline int device_sm_count() {
  constexpr int kMax = 64;
  static int cached[kMax] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMax) return -1;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return -1;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace attn
