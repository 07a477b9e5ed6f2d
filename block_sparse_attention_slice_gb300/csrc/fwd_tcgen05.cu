// Masked attention forward on sm_103a: tcgen05 MMAs with tensor-memory
// accumulators, TMA-fed multi-stage mbarrier pipeline, Empty tiles skipped
// (only the tile list of the CSR metadata is visited), per-element masking
// only on MASKED tiles, conditional (lazy) softmax rescaling.
//
// Method: for a fixed query tile, merge the softmax summaries over its valid
// KV tiles (UltraAttn page, section 3.3) with the online update of the
// running max m, normaliser l and output accumulator o (section 3.2).  The
// rescale of o is skipped unless the running max grew by more than TAU
// (FlashAttention-4 page, "conditional softmax rescaling"); the final
// O = o / l uses the same reference, so the result is exact either way.
//
// CTA = 256 query rows of one head (two 128-row MMA tiles, t = 0, 1) and
// the KV-tile list of that 256-row query tile.  Warp roles (320 threads):
//   warps 0-3  softmax of tile 0 (thread = row = tensor-memory lane)
//   warps 4-7  softmax of tile 1
//   warp  8    TMA producer: Q once, then K_j, V_j through an NS-slot ring
//   warp  9    tensor-memory allocator and MMA issuer
// Tensor memory (512 columns): S_0 [0,128)  S_1 [128,256)  O_0 [256,256+D)
// O_1 [384,384+D).  P (bf16) overwrites the first 64 columns of S_t and is
// the A operand of O_t += P_t V_j read straight from tensor memory, so the
// probabilities never touch shared memory.  The MMA order per KV step j is
//   PV_0(j), QK_0(j+1), PV_1(j), QK_1(j+1)
// so the tensor core works on one tile while the softmax warps of the other
// tile run (FlashAttention-4 page: softmax overlapped with the MMAs).
// tcgen05 operations of one thread complete in issue order, so when the
// softmax of tile t sees S_t(j) its previous PV_t(j-1) has completed too.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {

__device__ unsigned int g_fwd_status;

constexpr int BM = 128;           // rows per MMA tile
constexpr int BN = 128;           // keys per KV tile
constexpr float TAU = 8.0f;       // lazy-rescale threshold, log2 units
constexpr int NTHREADS = 320;

struct FwdParams {
  const int32_t *row_ptr, *col_idx, *ref_ptr, *ref_idx, *sched;
  const uint8_t *kind;
  const attn_slice_t *slices;
  void *out;
  float *lse;
  int sq, sk, hq, hk;
  int out_f32;
  float scale_log2;               // scale * log2(e)
  unsigned long long wait_ns;
};

template <int D, int NS>
struct Layout {
  static constexpr int HALF = 128 * 64 * 2;          // 128 rows x 64 bf16 (one swizzle span)
  static constexpr int NHALF = D / 64;
  static constexpr int TILE = NHALF * HALF;          // 128 x D bf16
  static constexpr int Q_OFF = 0;
  static constexpr int KV_OFF = 2 * TILE;
  static constexpr int BAR_OFF = KV_OFF + NS * TILE;
  // barriers: q_full | full[NS] | empty[NS] | s_full[2] | p_full[2] | o_full[2] | drain
  static constexpr int B_Q = 0, B_FULL = 1, B_EMPTY = 1 + NS, B_S = 1 + 2 * NS,
                       B_P = B_S + 2, B_O = B_P + 2, B_DRAIN = B_O + 2, NBAR = B_DRAIN + 1;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int BYTES = MISC_OFF + 16;
  static constexpr int ALLOC = BYTES + 1024;
};

__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity, volatile int *abort,
                                         uint64_t deadline) {
  bool ok = mbar_wait_bounded(bar, parity, abort, deadline);
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
  if (s.type == 1 || s.type == 3) h = min(h, a + (lk - lq) + 1);
  if (s.type == 2 || s.type == 3) l = max(l, a);
  if (h < l) h = l;
  lo = s.k_start + l;
  hi = s.k_start + h;
}

template <int D, int NS>
__global__ void __launch_bounds__(NTHREADS, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using L = Layout<D, NS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + L::BAR_OFF + 8u * i; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::MISC_OFF);
  volatile int *abort = reinterpret_cast<volatile int *>(smem + L::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = blockIdx.x;
  const int qt = p.sched[item / p.hq];
  const int h = item % p.hq;
  const int g = h / (p.hq / p.hk);
  const int e0 = p.row_ptr[qt];
  const int n = p.row_ptr[qt + 1] - e0;
  const uint64_t deadline = globaltimer_ns() + p.wait_ns;
  const uint32_t q_smem = sb + L::Q_OFF, kv_smem = sb + L::KV_OFF;

  if (threadIdx.x == 0) {
    mbar_init(bar(L::B_Q), 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(L::B_FULL + s), 1);
      mbar_init(bar(L::B_EMPTY + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(L::B_S + t), 1);
      mbar_init(bar(L::B_P + t), 128);
      mbar_init(bar(L::B_O + t), 1);
    }
    mbar_init(bar(L::B_DRAIN), 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n > 0) {
      mbar_arrive_expect_tx(bar(L::B_Q), 2 * L::TILE);
      for (int t = 0; t < 2; ++t)
        for (int hh = 0; hh < L::NHALF; ++hh)
          tma_load_2d(q_smem + t * L::TILE + hh * L::HALF, &tm_q, bar(L::B_Q), h * D + hh * 64,
                      qt * 256 + t * BM);
      int issued = 0;
      for (int i = 0; i < 2 * n; ++i) {
        const int slot = i % NS;
        const uint32_t use = i / NS;
        if (use > 0 && !mbar_wait_bounded(bar(L::B_EMPTY + slot), (use - 1) & 1, abort, deadline))
          break;
        const int kt = p.col_idx[e0 + (i >> 1)];
        const CUtensorMap *tm = (i & 1) ? &tm_v : &tm_k;
        mbar_arrive_expect_tx(bar(L::B_FULL + slot), L::TILE);
        for (int hh = 0; hh < L::NHALF; ++hh)
          tma_load_2d(kv_smem + slot * L::TILE + hh * L::HALF, tm, bar(L::B_FULL + slot),
                      g * D + hh * 64, kt * BN);
        issued = i + 1;
      }
      if (*abort) {
        // let the loads already in flight land before the CTA retires
        wait_drain(bar(L::B_Q), 0, 20000000ull);
        for (int i = (issued > NS ? issued - NS : 0); i < issued; ++i)
          wait_drain(bar(L::B_FULL + i % NS), (i / NS) & 1, 20000000ull);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n > 0) {
      constexpr uint32_t IDESC_QK = idesc_bf16_f32(BM, BN, 0);
      constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, D, 1);
      auto issue_qk = [&](int t, int slot) {
        const uint32_t d_tmem = tmem + t * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::HALF + (kk & 3) * 32;
          mma_ss(d_tmem, smem_desc_sw128(q_smem + t * L::TILE + off, 16, 1024),
                 smem_desc_sw128(kv_smem + slot * L::TILE + off, 16, 1024), IDESC_QK, kk > 0);
        }
      };
      auto issue_pv = [&](int t, int slot, bool first) {
        const uint32_t d_tmem = tmem + 256 + t * 128;
        const uint32_t a_tmem = tmem + t * 128;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts(d_tmem, a_tmem + kk * 8,
                 smem_desc_sw128(kv_smem + slot * L::TILE + kk * 16 * 128, L::HALF, 1024), IDESC_PV,
                 (first && kk == 0) ? 0u : 1u);
      };
      bool ok = mbar_wait_bounded(bar(L::B_Q), 0, abort, deadline);
      if (ok) ok = mbar_wait_bounded(bar(L::B_FULL + 0), 0, abort, deadline);
      if (ok) {
        tc_fence_after();
        issue_qk(0, 0);
        mma_commit(bar(L::B_S + 0));
        issue_qk(1, 0);
        mma_commit(bar(L::B_S + 1));
        mma_commit(bar(L::B_EMPTY + 0));
      }
      for (int j = 0; ok && j < n; ++j) {
        const int iv = 2 * j + 1, ik = 2 * j + 2;
        const int sv = iv % NS, sk = ik % NS;
        if (!mbar_wait_bounded(bar(L::B_FULL + sv), (iv / NS) & 1, abort, deadline)) break;
        if (!mbar_wait_bounded(bar(L::B_P + 0), j & 1, abort, deadline)) break;
        tc_fence_after();
        issue_pv(0, sv, j == 0);
        if (j == n - 1) mma_commit(bar(L::B_O + 0));
        const bool more = j + 1 < n;
        if (more) {
          if (!mbar_wait_bounded(bar(L::B_FULL + sk), (ik / NS) & 1, abort, deadline)) break;
          tc_fence_after();
          issue_qk(0, sk);
          mma_commit(bar(L::B_S + 0));
        }
        if (!mbar_wait_bounded(bar(L::B_P + 1), j & 1, abort, deadline)) break;
        tc_fence_after();
        issue_pv(1, sv, j == 0);
        mma_commit(bar(L::B_EMPTY + sv));
        if (j == n - 1) mma_commit(bar(L::B_O + 1));
        if (more) {
          issue_qk(1, sk);
          mma_commit(bar(L::B_S + 1));
          mma_commit(bar(L::B_EMPTY + sk));
        }
      }
      // every MMA this thread issued completes before tensor memory is freed
      mma_commit(bar(L::B_DRAIN));
      wait_drain(bar(L::B_DRAIN), 0, 20000000ull);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2, wl = warp & 3;
    const int row = qt * 256 + t * BM + wl * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wl * 32) << 16;
    const uint32_t tS = tmem + lane_off + t * 128;
    const uint32_t tO = tmem + lane_off + 256 + t * 128;
    const float sl2 = p.scale_log2;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int e = e0 + j;
      const int kt = __ldg(p.col_idx + e);
      const int kd = __ldg(p.kind + e);
      if (!wait_all(bar(L::B_S + t), j & 1, abort, deadline)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld32_wait(tS + c * 32, r);
#pragma unroll
        for (int k = 0; k < 32; ++k) s[c * 32 + k] = __uint_as_float(r[k]);
      }
      if (kd == 2) {
        // MASKED tile: union of the referenced slices' row intervals as a
        // 128-bit mask, then a predicated select per element.
        uint32_t w[BN / 32] = {0u, 0u, 0u, 0u};
        const int r0 = __ldg(p.ref_ptr + e), r1 = __ldg(p.ref_ptr + e + 1);
        const int c0 = kt * BN;
        for (int r = r0; r < r1; ++r) {
          const attn_slice_t sl = p.slices[__ldg(p.ref_idx + r)];
          int lo, hi;
          slice_interval(sl, row, lo, hi);
          lo = min(max(lo - c0, 0), BN);
          hi = min(max(hi - c0, 0), BN);
          if (hi <= lo) continue;
#pragma unroll
          for (int c = 0; c < BN / 32; ++c) {
            const int a = min(max(lo - 32 * c, 0), 32), b = min(max(hi - 32 * c, 0), 32);
            w[c] |= bits_below(b) & ~bits_below(a);
          }
        }
#pragma unroll
        for (int k = 0; k < BN; ++k)
          if (!((w[k >> 5] >> (k & 31)) & 1u)) s[k] = -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int k = 1; k < BN; ++k) mx = fmaxf(mx, s[k]);
      const float mx2 = mx * sl2;
      const float m_old = m_ref;
      const bool grow = mx2 > m_ref + TAU;
      if (grow) m_ref = mx2;
      const float factor = grow ? ex2_approx(m_old - m_ref) : 1.f;
      l *= factor;
      const float mb = (m_ref == -INFINITY) ? 0.f : m_ref;
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float p0 = ex2_approx(fmaf(s[c * 32 + 2 * k], sl2, -mb));
          const float p1 = ex2_approx(fmaf(s[c * 32 + 2 * k + 1], sl2, -mb));
          l += p0 + p1;
          pk[k] = pack_bf16x2(p0, p1);
        }
        tmem_st16(tS + c * 16, pk);
      }
      const bool rescale = grow && (m_old != -INFINITY) && j > 0;
      if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32_wait(tO + c * 32, r);
#pragma unroll
          for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * factor);
          tmem_st32(tO + c * 32, r);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(L::B_P + t));
    }
    // ------------------------------------------------------------ epilogue
    if (n > 0 && ok) ok = wait_all(bar(L::B_O + t), 0, abort, deadline);
    if (ok) {
      tc_fence_after();
      const bool live = row < p.sq;
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        if (n > 0) {
          tmem_ld32_wait(tO + c * 32, r);
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) r[k] = 0u;
        }
        if (!live) continue;
        const size_t base = (static_cast<size_t>(row) * p.hq + h) * D + c * 32;
        if (p.out_f32) {
          float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + base);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            dst[k] = make_float4(__uint_as_float(r[4 * k]) * inv, __uint_as_float(r[4 * k + 1]) * inv,
                                 __uint_as_float(r[4 * k + 2]) * inv,
                                 __uint_as_float(r[4 * k + 3]) * inv);
        } else {
          uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.out) + base);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(r[8 * k + 0]) * inv, __uint_as_float(r[8 * k + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(r[8 * k + 2]) * inv, __uint_as_float(r[8 * k + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(r[8 * k + 4]) * inv, __uint_as_float(r[8 * k + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(r[8 * k + 6]) * inv, __uint_as_float(r[8 * k + 7]) * inv);
            dst[k] = v;
          }
        }
      }
      if (live)
        p.lse[static_cast<size_t>(h) * p.sq + row] =
            l > 0.f ? (m_ref + __log2f(l)) * 0.69314718055994531f : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tmem, 512);
  if (threadIdx.x == 0 && *abort) atomicExch(&g_fwd_status, static_cast<unsigned>(ATTN_ERR_TIMEOUT));
}

// ------------------------------------------------------------------ host side

static PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
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

// 2-D bf16 map over a [rows, cols] row-major matrix, 64 x 128 boxes with
// the 128-byte swizzle the MMA descriptors expect.
static int make_map(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows) {
  auto enc = get_encode_fn();
  if (!enc) return ATTN_ERR_CUDA;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

static unsigned long long g_wait_ns = 4000000000ull;

template <int D, int NS>
static int launch_fwd(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                      const FwdParams &p, int grid, cudaStream_t s) {
  using L = Layout<D, NS>;
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(fwd_kernel<D, NS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::ALLOC) != cudaSuccess)
      return ATTN_ERR_CUDA;
    configured = true;
  }
  fwd_kernel<D, NS><<<grid, NTHREADS, L::ALLOC, s>>>(mq, mk, mv, p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int fwd_launch(const void *q, const void *k, const void *v, int sq, int sk, int hq, int hk, int d,
               float scale, const attn_tiles_t *tiles, void *out, int out_dtype, float *lse,
               cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  int rc;
  if ((rc = make_map(&mq, q, static_cast<uint64_t>(hq) * d, sq)) != ATTN_OK) return rc;
  if ((rc = make_map(&mk, k, static_cast<uint64_t>(hk) * d, sk)) != ATTN_OK) return rc;
  if ((rc = make_map(&mv, v, static_cast<uint64_t>(hk) * d, sk)) != ATTN_OK) return rc;
  FwdParams p;
  p.row_ptr = tiles->row_ptr;
  p.col_idx = tiles->col_idx;
  p.ref_ptr = tiles->ref_ptr;
  p.ref_idx = tiles->ref_idx;
  p.sched = tiles->sched;
  p.kind = tiles->kind;
  p.slices = tiles->slices;
  p.out = out;
  p.lse = lse;
  p.sq = sq;
  p.sk = sk;
  p.hq = hq;
  p.hk = hk;
  p.out_f32 = out_dtype == ATTN_DTYPE_F32;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.wait_ns = g_wait_ns;
  const int grid = tiles->n_qtiles * hq;
  if (grid == 0) return ATTN_OK;
  if (d == 128) return launch_fwd<128, 4>(mq, mk, mv, p, grid, stream);
  return launch_fwd<64, 8>(mq, mk, mv, p, grid, stream);
}

int fwd_status_take(unsigned int *status) {
  unsigned int zero = 0;
  if (cudaMemcpyFromSymbol(status, g_fwd_status, sizeof(unsigned int)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (*status && cudaMemcpyToSymbol(g_fwd_status, &zero, sizeof(unsigned int)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

void fwd_set_wait_ns(unsigned long long ns) { g_wait_ns = ns; }

// One thread waits on a barrier that nothing will complete; the bounded wait
// gives up after the configured limit and records a timeout.
__global__ void selftest_timeout_kernel(unsigned long long wait_ns) {
  __shared__ __align__(8) uint64_t b;
  __shared__ int abort_flag;
  const uint32_t a = smem_u32(&b);
  mbar_init(a, 1);
  abort_flag = 0;
  fence_mbar_init();
  const uint64_t dl = globaltimer_ns() + wait_ns;
  if (!mbar_wait_bounded(a, 0, reinterpret_cast<volatile int *>(&abort_flag), dl))
    atomicExch(&g_fwd_status, static_cast<unsigned>(ATTN_ERR_TIMEOUT));
}

int selftest_timeout_launch(cudaStream_t s) {
  selftest_timeout_kernel<<<1, 1, 0, s>>>(g_wait_ns);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn
