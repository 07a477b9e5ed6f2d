// Backward pass of masked attention on sm_103a: dQ, dK, dV from Q, K, V, the
// forward output O and its LSE, and the output gradient dO, for the same
// slice masks and tile metadata as the forward.
//
// With P = softmax(scale Q K^T + mask) recomputed from the saved LSE:
//   D   = rowsum(dO * O)                       (bwd_delta_kernel)
//   dP  = dO V^T,  dS = P * (dP - D)
//   dV  = P^T dO,  dK = scale dS^T Q            (bwd_kv_kernel, per key tile)
//   dQ  = scale dS K                            (bwd_q_kernel, per query tile)
// The key-tile kernel walks a transposed copy of the CSR tile lists (per
// key tile: the query tiles that have it, ascending), built deterministically
// by csc_count_kernel / csc_fill_kernel; dK and dV of a key tile accumulate
// in tensor memory over every query tile and every query head of its GQA
// group, so each is written once.  dQ is computed by a second walk of the
// forward's per-query-tile lists, so no kernel needs atomics.
//
// All MMAs have the forward's two forms: S^T = K Q^T and dP^T = V dO^T (both
// operands K-major in shared memory), dV += P^T dO and dK += dS^T Q (A read
// from tensor memory, B MN-major in shared memory); likewise S = Q K^T,
// dP = dO V^T and dQ += dS K in the query-tile kernel.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "attn_device.cuh"
#include "attn_internal.h"

namespace attn {

// First failure status of backward launches on this device (0 = none): a
// bounded wait that ran out, or metadata whose build did not finish with
// ATTN_OK.  Read and cleared by attn_last_device_error().
__device__ unsigned int g_bwd_status;

constexpr int Q_THREADS = 192;     // dQ kernel: warps 0-3 element-wise, 4 producer, 5 MMA issuer
constexpr int KV_THREADS = 320;    // dK/dV kernel: warps 0-7 element-wise, 8 producer, 9 MMA issuer
constexpr int B_TILE_Q = 256;      // query rows per tile of the metadata
constexpr float LOG2E = 1.4426950408889634f;

struct BwdParams {
  const int32_t *row_ptr, *col_idx, *ref_ptr, *ref_idx, *sched;
  const uint8_t *kind;
  const attn_slice_t *slices;
  const int32_t *col_ptr, *col_q, *col_e, *col_sched;
  const float *lse, *delta;
  void *dq, *dk, *dv;
  int sq, sk, hq, hk, n_qtiles, n_ktiles;
  int grad_f32;
  float scale, scale_log2;
  unsigned long long wait_ns;
  const long long *meta_status;   // the metadata build's status word (totals[3])
};

// True when the metadata's build did not finish with ATTN_OK: the kernel
// then reads none of it and returns at once (uniformly for the whole CTA,
// before any barrier or tensor memory is set up); the first CTA records the
// status.
__device__ __forceinline__ bool meta_refused(const BwdParams &p) {
  const long long st = *p.meta_status;
  if (st == ATTN_OK) return false;
  if (blockIdx.x == 0 && threadIdx.x == 0) atomicCAS(&g_bwd_status, 0u, static_cast<unsigned>(st));
  return true;
}

// ------------------------------------------------------------------ D = rowsum(dO * O)
// One thread per 8 consecutive elements (one 16-byte load of dO, one or two
// of O; rows are 16-byte aligned), D / 8 neighbouring lanes per row, summed
// by shuffles within those lanes.
template <int D, bool O_F32>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const void *out, const uint16_t *dout,
                                                         float *delta, int sq, int hq) {
  constexpr int TPR = D / 8;   // threads per row
  static_assert(32 % TPR == 0, "a row's lanes share one warp");
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long r = t / TPR;   // row (i, h) at i * hq + h
  const bool valid = r < static_cast<long long>(sq) * hq;
  float acc = 0.f;
  if (valid) {
    const size_t base = static_cast<size_t>(t) * 8;
    const uint4 g = *reinterpret_cast<const uint4 *>(dout + base);
    const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
    float o[8];
    if (O_F32) {
      const float4 a = *reinterpret_cast<const float4 *>(static_cast<const float *>(out) + base);
      const float4 b = *reinterpret_cast<const float4 *>(static_cast<const float *>(out) + base + 4);
      o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
      o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
    } else {
      const uint4 ov = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(out) + base);
      const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        o[2 * k] = __uint_as_float(ow[k] << 16);
        o[2 * k + 1] = __uint_as_float(ow[k] & 0xffff0000u);
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      acc = fmaf(__uint_as_float(gw[k] << 16), o[2 * k], acc);
      acc = fmaf(__uint_as_float(gw[k] & 0xffff0000u), o[2 * k + 1], acc);
    }
  }
#pragma unroll
  for (int m = TPR / 2; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
  if (valid && (t % TPR) == 0) {
    const int i = static_cast<int>(r / hq), h = static_cast<int>(r % hq);
    delta[static_cast<size_t>(h) * sq + i] = acc;
  }
}

// ------------------------------------------------------------------ transposed lists
// Position of key tile kt in query tile qt's sorted list, or -1.
__device__ __forceinline__ int find_entry(const BwdParams &p, int qt, int kt) {
  int lo = p.row_ptr[qt], hi = p.row_ptr[qt + 1];
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    const int c = p.col_idx[mid];
    if (c == kt) return mid;
    if (c < kt) lo = mid + 1; else hi = mid;
  }
  return -1;
}

__device__ long long block_sum_ll(long long v, long long *red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  long long t = 0;
  for (int u = 0; u < static_cast<int>(blockDim.x >> 5); ++u) t += red[u];
  return t;
}

__global__ void __launch_bounds__(256) csc_count_kernel(BwdParams p, int32_t *colcnt) {
  if (meta_refused(p)) return;
  __shared__ long long red[8];
  const int kt = blockIdx.x;
  long long c = 0;
  for (int qt = threadIdx.x; qt < p.n_qtiles; qt += blockDim.x) c += find_entry(p, qt, kt) >= 0;
  c = block_sum_ll(c, red);
  if (threadIdx.x == 0) colcnt[kt] = static_cast<int32_t>(c);
}

__global__ void __launch_bounds__(256) csc_fill_kernel(BwdParams p, const int32_t *colcnt,
                                                       int32_t *col_ptr, int32_t *col_q,
                                                       int32_t *col_e, int32_t *col_sched) {
  if (meta_refused(p)) return;
  __shared__ long long red[8];
  __shared__ int scan[256];
  const int kt = blockIdx.x, me = colcnt[kt];
  long long before = 0, all = 0, rank = 0;
  for (int u = threadIdx.x; u < p.n_ktiles; u += blockDim.x) {
    const int cu = colcnt[u];
    if (u < kt) before += cu;
    all += cu;
    rank += (cu > me || (cu == me && u < kt)) ? 1 : 0;
  }
  before = block_sum_ll(before, red);
  all = block_sum_ll(all, red);
  rank = block_sum_ll(rank, red);
  if (threadIdx.x == 0) {
    col_ptr[kt] = static_cast<int32_t>(before);
    col_sched[rank] = kt;
    if (kt == 0) col_ptr[p.n_ktiles] = static_cast<int32_t>(all);
  }
  // ascending query tiles, 256 at a time
  int out = static_cast<int>(before);
  for (int base = 0; base < p.n_qtiles; base += blockDim.x) {
    const int qt = base + threadIdx.x;
    const int e = qt < p.n_qtiles ? find_entry(p, qt, kt) : -1;
    scan[threadIdx.x] = e >= 0;
    __syncthreads();
    for (int o = 1; o < static_cast<int>(blockDim.x); o <<= 1) {
      const int v = threadIdx.x >= static_cast<unsigned>(o) ? scan[threadIdx.x - o] : 0;
      __syncthreads();
      scan[threadIdx.x] += v;
      __syncthreads();
    }
    if (e >= 0) {
      const int pos = out + scan[threadIdx.x] - 1;
      col_q[pos] = qt;
      col_e[pos] = e;
    }
    out += scan[blockDim.x - 1];
    __syncthreads();
  }
}

// ------------------------------------------------------------------ shared pieces
template <int D>
struct BLayout {
  static constexpr int HALF = 128 * 64 * 2;
  static constexpr int NHALF = D / 64;
  static constexpr int TILE = NHALF * HALF;
};

template <int D>
__device__ __forceinline__ void store_rows(void *base_ptr, bool f32, size_t off, const uint32_t (&r)[32],
                                           float mul) {
  if (f32) {
    float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(base_ptr) + off);
#pragma unroll
    for (int k = 0; k < 8; ++k)
      dst[k] = make_float4(__uint_as_float(r[4 * k]) * mul, __uint_as_float(r[4 * k + 1]) * mul,
                           __uint_as_float(r[4 * k + 2]) * mul, __uint_as_float(r[4 * k + 3]) * mul);
  } else {
    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(base_ptr) + off);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint4 v;
      v.x = pack_bf16x2(__uint_as_float(r[8 * k + 0]) * mul, __uint_as_float(r[8 * k + 1]) * mul);
      v.y = pack_bf16x2(__uint_as_float(r[8 * k + 2]) * mul, __uint_as_float(r[8 * k + 3]) * mul);
      v.z = pack_bf16x2(__uint_as_float(r[8 * k + 4]) * mul, __uint_as_float(r[8 * k + 5]) * mul);
      v.w = pack_bf16x2(__uint_as_float(r[8 * k + 6]) * mul, __uint_as_float(r[8 * k + 7]) * mul);
      dst[k] = v;
    }
  }
}

// ------------------------------------------------------------------ dK, dV per key tile
// Work item: (key tile kt, KV head g).  Steps: every query tile of kt's
// column, every query head of group g, both 128-row halves.  Tensor memory:
// S^T [0,128)  dP^T [128,256)  dV [256,256+D)  dK [384,384+D); P^T and dS^T
// (bf16) overwrite the first 64 columns of S^T and dP^T.
//
// The step is pipelined across two element-wise phases with their own
// arrivals: phase P (P^T from S^T) and phase dS (dS^T from dP^T and P, kept
// in registers).  The MMA lane issues, for step s,
//   [P(s-1) arrived]  dV += P^T(s-1) dO(s-1),  S^T(s) = K Q(s)^T
//   [dS(s-1) arrived] dK += dS^T(s-1) Q(s-1),  dP^T(s) = V dO(s)^T
// so the tensor core computes dV and the next S^T while the element-wise
// warps form dS, and dK and the next dP^T while they form the next P.  Each
// new S^T (dP^T) overwrites columns the MMA issued just before it reads;
// tcgen05 MMAs of one thread execute in issue order, and the element-wise
// warps have read the old values before their arrival.  Q and dO stream
// through two stages each, freed separately (dO after dV, Q after dK).
template <int D>
struct KVLayout {
  using B = BLayout<D>;
  static constexpr int K_OFF = 0, V_OFF = B::TILE;
  static constexpr int Q_OFF = 2 * B::TILE, DO_OFF = 4 * B::TILE;            // 2 stages each
  static constexpr int VEC_OFF = 6 * B::TILE;                                 // [2][lse2 128 | D 128]
  static constexpr int BAR_OFF = VEC_OFF + 2 * 256 * 4;
  // kv | q_full[2] | q_empty[2] | do_full[2] | do_empty[2] | s_ready | dp_ready |
  // p_done | ds_done | o_full | drain | vec
  static constexpr int B_KV = 0, B_QF = 1, B_QE = 3, B_DF = 5, B_DE = 7, B_SR = 9, B_DPR = 10,
                       B_PA = 11, B_DS = 12, B_O = 13, B_DR = 14, B_VEC = 15, NBAR = 16;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int ALLOC = MISC_OFF + 16 + 1024;
  static_assert(ALLOC <= 232448, "shared memory per CTA");
};

template <int D>
__global__ void __launch_bounds__(KV_THREADS, 1)
    bwd_kv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const BwdParams p) {
  if (meta_refused(p)) return;
  using L = KVLayout<D>;
  using BL = BLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + L::BAR_OFF + 8u * i; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::MISC_OFF);
  volatile int *abort = reinterpret_cast<volatile int *>(smem + L::MISC_OFF + 4);
  float *vec = reinterpret_cast<float *>(smem + L::VEC_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t lim = p.wait_ns;

  const int kt = p.col_sched[blockIdx.x / p.hk];
  const int g = blockIdx.x % p.hk;
  const int G = p.hq / p.hk;
  const int c0 = p.col_ptr[kt], nc = p.col_ptr[kt + 1] - c0;

  if (threadIdx.x == 0) {
    mbar_init(bar(L::B_KV), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::B_QF + s), 1);
      mbar_init(bar(L::B_QE + s), 1);
      mbar_init(bar(L::B_DF + s), 1);
      mbar_init(bar(L::B_DE + s), 1);
    }
    mbar_init(bar(L::B_SR), 1);
    mbar_init(bar(L::B_DPR), 1);
    mbar_init(bar(L::B_PA), 256);
    mbar_init(bar(L::B_DS), 256);
    mbar_init(bar(L::B_O), 1);
    mbar_init(bar(L::B_DR), 1);
    mbar_init(bar(L::B_VEC), 256);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the steps of this item: (column entry c, head offset gh, half t) with
  // the half inside the query sequence, in this order
  // (the first half of a query tile always lies inside S_q: only the second
  // one needs the tile's index)
  auto half_ok = [&](int c, int t) { return t == 0 || p.col_q[c0 + c] * B_TILE_Q + 128 < p.sq; };
  // moves (c, gh, t) to the next step; false past the last one
  auto advance = [&](int &c, int &gh, int &t) -> bool {
    do {
      if (++t == 2) {
        t = 0;
        if (++gh == G) {
          gh = 0;
          ++c;
        }
      }
      if (c >= nc) return false;
    } while (!half_ok(c, t));
    return true;
  };

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && nc > 0) {
      mbar_arrive_expect_tx(bar(L::B_KV), 2 * BL::TILE);
      for (int hh = 0; hh < BL::NHALF; ++hh) {
        tma_load_2d(sb + L::K_OFF + hh * BL::HALF, &tm_k, bar(L::B_KV), g * D + hh * 64, kt * 128);
        tma_load_2d(sb + L::V_OFF + hh * BL::HALF, &tm_v, bar(L::B_KV), g * D + hh * 64, kt * 128);
      }
      uint32_t s = 0;
      bool ok = true;
      int c = 0, gh = 0, t = -1;
      while (ok && advance(c, gh, t)) {
        const int st = s & 1;
        const int h = g * G + gh, q0 = p.col_q[c0 + c] * B_TILE_Q + t * 128;
        // Q(s) once dK(s-2) has read stage st, dO(s) once dV(s-2) has
        if (s >= 2 && !mbar_wait_bounded(bar(L::B_QE + st), ((s >> 1) - 1) & 1, abort, lim)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(L::B_QF + st), BL::TILE);
        for (int hh = 0; hh < BL::NHALF; ++hh)
          tma_load_2d(sb + L::Q_OFF + st * BL::TILE + hh * BL::HALF, &tm_q, bar(L::B_QF + st),
                      h * D + hh * 64, q0);
        if (s >= 2 && !mbar_wait_bounded(bar(L::B_DE + st), ((s >> 1) - 1) & 1, abort, lim)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(L::B_DF + st), BL::TILE);
        for (int hh = 0; hh < BL::NHALF; ++hh)
          tma_load_2d(sb + L::DO_OFF + st * BL::TILE + hh * BL::HALF, &tm_do, bar(L::B_DF + st),
                      h * D + hh * 64, q0);
        ++s;
      }
      if (*abort) {
        // let the loads already in flight land before the CTA retires
        wait_drain(bar(L::B_KV), 0, 20000000ull);
        for (uint32_t i = (s > 2 ? s - 2 : 0); i < s; ++i) {
          wait_drain(bar(L::B_QF + (i & 1)), (i >> 1) & 1, 20000000ull);
          wait_drain(bar(L::B_DF + (i & 1)), (i >> 1) & 1, 20000000ull);
        }
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nc > 0) {
      constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 128, 0);
      constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, D, 1);
      const uint32_t ks = sb + L::K_OFF, vs = sb + L::V_OFF;
      auto qst = [&](uint32_t s) { return sb + L::Q_OFF + (s & 1) * BL::TILE; };
      auto dost = [&](uint32_t s) { return sb + L::DO_OFF + (s & 1) * BL::TILE; };
      // dV += P^T(s) dO(s), then dO's stage is free
      auto issue_dv = [&](uint32_t s) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + 256, tmem + (kk >> 2) * 64 + (kk & 3) * 8,
                 smem_desc_sw128(dost(s) + kk * 16 * 128, BL::HALF, 1024),
                 IDESC_PV, (s > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(L::B_DE + (s & 1)));
      };
      // dK += dS^T(s) Q(s), then Q's stage is free
      auto issue_dk = [&](uint32_t s) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + 384, tmem + 128 + (kk >> 2) * 64 + (kk & 3) * 8,
                 smem_desc_sw128(qst(s) + kk * 16 * 128, BL::HALF, 1024),
                 IDESC_PV, (s > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(L::B_QE + (s & 1)));
      };
      bool ok = mbar_wait_bounded(bar(L::B_KV), 0, abort, lim);
      // The issuer needs only the number of steps: every column entry has
      // both halves for each of the G heads, except that the last query tile
      // (the column's last entry, if it has it) may lack its second half.
      const int last_q = (p.sq - 1) / B_TILE_Q;
      const bool short_last = p.col_q[c0 + nc - 1] == last_q && !half_ok(nc - 1, 1);
      const uint32_t nsteps = static_cast<uint32_t>(nc * 2 * G - (short_last ? G : 0));
      uint32_t s = 0;
      for (; ok && s < nsteps;) {
        // each group's dependency is tested (blocking) together with a
        // non-blocking look at the next group's: their latencies overlap,
        // and the next wait is skipped when the look found it complete
        bool have_q = false, have_do = false;
        if (s > 0) {
          const bool have_p = mbar_try_wait(bar(L::B_PA), (s - 1) & 1);
          have_q = mbar_test_wait(bar(L::B_QF + (s & 1)), (s >> 1) & 1);
          if (!have_p && !mbar_wait_bounded(bar(L::B_PA), (s - 1) & 1, abort, lim)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_dv(s - 1);
        }
        if (!have_q && !mbar_wait_bounded(bar(L::B_QF + (s & 1)), (s >> 1) & 1, abort, lim)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // S^T(s) = K Q(s)^T
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * BL::HALF + (kk & 3) * 32;
          mma_ss(tmem, smem_desc_sw128(ks + off, 16, 1024), smem_desc_sw128(qst(s) + off, 16, 1024),
                 IDESC_QK, kk > 0);
        }
        mma_commit(bar(L::B_SR));
        if (s > 0) {
          const bool have_ds = mbar_try_wait(bar(L::B_DS), (s - 1) & 1);
          have_do = mbar_test_wait(bar(L::B_DF + (s & 1)), (s >> 1) & 1);
          if (!have_ds && !mbar_wait_bounded(bar(L::B_DS), (s - 1) & 1, abort, lim)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_dk(s - 1);
        }
        if (!have_do && !mbar_wait_bounded(bar(L::B_DF + (s & 1)), (s >> 1) & 1, abort, lim)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // dP^T(s) = V dO(s)^T
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * BL::HALF + (kk & 3) * 32;
          mma_ss(tmem + 128, smem_desc_sw128(vs + off, 16, 1024), smem_desc_sw128(dost(s) + off, 16, 1024),
                 IDESC_QK, kk > 0);
        }
        mma_commit(bar(L::B_DPR));
        ++s;
      }
      if (ok && s > 0) {
        // the last step's dV and dK
        ok = mbar_wait_bounded(bar(L::B_PA), (s - 1) & 1, abort, lim);
        if (ok) {
          tc_fence_after();
          issue_dv(s - 1);
          ok = mbar_wait_bounded(bar(L::B_DS), (s - 1) & 1, abort, lim);
        }
        if (ok) {
          tc_fence_after();
          issue_dk(s - 1);
          mma_commit(bar(L::B_O));
        }
      }
      // every MMA this thread issued completes before tensor memory is freed
      mma_commit(bar(L::B_DR));
      wait_drain(bar(L::B_DR), 0, 20000000ull);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ element-wise (thread = key row)
    // warps 0-3 and 4-7 take the same 128 key rows (tensor-memory lanes
    // 32 (warp % 4) ...), columns (queries) [64 hc, 64 hc + 64) each
    const int r = (warp & 3) * 32 + lane, hc = warp >> 2;
    const int key = kt * 128 + r;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + lane_off + hc * 64, t_dp = t_s + 128;
    const float sl2 = p.scale_log2;
    uint32_t s = 0;
    bool ok = true, any = false;
    // statistics of query row q0 + r of a step (warps 0-3 stage all 128):
    // log2-domain lse (+inf past S_q, so that P = 0 there) and D
    auto load_stats = [&](int c, int gh, int t, float &lv, float &dv) {
      const int h = g * G + gh, i = p.col_q[c0 + c] * B_TILE_Q + t * 128 + r;
      const float l = i < p.sq ? p.lse[static_cast<size_t>(h) * p.sq + i] : -INFINITY;
      lv = l == -INFINITY ? INFINITY : l * LOG2E;
      dv = i < p.sq ? p.delta[static_cast<size_t>(h) * p.sq + i] : 0.f;
    };
    int c = 0, gh = 0, t = -1;
    bool have = advance(c, gh, t);
    float lv = 0.f, dv = 0.f;
    if (have && hc == 0) load_stats(c, gh, t, lv, dv);
    while (ok && have) {
      const int q0 = p.col_q[c0 + c] * B_TILE_Q + t * 128, e = p.col_e[c0 + c];
      const float *vl = vec + (s & 1) * 256 + hc * 64, *vd = vl + 128;
      // the statistics of this step are staged (the buffer of step s - 2 is
      // free: every element-wise thread got past step s - 1's barrier, after
      // its last reads of it)
      if (hc == 0) {
        vec[(s & 1) * 256 + r] = lv;
        vec[(s & 1) * 256 + 128 + r] = dv;
      }
      mbar_arrive(bar(L::B_VEC));
      if (!wait_all(bar(L::B_VEC), s & 1, abort, lim)) {
        ok = false;
        break;
      }
      uint32_t w[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
      if (p.kind[e] == ATTN_TILE_MASKED) {
        w[0] = w[1] = w[2] = w[3] = 0u;
        const int r0 = p.ref_ptr[e], r1 = p.ref_ptr[e + 1];
        for (int q = r0; q < r1; ++q) add_col_mask(p.slices[p.ref_idx[q]], key, q0, w);
      }
      const uint32_t wm[2] = {hc ? w[2] : w[0], hc ? w[3] : w[1]};
      // ---- phase P: P = exp2(S scale log2e - lse2) on the valid columns,
      // kept in f32 for phase dS; P^T (bf16) over the first 32 of this
      // warp's 64 S^T columns
      if (!wait_all(bar(L::B_SR), s & 1, abort, lim)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float P[64];
      {
        uint32_t x[64];
        tmem_ld32(t_s, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
        tmem_ld32(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(&x[32]));
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 64; ++k) {
          asm volatile("" : "+r"(x[k]));
          P[k] = __uint_as_float(x[k]);
        }
      }
      {
        uint32_t pk[32];
#pragma unroll
        for (int k = 0; k < 64; ++k) {
          const bool okc = (wm[k >> 5] >> (k & 31)) & 1u;
          const float ev = ex2_approx(fmaf(P[k], sl2, -vl[k]));
          P[k] = okc ? ev : 0.f;
        }
#pragma unroll
        for (int k = 0; k < 32; ++k) pk[k] = pack_bf16x2(P[2 * k], P[2 * k + 1]);
        tmem_st16(t_s, *reinterpret_cast<const uint32_t(*)[16]>(&pk[0]));
        tmem_st16(t_s + 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16]));
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(L::B_PA));
      // the next step's statistics load while phase dS runs
      int c2 = c, gh2 = gh, t2 = t;
      const bool have2 = advance(c2, gh2, t2);
      if (have2 && hc == 0) load_stats(c2, gh2, t2, lv, dv);
      // ---- phase dS: dS = P (dP - D); dS^T (bf16) over the first 32 of this
      // warp's 64 dP^T columns
      if (!wait_all(bar(L::B_DPR), s & 1, abort, lim)) {
        ok = false;
        break;
      }
      tc_fence_after();
      {
        uint32_t y[64];
        tmem_ld32(t_dp, *reinterpret_cast<uint32_t(*)[32]>(&y[0]));
        tmem_ld32(t_dp + 32, *reinterpret_cast<uint32_t(*)[32]>(&y[32]));
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 64; ++k) asm volatile("" : "+r"(y[k]));
        uint32_t dk[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float d0 = P[2 * k] * (__uint_as_float(y[2 * k]) - vd[2 * k]);
          const float d1 = P[2 * k + 1] * (__uint_as_float(y[2 * k + 1]) - vd[2 * k + 1]);
          dk[k] = pack_bf16x2(d0, d1);
        }
        tmem_st16(t_dp, *reinterpret_cast<const uint32_t(*)[16]>(&dk[0]));
        tmem_st16(t_dp + 16, *reinterpret_cast<const uint32_t(*)[16]>(&dk[16]));
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(L::B_DS));
      any = true;
      ++s;
      c = c2;
      gh = gh2;
      t = t2;
      have = have2;
    }
    // ---------------------------------------------------------- epilogue
    // columns [hc D / 2, hc D / 2 + D / 2) of this row's dV and dK
    bool have_o = ok && any;
    if (have_o) {
      have_o = wait_all(bar(L::B_O), 0, abort, lim);
      tc_fence_after();
    }
    if (ok) {
      // tensor-memory loads stay warp-uniform; only the stores depend on the row
      const size_t off = (static_cast<size_t>(key) * p.hk + g) * D;
      const uint32_t row_t = tmem + lane_off;
#pragma unroll 1
      for (int cc = hc * (D / 64); cc < (hc + 1) * (D / 64); ++cc) {
        uint32_t rv[32], rk[32];
        if (have_o) {
          tmem_ld32_wait(row_t + 256 + cc * 32, rv);
          tmem_ld32_wait(row_t + 384 + cc * 32, rk);
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) rv[k] = rk[k] = 0u;
        }
        if (key < p.sk) {
          store_rows<D>(p.dv, p.grad_f32, off + cc * 32, rv, 1.f);
          store_rows<D>(p.dk, p.grad_f32, off + cc * 32, rk, p.scale);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tmem, 512);
  if (threadIdx.x == 0 && *abort) atomicCAS(&g_bwd_status, 0u, static_cast<unsigned>(ATTN_ERR_TIMEOUT));
}

// ------------------------------------------------------------------ dQ per query tile
// Work item: (query tile, head) as in the forward; the two 128-row halves in
// turn.  Tensor memory: S_a [0,128)  dP [128,256)  dQ [256,256+D)
// S_b [384,512).  S of key tile j goes to S_a for even j, S_b for odd j, and
// dS (bf16) overwrites the first 64 columns of that S.  The element-wise
// warps read all of dP(j) first and say so (dp_read), so the tensor core
// computes dP(j+1) and S(j+2) while they form dS(j).  MMA order per key
// tile j: dP(j+1) after dp_read(j), dQ += dS(j) K_j after p_done(j), then
// S(j+2) into the S block dQ has just read.
template <int D, int NS>
struct QLayout {
  using B = BLayout<D>;
  static constexpr int Q_OFF = 0, DO_OFF = B::TILE, KV_OFF = 2 * B::TILE;
  static constexpr int BAR_OFF = KV_OFF + NS * B::TILE;
  // q_full | q_empty | full[NS] | empty[NS] | s_full | p_done | o_full | drain | dp_read
  static constexpr int B_Q = 0, B_QE = 1, B_FULL = 2, B_EMPTY = 2 + NS, B_S = 2 + 2 * NS,
                       B_P = B_S + 1, B_O = B_P + 1, B_DR = B_O + 1, B_DPR = B_DR + 1,
                       NBAR = B_DPR + 1;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int ALLOC = MISC_OFF + 16 + 1024;
  static_assert(ALLOC <= 232448, "shared memory per CTA");
};

// Column block of S(j) in the dQ kernel's tensor memory.
__device__ __forceinline__ uint32_t q_s_col(int j) { return (j & 1) ? 384u : 0u; }

// The dQ kernel's element-wise step for one query row: all 128 columns of dP
// into registers first (then dp_read), then S in 32-column chunks; dS =
// P (dP - D) with P = exp2(S scale log2e - lse2) goes back over the first 64
// columns of S as bf16 pairs.  Arithmetic on f32 pairs; only MASKED tiles
// pay for the per-element select by the mask bits w.
__device__ __forceinline__ void ds_step_dp_first(uint32_t t_s, uint32_t t_dp, bool masked, const uint32_t (&w)[4],
                                                 float sl2, float lse2, float dlt, uint32_t dp_read) {
  uint32_t y[128];
#pragma unroll
  for (int c = 0; c < 4; ++c) tmem_ld32(t_dp + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&y[c * 32]));
  tmem_wait_ld();
#pragma unroll
  for (int k = 0; k < 128; ++k) asm volatile("" : "+r"(y[k]));
  tc_fence_before();
  mbar_arrive(dp_read);
  const uint64_t sc2 = f2_make(sl2, sl2), nl2 = f2_make(-lse2, -lse2), nd2 = f2_make(-dlt, -dlt);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t x[32];
    tmem_ld32(t_s + c * 32, x);
    tmem_wait_ld();
#pragma unroll
    for (int k = 0; k < 32; ++k) asm volatile("" : "+r"(x[k]));
    uint32_t dk[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const int col = c * 32 + 2 * k;
      float a0, a1;
      f2_split(f2_fma(f2_make_u(x[2 * k], x[2 * k + 1]), sc2, nl2), a0, a1);
      float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
      if (masked) {
        if (!((w[c] >> (2 * k)) & 1u)) p0 = 0.f;
        if (!((w[c] >> (2 * k + 1)) & 1u)) p1 = 0.f;
      }
      float d0, d1;
      f2_split(f2_mul(f2_make(p0, p1), f2_add(f2_make_u(y[col], y[col + 1]), nd2)), d0, d1);
      dk[k] = pack_bf16x2(d0, d1);
    }
    tmem_st16(t_s + c * 16, dk);
  }
}

template <int D, int NS>
__global__ void __launch_bounds__(Q_THREADS, 1)
    bwd_q_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                 const BwdParams p) {
  if (meta_refused(p)) return;
  using L = QLayout<D, NS>;
  using BL = BLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + L::BAR_OFF + 8u * i; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::MISC_OFF);
  volatile int *abort = reinterpret_cast<volatile int *>(smem + L::MISC_OFF + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t lim = p.wait_ns;

  const int qt = p.sched[blockIdx.x / p.hq];
  const int h = blockIdx.x % p.hq;
  const int g = h / (p.hq / p.hk);
  const int e0 = p.row_ptr[qt], n = p.row_ptr[qt + 1] - e0;
  const int halves = (qt * B_TILE_Q + 128 < p.sq) ? 2 : 1;

  if (threadIdx.x == 0) {
    mbar_init(bar(L::B_Q), 1);
    mbar_init(bar(L::B_QE), 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(L::B_FULL + s), 1);
      mbar_init(bar(L::B_EMPTY + s), 1);
    }
    mbar_init(bar(L::B_S), 1);
    mbar_init(bar(L::B_P), 128);
    mbar_init(bar(L::B_O), 1);
    mbar_init(bar(L::B_DR), 1);
    mbar_init(bar(L::B_DPR), 128);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    if (lane == 0 && n > 0) {
      uint32_t ld = 0;
      bool ok = true;
      for (int t = 0; ok && t < halves; ++t) {
        if (t > 0 && !mbar_wait_bounded(bar(L::B_QE), (t - 1) & 1, abort, lim)) {
          ok = false;
          break;
        }
        const int q0 = qt * B_TILE_Q + t * 128;
        mbar_arrive_expect_tx(bar(L::B_Q), 2 * BL::TILE);
        for (int hh = 0; hh < BL::NHALF; ++hh) {
          tma_load_2d(sb + L::Q_OFF + hh * BL::HALF, &tm_q, bar(L::B_Q), h * D + hh * 64, q0);
          tma_load_2d(sb + L::DO_OFF + hh * BL::HALF, &tm_do, bar(L::B_Q), h * D + hh * 64, q0);
        }
        for (int i = 0; ok && i < 2 * n; ++i, ++ld) {
          const int slot = ld % NS;
          const uint32_t use = ld / NS;
          if (use > 0 && !mbar_wait_bounded(bar(L::B_EMPTY + slot), (use - 1) & 1, abort, lim)) {
            ok = false;
            break;
          }
          const int kt = p.col_idx[e0 + (i >> 1)];
          mbar_arrive_expect_tx(bar(L::B_FULL + slot), BL::TILE);
          for (int hh = 0; hh < BL::NHALF; ++hh)
            tma_load_2d(sb + L::KV_OFF + slot * BL::TILE + hh * BL::HALF, (i & 1) ? &tm_v : &tm_k,
                        bar(L::B_FULL + slot), g * D + hh * 64, kt * 128);
        }
      }
      if (*abort) {
        wait_drain(bar(L::B_Q), 0, 20000000ull);
        const uint32_t from = ld > static_cast<uint32_t>(NS) ? ld - NS : 0;
        for (uint32_t i = from; i < ld; ++i) wait_drain(bar(L::B_FULL + i % NS), (i / NS) & 1, 20000000ull);
      }
    }
  } else if (warp == 5) {
    if (lane == 0 && n > 0) {
      constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 128, 0);
      constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, D, 1);
      const uint32_t qs = sb + L::Q_OFF, dos = sb + L::DO_OFF;
      // S(j) = Q K^T and dP = dO V^T (SS); dQ += dS(j) K (TS, K MN-major)
      auto mma_s = [=](int j, uint32_t kb) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * BL::HALF + (kk & 3) * 32;
          mma_ss(tmem + q_s_col(j), smem_desc_sw128(qs + off, 16, 1024), smem_desc_sw128(kb + off, 16, 1024),
                 IDESC_QK, kk > 0);
        }
      };
      auto mma_dp = [=](uint32_t vb) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * BL::HALF + (kk & 3) * 32;
          mma_ss(tmem + 128, smem_desc_sw128(dos + off, 16, 1024), smem_desc_sw128(vb + off, 16, 1024),
                 IDESC_QK, kk > 0);
        }
      };
      auto mma_dq = [=](int j, uint32_t kb) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + 256, tmem + q_s_col(j) + kk * 8, smem_desc_sw128(kb + kk * 16 * 128, BL::HALF, 1024),
                 IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
      };
      // ring positions of a half: K_j at ld + 2j, V_j at ld + 2j + 1.  The
      // position ld + 2j is kept as (slot bs, round br), advanced by 2 per
      // key tile, and ld + 2j + off (off <= 4 < NS) as one conditional
      // subtraction: no division by NS on the issuing thread's path.
      uint32_t bs = 0, br = 0, s = 0;
      auto at = [&](uint32_t off, uint32_t &sl, uint32_t &ph) {
        sl = bs + off;
        uint32_t r = br;
        if (sl >= static_cast<uint32_t>(NS)) {
          sl -= NS;
          ++r;
        }
        ph = r & 1u;
      };
      auto full_at = [&](uint32_t off, uint32_t &sl) -> bool {
        uint32_t ph;
        at(off, sl, ph);
        return mbar_wait_bounded(bar(L::B_FULL + sl), ph, abort, lim);
      };
      auto kv_at = [=](uint32_t sl) -> uint32_t { return sb + L::KV_OFF + sl * BL::TILE; };
      auto step2 = [&]() {
        bs += 2;
        if (bs >= static_cast<uint32_t>(NS)) {
          bs -= NS;
          ++br;
        }
      };
      bool ok = true;
      for (int t = 0; ok && t < halves; ++t) {
        uint32_t s0, s1;
        ok = mbar_wait_bounded(bar(L::B_Q), t & 1, abort, lim) && full_at(0, s0) && full_at(1, s1);
        if (!ok) break;
        tc_fence_after();
        mma_s(0, kv_at(s0));
        mma_dp(kv_at(s1));
        mma_commit(bar(L::B_S));
        mma_commit(bar(L::B_EMPTY + s1));
        if (n == 1) mma_commit(bar(L::B_QE));
        if (n > 1) {
          uint32_t s2;
          if (!full_at(2, s2)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_s(1, kv_at(s2));
        }
        for (int j = 0; j < n; ++j, ++s, step2()) {
          bool have_p = false, look_k = false;
          if (j + 1 < n) {
            // dP(j+1) once dP(j) is in the element-wise warps' registers;
            // this commit also covers S(j+1), issued one key tile earlier.
            // Both dependencies are tested together (blocking), with a
            // non-blocking look at P(j) for the group after.
            uint32_t s3, ph3;
            at(3, s3, ph3);
            const bool have_v = mbar_try_wait(bar(L::B_FULL + s3), ph3);
            const bool have_dpr = mbar_try_wait(bar(L::B_DPR), s & 1);
            have_p = mbar_test_wait(bar(L::B_P), s & 1);
            if (j + 2 < n) {
              uint32_t s4l, ph4l;
              at(4, s4l, ph4l);
              look_k = mbar_test_wait(bar(L::B_FULL + s4l), ph4l);
            }
            if ((!have_v && !mbar_wait_bounded(bar(L::B_FULL + s3), ph3, abort, lim)) ||
                (!have_dpr && !mbar_wait_bounded(bar(L::B_DPR), s & 1, abort, lim))) {
              ok = false;
              break;
            }
            tc_fence_after();
            mma_dp(kv_at(s3));
            mma_commit(bar(L::B_S));
            mma_commit(bar(L::B_EMPTY + s3));
            if (j + 2 == n) mma_commit(bar(L::B_QE));   // the half's last reads of Q and dO
          }
          if (!have_p && !mbar_wait_bounded(bar(L::B_P), s & 1, abort, lim)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_dq(j, kv_at(bs));
          mma_commit(bar(L::B_EMPTY + bs));
          if (j + 2 < n) {
            uint32_t s4, ph4;
            at(4, s4, ph4);
            if (!look_k && !mbar_wait_bounded(bar(L::B_FULL + s4), ph4, abort, lim)) {
              ok = false;
              break;
            }
            tc_fence_after();
            mma_s(j + 2, kv_at(s4));
          }
        }
        if (ok) mma_commit(bar(L::B_O));
      }
      mma_commit(bar(L::B_DR));
      wait_drain(bar(L::B_DR), 0, 20000000ull);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ element-wise (thread = query row)
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const float sl2 = p.scale_log2;
    uint32_t s = 0;
    bool ok = true;
    for (int t = 0; ok && t < halves; ++t) {
      const int row = qt * B_TILE_Q + t * 128 + warp * 32 + lane;
      const bool live = row < p.sq;
      const float lv = live ? p.lse[static_cast<size_t>(h) * p.sq + row] : -INFINITY;
      const float lse2 = lv == -INFINITY ? INFINITY : lv * LOG2E;
      const float dlt = live ? p.delta[static_cast<size_t>(h) * p.sq + row] : 0.f;
      for (int j = 0; j < n; ++j, ++s) {
        const int e = e0 + j;
        const int kt = p.col_idx[e];
        uint32_t w[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
        if (p.kind[e] == ATTN_TILE_MASKED) {
          w[0] = w[1] = w[2] = w[3] = 0u;
          for (int q = p.ref_ptr[e]; q < p.ref_ptr[e + 1]; ++q)
            add_mask(p.slices[p.ref_idx[q]], row, kt * 128, w);
        }
        if (!wait_all(bar(L::B_S), s & 1, abort, lim)) {
          ok = false;
          break;
        }
        tc_fence_after();
        ds_step_dp_first(tmem + lane_off + q_s_col(j), tmem + lane_off + 128,
                         p.kind[e] == ATTN_TILE_MASKED, w, sl2, lse2, dlt, bar(L::B_DPR));
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(L::B_P));
      }
      if (!ok) break;
      bool have = n > 0;
      if (have) {
        if (!wait_all(bar(L::B_O), t & 1, abort, lim)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t r[32];
        if (have) {
          tmem_ld32_wait(tmem + lane_off + 256 + cc * 32, r);
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) r[k] = 0u;
        }
        if (live) store_rows<D>(p.dq, p.grad_f32, (static_cast<size_t>(row) * p.hq + h) * D + cc * 32, r, p.scale);
      }
      tc_fence_before();
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, 512);
  if (threadIdx.x == 0 && *abort) atomicCAS(&g_bwd_status, 0u, static_cast<unsigned>(ATTN_ERR_TIMEOUT));
}

// ------------------------------------------------------------------ host side

template <typename KernelT>
static int set_smem(KernelT k, int bytes) {
  return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess
             ? ATTN_OK
             : ATTN_ERR_CUDA;
}

template <int D>
static int launch_bwd_main(const CUtensorMap *m, const BwdParams &p, cudaStream_t s) {
  constexpr int NS = D == 128 ? 5 : 8;   // the dQ kernel's K/V ring
  int rc;
  if ((rc = set_smem(bwd_kv_kernel<D>, KVLayout<D>::ALLOC)) != ATTN_OK) return rc;
  if ((rc = set_smem(bwd_q_kernel<D, NS>, QLayout<D, NS>::ALLOC)) != ATTN_OK) return rc;
  if (p.n_ktiles > 0)
    bwd_kv_kernel<D><<<p.n_ktiles * p.hk, KV_THREADS, KVLayout<D>::ALLOC, s>>>(m[0], m[1], m[2], m[3], p);
  if (p.n_qtiles > 0)
    bwd_q_kernel<D, NS><<<p.n_qtiles * p.hq, Q_THREADS, QLayout<D, NS>::ALLOC, s>>>(m[0], m[1], m[2], m[3], p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

size_t bwd_workspace_bytes(int sq, int hq, int n_ktiles, int64_t cap_entries) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  return up(sizeof(float) * static_cast<size_t>(sq) * hq) + up(sizeof(int32_t) * n_ktiles) +
         up(sizeof(int32_t) * (n_ktiles + 1)) + up(sizeof(int32_t) * n_ktiles) +
         2 * up(sizeof(int32_t) * static_cast<size_t>(cap_entries > 0 ? cap_entries : 1));
}

int bwd_launch(const void *q, const void *k, const void *v, const void *out, int out_dtype,
               const void *dout, const float *lse, int sq, int sk, int hq, int hk, int d, float scale,
               const attn_tiles_t *tiles, void *dq, void *dk, void *dv, int grad_dtype, void *d_ws,
               cudaStream_t stream) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  uint8_t *ws = static_cast<uint8_t *>(d_ws);
  const int nk = tiles->n_ktiles;
  float *delta = reinterpret_cast<float *>(ws);
  ws += up(sizeof(float) * static_cast<size_t>(sq) * hq);
  int32_t *colcnt = reinterpret_cast<int32_t *>(ws);
  ws += up(sizeof(int32_t) * nk);
  int32_t *col_ptr = reinterpret_cast<int32_t *>(ws);
  ws += up(sizeof(int32_t) * (nk + 1));
  int32_t *col_sched = reinterpret_cast<int32_t *>(ws);
  ws += up(sizeof(int32_t) * nk);
  const size_t cap = up(sizeof(int32_t) * static_cast<size_t>(tiles->cap_entries > 0 ? tiles->cap_entries : 1));
  int32_t *col_q = reinterpret_cast<int32_t *>(ws);
  int32_t *col_e = reinterpret_cast<int32_t *>(ws + cap);

  BwdParams p;
  p.row_ptr = tiles->row_ptr;
  p.col_idx = tiles->col_idx;
  p.ref_ptr = tiles->ref_ptr;
  p.ref_idx = tiles->ref_idx;
  p.sched = tiles->sched;
  p.kind = tiles->kind;
  p.slices = tiles->slices;
  p.col_ptr = col_ptr;
  p.col_q = col_q;
  p.col_e = col_e;
  p.col_sched = col_sched;
  p.lse = lse;
  p.delta = delta;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.sq = sq;
  p.sk = sk;
  p.hq = hq;
  p.hk = hk;
  p.n_qtiles = tiles->n_qtiles;
  p.n_ktiles = nk;
  p.grad_f32 = grad_dtype == ATTN_DTYPE_F32;
  p.scale = scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.wait_ns = wait_limit_ns();
  p.meta_status = reinterpret_cast<const long long *>(tiles->totals + 3);

  const long long dthreads = static_cast<long long>(sq) * hq * (d / 8);
  const unsigned dgrid = static_cast<unsigned>((dthreads + 255) / 256);
  const uint16_t *dob = static_cast<const uint16_t *>(dout);
  if (d == 128) {
    if (out_dtype == ATTN_DTYPE_F32) bwd_delta_kernel<128, true><<<dgrid, 256, 0, stream>>>(out, dob, delta, sq, hq);
    else bwd_delta_kernel<128, false><<<dgrid, 256, 0, stream>>>(out, dob, delta, sq, hq);
  } else {
    if (out_dtype == ATTN_DTYPE_F32) bwd_delta_kernel<64, true><<<dgrid, 256, 0, stream>>>(out, dob, delta, sq, hq);
    else bwd_delta_kernel<64, false><<<dgrid, 256, 0, stream>>>(out, dob, delta, sq, hq);
  }
  if (nk > 0) {
    csc_count_kernel<<<nk, 256, 0, stream>>>(p, colcnt);
    csc_fill_kernel<<<nk, 256, 0, stream>>>(p, colcnt, col_ptr, col_q, col_e, col_sched);
  }
  CUtensorMap m[4];
  int rc;
  if ((rc = make_tma_2d(&m[0], q, static_cast<uint64_t>(hq) * d, sq)) != ATTN_OK) return rc;
  if ((rc = make_tma_2d(&m[1], k, static_cast<uint64_t>(hk) * d, sk)) != ATTN_OK) return rc;
  if ((rc = make_tma_2d(&m[2], v, static_cast<uint64_t>(hk) * d, sk)) != ATTN_OK) return rc;
  if ((rc = make_tma_2d(&m[3], dout, static_cast<uint64_t>(hq) * d, sq)) != ATTN_OK) return rc;
  if (d == 128) return launch_bwd_main<128>(m, p, stream);
  return launch_bwd_main<64>(m, p, stream);
}

int bwd_status_take(unsigned int *status) {
  unsigned int zero = 0;
  if (cudaMemcpyFromSymbol(status, g_bwd_status, sizeof(unsigned int)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (*status && cudaMemcpyToSymbol(g_bwd_status, &zero, sizeof(unsigned int)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

}  // namespace attn
