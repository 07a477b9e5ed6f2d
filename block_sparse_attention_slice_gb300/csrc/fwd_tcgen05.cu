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
// Persistent kernel: one CTA per SM takes work items (query tile, head) in
// longest-processing-time order from a global counter (the producer lane
// fetches and publishes each item id to the CTA's other roles through a
// small shared-memory queue), so the CTAs finish together and the next
// item's Q load and first QK overlap the previous item's epilogue.  A work item is 256
// query rows of one head (two 128-row MMA tiles, t = 0, 1) against the
// KV-tile list of that 256-row query tile.  Warp roles (352 threads):
//   warps 0-3  softmax of tile 0 (thread = row = tensor-memory lane)
//   warps 4-7  softmax of tile 1
//   warp  8    TMA producer: Q of each item, then K_j, V_j through an NS-slot ring
//   warp  9    tensor-memory allocator and MMA issuer
//   warp 10    metadata: resolves each tile entry (key tile, kind, the first
//              two referenced slices) 32 entries at a time into a shared
//              ring of records, so the softmax never waits on global memory
// Tensor memory (512 columns): S_0 [0,128)  S_1 [128,256)  O_0 [256,256+D)
// O_1 [384,384+D).  P (bf16) overwrites the first 64 columns of S_t and is
// the A operand of O_t += P_t V_j read straight from tensor memory, so the
// probabilities never touch shared memory.  The MMA order per KV step j is
//   PV_0(j), QK_0(j+1), PV_1(j), QK_1(j+1)
// so the tensor core works on one tile while the softmax warps of the other
// tile run (FlashAttention-4 page: softmax overlapped with the MMAs).
// The epilogue of a bf16 output stages O_t / l in the tile's own 128 x D
// shared-memory buffer (each 64-column half in the 128-byte swizzle of the
// output's tensor map) and leaves it with one TMA store per half, which
// writes whole rows and clips the rows past S_q; nothing waits for the
// stores until the buffer is needed again.  f32 partial outputs keep one
// thread per row.
// tcgen05 operations of one thread complete in issue order, so when the
// softmax of tile t sees S_t(j) its previous PV_t(j-1) has completed too,
// and the next item's first QK may be issued while the softmax warps are
// still storing the previous item's O (its first PV waits for their P).
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>
#include <type_traits>

#include "attn_device.cuh"
#include "attn_internal.h"

namespace attn {

// First failure status of forward launches on this device (0 = none): a
// bounded wait that ran out (ATTN_ERR_TIMEOUT), or metadata whose build did
// not finish with ATTN_OK (its status code).  Read and cleared by
// attn_last_device_error().
__device__ unsigned int g_fwd_status;

constexpr int BM = 128;           // rows per MMA tile
constexpr int BN = 128;           // keys per KV tile
constexpr float TAU = 8.0f;       // lazy-rescale threshold, log2 units
constexpr int NTHREADS = 352;
constexpr int RING = 16;          // metadata records in flight
constexpr int IQ = 4;             // queued work-item ids
constexpr int SCHED_SLOTS = 4096; // work counters, one per launch in flight

// Work counters of forward launches: each launch takes the next slot (host
// side, round robin).  Slot i holds the item counter at [i] and the count of
// retired CTAs at [SCHED_SLOTS + i]; both start at 0 (static device memory)
// and the launch's last CTA to retire puts both back to 0, so no launch needs
// a memset before it.
__device__ unsigned int g_sched_counter[2 * SCHED_SLOTS];

struct FwdParams {
  const int32_t *row_ptr, *col_idx, *ref_ptr, *ref_idx, *sched;
  const uint8_t *kind;
  const attn_slice_t *slices;
  void *out;
  float *lse;
  int sq, sk, hq, hk, n_items;
  int out_f32;                    // f32 O by direct stores, else bf16 O by TMA stores
  float scale_log2;               // scale * log2(e)
  unsigned long long wait_ns;
  unsigned int *counter;          // this launch's work counter (0 at launch, reset by its last CTA)
  const long long *meta_status;   // the metadata build's status word (totals[3])
  int test_stall;                 // failure-path test: leave one ring slot unarmed (see below)
};

// One resolved tile entry: key tile, kind, reference range and up to two
// referenced slices inline (more are read from global memory).
struct __align__(16) Rec {
  int kt, kind, r0, r1;
  attn_slice_t s[2];
  int pad[2];
};
static_assert(sizeof(Rec) == 64, "record size");

template <int D, int NS>
struct Layout {
  static constexpr int HALF = 128 * 64 * 2;          // 128 rows x 64 bf16 (one swizzle span)
  static constexpr int NHALF = D / 64;
  static constexpr int TILE = NHALF * HALF;          // 128 x D bf16
  static constexpr int Q_OFF = 0;
  static constexpr int KV_OFF = 2 * TILE;
  static constexpr int ST_OFF = KV_OFF + NS * TILE;   // bf16 O staging: one 128 x D tile per MMA tile
  static constexpr int REC_OFF = ST_OFF + 2 * TILE;
  static constexpr int IQ_OFF = REC_OFF + RING * 64;
  static constexpr int BAR_OFF = IQ_OFF + IQ * 16;
  // q_full | q_empty | full[NS] | empty[NS] | s_full[2] | p_full[2] | o_full[2] | drain |
  // rec_full[RING] | rec_empty[RING] | iq_full[IQ] | iq_empty[IQ] | stage_full[2] |
  // stage_free[2]
  static constexpr int B_Q = 0, B_QE = 1, B_FULL = 2, B_EMPTY = 2 + NS, B_S = 2 + 2 * NS,
                       B_P = B_S + 2, B_O = B_P + 2, B_DRAIN = B_O + 2, B_RF = B_DRAIN + 1,
                       B_RE = B_RF + RING, B_IF = B_RE + RING, B_IE = B_IF + IQ,
                       B_EF = B_IE + IQ, B_EE = B_EF + 2, NBAR = B_EE + 2;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int BYTES = MISC_OFF + 16;
  static constexpr int ALLOC = BYTES + 1024;
  static_assert(ST_OFF % 1024 == 0, "swizzled staging alignment");
  static_assert(ALLOC <= 232448, "shared memory per CTA");
};

struct Item {
  int qt, h, g, e0, n;
};

__device__ __forceinline__ Item decode(const FwdParams &p, int item) {
  Item it;
  it.qt = __ldg(p.sched + item / p.hq);
  it.h = item % p.hq;
  it.g = it.h / (p.hq / p.hk);
  it.e0 = __ldg(p.row_ptr + it.qt);
  it.n = __ldg(p.row_ptr + it.qt + 1) - it.e0;
  return it;
}

// POLY = 0: every exponential on the special-function unit; POLY = k > 0:
// on FULL tiles, every k-th pair of a row's exponentials on the FMA-pipe
// polynomial (exp2_poly2), the rest on the special-function unit.
template <int D, int NS, int POLY>
__global__ void __launch_bounds__(NTHREADS, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
               const FwdParams p) {
  using L = Layout<D, NS>;
  static_assert(POLY == 0 || (POLY > 0 && 16 % POLY == 0), "polynomial period");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + L::BAR_OFF + 8u * i; };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::MISC_OFF);
  volatile int *abort = reinterpret_cast<volatile int *>(smem + L::MISC_OFF + 4);
  volatile int *meta_bad = reinterpret_cast<volatile int *>(smem + L::MISC_OFF + 8);
  Rec *recs = reinterpret_cast<Rec *>(smem + L::REC_OFF);
  volatile int *iq = reinterpret_cast<volatile int *>(smem + L::IQ_OFF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t lim = p.wait_ns;
  const uint32_t q_smem = sb + L::Q_OFF, kv_smem = sb + L::KV_OFF;

  if (threadIdx.x == 0) {
    mbar_init(bar(L::B_Q), 1);
    mbar_init(bar(L::B_QE), 1);
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
    for (int r = 0; r < RING; ++r) {
      mbar_init(bar(L::B_RF + r), 1);
      mbar_init(bar(L::B_RE + r), 8);
    }
    // item ids are read by the MMA lane, the metadata warp and 8 softmax warps
    for (int u = 0; u < IQ; ++u) {
      mbar_init(bar(L::B_IF + u), 1);
      mbar_init(bar(L::B_IE + u), 10);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(L::B_EF + t), 128);
      mbar_init(bar(L::B_EE + t), 1);
    }
    *abort = 0;
    // metadata whose build failed (a grid barrier that ran out, capacity) is
    // not read at all: every CTA skips its work and the status is recorded
    const long long ms = *p.meta_status;
    *meta_bad = ms != ATTN_OK;
    if (ms != ATTN_OK) atomicCAS(&g_fwd_status, 0u, static_cast<unsigned>(ms));
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

  if (*meta_bad) {
    // nothing to do: no item is fetched, so the work counter stays at 0
  } else if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t ld = 0, nonempty = 0, qpos = 0;
      bool ok = true;
      while (ok) {
        // fetch the next item and publish it to the other roles
        const int qs = qpos % IQ;
        if (qpos >= IQ && !mbar_wait_bounded(bar(L::B_IE + qs), (qpos / IQ - 1) & 1, abort, lim)) {
          ok = false;
          break;
        }
        const int item = static_cast<int>(atomicAdd(p.counter, 1u));
        iq[qs] = item;
        mbar_arrive(bar(L::B_IF + qs));
        ++qpos;
        if (item >= p.n_items) break;
        const Item it = decode(p, item);
        if (it.n == 0) continue;
        if (nonempty > 0 && !mbar_wait_bounded(bar(L::B_QE), (nonempty - 1) & 1, abort, lim)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(L::B_Q), 2 * L::TILE);
        for (int t = 0; t < 2; ++t)
          for (int hh = 0; hh < L::NHALF; ++hh)
            tma_load_2d(q_smem + t * L::TILE + hh * L::HALF, &tm_q, bar(L::B_Q), it.h * D + hh * 64,
                        it.qt * 256 + t * BM);
        ++nonempty;
        // key-tile index of the next entry is fetched one entry ahead
        int kt = 0, kt_next = __ldg(p.col_idx + it.e0);
        for (int i = 0; i < 2 * it.n; ++i, ++ld) {
          if (!(i & 1)) {
            kt = kt_next;
            if ((i >> 1) + 1 < it.n) kt_next = __ldg(p.col_idx + it.e0 + (i >> 1) + 1);
          }
          const int slot = ld % NS;
          const uint32_t use = ld / NS;
          if (use > 0 && !mbar_wait_bounded(bar(L::B_EMPTY + slot), (use - 1) & 1, abort, lim)) {
            ok = false;
            break;
          }
          // failure-path test only: the CTA's second K/V load (V of its first
          // step) is neither armed nor issued, so the MMA lane's bounded wait
          // for that slot runs out and the whole abort path runs
          if (p.test_stall && ld == 1) continue;
          mbar_arrive_expect_tx(bar(L::B_FULL + slot), L::TILE);
          for (int hh = 0; hh < L::NHALF; ++hh)
            tma_load_2d(kv_smem + slot * L::TILE + hh * L::HALF, (i & 1) ? &tm_v : &tm_k,
                        bar(L::B_FULL + slot), it.g * D + hh * 64, kt * BN);
        }
      }
      if (*abort) {
        // let the loads already in flight land before the CTA retires
        if (nonempty > 0) wait_drain(bar(L::B_Q), (nonempty - 1) & 1, 20000000ull);
        const uint32_t from = ld > static_cast<uint32_t>(NS) ? ld - NS : 0;
        for (uint32_t i = from; i < ld; ++i)
          wait_drain(bar(L::B_FULL + i % NS), (i / NS) & 1, 20000000ull);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_QK = idesc_bf16_f32(BM, BN, 0);
      constexpr uint32_t IDESC_PV = idesc_bf16_f32(BM, D, 1);
      auto issue_qk = [=](int t, int slot) {
        const uint32_t d_tmem = tmem + t * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::HALF + (kk & 3) * 32;
          mma_ss(d_tmem, smem_desc_sw128(q_smem + t * L::TILE + off, 16, 1024),
                 smem_desc_sw128(kv_smem + slot * L::TILE + off, 16, 1024), IDESC_QK, kk > 0);
        }
      };
      auto issue_pv = [=](int t, int slot, bool first) {
        const uint32_t d_tmem = tmem + 256 + t * 128;
        const uint32_t a_tmem = tmem + t * 128;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts(d_tmem, a_tmem + kk * 8,
                 smem_desc_sw128(kv_smem + slot * L::TILE + kk * 16 * 128, L::HALF, 1024), IDESC_PV,
                 (first && kk == 0) ? 0u : 1u);
      };
      uint32_t ld = 0, nonempty = 0, step = 0;
      bool ok = true;
      uint32_t qpos = 0;
      while (ok) {
        const int qs = qpos % IQ;
        if (!mbar_wait_bounded(bar(L::B_IF + qs), (qpos / IQ) & 1, abort, lim)) {
          ok = false;
          break;
        }
        const int item = iq[qs];
        mbar_arrive(bar(L::B_IE + qs));
        ++qpos;
        if (item >= p.n_items) break;
        const Item it = decode(p, item);
        const int n = it.n;
        if (n == 0) continue;
        ok = mbar_wait_bounded(bar(L::B_Q), nonempty & 1, abort, lim) &&
             mbar_wait_bounded(bar(L::B_FULL + ld % NS), (ld / NS) & 1, abort, lim);
        if (!ok) break;
        tc_fence_after();
        issue_qk(0, ld % NS);
        mma_commit(bar(L::B_S + 0));
        issue_qk(1, ld % NS);
        mma_commit(bar(L::B_S + 1));
        mma_commit(bar(L::B_EMPTY + ld % NS));
        if (n == 1) mma_commit(bar(L::B_QE));
        ++ld;
        for (int j = 0; j < n; ++j, ++step) {
          const uint32_t vpos = ld, kpos = ld + 1;
          const bool more = j + 1 < n;
          if (!mbar_wait_bounded(bar(L::B_FULL + vpos % NS), (vpos / NS) & 1, abort, lim) ||
              !mbar_wait_bounded(bar(L::B_P + 0), step & 1, abort, lim)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(0, vpos % NS, j == 0);
          if (!more) mma_commit(bar(L::B_O + 0));
          if (more) {
            if (!mbar_wait_bounded(bar(L::B_FULL + kpos % NS), (kpos / NS) & 1, abort, lim)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_qk(0, kpos % NS);
            mma_commit(bar(L::B_S + 0));
          }
          if (!mbar_wait_bounded(bar(L::B_P + 1), step & 1, abort, lim)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(1, vpos % NS, j == 0);
          mma_commit(bar(L::B_EMPTY + vpos % NS));
          if (!more) mma_commit(bar(L::B_O + 1));
          if (more) {
            issue_qk(1, kpos % NS);
            mma_commit(bar(L::B_S + 1));
            mma_commit(bar(L::B_EMPTY + kpos % NS));
            if (j + 2 == n) mma_commit(bar(L::B_QE));
          }
          ld += more ? 2 : 1;
        }
        ++nonempty;
      }
      // every MMA this thread issued completes before tensor memory is freed
      mma_commit(bar(L::B_DRAIN));
      wait_drain(bar(L::B_DRAIN), 0, 20000000ull);
    }
    __syncwarp();
  } else if (warp == 10) {
    // ------------------------------------------------------------ metadata
    uint32_t rpos = 0;
    bool ok = true;
    uint32_t qpos = 0;
    while (ok) {
      const int qs = qpos % IQ;
      if (!wait_all(bar(L::B_IF + qs), (qpos / IQ) & 1, abort, lim)) {
        ok = false;
        break;
      }
      const int item = iq[qs];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::B_IE + qs));
      ++qpos;
      if (item >= p.n_items) break;
      const Item it = decode(p, item);
      for (int base = 0; ok && base < it.n; base += 32) {
        const int j = base + lane, cnt = min(32, it.n - base);
        Rec r;
        r.kt = r.kind = r.r0 = r.r1 = r.pad[0] = r.pad[1] = 0;
        r.s[0] = attn_slice_t{0, 0, 0, 0, 0};
        r.s[1] = attn_slice_t{0, 0, 0, 0, 0};
        if (j < it.n) {
          const int e = it.e0 + j;
          r.kt = __ldg(p.col_idx + e);
          r.kind = __ldg(p.kind + e);
          r.r0 = __ldg(p.ref_ptr + e);
          r.r1 = __ldg(p.ref_ptr + e + 1);
          if (r.r1 > r.r0) r.s[0] = p.slices[__ldg(p.ref_idx + r.r0)];
          if (r.r1 > r.r0 + 1) r.s[1] = p.slices[__ldg(p.ref_idx + r.r0 + 1)];
        }
        // records go out in order; lane 0 alone waits for each slot to be
        // released (the others park at the shuffle), then lane l writes
        for (int l = 0; l < cnt; ++l, ++rpos) {
          const int slot = rpos % RING;
          bool free_ok = true;
          if (lane == 0 && rpos >= RING)
            free_ok = mbar_wait_bounded(bar(L::B_RE + slot), (rpos / RING - 1) & 1, abort, lim);
          if (!__shfl_sync(0xffffffffu, free_ok ? 1 : 0, 0)) {
            ok = false;
            break;
          }
          if (lane == l) {
            recs[slot] = r;
            mbar_arrive(bar(L::B_RF + slot));
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2, wl = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(wl * 32) << 16;
    const uint32_t tS = tmem + lane_off + t * 128;
    const uint32_t tO = tmem + lane_off + 256 + t * 128;
    const float sl2 = p.scale_log2;
    const bool elected = wl == 0 && lane == 0;   // issues this tile's output stores
    bool ee_due = false;   // elected: the last stores' staging release is not yet signalled
    uint32_t step = 0, rpos = 0, nonempty = 0, ep = 0;
    bool ok = true;
    uint32_t qpos = 0;
    while (ok) {
      const int qs = qpos % IQ;
      if (!wait_all(bar(L::B_IF + qs), (qpos / IQ) & 1, abort, lim)) {
        ok = false;
        break;
      }
      const int item = iq[qs];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::B_IE + qs));
      ++qpos;
      if (item >= p.n_items) break;
      const Item it = decode(p, item);
      const int row = it.qt * 256 + t * BM + wl * 32 + lane;
      const bool live = row < p.sq;
      const size_t obase = (static_cast<size_t>(row) * p.hq + it.h) * D;
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < it.n; ++j, ++step, ++rpos) {
        const int slot = rpos % RING;
        if (!wait_all(bar(L::B_RF + slot), (rpos / RING) & 1, abort, lim)) {
          ok = false;
          break;
        }
        const Rec &rc = recs[slot];
        const int kt = rc.kt, kd = rc.kind, r0 = rc.r0, r1 = rc.r1;
        uint32_t w[BN / 32] = {0u, 0u, 0u, 0u};
        if (kd == ATTN_TILE_MASKED) {
          // MASKED tile: union of the referenced slices' row intervals as a
          // 128-bit mask, then a predicated select per element.
          const int c0 = kt * BN;
          if (r1 > r0) add_mask(rc.s[0], row, c0, w);
          if (r1 > r0 + 1) add_mask(rc.s[1], row, c0, w);
          for (int r = r0 + 2; r < r1; ++r) add_mask(p.slices[__ldg(p.ref_idx + r)], row, c0, w);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::B_RE + slot));
        if (!wait_all(bar(L::B_S + t), step & 1, abort, lim)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float s[BN];
        {
          // all four 32-column loads in flight, one wait
          uint32_t r[BN];
#pragma unroll
          for (int c = 0; c < BN / 32; ++c)
            tmem_ld32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&r[c * 32]));
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < BN; ++k) {
            asm volatile("" : "+r"(r[k]));
            s[k] = __uint_as_float(r[k]);
          }
        }
        if (kd == ATTN_TILE_MASKED) {
#pragma unroll
          for (int k = 0; k < BN; ++k)
            if (!((w[k >> 5] >> (k & 31)) & 1u)) s[k] = -INFINITY;
        }
        // row max: four independent chains of three-input maxima, seeded
        // with s[0..7] and covering s[8..BN) in rounds of eight
        static_assert(BN % 8 == 0, "row max rounds");
        float m4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) m4[u] = fmaxf(s[2 * u], s[2 * u + 1]);
#pragma unroll
        for (int k = 8; k < BN; k += 8) {
#pragma unroll
          for (int u = 0; u < 4; ++u) m4[u] = max3f(m4[u], s[k + 2 * u], s[k + 2 * u + 1]);
        }
        const float mx = max3f(m4[0], m4[1], fmaxf(m4[2], m4[3]));
        const float mx2 = mx * sl2;
        const float m_old = m_ref;
        const bool grow = mx2 > m_ref + TAU;
        if (grow) m_ref = mx2;
        const float factor = grow ? ex2_approx(m_old - m_ref) : 1.f;
        l *= factor;
        const float mb = (m_ref == -INFINITY) ? 0.f : m_ref;
        // exponent arguments and row sums on f32 pairs: four independent
        // two-wide partial sums
        const uint64_t sc2 = f2_make(sl2, sl2), nb2 = f2_make(-mb, -mb);
        uint64_t l2[4] = {0ull, 0ull, 0ull, 0ull};
        // USE_POLY: FULL tile with the polynomial enabled (all arguments
        // finite); MASKED tiles keep the special-function unit, which maps
        // a masked -inf to exactly 0
        auto exps = [&](auto use_poly) {
          constexpr bool USE_POLY = decltype(use_poly)::value;
#pragma unroll
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t pk[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const uint64_t a2 = f2_fma(f2_make(s[c * 32 + 2 * k], s[c * 32 + 2 * k + 1]), sc2, nb2);
              float p0, p1;
              if (USE_POLY && (k % (POLY > 0 ? POLY : 1)) == (POLY > 0 ? POLY : 1) - 1) {
                f2_split(exp2_poly2(a2), p0, p1);
              } else {
                float a0, a1;
                f2_split(a2, a0, a1);
                p0 = ex2_approx(a0);
                p1 = ex2_approx(a1);
              }
              l2[k & 3] = f2_add(l2[k & 3], f2_make(p0, p1));
              pk[k] = pack_bf16x2(p0, p1);
            }
            tmem_st16(tS + c * 16, pk);
          }
        };
        if (POLY > 0 && kd == ATTN_TILE_FULL)
          exps(std::true_type{});
        else
          exps(std::false_type{});
        {
          float x0, x1;
          f2_split(f2_add(f2_add(l2[0], l2[1]), f2_add(l2[2], l2[3])), x0, x1);
          l += x0 + x1;
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
        if (ee_due) {
          // a KV step after the last item's stores were issued: they have read
          // the staging by now, normally without waiting
          bulk_wait_read_all();
          mbar_arrive(bar(L::B_EE + t));
          ee_due = false;
        }
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      if (it.n > 0) {
        if (!wait_all(bar(L::B_O + t), nonempty & 1, abort, lim)) {
          ok = false;
          break;
        }
        ++nonempty;
        tc_fence_after();
      }
      const float inv = l > 0.f ? 1.f / l : 0.f;
      if (!p.out_f32) {
        // bf16 O through this tile's 128 x D shared-memory staging, each
        // 64-column half in the 128-byte swizzle of the output's tensor map
        // (16-byte chunk c of row r at chunk c ^ (r & 7)), one TMA store per
        // half; the store clips the rows past S_q.  Nothing here waits for
        // the stores: the elected thread confirms that they have read the
        // staging during the next item's first KV step (or at the next
        // epilogue, if that comes first).
        const uint32_t stg = sb + L::ST_OFF + t * L::TILE;
        const int r = wl * 32 + lane;
        const int y0 = it.qt * 256 + t * BM;
        if (ep > 0) {
          if (ee_due) {
            bulk_wait_read_all();
            mbar_arrive(bar(L::B_EE + t));
            ee_due = false;
          }
          if (!wait_all(bar(L::B_EE + t), (ep - 1) & 1, abort, lim)) {
            ok = false;
            break;
          }
        }
#pragma unroll 1
        for (int hh = 0; hh < L::NHALF; ++hh) {
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) {
            uint32_t x[32];
            if (it.n > 0) {
              tmem_ld32_wait(tO + hh * 64 + c2 * 32, x);
            } else {
#pragma unroll
              for (int k = 0; k < 32; ++k) x[k] = 0u;
            }
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(x[8 * q4 + 0]) * inv, __uint_as_float(x[8 * q4 + 1]) * inv);
              v.y = pack_bf16x2(__uint_as_float(x[8 * q4 + 2]) * inv, __uint_as_float(x[8 * q4 + 3]) * inv);
              v.z = pack_bf16x2(__uint_as_float(x[8 * q4 + 4]) * inv, __uint_as_float(x[8 * q4 + 5]) * inv);
              v.w = pack_bf16x2(__uint_as_float(x[8 * q4 + 6]) * inv, __uint_as_float(x[8 * q4 + 7]) * inv);
              st_shared_v4(stg + hh * L::HALF + r * 128 + (((c2 * 4 + q4) ^ (r & 7)) << 4), v);
            }
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(L::B_EF + t));
        if (elected) {
          if (mbar_wait_bounded(bar(L::B_EF + t), ep & 1, abort, lim) && y0 < p.sq) {
            for (int hh = 0; hh < L::NHALF; ++hh)
              tma_store_2d(&tm_o, stg + hh * L::HALF, it.h * D + hh * 64, y0);
            bulk_commit_group();
          }
          ee_due = true;
        }
        ++ep;
      } else {
        // f32 O (KV-split partials): one thread per row, 16-byte stores
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          if (it.n > 0) {
            tmem_ld32_wait(tO + c * 32, r);
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) r[k] = 0u;
          }
          if (!live) continue;
          float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + obase + c * 32);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            dst[k] = make_float4(__uint_as_float(r[4 * k]) * inv, __uint_as_float(r[4 * k + 1]) * inv,
                                 __uint_as_float(r[4 * k + 2]) * inv,
                                 __uint_as_float(r[4 * k + 3]) * inv);
        }
      }
      if (live)
        p.lse[static_cast<size_t>(it.h) * p.sq + row] =
            l > 0.f ? (m_ref + __log2f(l)) * 0.69314718055994531f : -INFINITY;
      // tensor-memory reads of O finish before the next item's first PV
      tc_fence_before();
    }
    // the output stores have completed before the CTA retires
    if (wl == 0 && lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tmem, 512);
  if (threadIdx.x == 0) {
    if (*abort) atomicCAS(&g_fwd_status, 0u, static_cast<unsigned>(ATTN_ERR_TIMEOUT));
    // every CTA has fetched its last item id once it gets here: the last one
    // to retire resets this launch's slot for its next use
    __threadfence();
    if (atomicAdd(p.counter + SCHED_SLOTS, 1u) == gridDim.x - 1) {
      atomicExch(p.counter, 0u);
      atomicExch(p.counter + SCHED_SLOTS, 0u);
    }
  }
}

// ------------------------------------------------------------------ host side

static unsigned long long g_wait_ns = 4000000000ull;
static int g_exp2_poly = 0;   // 0, 4 or 8: see fwd_kernel's POLY
constexpr int kMaxDev = 64;
static std::atomic<unsigned int> g_launch_seq{0};

// Device address of this launch's work counter (g_sched_counter on the
// current device, looked up once per device).
static unsigned int *next_counter() {
  static unsigned int *base[kMaxDev] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!base[dev]) {
      void *ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_sched_counter) != cudaSuccess) return nullptr;
      base[dev] = static_cast<unsigned int *>(ptr);
    }
  }
  return base[dev] + (g_launch_seq.fetch_add(1) % SCHED_SLOTS);
}

template <int D, int NS, int POLY>
static int launch_fwd(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                      const CUtensorMap &mo, const FwdParams &p, int grid, cudaStream_t s) {
  using L = Layout<D, NS>;
  static bool configured[kMaxDev] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return ATTN_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!configured[dev]) {
      if (cudaFuncSetAttribute(fwd_kernel<D, NS, POLY>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               L::ALLOC) != cudaSuccess)
        return ATTN_ERR_CUDA;
      configured[dev] = true;
    }
  }
  fwd_kernel<D, NS, POLY><<<grid, NTHREADS, L::ALLOC, s>>>(mq, mk, mv, mo, p);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int fwd_launch(const void *q, const void *k, const void *v, int sq, int sk, int hq, int hk, int d,
               float scale, const attn_tiles_t *tiles, void *out, int out_dtype, float *lse,
               cudaStream_t stream) {
  CUtensorMap mq, mk, mv, mo;
  int rc;
  if ((rc = make_tma_2d(&mq, q, static_cast<uint64_t>(hq) * d, sq)) != ATTN_OK) return rc;
  if ((rc = make_tma_2d(&mk, k, static_cast<uint64_t>(hk) * d, sk)) != ATTN_OK) return rc;
  if ((rc = make_tma_2d(&mv, v, static_cast<uint64_t>(hk) * d, sk)) != ATTN_OK) return rc;
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
  // bf16 O is stored by TMA through the same 64 x 128 box format as Q; the
  // f32 path (partials) keeps one thread per row and needs no map
  if (!p.out_f32) {
    if ((rc = make_tma_2d(&mo, out, static_cast<uint64_t>(hq) * d, sq)) != ATTN_OK) return rc;
  } else {
    mo = mq;
  }
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.wait_ns = g_wait_ns;
  const long long items = static_cast<long long>(tiles->n_qtiles) * hq;
  if (items == 0) return ATTN_OK;
  if (items >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
  p.n_items = static_cast<int>(items);
  const int sms = device_sm_count();
  if (sms <= 0) return ATTN_ERR_CUDA;
  const int grid = static_cast<int>(items < sms ? items : sms);
  p.counter = next_counter();
  if (!p.counter) return ATTN_ERR_CUDA;
  p.meta_status = reinterpret_cast<const long long *>(tiles->totals + 3);
  // ATTN_TEST_STALL_FWD=1 in the environment: every CTA leaves its second
  // K/V load unissued, so the launch ends by its bounded waits running out
  // (ATTN_ERR_TIMEOUT) -- the form in which the tests drive the forward's
  // own abort path without faulting or hanging the GPU
  const char *stall = std::getenv("ATTN_TEST_STALL_FWD");
  p.test_stall = stall && stall[0] == '1';
  const int poly = g_exp2_poly;
  if (d == 128) {
    if (poly == 4) return launch_fwd<128, 3, 4>(mq, mk, mv, mo, p, grid, stream);
    if (poly == 8) return launch_fwd<128, 3, 8>(mq, mk, mv, mo, p, grid, stream);
    return launch_fwd<128, 3, 0>(mq, mk, mv, mo, p, grid, stream);
  }
  if (poly == 4) return launch_fwd<64, 8, 4>(mq, mk, mv, mo, p, grid, stream);
  if (poly == 8) return launch_fwd<64, 8, 8>(mq, mk, mv, mo, p, grid, stream);
  return launch_fwd<64, 8, 0>(mq, mk, mv, mo, p, grid, stream);
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

void fwd_set_exp2_poly(int period) { g_exp2_poly = period; }

unsigned long long wait_limit_ns() { return g_wait_ns; }

// One thread waits on a barrier that nothing will complete; the bounded wait
// gives up after the configured limit and records a timeout.
__global__ void selftest_timeout_kernel(unsigned long long wait_ns) {
  __shared__ __align__(8) uint64_t b;
  __shared__ int abort_flag;
  const uint32_t a = smem_u32(&b);
  mbar_init(a, 1);
  abort_flag = 0;
  fence_mbar_init();
  if (!mbar_wait_bounded(a, 0, reinterpret_cast<volatile int *>(&abort_flag), wait_ns))
    atomicCAS(&g_fwd_status, 0u, static_cast<unsigned>(ATTN_ERR_TIMEOUT));
}

int selftest_timeout_launch(cudaStream_t s) {
  selftest_timeout_kernel<<<1, 1, 0, s>>>(g_wait_ns);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn
