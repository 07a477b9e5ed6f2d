// Exact merge of KV-split partial attention outputs (UltraAttn page,
// section 3.2): every KV shard contributes a summary that is rescaled to the
// global maximum before the sums are added, so the result equals the softmax
// over the concatenated keys.  A partial (O_i normalised, lse_i) is the
// summary (m = lse_i, l = 1, o = O_i):
//   m = max_i lse_i,  w_i = exp(lse_i - m),  L = sum_i w_i
//   lse = m + ln L,   O = sum_i (w_i / L) O_i
// HBM streaming: one warp per (head, row); each lane moves 16 bytes of every
// partial with one vector load, so a warp reads a whole 512-byte f32 row of
// d = 128 in one instruction per partial; consecutive warps take
// consecutive rows of one head so the lse reads coalesce too.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "attn_internal.h"

namespace attn {

struct MergeParams {
  const void *o[ATTN_MERGE_MAX_PARTS];
  const float *lse[ATTN_MERGE_MAX_PARTS];
  int n, S, H;
  void *out;
  float *lse_out;
};

template <int D, typename TI, bool OUT_F32>
__global__ void __launch_bounds__(256) merge_kernel(const MergeParams p) {
  constexpr int V = D / 32;                         // elements per lane
  const long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= static_cast<long long>(p.S) * p.H) return;
  const int h = static_cast<int>(w / p.S), s = static_cast<int>(w % p.S);
  const size_t lidx = static_cast<size_t>(h) * p.S + s;
  const float li = lane < p.n ? __ldg(p.lse[lane] + lidx) : -INFINITY;
  float m = li;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const size_t obase = (static_cast<size_t>(s) * p.H + h) * D + lane * V;
  if (m == -INFINITY) {
    if constexpr (OUT_F32) {
      float *dst = static_cast<float *>(p.out) + obase;
#pragma unroll
      for (int k = 0; k < V; ++k) dst[k] = 0.f;
    } else {
      uint16_t *dst = static_cast<uint16_t *>(p.out) + obase;
#pragma unroll
      for (int k = 0; k < V; ++k) dst[k] = 0;
    }
    if (lane == 0) p.lse_out[lidx] = -INFINITY;
    return;
  }
  const float wi = lane < p.n ? expf(li - m) : 0.f;
  float L = wi;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  const float invL = 1.f / L;
  float acc[V];
#pragma unroll
  for (int k = 0; k < V; ++k) acc[k] = 0.f;
  for (int i = 0; i < p.n; ++i) {
    const float c = __shfl_sync(0xffffffffu, wi, i) * invL;
    float x[V];
    if constexpr (sizeof(TI) == 4) {
      const float *src = static_cast<const float *>(p.o[i]) + obase;
      if constexpr (V == 4) {
        const float4 y = __ldcs(reinterpret_cast<const float4 *>(src));
        x[0] = y.x; x[1] = y.y; x[2] = y.z; x[3] = y.w;
      } else {
        const float2 y = __ldcs(reinterpret_cast<const float2 *>(src));
        x[0] = y.x; x[1] = y.y;
      }
    } else {
      const uint16_t *src = static_cast<const uint16_t *>(p.o[i]) + obase;
      uint32_t u[V / 2];
      if constexpr (V == 4) {
        const uint2 y = __ldcs(reinterpret_cast<const uint2 *>(src));
        u[0] = y.x; u[1] = y.y;
      } else {
        u[0] = __ldcs(reinterpret_cast<const unsigned int *>(src));
      }
#pragma unroll
      for (int k = 0; k < V / 2; ++k) {
        x[2 * k] = __uint_as_float(u[k] << 16);
        x[2 * k + 1] = __uint_as_float(u[k] & 0xffff0000u);
      }
    }
#pragma unroll
    for (int k = 0; k < V; ++k) acc[k] = fmaf(c, x[k], acc[k]);
  }
  if constexpr (OUT_F32) {
    float *dst = static_cast<float *>(p.out) + obase;
    if constexpr (V == 4)
      *reinterpret_cast<float4 *>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    else
      *reinterpret_cast<float2 *>(dst) = make_float2(acc[0], acc[1]);
  } else {
    uint16_t *dst = static_cast<uint16_t *>(p.out) + obase;
    uint32_t pk[V / 2];
#pragma unroll
    for (int k = 0; k < V / 2; ++k)
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(pk[k]) : "f"(acc[2 * k + 1]), "f"(acc[2 * k]));
    if constexpr (V == 4)
      *reinterpret_cast<uint2 *>(dst) = make_uint2(pk[0], pk[1]);
    else
      *reinterpret_cast<uint32_t *>(dst) = pk[0];
  }
  if (lane == 0) p.lse_out[lidx] = m + logf(L);
}

template <int D>
static void launch_d(const MergeParams &p, int part_dtype, int out_dtype, unsigned grid,
                     cudaStream_t s) {
  const bool in32 = part_dtype == ATTN_DTYPE_F32, out32 = out_dtype == ATTN_DTYPE_F32;
  if (in32 && out32) merge_kernel<D, float, true><<<grid, 256, 0, s>>>(p);
  if (in32 && !out32) merge_kernel<D, float, false><<<grid, 256, 0, s>>>(p);
  if (!in32 && out32) merge_kernel<D, uint16_t, true><<<grid, 256, 0, s>>>(p);
  if (!in32 && !out32) merge_kernel<D, uint16_t, false><<<grid, 256, 0, s>>>(p);
}

int merge_launch(const void *const *o_parts, const float *const *lse_parts, int n_parts,
                 int part_dtype, int s_len, int h, int d, void *out, int out_dtype, float *lse,
                 cudaStream_t s) {
  MergeParams p;
  for (int i = 0; i < ATTN_MERGE_MAX_PARTS; ++i) {
    p.o[i] = i < n_parts ? o_parts[i] : nullptr;
    p.lse[i] = i < n_parts ? lse_parts[i] : nullptr;
  }
  p.n = n_parts;
  p.S = s_len;
  p.H = h;
  p.out = out;
  p.lse_out = lse;
  const long long warps = static_cast<long long>(s_len) * h;
  if (warps == 0) return ATTN_OK;
  const unsigned grid = static_cast<unsigned>((warps * 32 + 255) / 256);
  if (d == 128)
    launch_d<128>(p, part_dtype, out_dtype, grid, s);
  else
    launch_d<64>(p, part_dtype, out_dtype, grid, s);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn
