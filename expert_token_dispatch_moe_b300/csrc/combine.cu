// Step 7 of the MoE layer: unpermute, gate and combine ("Expert parallelism",
// step 7: undo the sort and scatter-add each row into its token with its
// gate).  The scatter-add is computed as a gather per token: one warp per
// token reads its k expert rows (16-byte vectors), accumulates gate * row in
// fp32 in slot order j = 0..k-1, adds the shared expert's row, and writes the
// bf16 result once.  Same sum as the scatter-add, with no atomics and a fixed
// order, so the output is deterministic.
#include "common.cuh"
#include "launch.h"

namespace moe {

__device__ __forceinline__ void fma_bf16x8(float (&acc)[8], const uint4& v, float g) {
  acc[0] = fmaf(g, bf16lo(v.x), acc[0]);
  acc[1] = fmaf(g, bf16hi(v.x), acc[1]);
  acc[2] = fmaf(g, bf16lo(v.y), acc[2]);
  acc[3] = fmaf(g, bf16hi(v.y), acc[3]);
  acc[4] = fmaf(g, bf16lo(v.z), acc[4]);
  acc[5] = fmaf(g, bf16hi(v.z), acc[5]);
  acc[6] = fmaf(g, bf16lo(v.w), acc[6]);
  acc[7] = fmaf(g, bf16hi(v.w), acc[7]);
}

// KT > 0: k known at compile time (loads of all k rows issued together),
// U vectors per lane per pass.
template <int KT, int U>
__global__ void __launch_bounds__(256) combine_kernel(const uint4* __restrict__ y_sorted,
                                                      const int32_t* __restrict__ inv,
                                                      const float* __restrict__ gate, int T,
                                                      int k_rt, int vec, int R, int has_shared,
                                                      uint4* __restrict__ y) {
  const int k = KT > 0 ? KT : k_rt;
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  const int my_row = (lane < k) ? __ldg(inv + size_t(t) * k + lane) : -1;
  // gate == nullptr: unit gates (the permute's backward sums the rows)
  const float my_g = (lane < k) ? (gate ? __ldg(gate + size_t(t) * k + lane) : 1.0f) : 0.0f;
  const uint4* shared_row = y_sorted + size_t(R + t) * vec;
  if (KT > 0) {
    int rows[KT > 0 ? KT : 1];
    float gs[KT > 0 ? KT : 1];
#pragma unroll
    for (int j = 0; j < KT; ++j) {
      rows[j] = __shfl_sync(0xffffffffu, my_row, j);
      gs[j] = __shfl_sync(0xffffffffu, my_g, j);
    }
    for (int v0 = lane; v0 < vec; v0 += 32 * U) {
      uint4 val[U][KT > 0 ? KT : 1];
      uint4 sv[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + 32 * u;
        if (v < vec) {
#pragma unroll
          for (int j = 0; j < KT; ++j)
            if (rows[j] >= 0) val[u][j] = __ldg(y_sorted + size_t(rows[j]) * vec + v);
          if (has_shared) sv[u] = __ldg(shared_row + v);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + 32 * u;
        if (v >= vec) break;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < KT; ++j)
          if (rows[j] >= 0) fma_bf16x8(acc, val[u][j], gs[j]);
        if (has_shared) fma_bf16x8(acc, sv[u], 1.0f);
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        y[size_t(t) * vec + v] = o;
      }
    }
  } else {
    // warp-uniform trip count: every lane takes part in the broadcasts
    for (int v0 = 0; v0 < vec; v0 += 32) {
      const int v = v0 + lane;
      const bool active = v < vec;
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int j = 0; j < k; ++j) {
        const int row = __shfl_sync(0xffffffffu, my_row, j);
        const float g = __shfl_sync(0xffffffffu, my_g, j);
        if (row >= 0 && active) fma_bf16x8(acc, __ldg(y_sorted + size_t(row) * vec + v), g);
      }
      if (!active) continue;
      if (has_shared) fma_bf16x8(acc, __ldg(shared_row + v), 1.0f);
      uint4 o;
      o.x = pack_bf16x2(acc[0], acc[1]);
      o.y = pack_bf16x2(acc[2], acc[3]);
      o.z = pack_bf16x2(acc[4], acc[5]);
      o.w = pack_bf16x2(acc[6], acc[7]);
      y[size_t(t) * vec + v] = o;
    }
  }
}

int launch_combine(const moe_cfg& c, const void* y_sorted, const int32_t* inv, const float* gate,
                   void* y, cudaStream_t st) {
  const int R = c.capacity ? c.E * c.capacity : c.T * c.k;
  const int vec = c.d / 8;
  const int blocks = (c.T + 7) / 8;
  const uint4* ys = static_cast<const uint4*>(y_sorted);
  uint4* out = static_cast<uint4*>(y);
  // row loads in flight per lane: 16 for rows longer than 256 vectors (a
  // Mixtral-shaped token's two 8 KB rows in two passes: 18.5 against 21.5 us),
  // 8 for shorter rows (more warps per SM: the skewed layer's combine ran 25
  // against 27 us with 8 than with 16)
  const bool long_rows = vec > 256;
#define MOE_COMBINE(K_, UL_, US_)                                                          \
  do {                                                                                     \
    if (long_rows)                                                                         \
      combine_kernel<K_, UL_><<<blocks, 256, 0, st>>>(ys, inv, gate, c.T, c.k, vec, R,     \
                                                    c.has_shared, out);                    \
    else                                                                                   \
      combine_kernel<K_, US_><<<blocks, 256, 0, st>>>(ys, inv, gate, c.T, c.k, vec, R,     \
                                                    c.has_shared, out);                    \
  } while (0)
  switch (c.k) {
    case 1: MOE_COMBINE(1, 16, 8); break;
    case 2: MOE_COMBINE(2, 8, 4); break;
    case 4: MOE_COMBINE(4, 4, 2); break;
    case 8: MOE_COMBINE(8, 2, 1); break;
    default:
      combine_kernel<0, 1><<<blocks, 256, 0, st>>>(ys, inv, gate, c.T, c.k, vec, R, c.has_shared,
                                                   out);
      break;
  }
#undef MOE_COMBINE
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_E_CUDA;
}

}  // namespace moe
