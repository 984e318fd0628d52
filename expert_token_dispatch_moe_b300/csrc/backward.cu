// Backward of the MoE layer with the routing held fixed ("Expert parallelism":
// the dispatch and the combine run "twice more in the backward pass").
//
//   step 7 backward (combine_backward_kernel): every kept assignment a of token
//     t receives d_o[row(a)] = gate[a] * dy[t] (a dispatch of dy into expert
//     order) and its gate receives dgate[a] = <dy[t], o[row(a)]>; the shared
//     expert's rows receive dy itself.
//   step 5 backward (the grouped GEMM kernel, launched from moe_api.cu):
//     g1 = x W13^T recomputed; dh = d_o W2 with the SwiGLU derivative fused
//     into its epilogue (-> dg1, packed like W13); dx_sorted = dg1 W13; the
//     weight gradients dW2 = d_o^T h and dW13 = dg1^T x reduce over each
//     expert's rows, read from transposed copies whose segments start on
//     64-column boundaries (transpose_segments_kernel, kpad_offsets_kernel).
//   step 2 backward: each token sums its rows' dx_sorted (the combine kernel
//     with unit gates).
#include "common.cuh"
#include "launch.h"

namespace moe {

// ---------------------------------------------------------------------------
// step 7 backward: one warp per token.  KT > 0 (k known at compile time): per
// pass a lane loads U vectors of dy once and the matching vectors of all k
// expert rows together, so about 8-16 loads are in flight per lane; KT == 0
// walks the k rows one after another.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 scale_dot_bf16x8(const uint4& dv, const uint4& ov, float g,
                                                  float& dot) {
  const uint32_t dw[4] = {dv.x, dv.y, dv.z, dv.w}, ow[4] = {ov.x, ov.y, ov.z, ov.w};
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float d0 = bf16lo(dw[i]), d1 = bf16hi(dw[i]);
    dot = fmaf(d0, bf16lo(ow[i]), dot);
    dot = fmaf(d1, bf16hi(ow[i]), dot);
    out[i] = pack_bf16x2(g * d0, g * d1);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

template <int KT>
__global__ void __launch_bounds__(256) combine_backward_kernel(
    const uint4* __restrict__ dy, const uint4* __restrict__ y_sorted,
    const int32_t* __restrict__ inv, const float* __restrict__ gate, int T, int k_rt, int vec,
    int R, int has_shared, uint4* __restrict__ d_o, float* __restrict__ dgate) {
  const int k = KT > 0 ? KT : k_rt;
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  const uint4* dyr = dy + size_t(t) * vec;
  uint4* shared_row = d_o + size_t(R + t) * vec;
  if constexpr (KT > 0) {
    const int my_row = (lane < KT) ? __ldg(inv + size_t(t) * KT + lane) : -1;
    const float my_g = (lane < KT) ? __ldg(gate + size_t(t) * KT + lane) : 0.0f;
    int rows[KT];
    float gs[KT], dot[KT];
#pragma unroll
    for (int j = 0; j < KT; ++j) {
      rows[j] = __shfl_sync(0xffffffffu, my_row, j);
      gs[j] = __shfl_sync(0xffffffffu, my_g, j);
      dot[j] = 0.0f;
    }
    constexpr int U = KT <= 1 ? 8 : (KT <= 2 ? 4 : (KT <= 4 ? 2 : 1));
    for (int v0 = lane; v0 < vec; v0 += 32 * U) {
      uint4 dv[U], ov[U][KT];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + 32 * u;
        if (v < vec) {
          dv[u] = __ldg(dyr + v);
#pragma unroll
          for (int j = 0; j < KT; ++j)
            if (rows[j] >= 0) ov[u][j] = __ldg(y_sorted + size_t(rows[j]) * vec + v);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + 32 * u;
        if (v >= vec) break;
#pragma unroll
        for (int j = 0; j < KT; ++j)
          if (rows[j] >= 0)
            d_o[size_t(rows[j]) * vec + v] = scale_dot_bf16x8(dv[u], ov[u][j], gs[j], dot[j]);
        if (has_shared) shared_row[v] = dv[u];
      }
    }
#pragma unroll
    for (int j = 0; j < KT; ++j) {
      float d = dot[j];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
      if (lane == 0) dgate[size_t(t) * KT + j] = rows[j] >= 0 ? d : 0.0f;
    }
  } else {
    for (int j = 0; j < k; ++j) {
      const int a = t * k + j;
      const int row = __ldg(inv + a);
      if (row < 0) {
        if (lane == 0) dgate[a] = 0.0f;
        continue;
      }
      const float g = __ldg(gate + a);
      const uint4* orow = y_sorted + size_t(row) * vec;
      uint4* drow = d_o + size_t(row) * vec;
      float dot = 0.0f;
      for (int v = lane; v < vec; v += 32) drow[v] = scale_dot_bf16x8(__ldg(dyr + v), __ldg(orow + v), g, dot);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
      if (lane == 0) dgate[a] = dot;
    }
    if (has_shared)
      for (int v = lane; v < vec; v += 32) shared_row[v] = __ldg(dyr + v);
  }
}

// ---------------------------------------------------------------------------
// padded segment offsets for the weight gradients (one warp)
// ---------------------------------------------------------------------------
// kpad_off[g] = sum over g' < g of roundup(kept rows of g', 64), g over the
// routed experts and then the shared expert (T rows).
__global__ void __launch_bounds__(32) kpad_offsets_kernel(const int32_t* __restrict__ counts,
                                                          int capacity, int E, int has_shared,
                                                          int T, int32_t* __restrict__ kpad_off) {
  const int lane = threadIdx.x;
  const int n = E + has_shared;
  int carry = 0;
  for (int base = 0; base < n; base += 32) {
    const int g = base + lane;
    int v = 0;
    if (g < E) {
      const int c = __ldg(counts + g);
      v = capacity ? min(c, capacity) : c;
    } else if (g < n) {
      v = T;
    }
    v = (v + 63) & ~63;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    if (g < n) kpad_off[g] = carry + incl - v;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) kpad_off[n] = carry;
}

// ---------------------------------------------------------------------------
// Transposes through 64 x 64 shared-memory tiles
// ---------------------------------------------------------------------------
constexpr int kTr = 64;

// One 64 x 64 tile: src rows [0, 64) (row i valid when i < n_valid, else
// zero), columns [c0, c0 + 64) -> dst row c0 + c, columns [dc0, dc0 + 64).
// The tile sits in shared memory as 32-bit words, 33 per row (one spare word
// spreads a column's rows over the banks); each thread then writes two
// destination rows (a pair of source columns) of 8 elements each.
__device__ __forceinline__ void transpose_tile(const __nv_bfloat16* __restrict__ src, size_t ld_src,
                                               int n_valid, int c0, __nv_bfloat16* __restrict__ dst,
                                               size_t ld_dst, size_t dc0, uint32_t* tile) {
  constexpr int P = kTr / 2 + 1;  // words per tile row
  for (int i = threadIdx.x; i < kTr * (kTr / 8); i += blockDim.x) {
    const int r = i / (kTr / 8), cv = i % (kTr / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < n_valid) v = __ldg(reinterpret_cast<const uint4*>(src + size_t(r) * ld_src + c0) + cv);
    uint32_t* w = tile + r * P + cv * 4;
    w[0] = v.x;
    w[1] = v.y;
    w[2] = v.z;
    w[3] = v.w;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < (kTr / 2) * (kTr / 8); i += blockDim.x) {
    const int rv = i % (kTr / 8), c2 = i / (kTr / 8);  // rows 8rv..8rv+7, columns 2c2, 2c2+1
    uint32_t lo[4], hi[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t a = tile[(rv * 8 + 2 * q) * P + c2];
      const uint32_t b = tile[(rv * 8 + 2 * q + 1) * P + c2];
      lo[q] = (a & 0xffffu) | (b << 16);          // column 2c2 of rows 2q, 2q+1
      hi[q] = (a >> 16) | (b & 0xffff0000u);      // column 2c2+1
    }
    *reinterpret_cast<uint4*>(dst + size_t(c0 + 2 * c2) * ld_dst + dc0 + rv * 8) =
        make_uint4(lo[0], lo[1], lo[2], lo[3]);
    *reinterpret_cast<uint4*>(dst + size_t(c0 + 2 * c2 + 1) * ld_dst + dc0 + rv * 8) =
        make_uint4(hi[0], hi[1], hi[2], hi[3]);
  }
  __syncthreads();
}

// The kept rows of every segment of src [rows, C] (experts at offsets[g]; the
// shared expert's T rows at src_shared) transposed into dst [C, ld_dst] at
// columns [kpad_off[g], kpad_off[g+1]), zero past the kept rows.
// grid.x: 64-column blocks of dst (up to the upper bound ld_dst / 64), grid.y:
// groups of kTrGroup 64-row blocks of C.  A CTA loads the next tile of its
// group while it writes out the current one.
constexpr int kTrGroup = 4;

__global__ void __launch_bounds__(256) transpose_segments_kernel(
    const __nv_bfloat16* __restrict__ src, const __nv_bfloat16* __restrict__ src_shared, int C,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ counts, int capacity, int E,
    int has_shared, int T, const int32_t* __restrict__ kpad_off, __nv_bfloat16* __restrict__ dst,
    size_t ld_dst) {
  __shared__ uint32_t tile[kTr * (kTr / 2 + 1)];
  constexpr int P = kTr / 2 + 1;
  const int n = E + has_shared;
  const int col = blockIdx.x * kTr;
  if (col >= __ldg(kpad_off + n)) return;
  int lo = 0, hi = n;  // segment g with kpad_off[g] <= col < kpad_off[g+1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(kpad_off + mid) <= col) lo = mid; else hi = mid;
  }
  const int g = lo;
  const int i0 = col - __ldg(kpad_off + g);
  int kept;
  const __nv_bfloat16* base;
  if (g < E) {
    const int c = __ldg(counts + g);
    kept = capacity ? min(c, capacity) : c;
    base = src + size_t(__ldg(offsets + g)) * C;
  } else {
    kept = T;
    base = src_shared;
  }
  base += size_t(i0) * C;
  const int n_valid = kept - i0;  // source rows of this column block that exist
  const int cb0 = blockIdx.y * kTrGroup, cb1 = min(C / kTr, cb0 + kTrGroup);
  // this thread's two 16-byte vectors of a 64 x 64 tile: (row r, vector cv)
  constexpr int PER = kTr * (kTr / 8) / 256;  // 2
  uint4 buf[PER];
  auto load = [&](int cb) {
#pragma unroll
    for (int q = 0; q < PER; ++q) {
      const int i = threadIdx.x + q * 256;
      const int r = i / (kTr / 8), cv = i % (kTr / 8);
      buf[q] = r < n_valid
                   ? __ldg(reinterpret_cast<const uint4*>(base + size_t(r) * C + cb * kTr) + cv)
                   : make_uint4(0, 0, 0, 0);
    }
  };
  load(cb0);
  for (int cb = cb0; cb < cb1; ++cb) {
#pragma unroll
    for (int q = 0; q < PER; ++q) {
      const int i = threadIdx.x + q * 256;
      const int r = i / (kTr / 8), cv = i % (kTr / 8);
      uint32_t* w = tile + r * P + cv * 4;
      w[0] = buf[q].x;
      w[1] = buf[q].y;
      w[2] = buf[q].z;
      w[3] = buf[q].w;
    }
    __syncthreads();
    if (cb + 1 < cb1) load(cb + 1);  // in flight during the write-out below
    const int c0 = cb * kTr;
    for (int i = threadIdx.x; i < (kTr / 2) * (kTr / 8); i += blockDim.x) {
      const int rv = i % (kTr / 8), c2 = i / (kTr / 8);  // rows 8rv..8rv+7, columns 2c2, 2c2+1
      uint32_t lo4[4], hi4[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t a = tile[(rv * 8 + 2 * q) * P + c2];
        const uint32_t b = tile[(rv * 8 + 2 * q + 1) * P + c2];
        lo4[q] = (a & 0xffffu) | (b << 16);      // column 2c2 of rows 2q, 2q+1
        hi4[q] = (a >> 16) | (b & 0xffff0000u);  // column 2c2+1
      }
      *reinterpret_cast<uint4*>(dst + size_t(c0 + 2 * c2) * ld_dst + col + rv * 8) =
          make_uint4(lo4[0], lo4[1], lo4[2], lo4[3]);
      *reinterpret_cast<uint4*>(dst + size_t(c0 + 2 * c2 + 1) * ld_dst + col + rv * 8) =
          make_uint4(hi4[0], hi4[1], hi4[2], hi4[3]);
    }
    __syncthreads();
  }
}

// Batched transpose of dense matrices: src [n][rows][cols] -> dst [n][cols][rows]
// (rows, cols multiples of 64).  grid: (cols/64, rows/64, n).
__global__ void __launch_bounds__(256) transpose_batched_kernel(const __nv_bfloat16* __restrict__ src,
                                                                int rows, int cols,
                                                                __nv_bfloat16* __restrict__ dst) {
  __shared__ uint32_t tile[kTr * (kTr / 2 + 1)];
  const size_t mat = size_t(rows) * cols * blockIdx.z;
  const int r0 = blockIdx.y * kTr, c0 = blockIdx.x * kTr;
  transpose_tile(src + mat + size_t(r0) * cols, cols, kTr, c0, dst + mat, rows, size_t(r0), tile);
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
int launch_combine_backward(const moe_cfg& c, const void* dy, const void* y_sorted,
                            const int32_t* inv, const float* gate, void* d_o, float* dgate,
                            cudaStream_t st) {
  const int R = c.capacity ? c.E * c.capacity : c.T * c.k;
  const uint4* dyv = static_cast<const uint4*>(dy);
  const uint4* ys = static_cast<const uint4*>(y_sorted);
  uint4* dov = static_cast<uint4*>(d_o);
  const int blocks = (c.T + 7) / 8, vec = c.d / 8;
#define MOE_CB(KTV) \
  combine_backward_kernel<KTV><<<blocks, 256, 0, st>>>(dyv, ys, inv, gate, c.T, c.k, vec, R, \
                                                      c.has_shared, dov, dgate)
  switch (c.k) {
    case 1: MOE_CB(1); break;
    case 2: MOE_CB(2); break;
    case 4: MOE_CB(4); break;
    case 8: MOE_CB(8); break;
    default: MOE_CB(0); break;
  }
#undef MOE_CB
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_E_CUDA;
}

int launch_pack_backward(const moe_cfg& c, const void* W13, const void* W2, void* W13t, void* W2t,
                         cudaStream_t st) {
  const int n = c.E + c.has_shared;
  // W13 [n, 2f, d] -> W13t [n, d, 2f];  W2 [n, d, f] -> W2t [n, f, d]
  transpose_batched_kernel<<<dim3(c.d / kTr, 2 * c.f / kTr, n), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(W13), 2 * c.f, c.d, static_cast<__nv_bfloat16*>(W13t));
  transpose_batched_kernel<<<dim3(c.f / kTr, c.d / kTr, n), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(W2), c.d, c.f, static_cast<__nv_bfloat16*>(W2t));
  note_launches(2);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_E_CUDA;
}

int launch_kpad_offsets(const moe_cfg& c, const int32_t* counts, int32_t* kpad_off,
                        cudaStream_t st) {
  kpad_offsets_kernel<<<1, 32, 0, st>>>(counts, c.capacity, c.E, c.has_shared, c.T, kpad_off);
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_E_CUDA;
}

int launch_transpose_segments(const moe_cfg& c, const void* src, const void* src_shared, int C,
                              const int32_t* offsets, const int32_t* counts,
                              const int32_t* kpad_off, void* dst, size_t ld_dst,
                              cudaStream_t st) {
  const dim3 grid(unsigned(ld_dst / kTr), unsigned((C / kTr + kTrGroup - 1) / kTrGroup));
  transpose_segments_kernel<<<grid, 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(src), static_cast<const __nv_bfloat16*>(src_shared), C,
      offsets, counts, c.capacity, c.E, c.has_shared, c.T, kpad_off,
      static_cast<__nv_bfloat16*>(dst), ld_dst);
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_E_CUDA;
}

}  // namespace moe
