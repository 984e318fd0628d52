// FP8 dispatch: the expert-parallel send buffer in e4m3 with one fp32 scale
// per row, and the receiver's dequantization into the expert-grouped buffer
// ("Expert parallelism", "A worked example at DeepSeek-V3's shape": DeepSeek-V3
// dispatches in FP8, s = 1 byte per element, and combines in BF16; "Lower
// precision on the wire": FP8 halves the dispatch bytes).
//
// The format and scale granularity are not fixed by that description; this
// library uses e4m3 (largest finite value 448) with one scale per row:
//   scale = absmax(row) / 448 (1 for an all-zero row)
//   code  = e4m3_rn_satfinite(x * (448 / absmax))
//   value = bf16_rn(float(code) * scale)
// Each factor is one correctly rounded fp32 division per row; each element one
// fp32 product and one hardware conversion, so the codes are reproducible
// bit for bit.
#include <cuda_fp8.h>

#include "common.cuh"
#include "launch.h"

namespace moe {

__device__ __forceinline__ uint32_t fp8x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

// One warp per token: absmax of x[t] (first pass), then the codes of the row
// (second pass, the row is re-read from L1/L2) written to each of the token's
// kept send slots, with the row's scale.
__global__ void __launch_bounds__(256) fp8_pack_kernel(const uint4* __restrict__ x, int T,
                                                       int vec_per_row, int k,
                                                       const int32_t* __restrict__ send_pos,
                                                       uint2* __restrict__ send_fp8,
                                                       float* __restrict__ send_scale) {
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  const uint4* src = x + size_t(t) * vec_per_row;
  float amax = 0.0f;
  constexpr int U = 4;  // vectors in flight per lane
  for (int v0 = lane; v0 < vec_per_row; v0 += 32 * U) {
    uint4 w[U];
#pragma unroll
    for (int q = 0; q < U; ++q)
      w[q] = (v0 + 32 * q < vec_per_row) ? __ldg(src + v0 + 32 * q) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int q = 0; q < U; ++q) {
      const uint32_t u[4] = {w[q].x, w[q].y, w[q].z, w[q].w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        amax = fmaxf(amax, fmaxf(fabsf(bf16lo(u[i])), fabsf(bf16hi(u[i]))));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float scale = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  const float inv = amax > 0.0f ? __fdiv_rn(448.0f, amax) : 1.0f;
  const int my_slot = (lane < k) ? __ldg(send_pos + size_t(t) * k + lane) : -1;
  if (lane < k && my_slot >= 0) send_scale[my_slot] = scale;
  for (int v0 = 0; v0 < vec_per_row; v0 += 32) {
    const int v = v0 + lane;
    uint2 code = make_uint2(0, 0);
    if (v < vec_per_row) {
      const uint4 w = __ldg(src + v);
      code.x = fp8x4(__fmul_rn(bf16lo(w.x), inv), __fmul_rn(bf16hi(w.x), inv),
                     __fmul_rn(bf16lo(w.y), inv), __fmul_rn(bf16hi(w.y), inv));
      code.y = fp8x4(__fmul_rn(bf16lo(w.z), inv), __fmul_rn(bf16hi(w.z), inv),
                     __fmul_rn(bf16lo(w.w), inv), __fmul_rn(bf16hi(w.w), inv));
    }
    for (int j = 0; j < k; ++j) {
      const int slot = __shfl_sync(0xffffffffu, my_slot, j);
      if (slot >= 0 && v < vec_per_row) send_fp8[size_t(slot) * vec_per_row + v] = code;
    }
  }
}

// Empty send slots (past a rank's kept rows): zero codes, scale 0.  One warp
// per slot, grid-stride.
__global__ void __launch_bounds__(256) fp8_pad_kernel(const int32_t* __restrict__ send_idx, int A,
                                                      int vec_per_row, uint2* __restrict__ send_fp8,
                                                      float* __restrict__ send_scale) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int p = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; p < A; p += warps) {
    if (__ldg(send_idx + p) >= 0) continue;
    if (lane == 0) send_scale[p] = 0.0f;
    uint2* row = send_fp8 + size_t(p) * vec_per_row;
    for (int v = lane; v < vec_per_row; v += 32) row[v] = make_uint2(0, 0);
  }
}

__device__ __forceinline__ uint32_t deq2(uint32_t codes2, float scale) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(__nv_fp8x2_storage_t(codes2), __NV_E4M3);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
  return pack_bf16x2(__fmul_rn(f.x, scale), __fmul_rn(f.y, scale));
}

// The receiver: slot p of the send buffers carries assignment a = send_idx[p],
// whose row in the expert-grouped buffer is inv[a]; write its dequantized row
// there.  One warp per slot, grid-stride.
__global__ void __launch_bounds__(256) fp8_recv_kernel(const uint4* __restrict__ send_fp8,
                                                       const float* __restrict__ send_scale,
                                                       const int32_t* __restrict__ send_idx,
                                                       const int32_t* __restrict__ inv, int A,
                                                       int vec16_per_row,
                                                       uint4* __restrict__ x_sorted) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int p = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; p < A; p += warps) {
    const int a = __ldg(send_idx + p);
    if (a < 0) continue;
    const int row = __ldg(inv + a);
    if (row < 0) continue;
    const float scale = __ldg(send_scale + p);
    const uint4* src = send_fp8 + size_t(p) * vec16_per_row;  // 16 codes per vector
    uint4* dst = x_sorted + size_t(row) * 2 * vec16_per_row;   // 8 bf16 per vector
    // four code vectors in flight per lane, then their conversions
    constexpr int U = 4;
    for (int v0 = lane; v0 < vec16_per_row; v0 += 32 * U) {
      uint4 c[U];
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (v0 + 32 * u < vec16_per_row) c[u] = __ldg(src + v0 + 32 * u);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + 32 * u;
        if (v >= vec16_per_row) break;
        uint4 o0, o1;
        o0.x = deq2(c[u].x & 0xffffu, scale);
        o0.y = deq2(c[u].x >> 16, scale);
        o0.z = deq2(c[u].y & 0xffffu, scale);
        o0.w = deq2(c[u].y >> 16, scale);
        o1.x = deq2(c[u].z & 0xffffu, scale);
        o1.y = deq2(c[u].z >> 16, scale);
        o1.z = deq2(c[u].w & 0xffffu, scale);
        o1.w = deq2(c[u].w >> 16, scale);
        dst[2 * v] = o0;
        dst[2 * v + 1] = o1;
      }
    }
  }
}

static int grid_rows(long long rows) {
  const long long want = (rows + 7) / 8;
  const long long cap = 8LL * device_sm_count();
  return int(want < cap ? (want > 0 ? want : 1) : cap);
}

int launch_fp8_pack(const moe_cfg& c, const void* x, const int32_t* send_idx, void* send_fp8,
                    float* send_scale, void* ws, cudaStream_t st) {
  const WsLayout L = ws_layout(c);
  const int A = c.T * c.k;
  const int32_t* send_pos = ws_ptr<int32_t>(ws, L.send_pos);
  fp8_pack_kernel<<<(c.T + 7) / 8, 256, 0, st>>>(static_cast<const uint4*>(x), c.T, c.d / 8, c.k,
                                                 send_pos, static_cast<uint2*>(send_fp8),
                                                 send_scale);
  note_launches(1);
  if (c.capacity) {
    fp8_pad_kernel<<<grid_rows(A), 256, 0, st>>>(send_idx, A, c.d / 8,
                                                 static_cast<uint2*>(send_fp8), send_scale);
    note_launches(1);
  }
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_E_CUDA;
}

int launch_fp8_recv(const moe_cfg& c, const void* send_fp8, const float* send_scale,
                    const int32_t* send_idx, const int32_t* inv, void* x_sorted,
                    cudaStream_t st) {
  const int A = c.T * c.k;
  fp8_recv_kernel<<<grid_rows(A), 256, 0, st>>>(static_cast<const uint4*>(send_fp8), send_scale,
                                                send_idx, inv, A, c.d / 16,
                                                static_cast<uint4*>(x_sorted));
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_E_CUDA;
}

}  // namespace moe
