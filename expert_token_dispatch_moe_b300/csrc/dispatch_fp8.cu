// FP8 dispatch: the receiver's dequantization into the expert-grouped buffer
// (the sender's quantization runs inside the EP layout kernel, permute.cu)
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
#include "common.cuh"
#include "launch.h"

namespace moe {

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
    // eight code vectors in flight per lane (a row of up to 4096 elements at
    // once), then their conversions.  Two other arrangements measured no
    // better: items of 512 codes strided over all warps, four in flight (0.48
    // against 0.50 of the copy peak on the Mixtral shape, 0.66 against 0.75 on
    // the skewed layer); and a one-wave grid whose warps resolve 32 slots'
    // indices at once and stream their rows through two register buffers
    // (Mixtral shape 28.5 against 27.4 us, DS-V3 284 against 297 us).
    constexpr int U = 8;
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
