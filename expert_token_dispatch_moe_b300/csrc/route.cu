// Step 1 of the MoE layer: router logits and top-k routing.
//
// router_logits_small / router_logits_tiled:  l = x W_r (+ bias) in fp32 SIMT
//   arithmetic ("Expert parallelism", step 1 "Route": compute the router).
// route_topk: one warp per token; top-k by iterated warp arg-max with the
//   order (value desc, expert asc), optional selection bias and group-limited
//   (node-limited) pre-selection ("What DeepSeek-V3 did about it"), then
//   softmax or (normalised) sigmoid gates.
#include "common.cuh"
#include "launch.h"

namespace moe {

// ---------------------------------------------------------------------------
// Order key of an fp32 value: larger value -> larger key; -0.0 and +0.0 give
// the same key; every NaN gets key 1, below -inf (whose key is 0x007FFFFF);
// key 0 is reserved for "not selectable".
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t order_key(float v) {
  if (v != v) return 1u;
  if (v == 0.0f) v = 0.0f;  // canonical +0
  uint32_t b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  if (k == 1u) return __uint_as_float(0x7fc00000u);  // NaN
  uint32_t b = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(b);
}

template <int EPL>
__global__ void __launch_bounds__(256) route_topk_kernel(
    const float* __restrict__ scores, const float* __restrict__ bias, int T, int E, int k,
    int score_fn, int norm_topk, int n_groups, int topk_groups, int32_t* __restrict__ topk_idx,
    float* __restrict__ topk_gate) {
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;  // uniform per warp
  const float* row = scores + size_t(t) * E;

  float s[EPL];
  uint32_t key[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane * EPL + i;
    if (e < E) {
      s[i] = __ldg(row + e);
      const float v = bias ? __fadd_rn(s[i], __ldg(bias + e)) : s[i];
      key[i] = order_key(v);
    } else {
      s[i] = 0.0f;
      key[i] = 0u;
    }
  }

  // Group-limited pre-selection: group score = top1 + top2 (one fp32 add).
  if (n_groups > 1) {
    const int gs = E / n_groups;
    uint32_t my_gkey = 0u;  // lane g holds group g's score key
    const int lpg = gs / EPL;  // lanes per group when groups are whole lanes
    if (gs % EPL == 0 && (lpg & (lpg - 1)) == 0) {
      // each lane's local top-2, then a reduction inside each aligned run of
      // lpg lanes (xor offsets below lpg never leave the run)
      uint32_t t1 = 0u, t2 = 0u;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const uint32_t kk = key[i];
        if (kk > t1) { t2 = t1; t1 = kk; } else if (kk > t2) { t2 = kk; }
      }
      for (int off = 1; off < lpg; off <<= 1) {
        const uint32_t o1 = __shfl_xor_sync(0xffffffffu, t1, off);
        const uint32_t o2 = __shfl_xor_sync(0xffffffffu, t2, off);
        const uint32_t hi = max(t1, o1), lo = min(t1, o1);
        t1 = hi;
        t2 = max(lo, max(t2, o2));
      }
      const float gsum = __fadd_rn(key_value(t1), key_value(t2));
      const uint32_t gk = order_key(gsum);
      const uint32_t from = __shfl_sync(0xffffffffu, gk, (lane * lpg) & 31);
      if (lane < n_groups) my_gkey = from;
    } else {
      for (int g = 0; g < n_groups; ++g) {
        uint32_t t1 = 0u, t2 = 0u;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
          const int e = lane * EPL + i;
          if (e < E && e / gs == g) {
            const uint32_t kk = key[i];
            if (kk > t1) { t2 = t1; t1 = kk; } else if (kk > t2) { t2 = kk; }
          }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          const uint32_t o1 = __shfl_xor_sync(0xffffffffu, t1, off);
          const uint32_t o2 = __shfl_xor_sync(0xffffffffu, t2, off);
          const uint32_t hi = max(t1, o1), lo = min(t1, o1);
          t1 = hi;
          t2 = max(lo, max(t2, o2));
        }
        const float gsum = __fadd_rn(key_value(t1), key_value(t2));
        if (lane == g) my_gkey = order_key(gsum);
      }
    }
    uint32_t kept = 0u;
    for (int r = 0; r < topk_groups; ++r) {
      const uint32_t kmax = __reduce_max_sync(0xffffffffu, my_gkey);
      const uint32_t cand = (my_gkey == kmax) ? uint32_t(lane) : 32u;
      const uint32_t g = __reduce_min_sync(0xffffffffu, cand);
      kept |= 1u << g;
      if (uint32_t(lane) == g) my_gkey = 0u;
    }
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane * EPL + i;
      if (e < E && !((kept >> (e / gs)) & 1u)) key[i] = 0u;
    }
  }

  // Top-k by iterated warp arg-max.
  int my_idx = 0;
  float my_s = 0.0f;
  for (int j = 0; j < k; ++j) {
    uint32_t bk = 0u;
    int bi = 0x7fffffff;
    float bs = 0.0f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      if (key[i] > bk) { bk = key[i]; bi = lane * EPL + i; bs = s[i]; }
    }
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
    const uint32_t cand = (bk == kmax) ? uint32_t(bi) : 0xffffffffu;
    const int win = int(__reduce_min_sync(0xffffffffu, cand));
    const int owner = win / EPL;
    const float ws = __shfl_sync(0xffffffffu, bs, owner);
    if (lane == owner) {
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (lane * EPL + i == win) key[i] = 0u;
    }
    if (lane == j) { my_idx = win; my_s = ws; }
  }

  // Gates.
  float g;
  if (score_fn == MOE_SOFTMAX) {
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (lane * EPL + i < E) m = fmaxf(m, s[i]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float z = 0.0f;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (lane * EPL + i < E) z += expf(s[i] - m);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    g = expf(my_s - m) / z;
  } else {
    g = my_s;
  }
  if (norm_topk) {
    float sum = (lane < k) ? g : 0.0f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    g = g / sum;
  }
  if (lane < k) {
    topk_idx[size_t(t) * k + lane] = my_idx;
    topk_gate[size_t(t) * k + lane] = g;
  }
}

// ---------------------------------------------------------------------------
// Router logits, E <= 16: each warp handles 4 tokens; W_r is staged through
// shared memory in pieces of 1024 rows (rows padded so that the 8 rows a lane
// reads start on distinct banks).
// ---------------------------------------------------------------------------
constexpr int kRlTok = 4;       // tokens per warp
constexpr int kRlPiece = 1024;  // W_r rows per shared-memory piece

template <int EP>
__global__ void __launch_bounds__(256) router_logits_small_kernel(
    const __nv_bfloat16* __restrict__ x, const float* __restrict__ W, const float* __restrict__ lbias,
    int T, int d, int E, int score_fn, float* __restrict__ out) {
  extern __shared__ float wsm[];  // kRlPiece rows, row r at r*EP + (r/8)*4
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t0 = (blockIdx.x * 8 + warp) * kRlTok;
  float acc[kRlTok][EP];
#pragma unroll
  for (int a = 0; a < kRlTok; ++a)
#pragma unroll
    for (int e = 0; e < EP; ++e) acc[a][e] = 0.0f;

  for (int p0 = 0; p0 < d; p0 += kRlPiece) {
    __syncthreads();
    for (int i = threadIdx.x; i < kRlPiece * EP; i += blockDim.x) {
      const int r = i / EP, e = i % EP;
      const int dr = p0 + r;
      wsm[r * EP + (r >> 3) * 4 + e] = (dr < d && e < E) ? __ldg(W + size_t(dr) * E + e) : 0.0f;
    }
    __syncthreads();
    for (int r0 = 0; r0 < kRlPiece; r0 += 256) {
      const int dcol = p0 + r0 + lane * 8;
      if (dcol >= d) break;  // d % 8 == 0: a lane's 8 values are all in or all out
      uint4 xv[kRlTok];
#pragma unroll
      for (int a = 0; a < kRlTok; ++a) {
        const int t = t0 + a;
        xv[a] = (t < T) ? __ldg(reinterpret_cast<const uint4*>(x + size_t(t) * d + dcol))
                        : make_uint4(0, 0, 0, 0);
      }
      const float* wr = wsm + (r0 + lane * 8) * EP + ((r0 + lane * 8) >> 3) * 4;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float w[EP];
#pragma unroll
        for (int e = 0; e < EP; e += 4) {
          const float4 q = *reinterpret_cast<const float4*>(wr + i * EP + e);
          w[e] = q.x; w[e + 1] = q.y; w[e + 2] = q.z; w[e + 3] = q.w;
        }
#pragma unroll
        for (int a = 0; a < kRlTok; ++a) {
          const uint32_t word = (&xv[a].x)[i >> 1];
          const float xf = (i & 1) ? bf16hi(word) : bf16lo(word);
#pragma unroll
          for (int e = 0; e < EP; ++e) acc[a][e] = fmaf(xf, w[e], acc[a][e]);
        }
      }
    }
  }
#pragma unroll
  for (int a = 0; a < kRlTok; ++a)
#pragma unroll
    for (int e = 0; e < EP; ++e) {
      float v = acc[a][e];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      acc[a][e] = v;
    }
  if (lane < kRlTok) {
    const int t = t0 + lane;
    if (t < T) {
#pragma unroll
      for (int a = 0; a < kRlTok; ++a) {
        if (a != lane) continue;
#pragma unroll
        for (int e = 0; e < EP; ++e) {
          if (e >= E) break;
          float l = acc[a][e];
          if (lbias) l += __ldg(lbias + e);
          if (score_fn == MOE_SIGMOID) l = 1.0f / (1.0f + expf(-l));
          out[size_t(t) * E + e] = l;
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Router logits, E > 16: 64 x 64 output tiles, 4 x 4 per thread, K step 16.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) router_logits_tiled_kernel(
    const __nv_bfloat16* __restrict__ x, const float* __restrict__ W, const float* __restrict__ lbias,
    int T, int d, int E, int score_fn, float* __restrict__ out) {
  __shared__ __align__(16) float As[16][64 + 4];  // [k][token]
  __shared__ __align__(16) float Bs[16][64 + 4];  // [k][expert]
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.x * 64, n0 = blockIdx.y * 64;
  float acc[4][4] = {};
  // loader roles
  const int xr = threadIdx.x >> 2, xc = (threadIdx.x & 3) * 4;  // x tile: 64 rows x 16 cols
  const int wr = threadIdx.x >> 4, wc = (threadIdx.x & 15) * 4; // W tile: 16 rows x 64 cols
  for (int k0 = 0; k0 < d; k0 += 16) {
    {
      const int t = m0 + xr;
      uint2 v = make_uint2(0, 0);
      if (t < T) v = __ldg(reinterpret_cast<const uint2*>(x + size_t(t) * d + k0 + xc));
      As[xc + 0][xr] = bf16lo(v.x);
      As[xc + 1][xr] = bf16hi(v.x);
      As[xc + 2][xr] = bf16lo(v.y);
      As[xc + 3][xr] = bf16hi(v.y);
      const float* wp = W + size_t(k0 + wr) * E + n0 + wc;
#pragma unroll
      for (int j = 0; j < 4; ++j) Bs[wr][wc + j] = (n0 + wc + j < E) ? __ldg(wp + j) : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      const float4 b = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = m0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = n0 + tx * 4 + j;
      if (e >= E) continue;
      float l = acc[i][j];
      if (lbias) l += __ldg(lbias + e);
      if (score_fn == MOE_SIGMOID) l = 1.0f / (1.0f + expf(-l));
      out[size_t(t) * E + e] = l;
    }
  }
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
int launch_router_logits(const moe_cfg& c, const void* x, const float* W, const float* lbias,
                         float* out, cudaStream_t st) {
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  if (c.E <= 16) {
    const int blocks = (c.T + 8 * kRlTok - 1) / (8 * kRlTok);
    if (c.E <= 8) {
      const size_t sm = size_t(kRlPiece) * 8 * 4 + (kRlPiece / 8) * 16;
      router_logits_small_kernel<8><<<blocks, 256, sm, st>>>(xb, W, lbias, c.T, c.d, c.E,
                                                             c.score_fn, out);
    } else {
      const size_t sm = size_t(kRlPiece) * 16 * 4 + (kRlPiece / 8) * 16;
      static bool attr = false;
      if (!attr) {
        cudaFuncSetAttribute(router_logits_small_kernel<16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, int(sm));
        attr = true;
      }
      router_logits_small_kernel<16><<<blocks, 256, sm, st>>>(xb, W, lbias, c.T, c.d, c.E,
                                                              c.score_fn, out);
    }
  } else {
    dim3 grid((c.T + 63) / 64, (c.E + 63) / 64);
    router_logits_tiled_kernel<<<grid, 256, 0, st>>>(xb, W, lbias, c.T, c.d, c.E, c.score_fn, out);
  }
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_E_CUDA;
}

int launch_route(const moe_cfg& c, const float* scores, const float* bias, int32_t* idx,
                 float* gate, cudaStream_t st) {
  const int blocks = (c.T + 7) / 8;
#define MOE_ROUTE(EPL)                                                                   \
  route_topk_kernel<EPL><<<blocks, 256, 0, st>>>(scores, bias, c.T, c.E, c.k, c.score_fn, \
                                                  c.norm_topk, c.n_groups, c.topk_groups, idx, gate)
  if (c.E <= 32) MOE_ROUTE(1);
  else if (c.E <= 64) MOE_ROUTE(2);
  else if (c.E <= 128) MOE_ROUTE(4);
  else if (c.E <= 256) MOE_ROUTE(8);
  else if (c.E <= 512) MOE_ROUTE(16);
  else MOE_ROUTE(32);
#undef MOE_ROUTE
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_E_CUDA;
}

}  // namespace moe
