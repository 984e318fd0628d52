// Step 1 of the MoE layer: router logits and top-k routing.
//
// router_logits_small / router_logits_tiled:  l = x W_r (+ bias) in fp32 SIMT
//   arithmetic ("Expert parallelism", step 1 "Route": compute the router).
// route_topk: one warp per token; top-k by iterated warp arg-max with the
//   order (value desc, expert asc), optional selection bias and group-limited
//   (node-limited) pre-selection ("What DeepSeek-V3 did about it"), then
//   softmax or (normalised) sigmoid gates.
#include <mutex>

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
// Router logits, E <= 16, fp32 SIMT.  Every lane keeps a COLS x EP block of W_r
// in registers (COLS = 64 / EP columns of d: column pairs 2L, 2L + 1 of each
// 64-column group of its warp, so that the warp's loads of W_r rows and its
// shared-memory reads of x are both contiguous); a warp covers 32 * COLS
// columns and a block of kRlWarps warps a column tile of 512 * COLS (4096
// columns at EP = 8).  The block's tokens stream through a
// ring of shared-memory stages filled by bulk copies (TB = 32 / EP token rows
// of one column tile per stage, 128 KB in flight), so the loads of later
// tokens overlap the arithmetic of earlier ones.  Per stage a lane holds
// TB * EP = 32 partial sums; a butterfly transpose-reduce over the warp (31
// shuffles) leaves lane L with the warp's sum for token L / EP, expert L % EP.
// Warp sums accumulate in shared memory, one slot per warp; the block adds the
// warps in index order at the end, so the result does not depend on timing.
// Waits are bounded (1 s): on time-out the block records
// MOE_E_DEVICE_TIMEOUT (when given a status word), drains its copies and
// writes nothing.
// ---------------------------------------------------------------------------
constexpr int kRlWarps = 16;
constexpr int kRlMaxTok = 64;               // tokens per block at most
constexpr uint32_t kRlRingBytes = 128 * 1024;
constexpr uint64_t kRlWaitNs = 1000000000ull;
constexpr uint64_t kRlDrainNs = 100000000ull;

template <int EP>
struct RlShape {
  static constexpr int COLS = 64 / EP;                   // columns of d per lane
  static constexpr int TB = 32 / EP;                     // tokens per stage
  static constexpr int SPAN = kRlWarps * 32 * COLS;      // columns per tile
  static constexpr uint32_t STAGE = TB * SPAN * 2;       // bytes per stage
  static constexpr int NS = int(kRlRingBytes / STAGE);   // stages
};

// one butterfly step over N values: lanes with bit o set keep the upper half
template <int N>
__device__ __forceinline__ void transpose_reduce_step(float (&v)[32], int lane, int o) {
  const bool up = (lane & o) != 0;
#pragma unroll
  for (int i = 0; i < N / 2; ++i) {
    const float send = up ? v[i] : v[i + N / 2];
    const float keep = up ? v[i + N / 2] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
  }
}

__device__ __forceinline__ bool rl_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                        int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*abort) return false;
      if (global_ns() - t0 > kRlWaitNs) {
        *abort = 1;
        if (status) report_status(status, MOE_E_DEVICE_TIMEOUT);
        return false;
      }
    }
  }
}

template <int EP>
__global__ void __launch_bounds__(kRlWarps * 32, 1) router_logits_small_kernel(
    const __nv_bfloat16* __restrict__ x, const float* __restrict__ W, const float* __restrict__ lbias,
    int T, int d, int E, int score_fn, int tpb, int* status, float* __restrict__ out) {
  using S = RlShape<EP>;
  constexpr int COLS = S::COLS, TB = S::TB, SPAN = S::SPAN, NS = S::NS;
  extern __shared__ __align__(128) uint8_t smem_rl[];
  uint8_t* ring = smem_rl;                                             // [NS][TB][SPAN] bf16
  float* part = reinterpret_cast<float*>(smem_rl + size_t(NS) * S::STAGE);  // [warps][tpb][EP]
  __shared__ uint64_t full[NS], empty[NS];
  __shared__ int abort_flag;
  volatile int* abort = &abort_flag;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t0 = blockIdx.x * tpb;
  const int n_tok = min(T - t0, tpb);
  const int n_b = (n_tok + TB - 1) / TB;   // stages per column tile
  const int n_j = n_b * ((d + SPAN - 1) / SPAN);
  float* mine = part + size_t(warp) * tpb * EP;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kRlWarps);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // stage j: column tile j / n_b, tokens (j % n_b) * TB .. + TB (thread 0 only)
  auto issue = [&](int j) {
    const int q = j % NS, ct = j / n_b, b = j - ct * n_b;
    const int rows = min(TB, n_tok - b * TB);
    const uint32_t bytes = uint32_t(min(SPAN, d - ct * SPAN)) * 2;
    mbar_arrive_expect_tx(&full[q], bytes * rows);
    for (int a = 0; a < rows; ++a)
      bulk_load_1d(ring + size_t(q) * S::STAGE + size_t(a) * SPAN * 2,
                   x + size_t(t0 + b * TB + a) * d + size_t(ct) * SPAN, bytes, &full[q]);
  };
  int issued = 0;
  if (threadIdx.x == 0)
    for (; issued < min(NS, n_j); ++issued) issue(issued);

  float2 w[COLS][EP / 2];  // expert pairs (e, e + 1), for packed fp32 FMAs
  int ct_w = -1;
  for (int j = 0; j < n_j; ++j) {
    const int q = j % NS, ct = j / n_b, b = j - ct * n_b;
    const uint32_t ph = uint32_t(j / NS) & 1u;
    // this warp's first column in the tile; d % 64 == 0, so each 64-column
    // group lies wholly inside or wholly past d.  Lane L takes columns
    // g + 2L and g + 2L + 1 of each group g = cw + 64 i, i < COLS / 2.
    const int cw = warp * 32 * COLS;
    if (ct != ct_w) {
#pragma unroll
      for (int i = 0; i < COLS / 2; ++i) {
        const int c = ct * SPAN + cw + 64 * i + 2 * lane;  // even column
        const bool in = c < d;
        if (E == EP) {
          // rows c, c + 1: 2 * EP consecutive floats
          const float4* src = reinterpret_cast<const float4*>(W + size_t(c) * EP);
#pragma unroll
          for (int v4 = 0; v4 < EP / 2; ++v4) {
            const float4 f = in ? __ldg(src + v4) : make_float4(0.f, 0.f, 0.f, 0.f);
            const int k = (4 * v4) / EP, e2 = ((4 * v4) % EP) / 2;
            w[2 * i + k][e2] = make_float2(f.x, f.y);
            w[2 * i + k][e2 + 1] = make_float2(f.z, f.w);
          }
        } else {
#pragma unroll
          for (int k = 0; k < 2; ++k)
#pragma unroll
            for (int e2 = 0; e2 < EP / 2; ++e2) {
              const int e = 2 * e2;
              w[2 * i + k][e2] =
                  make_float2((in && e < E) ? __ldg(W + size_t(c + k) * E + e) : 0.0f,
                              (in && e + 1 < E) ? __ldg(W + size_t(c + k) * E + e + 1) : 0.0f);
            }
        }
      }
      ct_w = ct;
    }
    const bool got = rl_wait(&full[q], ph, abort, status);
    if (!__all_sync(0xffffffffu, got)) break;
    // x words (bf16 pairs) of this lane's columns, token rows of the stage
    const uint32_t* stg =
        reinterpret_cast<const uint32_t*>(ring + size_t(q) * S::STAGE) + (cw >> 1) + lane;
    uint32_t xw[TB][COLS / 2];
#pragma unroll
    for (int a = 0; a < TB; ++a) {
      const bool row_in = b * TB + a < n_tok;
#pragma unroll
      for (int i = 0; i < COLS / 2; ++i) {
        const bool ok = row_in && ct * SPAN + cw + 64 * i < d;
        xw[a][i] = ok ? stg[a * (SPAN / 2) + 32 * i] : 0u;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[q]);
    float v[32];
#pragma unroll
    for (int a = 0; a < TB; ++a)
#pragma unroll
      for (int e2 = 0; e2 < EP / 2; ++e2) {
        float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int i = 0; i < COLS; ++i) {
          const float xf = (i & 1) ? bf16hi(xw[a][i >> 1]) : bf16lo(xw[a][i >> 1]);
          acc = __ffma2_rn(make_float2(xf, xf), w[i][e2], acc);  // two fmaf in one
        }
        v[a * EP + 2 * e2] = acc.x;
        v[a * EP + 2 * e2 + 1] = acc.y;
      }
    transpose_reduce_step<32>(v, lane, 16);
    transpose_reduce_step<16>(v, lane, 8);
    transpose_reduce_step<8>(v, lane, 4);
    transpose_reduce_step<4>(v, lane, 2);
    transpose_reduce_step<2>(v, lane, 1);
    {
      const int a = lane / EP, e = lane % EP;
      if (b * TB + a < n_tok) {
        float* slot = mine + (b * TB + a) * EP + e;
        *slot = ct == 0 ? v[0] : *slot + v[0];
      }
    }
    // refill this stage once every warp has read it
    if (warp == 0 && j + NS < n_j) {
      bool freed = true;
      if (lane == 0) {
        freed = rl_wait(&empty[q], ph, abort, status);
        if (freed) issue(issued++);
      }
      if (!__shfl_sync(0xffffffffu, freed ? 1 : 0, 0)) break;
    }
  }
  if (threadIdx.x == 0 && *abort) {
    // copies still in flight land before the block exits
    for (int k = max(0, issued - NS); k < issued; ++k)
      mbar_wait_bounded(&full[k % NS], uint32_t(k / NS) & 1u, kRlDrainNs);
  }
  __syncthreads();
  if (*abort) return;
  for (int i = threadIdx.x; i < n_tok * E; i += blockDim.x) {
    const int a = i / E, e = i - a * E;
    float l = 0.0f;
#pragma unroll
    for (int w2 = 0; w2 < kRlWarps; ++w2) l += part[(size_t(w2) * tpb + a) * EP + e];
    if (lbias) l += __ldg(lbias + e);
    if (score_fn == MOE_SIGMOID) l = 1.0f / (1.0f + expf(-l));
    out[size_t(t0 + a) * E + e] = l;
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
                         float* out, int* status, cudaStream_t st) {
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  if (c.E <= 16) {
    // tokens per block: the tokens spread over the SMs, whole stages, at most kRlMaxTok
    const int sms = device_sm_count();
    if (sms <= 0) return MOE_E_CUDA;
    const int ep = c.E <= 8 ? 8 : 16;
    const int tb = 32 / ep;
    int tpb = (c.T + sms - 1) / sms;
    tpb = (tpb + tb - 1) / tb * tb;
    if (tpb > kRlMaxTok) tpb = kRlMaxTok;
    const int blocks = (c.T + tpb - 1) / tpb;
    const size_t sm = kRlRingBytes + size_t(kRlWarps) * tpb * ep * 4;
    static PerDeviceOnce once;
    const int attr_rc = once.run([] {
      const int mx = int(kRlRingBytes + size_t(kRlWarps) * kRlMaxTok * 16 * 4);
      cudaError_t e = cudaFuncSetAttribute(router_logits_small_kernel<8>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(router_logits_small_kernel<16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
      if (e != cudaSuccess) cudaGetLastError();
      return e == cudaSuccess ? MOE_OK : MOE_E_CUDA;
    });
    if (attr_rc != MOE_OK) return attr_rc;
    if (ep == 8)
      router_logits_small_kernel<8><<<blocks, kRlWarps * 32, sm, st>>>(
          xb, W, lbias, c.T, c.d, c.E, c.score_fn, tpb, status, out);
    else
      router_logits_small_kernel<16><<<blocks, kRlWarps * 32, sm, st>>>(
          xb, W, lbias, c.T, c.d, c.E, c.score_fn, tpb, status, out);
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
