// Step 5 of the MoE layer: the experts as one grouped product ("Expert
// parallelism" page, "Token permutation and grouped GEMMs": one kernel that
// receives the list of problem sizes and schedules the output tiles of all
// experts across the GPU; SwiGLU experts with three d x d_e matrices).
//
// Persistent tcgen05 kernel, one CTA per SM, 192 threads:
//   warp 0      TMA producer: 128x64 A tiles and 256x64 B tiles (bf16,
//               128-byte swizzle) into a 4-stage shared-memory ring
//   warp 1      MMA issuer (one thread): tcgen05.mma kind::f16, M=128 N=256
//               K=16, fp32 accumulators in tensor memory (two 256-column
//               buffers, so the epilogue of one tile overlaps the next).
//               A segment's last M block with at most 64 valid rows is a
//               half tile: 64-row A loads and M=64 MMAs (same issue time as
//               M=128 but half the tensor work, which matters when the clock
//               is held down by the power limit).
//   warps 2-5   epilogue: tcgen05.ld of the accumulator, SwiGLU (GEMM 1) or
//               plain conversion (GEMM 2), bf16 stores of the valid rows
// Tiles come from a device-side schedule built from the expert counts and
// offsets (no host sync): segment g (expert, or the shared expert last) has
// ceil(rows_g/128) x ceil(N/256) tiles, numbered expert-major, then by N
// block, then by M block, so CTAs running at the same time share weight tiles
// through L2.  Rows past a segment's end are computed but never stored.
// Every wait is bounded (1 s); on time-out the CTA records
// MOE_E_DEVICE_TIMEOUT, stops issuing work, drains its copies and MMAs, frees
// tensor memory and returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace moe {
namespace gg {
constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr uint32_t A_BYTES = BM * BK * 2;
constexpr uint32_t B_BYTES = BN * BK * 2;
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr int MAX_SEG = 1025;
constexpr uint64_t WAIT_NS = 1000000000ull;
constexpr uint64_t DRAIN_NS = 100000000ull;
constexpr size_t DYN_SMEM = size_t(STAGES) * STAGE_BYTES + 1024;
}  // namespace gg

enum { kEpiSwiglu = 0, kEpiBf16 = 1, kEpiF32 = 2 };

struct GroupedParams {
  const int32_t* counts;  // nullptr: one dense segment of dense_rows rows at row 0
  const int32_t* offsets;
  int E, capacity, has_shared, T, R;
  int dense_rows;
  int K;                  // reduction length of one pass
  int k_passes;           // passes over K: A re-read each pass, B advanced by b_pass_rows
  int b_pass_rows;
  int N;                  // weight rows per expert (output columns before SwiGLU)
  int mode;               // kEpiSwiglu: out[:, j] = silu(acc[:, gate j]) * acc[:, up j]
                          // kEpiBf16:   out = bf16(acc)
                          // kEpiF32:    out_f32 = acc + col_bias (sigmoid if set), fp32
  int shared_a_separate;  // 1: shared expert's A rows come from tmA_sh from row 0
  __nv_bfloat16* out;
  float* out_f32;
  const float* col_bias;
  int sigmoid;
  int ld_out;
  int* status;
};

struct GroupedCtl {
  uint64_t full[gg::STAGES];
  uint64_t empty[gg::STAGES];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t done;
  uint32_t tmem_base;
  volatile int abort;
  int warp_sum[8];
  int tile_start[gg::MAX_SEG + 1];
};

__device__ __forceinline__ void segment(const GroupedParams& p, int g, int& rows, int& a_row0,
                                        int& out_row0) {
  if (p.counts == nullptr) {
    rows = p.dense_rows;
    a_row0 = 0;
    out_row0 = 0;
  } else if (g < p.E) {
    const int c = __ldg(p.counts + g);
    rows = p.capacity ? min(c, p.capacity) : c;
    a_row0 = __ldg(p.offsets + g);
    out_row0 = a_row0;
  } else {
    rows = p.T;
    a_row0 = p.shared_a_separate ? 0 : p.R;
    out_row0 = p.R;
  }
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, GroupedCtl& ctl,
                                              int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (ctl.abort) return false;
      if (global_ns() - t0 > gg::WAIT_NS) {
        ctl.abort = 1;
        report_status(status, MOE_E_DEVICE_TIMEOUT);
        return false;
      }
    }
  }
}

// tmA / tmA_sh: 128-row A boxes; tmA64 / tmA_sh64: the same tensors with 64-row
// boxes for half tiles.
__global__ void __launch_bounds__(gg::THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmA_sh,
                        const __grid_constant__ CUtensorMap tmA64,
                        const __grid_constant__ CUtensorMap tmA_sh64,
                        const __grid_constant__ CUtensorMap tmB, const GroupedParams p) {
  using namespace gg;
  extern __shared__ uint8_t dyn_smem[];
  __shared__ GroupedCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) &
                                             ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_seg = p.counts ? p.E + p.has_shared : 1;
  const int n_blocks_n = (p.N + BN - 1) / BN;
  const int kb_per_pass = p.K / BK;
  const int num_kb = kb_per_pass * p.k_passes;

  // ---- device-side tile schedule: exclusive prefix of tiles per segment ----
  {
    const int per = (n_seg + THREADS - 1) / THREADS;
    const int g0 = tid * per;
    int local = 0;
    for (int i = 0; i < per; ++i) {
      const int g = g0 + i;
      if (g < n_seg) {
        int rows, ar, orow;
        segment(p, g, rows, ar, orow);
        local += ((rows + BM - 1) / BM) * n_blocks_n;
      }
    }
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    if (lane == 31) ctl.warp_sum[warp] = incl;
    if (tid == 0) {
      for (int s = 0; s < STAGES; ++s) {
        mbar_init(&ctl.full[s], 1);
        mbar_init(&ctl.empty[s], 1);
      }
      for (int b = 0; b < 2; ++b) {
        mbar_init(&ctl.acc_full[b], 1);
        mbar_init(&ctl.acc_empty[b], 128);
      }
      mbar_init(&ctl.done, 1);
      ctl.abort = 0;
      fence_mbar_init();
    }
    __syncthreads();
    int run = incl - local;
    for (int w = 0; w < warp; ++w) run += ctl.warp_sum[w];
    for (int i = 0; i < per; ++i) {
      const int g = g0 + i;
      if (g < n_seg) {
        ctl.tile_start[g] = run;
        int rows, ar, orow;
        segment(p, g, rows, ar, orow);
        run += ((rows + BM - 1) / BM) * n_blocks_n;
      }
    }
    if (g0 < n_seg && g0 + per >= n_seg) ctl.tile_start[n_seg] = run;
  }
  if (warp == 1) {
    tmem_alloc(&ctl.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmA_sh);
    tma_prefetch_desc(&tmA64);
    tma_prefetch_desc(&tmA_sh64);
    tma_prefetch_desc(&tmB);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl.tmem_base;
  const int total = ctl.tile_start[n_seg];

  auto decode = [&](int t, int& g, int& m_blk, int& n_blk, int& rows, int& a_row0,
                    int& out_row0) {
    int lo = 0, hi = n_seg;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (ctl.tile_start[mid] <= t) lo = mid; else hi = mid;
    }
    g = lo;
    segment(p, g, rows, a_row0, out_row0);
    const int m_tiles = max((rows + BM - 1) / BM, 1);
    const int local = t - ctl.tile_start[g];
    n_blk = local / m_tiles;
    m_blk = local - n_blk * m_tiles;
  };
  // a half tile: the segment's last M block holds at most 64 valid rows
  auto is_half = [&](int rows, int m_blk) { return rows - m_blk * BM <= BM / 2; };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      uint32_t stage = 0, phase = 0;
      uint32_t issued = 0, last_phase = 0;  // per-stage bit masks
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        int g, m_blk, n_blk, rows, a_row0, out_row0;
        decode(t, g, m_blk, n_blk, rows, a_row0, out_row0);
        const bool sep = p.counts && g >= p.E && p.shared_a_separate;
        const bool half = is_half(rows, m_blk);
        const CUtensorMap* ma = half ? (sep ? &tmA_sh64 : &tmA64) : (sep ? &tmA_sh : &tmA);
        const uint32_t tx = half ? A_BYTES / 2 + B_BYTES : STAGE_BYTES;
        const int a_row = a_row0 + m_blk * BM;
        const int b_row = g * p.N + n_blk * BN;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wait_or_abort(&ctl.empty[stage], phase ^ 1u, ctl, p.status)) { ok = false; break; }
          uint8_t* sa = smem + stage * STAGE_BYTES;
          uint8_t* sb = sa + A_BYTES;
          const int pass = kb / kb_per_pass;
          const int ka = (kb - pass * kb_per_pass) * BK;
          mbar_arrive_expect_tx(&ctl.full[stage], tx);
          tma_load_2d(sa, ma, ka, a_row, &ctl.full[stage]);
          tma_load_2d(sb, &tmB, ka, b_row + pass * p.b_pass_rows, &ctl.full[stage]);
          issued |= 1u << stage;
          last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (ok && !ctl.abort) {
        // every stage released by the MMA warp: all its commits have landed
        for (int i = 0; i < STAGES; ++i) {
          if (!wait_or_abort(&ctl.empty[stage], phase ^ 1u, ctl, p.status)) break;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      } else {
        // aborted: wait (bounded) for the copies still in flight
        for (int s = 0; s < STAGES; ++s)
          if (issued & (1u << s))
            mbar_wait_bounded(&ctl.full[s], (last_phase >> s) & 1u, DRAIN_NS);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        int g, m_blk, n_blk, rows, a_row0, out_row0;
        decode(t, g, m_blk, n_blk, rows, a_row0, out_row0);
        const uint32_t idesc = is_half(rows, m_blk) ? idesc_bf16_f32(BM / 2, BN)
                                                    : idesc_bf16_f32(BM, BN);
        if (!wait_or_abort(&ctl.acc_empty[acc], acc_phase ^ 1u, ctl, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wait_or_abort(&ctl.full[stage], phase, ctl, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint8_t* sa = smem + stage * STAGE_BYTES;
          const uint64_t a_desc = smem_desc_k128(sa);
          const uint64_t b_desc = smem_desc_k128(sa + A_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            umma_bf16(d_tmem, a_desc + 2 * kk, b_desc + 2 * kk, idesc, (kb | kk) != 0);
          umma_commit(&ctl.empty[stage]);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit(&ctl.acc_full[acc]);
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      // all MMAs issued by this thread have completed before tensor memory is freed
      umma_commit(&ctl.done);
      mbar_wait_bounded(&ctl.done, 0, DRAIN_NS);
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    // Warp w may access tensor-memory lanes [32*(w%4), 32*(w%4)+32).  An M=128
    // accumulator keeps row r in lane r; an M=64 accumulator keeps rows
    // 16q..16q+15 in lanes 32q..32q+15.
    const int quarter = warp & 3;
    uint32_t acc = 0, acc_phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      int g, m_blk, n_blk, rows, a_row0, out_row0;
      decode(t, g, m_blk, n_blk, rows, a_row0, out_row0);
      if (!wait_or_abort(&ctl.acc_full[acc], acc_phase, ctl, p.status)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + acc * BN + (uint32_t(quarter * 32) << 16);
      const bool half = is_half(rows, m_blk);
      const int r = m_blk * BM + (half ? quarter * 16 + lane : quarter * 32 + lane);
      const bool valid = (!half || lane < 16) && r < rows;
      const size_t orow_idx = size_t(out_row0 + (valid ? r : 0)) * p.ld_out;
      __nv_bfloat16* orow = p.out + orow_idx;
      if (p.mode == kEpiF32) {
        const int col0 = n_blk * BN;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t v[32];
          tmem_ld32(taddr + c, v);
          tmem_ld_wait();
          if (valid && col0 + c < p.N) {
            float* dst = p.out_f32 + orow_idx + col0 + c;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int col = col0 + c + i;
              if (col < p.N) {
                float l = __uint_as_float(v[i]);
                if (p.col_bias) l += __ldg(p.col_bias + col);
                if (p.sigmoid) l = 1.0f / (1.0f + expf(-l));
                dst[i] = l;
              }
            }
          }
        }
      } else if (p.mode == kEpiSwiglu) {
        const int col0 = n_blk * (BN / 2);
#pragma unroll 1
        for (int c = 0; c < BN / 2; c += 32) {
          uint32_t gv[32], uv[32];
          tmem_ld32(taddr + c, gv);
          tmem_ld32(taddr + BN / 2 + c, uv);
          tmem_ld_wait();
          if (valid) {
            uint32_t packed[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float g0 = __uint_as_float(gv[2 * i]), g1 = __uint_as_float(gv[2 * i + 1]);
              const float u0 = __uint_as_float(uv[2 * i]), u1 = __uint_as_float(uv[2 * i + 1]);
              const float h0 = g0 / (1.0f + __expf(-g0)) * u0;
              const float h1 = g1 / (1.0f + __expf(-g1)) * u1;
              packed[i] = pack_bf16x2(h0, h1);
            }
            uint4* dst = reinterpret_cast<uint4*>(orow + col0 + c);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
          }
        }
      } else {
        const int col0 = n_blk * BN;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t v[32];
          tmem_ld32(taddr + c, v);
          tmem_ld_wait();
          if (valid && col0 + c < p.N) {
            uint32_t packed[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              packed[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
            uint4* dst = reinterpret_cast<uint4*>(orow + col0 + c);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&ctl.acc_empty[acc]);
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// One-time weight packing: interleave 128-row blocks of W1 and W3.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) pack_w13_kernel(const uint4* __restrict__ W1,
                                                       const uint4* __restrict__ W3, int n_exp,
                                                       int f, int vec, uint4* __restrict__ W13) {
  const int lane = threadIdx.x & 31;
  const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (row >= (long long)n_exp * 2 * f) return;
  const int e = int(row / (2 * f));
  const int r = int(row % (2 * f));
  const int b = r / 256, i = r % 256;
  const uint4* src = (i < 128) ? W1 + (size_t(e) * f + b * 128 + i) * vec
                               : W3 + (size_t(e) * f + b * 128 + (i - 128)) * vec;
  uint4* dst = W13 + size_t(row) * vec;
  for (int v = lane; v < vec; v += 32) dst[v] = __ldg(src + v);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;

static bool get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// 2-D bf16 row-major [rows, cols] tensor, box = 64 columns x box_rows rows,
// 128-byte swizzle, out-of-bounds elements read as zero.
static bool make_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols,
                     uint32_t box_rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int set_smem_attr() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(grouped_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               int(gg::DYN_SMEM));
  });
  return err == cudaSuccess ? MOE_OK : MOE_E_CUDA;
}

static int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

int launch_pack_w13(const moe_cfg& c, const void* W1, const void* W3, void* W13, cudaStream_t st) {
  const int n_exp = c.E + c.has_shared;
  const long long rows = (long long)n_exp * 2 * c.f;
  const long long blocks = (rows + 7) / 8;
  pack_w13_kernel<<<unsigned(blocks), 256, 0, st>>>(static_cast<const uint4*>(W1),
                                                    static_cast<const uint4*>(W3), n_exp, c.f,
                                                    c.d / 8, static_cast<uint4*>(W13));
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_E_CUDA;
}

// Router logits on the tensor cores: x [T, d] (bf16) times the three bf16
// terms of W_r (W_r = hi + mid + lo exactly, stored [3][E][d]), accumulated in
// fp32 in tensor memory over 3 passes of K, + logit bias, sigmoid if asked.
int launch_router_tc(const moe_cfg& c, const void* x, const void* W_split, const float* lbias,
                     float* out, int* status, cudaStream_t st) {
  using namespace gg;
  if (!get_encoder()) return MOE_E_CUDA;
  if (set_smem_attr() != MOE_OK) return MOE_E_CUDA;
  CUtensorMap mA, mA64, mB;
  if (!make_map(&mA, x, uint64_t(c.T), c.d, BM)) return MOE_E_CUDA;
  if (!make_map(&mA64, x, uint64_t(c.T), c.d, BM / 2)) return MOE_E_CUDA;
  if (!make_map(&mB, W_split, uint64_t(3) * c.E, c.d, BN)) return MOE_E_CUDA;
  const int sms = sm_count();
  if (sms <= 0) return MOE_E_CUDA;
  GroupedParams p{};
  p.counts = nullptr;
  p.dense_rows = c.T;
  p.K = c.d;
  p.k_passes = 3;
  p.b_pass_rows = c.E;
  p.N = c.E;
  p.mode = kEpiF32;
  p.out_f32 = out;
  p.col_bias = lbias;
  p.sigmoid = c.score_fn == MOE_SIGMOID;
  p.ld_out = c.E;
  p.status = status;
  const long long tiles = (long long)((c.T + BM - 1) / BM) * ((c.E + BN - 1) / BN);
  const int grid = int(tiles < sms ? tiles : sms);
  grouped_gemm_kernel<<<grid, THREADS, DYN_SMEM, st>>>(mA, mA, mA64, mA64, mB, p);
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_E_CUDA;
}

// Exact three-term bf16 split of the fp32 router weights, transposed to
// K-major: out[s][e][i] for W_r[i][e] = hi + mid + lo.
__global__ void __launch_bounds__(256) pack_router_kernel(const float* __restrict__ W, int d, int E,
                                                          __nv_bfloat16* __restrict__ out) {
  const long long n = (long long)d * E;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < n;
       idx += (long long)gridDim.x * blockDim.x) {
    const int i = int(idx / E), e = int(idx % E);
    const float w = W[idx];
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
    const size_t o = size_t(e) * d + i;
    out[o] = hi;
    out[size_t(E) * d + o] = mid;
    out[size_t(2) * E * d + o] = lo;
  }
}

int launch_pack_router(const moe_cfg& c, const float* W, void* out, cudaStream_t st) {
  const long long n = (long long)c.d * c.E;
  const int blocks = int((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  pack_router_kernel<<<blocks, 256, 0, st>>>(W, c.d, c.E, static_cast<__nv_bfloat16*>(out));
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_E_CUDA;
}

int launch_grouped_ffn(const moe_cfg& c, const void* x_sorted, const void* x,
                       const int32_t* counts, const int32_t* offsets, const void* W13,
                       const void* W2, void* h, void* y_sorted, void* ws, cudaStream_t st) {
  using namespace gg;
  if (!get_encoder()) return MOE_E_CUDA;
  if (set_smem_attr() != MOE_OK) return MOE_E_CUDA;
  const WsLayout L = ws_layout(c);
  const int R = c.capacity ? c.E * c.capacity : c.T * c.k;
  const int n_exp = c.E + c.has_shared;
  const uint64_t rows_h = uint64_t(R) + (c.has_shared ? c.T : 0);

  CUtensorMap mA1, mA1s, mA1h, mA1sh, mB1, mA2, mA2h, mB2;
  const void* a1s = c.has_shared ? x : x_sorted;
  const uint64_t a1s_rows = c.has_shared ? uint64_t(c.T) : uint64_t(R);
  if (!make_map(&mA1, x_sorted, uint64_t(R), c.d, BM)) return MOE_E_CUDA;
  if (!make_map(&mA1h, x_sorted, uint64_t(R), c.d, BM / 2)) return MOE_E_CUDA;
  if (!make_map(&mA1s, a1s, a1s_rows, c.d, BM)) return MOE_E_CUDA;
  if (!make_map(&mA1sh, a1s, a1s_rows, c.d, BM / 2)) return MOE_E_CUDA;
  if (!make_map(&mB1, W13, uint64_t(n_exp) * 2 * c.f, c.d, BN)) return MOE_E_CUDA;
  if (!make_map(&mA2, h, rows_h, c.f, BM)) return MOE_E_CUDA;
  if (!make_map(&mA2h, h, rows_h, c.f, BM / 2)) return MOE_E_CUDA;
  if (!make_map(&mB2, W2, uint64_t(n_exp) * c.d, c.f, BN)) return MOE_E_CUDA;

  // grid: at most one CTA per SM, no more than an upper bound on the tiles
  const int sms = sm_count();
  if (sms <= 0) return MOE_E_CUDA;
  const long long mt_ub = rows_h / BM + n_exp + 1;

  GroupedParams p1{};
  p1.counts = counts;
  p1.offsets = offsets;
  p1.E = c.E;
  p1.capacity = c.capacity;
  p1.has_shared = c.has_shared;
  p1.T = c.T;
  p1.R = R;
  p1.K = c.d;
  p1.N = 2 * c.f;
  p1.k_passes = 1;
  p1.mode = kEpiSwiglu;
  p1.shared_a_separate = 1;
  p1.out = static_cast<__nv_bfloat16*>(h);
  p1.ld_out = c.f;
  p1.status = ws_ptr<int>(ws, L.status);
  const long long t1 = mt_ub * ((p1.N + BN - 1) / BN);
  const int grid1 = int(t1 < sms ? t1 : sms);
  grouped_gemm_kernel<<<grid1, THREADS, DYN_SMEM, st>>>(mA1, mA1s, mA1h, mA1sh, mB1, p1);

  GroupedParams p2 = p1;
  p2.K = c.f;
  p2.N = c.d;
  p2.mode = kEpiBf16;
  p2.shared_a_separate = 0;
  p2.out = static_cast<__nv_bfloat16*>(y_sorted);
  p2.ld_out = c.d;
  const long long t2 = mt_ub * ((p2.N + BN - 1) / BN);
  const int grid2 = int(t2 < sms ? t2 : sms);
  grouped_gemm_kernel<<<grid2, THREADS, DYN_SMEM, st>>>(mA2, mA2, mA2h, mA2h, mB2, p2);
  note_launches(2);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_E_CUDA;
}

}  // namespace moe
