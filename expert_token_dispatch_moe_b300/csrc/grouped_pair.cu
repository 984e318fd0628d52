// Step 5 of the MoE layer on SM pairs: the forward expert FFN as one grouped
// product per GEMM ("Expert parallelism" page, "Token permutation and grouped
// GEMMs": one kernel schedules the output tiles of every expert).
//
// Each tile is computed transposed, out^T = W * X^T: the expert's weight rows
// are the MMA's M side and the segment's token rows its N side.  A tile is
// 256 weight rows by up to 256 tokens, run by a cluster of two CTAs on two SMs
// with one tcgen05.mma.cta_group::2 (M = 256): each CTA stages 128 of the
// weight rows and half of the token rows, and keeps its 128 weight rows by all
// the tile's tokens in its own tensor memory.  Two things follow:
//   * the MMA's N is the tile's token count rounded up to 16, so the ragged
//     end of a segment costs about its own rows instead of a whole 128-row tile
//     (a DeepSeek-V3-shaped layer has 256 +- 20 rows per expert);
//   * each SM stages 32 KB per 64-deep k-block (16 KB of weights, 16 KB of
//     tokens) for the same tensor work as a one-SM 128 x 256 tile that stages
//     48 KB, so a 6-stage ring holds 50 % more k-blocks in flight.
//
// 192 threads per CTA:
//   warp 0    TMA producer (both CTAs): the CTA's weight rows and token rows
//             into its own ring; every copy counts on the leader CTA's "full"
//             barrier
//   warp 1    the leader CTA's MMA issuer (one thread): 4 MMAs (K = 16) per
//             k-block into one of two 256-column accumulators; commits release
//             the ring stage and the accumulator in both CTAs.  Warp 1 of both
//             CTAs allocates and frees the pair's tensor memory.
//   warps 2-5 epilogue (both CTAs): tcgen05.ld of the CTA's accumulator rows,
//             SwiGLU (GEMM 1) or conversion (GEMM 2), bf16 stores of the
//             tile's valid tokens; each warp then signals the leader.
// GEMM 1 takes each CTA's 128 rows of W13 as two 64-row boxes: the gate rows
// of 64 hidden columns, then their up rows (each TMA instruction costs the
// SM's copy engine about 40 cycles, so 16-row pieces cost more than the
// bytes).  Epilogue warps then hold gate (tensor-memory lanes 0-63) or up
// (lanes 64-127) pre-activations; warps with lanes 0-31 and 64-95, and with
// 32-63 and 96-127, trade half of each 32-token chunk through shared memory,
// and each activates its half.  Each CTA stages its token rows with one box
// whose height is a power of two, the tile's MMA N being twice that.
//
// Tiles come from a device-side schedule built from the expert counts and
// offsets (no host sync): segment g (expert, or the shared expert last) has
// ceil(rows/256) token blocks for each weight block, numbered expert-major,
// then by weight block, then by token block, so pairs running at the same time
// share a weight block through L2.  Every wait is bounded (1 s); on time-out
// the CTA records MOE_E_DEVICE_TIMEOUT and stops issuing work; both CTAs meet
// at a cluster barrier before the pair frees its tensor memory and exits.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"

namespace moe {
namespace gp {
constexpr int BW = 128;   // weight rows per CTA (M = 256 per pair)
constexpr int BT = 256;   // tokens per tile at most (the MMA's N)
constexpr int BK = 64;
constexpr int STAGES = 6;
constexpr uint32_t A_BYTES = BW * BK * 2;        // 16 KB of weight rows
constexpr uint32_t B_BYTES = (BT / 2) * BK * 2;  // 16 KB of token rows (half the tile's)
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr int MAX_SEG = 1025;
constexpr int NBOX = 5;   // token boxes of 128, 64, 32, 16 and 8 rows
constexpr uint64_t WAIT_NS = 1000000000ull;
constexpr uint64_t DRAIN_NS = 100000000ull;
// GEMM 1's epilogue exchange: per warp pair, two buffers of gate values and
// two of up values, 32 lanes x 16 fp32 each (row pitch 17 words: lane-wise
// writes and reads hit distinct banks)
constexpr int XPITCH = 17;
constexpr uint32_t XBUF_BYTES = 32 * XPITCH * 4;
constexpr uint32_t XCHG_BYTES = 2 * 2 * 2 * XBUF_BYTES;  // 2 pairs x 2 buffers x (gate, up)
constexpr size_t DYN_SMEM = size_t(STAGES) * STAGE_BYTES + XCHG_BYTES + 1024;
}  // namespace gp

struct PairMaps {
  CUtensorMap w;               // weights: 16-row boxes (GEMM 1) or 128-row boxes (GEMM 2)
  CUtensorMap tok[gp::NBOX];   // token rows of the grouped buffer, boxes of 128 .. 8 rows
  CUtensorMap tok_sh[gp::NBOX];  // the shared expert's token rows when they sit apart
};

struct PairParams {
  const int32_t* counts;
  const int32_t* offsets;
  int E, capacity, has_shared, T, R;
  int K;                 // reduction length
  int n_wblk;            // weight blocks per segment
  int w_rows;            // weight rows per segment in the weight tensor (2f or d)
  int swiglu;            // 1: GEMM 1 (gate/up pieces, SwiGLU epilogue); 0: plain bf16
  int n_out;             // output columns (f for GEMM 1, d for GEMM 2)
  int shared_tok_apart;  // 1: the shared expert's token rows are tok_sh from row 0
  __nv_bfloat16* out;
  int ld_out;
  int* status;
};

struct PairCtl {
  uint64_t full[gp::STAGES];   // leader only: both CTAs' copies of a stage
  uint64_t empty[gp::STAGES];  // both: the MMAs reading a stage have completed
  uint64_t acc_full[2];        // both: an accumulator holds a finished tile
  uint64_t acc_empty[2];       // leader only: 8 epilogue warps have read it
  uint64_t done;               // leader only: every MMA has completed
  uint32_t tmem_base;
  volatile int abort;
  int warp_sum[8];
  int tile_start[gp::MAX_SEG + 1];
};

__device__ __forceinline__ void pair_segment(const PairParams& p, int g, int& rows, int& tok_row0,
                                             int& out_row0) {
  if (g < p.E) {
    const int c = __ldg(p.counts + g);
    rows = p.capacity ? min(c, p.capacity) : c;
    tok_row0 = __ldg(p.offsets + g);
    out_row0 = tok_row0;
  } else {
    rows = p.T;
    tok_row0 = p.shared_tok_apart ? 0 : p.R;
    out_row0 = p.R;
  }
}

__device__ __forceinline__ bool pair_wait(uint64_t* bar, uint32_t parity, PairCtl& ctl,
                                          int* status) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (ctl.abort) return false;
      if (global_ns() - t0 > gp::WAIT_NS) {
        ctl.abort = 1;
        report_status(status, MOE_E_DEVICE_TIMEOUT);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// GEMM 1 epilogue of one chunk of W token columns (W = 32 or 16) at column c0.
// This warp holds the gate (gate = true) or up pre-activations of hidden
// column j for the chunk; its partner warp holds the other.  The gate warp
// activates the first W/2 tokens and the up warp the rest: each writes the
// half it does not activate to its buffer, both meet at a named barrier, and
// each reads the partner's half.  Neighbouring lanes then pair their columns
// into 4-byte stores.
template <int W>
__device__ __forceinline__ void epi_swiglu(const uint32_t* v, int lane, bool gate, int j, int c0,
                                           int n_valid, float* mine, const float* theirs,
                                           uint32_t bar_id, __nv_bfloat16* out_rows,
                                           int ld_out) {
  constexpr int H = W / 2;
#pragma unroll
  for (int m = 0; m < H; ++m) mine[lane * gp::XPITCH + m] = __uint_as_float(gate ? v[H + m] : v[m]);
  named_barrier(bar_id, 64);
  float hv[H];
#pragma unroll
  for (int m = 0; m < H; ++m) {
    const float r = theirs[lane * gp::XPITCH + m];
    const float g = gate ? __uint_as_float(v[m]) : r;
    const float u = gate ? r : __uint_as_float(v[H + m]);
    hv[m] = g / (1.0f + __expf(-g)) * u;
  }
  const bool odd = lane & 1;
  const int tbase = c0 + (gate ? 0 : H);
#pragma unroll
  for (int m = 0; m < H; m += 2) {
    const float send = odd ? hv[m] : hv[m + 1];
    const float r = __shfl_xor_sync(0xffffffffu, send, 1);
    const int tok = tbase + m + (odd ? 1 : 0);
    const float lo = odd ? r : hv[m];
    const float hi = odd ? hv[m + 1] : r;
    if (tok < n_valid)
      *reinterpret_cast<uint32_t*>(out_rows + size_t(tok) * ld_out + (odd ? j - 1 : j)) =
          pack_bf16x2(lo, hi);
  }
}

// The same for GEMM 2: lane i holds output column col for the chunk's tokens.
template <int W>
__device__ __forceinline__ void epi_plain(const uint32_t* v, int lane, int col, int c0,
                                          int n_valid, bool col_ok, __nv_bfloat16* out_rows,
                                          int ld_out) {
  const bool odd = lane & 1;
#pragma unroll
  for (int m = 0; m < W; m += 2) {
    const float a = __uint_as_float(v[m]), b = __uint_as_float(v[m + 1]);
    const float r = __shfl_xor_sync(0xffffffffu, odd ? a : b, 1);
    const int tok = c0 + m + (odd ? 1 : 0);
    const float lo = odd ? r : a;
    const float hi = odd ? b : r;
    if (col_ok && tok < n_valid)
      *reinterpret_cast<uint32_t*>(out_rows + size_t(tok) * ld_out + (odd ? col - 1 : col)) =
          pack_bf16x2(lo, hi);
  }
}

// Token box of a tile with n_valid tokens: index i of the 128 >> i rows each
// CTA stages, the smallest power of two (at least 8) holding half the tokens.
__device__ __forceinline__ int token_box(int n_valid) {
  const int need = (n_valid + 1) >> 1;
  int i = 0;
  while (i < gp::NBOX - 1 && (128 >> (i + 1)) >= need) ++i;
  return i;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(gp::THREADS, 1)
    grouped_pair_kernel(const __grid_constant__ PairMaps maps, const PairParams p) {
  using namespace gp;
  extern __shared__ uint8_t dyn_smem[];
  __shared__ PairCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) &
                                             ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();  // 0: the leader, which issues the MMAs
  const int pair = int(cluster_id_x()), n_pairs = int(cluster_count_x());
  const int n_seg = p.E + p.has_shared;

  // ---- device-side tile schedule: exclusive prefix of tiles per segment ----
  {
    const int per = (n_seg + THREADS - 1) / THREADS;
    const int g0 = tid * per;
    int local = 0;
    for (int i = 0; i < per; ++i) {
      const int g = g0 + i;
      if (g < n_seg) {
        int rows, tr, orow;
        pair_segment(p, g, rows, tr, orow);
        local += ((rows + BT - 1) / BT) * p.n_wblk;
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
        mbar_init(&ctl.acc_empty[b], 8);
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
        int rows, tr, orow;
        pair_segment(p, g, rows, tr, orow);
        run += ((rows + BT - 1) / BT) * p.n_wblk;
      }
    }
    if (g0 < n_seg && g0 + per >= n_seg) ctl.tile_start[n_seg] = run;
  }
  if (warp == 1) {
    tmem_alloc_pair(&ctl.tmem_base, TMEM_COLS);
    tmem_relinquish_pair();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.w);
    for (int i = 0; i < NBOX; ++i) {
      tma_prefetch_desc(&maps.tok[i]);
      if (p.shared_tok_apart) tma_prefetch_desc(&maps.tok_sh[i]);
    }
  }
  // barriers initialised and tensor memory allocated in both CTAs
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = ctl.tmem_base;
  const int total = ctl.tile_start[n_seg];
  const int num_kb = p.K / BK;

  // tile t -> segment g, weight block wb, token block tb
  auto decode = [&](int t, int& g, int& wb, int& tb, int& rows, int& tok_row0, int& out_row0) {
    int lo = 0, hi = n_seg;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (ctl.tile_start[mid] <= t) lo = mid; else hi = mid;
    }
    g = lo;
    pair_segment(p, g, rows, tok_row0, out_row0);
    const int nt = max((rows + BT - 1) / BT, 1);
    const int local = t - ctl.tile_start[g];
    wb = local / nt;
    tb = local - wb * nt;
  };

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    // Lane 0 waits for a free stage (and, in the leader, arms the stage's
    // barrier with both CTAs' bytes); lanes 0-7 copy the weight pieces, lanes
    // 8-12 the token boxes.
    const uint32_t full0 = map_to_rank(smem_u32(&ctl.full[0]), 0);
    uint32_t stage = 0, phase = 0;
    uint32_t issued = 0, last_phase = 0;  // leader's per-stage masks, for the drain
    bool ok = true;
    for (int t = pair; t < total && ok; t += n_pairs) {
      int g, wb, tb, rows, tok_row0, out_row0;
      decode(t, g, wb, tb, rows, tok_row0, out_row0);
      const int n_valid = min(BT, rows - tb * BT);
      const int bi = token_box(n_valid);
      const int half = 128 >> bi;                     // token rows this CTA stages
      const int tok0 = tok_row0 + tb * BT + int(rank) * half;
      const CUtensorMap* tmap = ((g >= p.E && p.shared_tok_apart) ? maps.tok_sh : maps.tok) + bi;
      const uint32_t tx = 2u * (A_BYTES + uint32_t(half) * BK * 2);
      const int wrow = g * p.w_rows + wb * 2 * BW + int(rank) * (p.swiglu ? BW / 2 : BW);
      for (int kb = 0; kb < num_kb; ++kb) {
        if (lane == 0) ok = pair_wait(&ctl.empty[stage], phase ^ 1u, ctl, p.status);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        uint8_t* sa = smem + stage * STAGE_BYTES;
        const int ka = kb * BK;
        const uint32_t bar = full0 + stage * 8u;
        if (rank == 0 && lane == 0) {
          mbar_arrive_expect_tx(&ctl.full[stage], tx);
          issued |= 1u << stage;
          last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
        }
        if (p.swiglu) {
          // 64 gate rows, then the 64 matching up rows
          if (lane < 2)
            tma_load_2d_pair(sa + lane * (BW / 2) * (BK * 2), &maps.w, ka, wrow + lane * BW, bar);
        } else if (lane == 0) {
          tma_load_2d_pair(sa, &maps.w, ka, wrow, bar);
        }
        if (lane == 2) tma_load_2d_pair(sa + A_BYTES, tmap, ka, tok0, bar);
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (lane == 0) {
      if (ok && !ctl.abort) {
        // every stage released by the MMAs: all of this CTA's copies were consumed
        for (int i = 0; i < STAGES; ++i) {
          if (!pair_wait(&ctl.empty[stage], phase ^ 1u, ctl, p.status)) break;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      } else if (rank == 0) {
        // aborted: wait (bounded) for the copies still in flight
        for (int s = 0; s < STAGES; ++s)
          if (issued & (1u << s))
            mbar_wait_bounded(&ctl.full[s], (last_phase >> s) & 1u, DRAIN_NS);
      }
    }
  } else if (warp == 1) {
    if (rank == 0 && lane == 0) {
      // ---------------- MMA issuer (leader CTA) ----------------
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int t = pair; t < total && ok; t += n_pairs) {
        int g, wb, tb, rows, tok_row0, out_row0;
        decode(t, g, wb, tb, rows, tok_row0, out_row0);
        const int n_valid = min(BT, rows - tb * BT);
        const int ntile = 2 * (128 >> token_box(n_valid));
        const uint32_t idesc = idesc_bf16_f32(2 * BW, ntile);
        if (!pair_wait(&ctl.acc_empty[acc], acc_phase ^ 1u, ctl, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BT;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!pair_wait(&ctl.full[stage], phase, ctl, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint8_t* sa = smem + stage * STAGE_BYTES;
          const uint64_t a_desc = smem_desc_k128(sa);
          const uint64_t b_desc = smem_desc_k128(sa + A_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            umma_bf16_pair(d_tmem, a_desc + 2 * kk, b_desc + 2 * kk, idesc, (kb | kk) != 0);
          umma_commit_pair_mc(&ctl.empty[stage], 0x3);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit_pair_mc(&ctl.acc_full[acc], 0x3);
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      // every MMA issued here has completed before tensor memory is freed
      umma_commit_pair(&ctl.done);
      mbar_wait_bounded(&ctl.done, 0, DRAIN_NS);
    }
  } else {
    // ---------------- epilogue (warps 2..5 of both CTAs) ----------------
    // Warp w reads tensor-memory lanes [32*(w%4), 32*(w%4)+32): this CTA's
    // weight rows, by the tile's token columns.
    const int quarter = warp & 3;
    const uint32_t acc_empty0 = map_to_rank(smem_u32(&ctl.acc_empty[0]), 0);
    // GEMM 1: quarters 0/2 and 1/3 are the gate/up warps of hidden columns
    // j0 + lane and j0 + 32 + lane
    const bool gate = quarter < 2;
    const int pi = quarter & 1;
    float* xchg = reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES) +
                  pi * 4 * (XBUF_BYTES / 4);
    uint32_t chunk = 0;
    uint32_t acc = 0, acc_phase = 0;
    for (int t = pair; t < total; t += n_pairs) {
      int g, wb, tb, rows, tok_row0, out_row0;
      decode(t, g, wb, tb, rows, tok_row0, out_row0);
      const int n_valid = min(BT, rows - tb * BT);
      if (!pair_wait(&ctl.acc_full[acc], acc_phase, ctl, p.status)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + acc * BT + (uint32_t(quarter * 32) << 16);
      __nv_bfloat16* out_rows = p.out + size_t(out_row0 + tb * BT) * p.ld_out;
      if (p.swiglu) {
        const int j = wb * BW + int(rank) * (BW / 2) + pi * 32 + lane;
#pragma unroll 1
        for (int c0 = 0; c0 < n_valid; c0 += 32, ++chunk) {
          // buffers of this chunk: [chunk parity][gate writes | up writes]
          float* base = xchg + (chunk & 1) * 2 * (XBUF_BYTES / 4);
          float* mine = base + (gate ? 0 : XBUF_BYTES / 4);
          const float* theirs = base + (gate ? XBUF_BYTES / 4 : 0);
          if (n_valid - c0 > 16) {
            uint32_t v[32];
            tmem_ld32(taddr + c0, v);
            tmem_ld_wait();
            epi_swiglu<32>(v, lane, gate, j, c0, n_valid, mine, theirs, 1 + pi, out_rows,
                           p.ld_out);
          } else {
            uint32_t v[16];
            tmem_ld16(taddr + c0, v);
            tmem_ld_wait();
            epi_swiglu<16>(v, lane, gate, j, c0, n_valid, mine, theirs, 1 + pi, out_rows,
                           p.ld_out);
          }
        }
      } else {
        const int col = wb * 2 * BW + int(rank) * BW + quarter * 32 + lane;
        const bool col_ok = (col | 1) < p.n_out;
#pragma unroll 1
        for (int c0 = 0; c0 < n_valid; c0 += 32) {
          if (n_valid - c0 > 16) {
            uint32_t v[32];
            tmem_ld32(taddr + c0, v);
            tmem_ld_wait();
            epi_plain<32>(v, lane, col, c0, n_valid, col_ok, out_rows, p.ld_out);
          } else {
            uint32_t v[16];
            tmem_ld16(taddr + c0, v);
            tmem_ld_wait();
            epi_plain<16>(v, lane, col, c0, n_valid, col_ok, out_rows, p.ld_out);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc_empty0 + acc * 8u);
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  // both CTAs: MMAs complete, accumulators read, remote arrivals done
  __syncwarp();
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static int pair_set_attr() {
  static PerDeviceOnce once;
  return once.run([] {
    const cudaError_t e = cudaFuncSetAttribute(
        grouped_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(gp::DYN_SMEM));
    if (e != cudaSuccess) cudaGetLastError();
    return e == cudaSuccess ? MOE_OK : MOE_E_CUDA;
  });
}

// Clusters of two that can run at once (cached per device).
static int pair_max_clusters() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 0;
  }
  if (cache[dev] == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 74, 1, 1);
    cfg.blockDim = dim3(gp::THREADS, 1, 1);
    cfg.dynamicSmemBytes = gp::DYN_SMEM;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, grouped_pair_kernel, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = device_sm_count() / 2;
    }
    cache[dev] = n;
  }
  return cache[dev];
}

static bool make_token_maps(CUtensorMap (&m)[gp::NBOX], const void* ptr, uint64_t rows,
                            uint64_t cols) {
  for (int i = 0; i < gp::NBOX; ++i)
    if (!make_bf16_map(&m[i], ptr, rows, cols, uint32_t(128 >> i))) return false;
  return true;
}

static int launch_pair(const PairMaps& maps, const PairParams& p, long long tiles_ub,
                       cudaStream_t st) {
  const int clusters = pair_max_clusters();
  if (clusters <= 0) return MOE_E_CUDA;
  const long long n = tiles_ub < clusters ? (tiles_ub > 0 ? tiles_ub : 1) : clusters;
  grouped_pair_kernel<<<unsigned(2 * n), gp::THREADS, gp::DYN_SMEM, st>>>(maps, p);
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_E_CUDA;
}

int launch_grouped_ffn_pair(const moe_cfg& c, const void* x_sorted, const void* x,
                            const int32_t* counts, const int32_t* offsets, const void* W13,
                            const void* W2, void* h, void* y_sorted, int* status,
                            cudaStream_t st) {
  using namespace gp;
  if (pair_set_attr() != MOE_OK) return MOE_E_CUDA;
  const int R = c.capacity ? c.E * c.capacity : c.T * c.k;
  const int n_exp = c.E + c.has_shared;
  const uint64_t rows_h = uint64_t(R) + (c.has_shared ? c.T : 0);
  const long long seg_ub = (long long)rows_h / BT + n_exp + 1;

  PairMaps m1, m2;
  if (!make_bf16_map(&m1.w, W13, uint64_t(n_exp) * 2 * c.f, c.d, 64)) return MOE_E_CUDA;
  if (!make_token_maps(m1.tok, x_sorted, uint64_t(R), c.d)) return MOE_E_CUDA;
  if (c.has_shared) {
    if (!make_token_maps(m1.tok_sh, x, uint64_t(c.T), c.d)) return MOE_E_CUDA;
  } else {
    for (int i = 0; i < NBOX; ++i) m1.tok_sh[i] = m1.tok[i];
  }
  PairParams p1{};
  p1.counts = counts;
  p1.offsets = offsets;
  p1.E = c.E;
  p1.capacity = c.capacity;
  p1.has_shared = c.has_shared;
  p1.T = c.T;
  p1.R = R;
  p1.K = c.d;
  p1.n_wblk = c.f / BW;          // 128 hidden columns (256 rows of W13) per block
  p1.w_rows = 2 * c.f;
  p1.swiglu = 1;
  p1.n_out = c.f;
  p1.shared_tok_apart = c.has_shared;
  p1.out = static_cast<__nv_bfloat16*>(h);
  p1.ld_out = c.f;
  p1.status = status;
  const int rc = launch_pair(m1, p1, seg_ub * p1.n_wblk, st);
  if (rc != MOE_OK) return rc;

  if (!make_bf16_map(&m2.w, W2, uint64_t(n_exp) * c.d, c.f, 128)) return MOE_E_CUDA;
  if (!make_token_maps(m2.tok, h, rows_h, c.f)) return MOE_E_CUDA;
  for (int i = 0; i < NBOX; ++i) m2.tok_sh[i] = m2.tok[i];
  PairParams p2 = p1;
  p2.K = c.f;
  p2.n_wblk = (c.d + 2 * BW - 1) / (2 * BW);  // 256 output columns per block
  p2.w_rows = c.d;
  p2.swiglu = 0;
  p2.n_out = c.d;
  p2.shared_tok_apart = 0;
  p2.out = static_cast<__nv_bfloat16*>(y_sorted);
  p2.ld_out = c.d;
  return launch_pair(m2, p2, seg_ub * p2.n_wblk, st);
}

}  // namespace moe
