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

#include <stdlib.h>
#include <string.h>

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
constexpr uint32_t EPI_STAGE_BYTES = 32 * 128;  // per epilogue warp: 32 rows x 64 bf16
constexpr size_t DYN_SMEM = size_t(STAGES) * STAGE_BYTES + 4 * EPI_STAGE_BYTES + 1024;
}  // namespace gg

enum { kEpiSwiglu = 0, kEpiBf16 = 1, kEpiF32 = 2, kEpiSwigluBwd = 3, kEpiCombine = 4 };

struct GroupedParams {
  const int32_t* counts;  // nullptr: one dense segment of dense_rows rows at row 0
  const int32_t* offsets;
  int E, capacity, has_shared, T, R;
  int dense_rows;
  int K;                  // reduction length of one pass
  int k_passes;           // passes over K (interleaved per k-block), B advanced by b_pass_rows
  int b_pass_rows;
  int k_split;            // dense mode: > 1 = segment g reduces K chunk g (length K) into
                          //   its own partial output rows [g*dense_rows, (g+1)*dense_rows)
  int merge_passes;       // 1 (with the kernel's kMerge): one pass over K; each k-block loads
                          //   A once and the k_passes B boxes side by side, and multiplies
                          //   A by each of them
  int N;                  // weight rows per expert (output columns before SwiGLU)
  int mode;               // kEpiSwiglu: out[:, j] = silu(acc[:, gate j]) * acc[:, up j]
                          // kEpiBf16:   out = bf16(acc)
                          // kEpiF32:    out_f32 = acc + col_bias (sigmoid if set), fp32
                          // kEpiSwigluBwd: acc = dh (columns j of the expert width);
                          //   with u, v = aux[:, gate j], aux[:, up j] (packed like W13)
                          //   and s = sigmoid(u): out[:, gate j] = dh v s (1 + u (1 - s)),
                          //   out[:, up j] = dh u s
                          // kEpiCombine: routed row r of assignment a = comb_order[r]
                          //   adds bf16(comb_gate[a] * acc) into comb_y[a / comb_k]; the
                          //   shared expert's row t adds bf16(acc) into comb_y[t]
  int shared_a_separate;  // 1: shared expert's A rows come from tmA_sh from row 0
  __nv_bfloat16* out;
  float* out_f32;
  const float* col_bias;
  int sigmoid;
  int ld_out;
  int* status;
  const int32_t* gather_order;  // non-null: a routed segment's A rows are gathered from the
  int gather_k;                 //   token rows, row r -> token gather_order[r] / gather_k
  const __nv_bfloat16* aux;     // kEpiSwigluBwd: the recomputed GEMM 1 output (u | v packed)
  int ld_aux;
  // Weight-gradient mode (kpad_off non-null): every segment g is an m_out x N
  // output block at rows g*m_out, reduced over columns [kpad_off[g],
  // kpad_off[g+1]) of the transposed operands (A [m_out, K_all], B [N, K_all],
  // shared by all segments; zero-padded to multiples of 64 per segment).
  const int32_t* kpad_off;
  int m_out;
  // kEpiBf16: 1 = groups of 32 rows whose rows are all valid leave through a
  // tensor store of tmOut (box 64 columns x 32 rows, 128-byte swizzle)
  int tma_store;
  // MMA width (N of each tcgen05.mma and columns of a tile): 0 = BN.  A narrower
  // width (a multiple of 16) serves outputs with few columns (the router).
  int n_mma;
  // kEpiSwiglu: non-null = also keep the pre-activations, aux_out[:, n_blk*BN + c]
  // = bf16(acc[:, c]) (gate and up columns packed like W13), ld_aux
  __nv_bfloat16* aux_out;
  // kEpiCombine: the assignment of each grouped row, the gates, top-k, and the
  // token-order output (zeroed before the launch; row stride ld_out)
  const int32_t* comb_order;
  const float* comb_gate;
  int comb_k;
  __nv_bfloat16* comb_y;
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
  if (p.kpad_off != nullptr) {
    rows = p.m_out;
    a_row0 = 0;
    out_row0 = g * p.m_out;
  } else if (p.counts == nullptr) {
    rows = p.dense_rows;
    a_row0 = 0;
    out_row0 = g * p.dense_rows;  // g > 0 only with k_split
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
template <bool kMerge>
__global__ void __launch_bounds__(gg::THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmA_sh,
                        const __grid_constant__ CUtensorMap tmA64,
                        const __grid_constant__ CUtensorMap tmA_sh64,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmOut, const GroupedParams p) {
  using namespace gg;
  extern __shared__ uint8_t dyn_smem[];
  __shared__ GroupedCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) &
                                             ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_seg = p.counts ? p.E + p.has_shared : (p.k_split > 1 ? p.k_split : 1);
  const int NM = p.n_mma ? p.n_mma : BN;                // tile width
  const uint32_t b_bytes = uint32_t(NM) * BK * 2;
  const int n_blocks_n = (p.N + NM - 1) / NM;
  const bool wgrad = p.kpad_off != nullptr;
  const int kb_per_pass = wgrad ? (1 << 30) : p.K / BK;
  const int n_b = kMerge ? p.k_passes : 1;  // B boxes per stage
  // passes over K taken k-block by k-block (pass = kb % n_pass): the passes'
  // B boxes of one k-block follow each other, so A's box is re-read from L2
  const int n_pass = kMerge || wgrad ? 1 : p.k_passes;
  const int num_kb = wgrad ? 0 : (kMerge ? kb_per_pass : kb_per_pass * p.k_passes);
  // first column and k-blocks of segment g's reduction
  auto tile_k = [&](int g, int& k0, int& nkb) {
    if (wgrad) {
      k0 = __ldg(p.kpad_off + g);
      nkb = (__ldg(p.kpad_off + g + 1) - k0) / BK;
    } else {
      k0 = p.counts == nullptr && p.k_split > 1 ? g * p.K : 0;
      nkb = num_kb;
    }
  };

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
    if (p.tma_store) tma_prefetch_desc(&tmOut);
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
    // ---------------- TMA producer ----------------
    // Lane 0 waits for free stages and issues the box copies.  With gathered
    // A rows (p.gather_order) the whole warp takes part: lane j copies rows
    // 4j..4j+3 of the tile with one four-row gather per k-block.
    uint32_t stage = 0, phase = 0;
    uint32_t issued = 0, last_phase = 0;  // per-stage bit masks (lane 0)
    bool ok = true;
    if (p.gather_order == nullptr) {
      if (lane == 0) {
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
          int g, m_blk, n_blk, rows, a_row0, out_row0;
          decode(t, g, m_blk, n_blk, rows, a_row0, out_row0);
          const bool sep = p.counts && g >= p.E && p.shared_a_separate;
          const bool half = is_half(rows, m_blk);
          const CUtensorMap* ma = half ? (sep ? &tmA_sh64 : &tmA64) : (sep ? &tmA_sh : &tmA);
          const uint32_t tx = (half ? A_BYTES / 2 : A_BYTES) + n_b * b_bytes;
          const int a_row = a_row0 + m_blk * BM;
          // per-segment weights (grouped mode); one shared B otherwise
          const int b_row = (wgrad || p.counts == nullptr ? 0 : g * p.N) + n_blk * NM;
          int k0, nkb;
          tile_k(g, k0, nkb);
          for (int kb = 0; kb < nkb; ++kb) {
            if (!wait_or_abort(&ctl.empty[stage], phase ^ 1u, ctl, p.status)) { ok = false; break; }
            uint8_t* sa = smem + stage * STAGE_BYTES;
            const int pass = kb % n_pass;
            const int ka = k0 + (kb / n_pass) * BK;
            mbar_arrive_expect_tx(&ctl.full[stage], tx);
            tma_load_2d(sa, ma, ka, a_row, &ctl.full[stage]);
            if (!kMerge) {
              tma_load_2d(sa + A_BYTES, &tmB, ka, b_row + pass * p.b_pass_rows, &ctl.full[stage]);
            } else {
              for (int j = 0; j < n_b; ++j)
                tma_load_2d(sa + A_BYTES + j * b_bytes, &tmB, ka, b_row + j * p.b_pass_rows,
                            &ctl.full[stage]);
            }
            issued |= 1u << stage;
            last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
        }
      }
    } else {
      for (int t = blockIdx.x; t < total; t += gridDim.x) {
        int g, m_blk, n_blk, rows, a_row0, out_row0;
        decode(t, g, m_blk, n_blk, rows, a_row0, out_row0);
        const bool sep = p.counts && g >= p.E && p.shared_a_separate;
        const bool gather = p.gather_order != nullptr && p.counts && g < p.E;
        const bool half = is_half(rows, m_blk);
        const int n_rows = half ? BM / 2 : BM;
        int tok[4] = {0, 0, 0, 0};
        if (gather && 4 * lane < n_rows) {
          // tokens of rows 4*lane .. 4*lane+3; rows past the segment repeat its first row
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = m_blk * BM + 4 * lane + i;
            const int src = a_row0 + (r < rows ? r : m_blk * BM);
            tok[i] = __ldg(p.gather_order + src) / p.gather_k;
          }
        }
        const CUtensorMap* ma = half ? (sep ? &tmA_sh64 : &tmA64) : (sep ? &tmA_sh : &tmA);
        const uint32_t tx = (half ? A_BYTES / 2 : A_BYTES) + b_bytes;
        const int a_row = a_row0 + m_blk * BM;
        const int b_row = g * p.N + n_blk * NM;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (lane == 0) ok = wait_or_abort(&ctl.empty[stage], phase ^ 1u, ctl, p.status);
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (!ok) break;
          uint8_t* sa = smem + stage * STAGE_BYTES;
          const int pass = kb % n_pass;
          const int ka = (kb / n_pass) * BK;
          if (lane == 0) mbar_arrive_expect_tx(&ctl.full[stage], tx);
          __syncwarp();
          if (gather) {
            if (4 * lane < n_rows)
              tma_gather4_2d(sa + lane * 4 * (BK * 2), &tmA, ka, tok[0], tok[1], tok[2], tok[3],
                             &ctl.full[stage]);
          } else if (lane == 0) {
            tma_load_2d(sa, ma, ka, a_row, &ctl.full[stage]);
          }
          if (lane == 0) {
            tma_load_2d(sa + A_BYTES, &tmB, ka, b_row + pass * p.b_pass_rows, &ctl.full[stage]);
            issued |= 1u << stage;
            last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
          }
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
      }
    }
    if (lane == 0) {
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
        const uint32_t idesc = is_half(rows, m_blk) ? idesc_bf16_f32(BM / 2, NM)
                                                    : idesc_bf16_f32(BM, NM);
        int k0, nkb;
        tile_k(g, k0, nkb);
        if (!wait_or_abort(&ctl.acc_empty[acc], acc_phase ^ 1u, ctl, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_or_abort(&ctl.full[stage], phase, ctl, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint8_t* sa = smem + stage * STAGE_BYTES;
          const uint64_t a_desc = smem_desc_k128(sa);
          for (int j = 0; j < n_b; ++j) {
            const uint64_t b_desc = smem_desc_k128(sa + A_BYTES + j * b_bytes);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              umma_bf16(d_tmem, a_desc + 2 * kk, b_desc + 2 * kk, idesc, (kb | kk | j) != 0);
          }
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
      int k0, nkb;
      tile_k(g, k0, nkb);
      if (nkb == 0) {
        // an empty reduction (a weight-gradient segment with no rows): zeros
        const int col0 = n_blk * BN;
        if (valid)
          for (int c = 0; c < BN && col0 + c < p.N; c += 8)
            *reinterpret_cast<uint4*>(orow + col0 + c) = make_uint4(0, 0, 0, 0);
      } else if (p.mode == kEpiSwigluBwd) {
        // accumulator columns are expert-width columns j = n_blk*BN + c; u and v
        // of column j sit at packed columns 256*(j/128) + j%128 and that + 128
        const __nv_bfloat16* arow = p.aux + size_t(out_row0 + (valid ? r : 0)) * p.ld_aux;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t dv32[32];
          tmem_ld32(taddr + c, dv32);
          tmem_ld_wait();
          const int j = n_blk * BN + c;
          if (valid && j < p.N) {
            const int pu = 256 * (j / 128) + (j % 128);
            const uint4* up = reinterpret_cast<const uint4*>(arow + pu);
            const uint4* vp = reinterpret_cast<const uint4*>(arow + pu + 128);
            uint4* dup = reinterpret_cast<uint4*>(orow + pu);
            uint4* dvp = reinterpret_cast<uint4*>(orow + pu + 128);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint4 uq = __ldg(up + q), vq = __ldg(vp + q);
              const uint32_t uw[4] = {uq.x, uq.y, uq.z, uq.w}, vw[4] = {vq.x, vq.y, vq.z, vq.w};
              uint32_t du_out[4], dv_out[4];
#pragma unroll
              for (int w = 0; w < 4; ++w) {
                float du2[2], dvv2[2];
#pragma unroll
                for (int hlf = 0; hlf < 2; ++hlf) {
                  const float u = hlf ? bf16hi(uw[w]) : bf16lo(uw[w]);
                  const float v = hlf ? bf16hi(vw[w]) : bf16lo(vw[w]);
                  const float dh = __uint_as_float(dv32[8 * q + 2 * w + hlf]);
                  const float sg = 1.0f / (1.0f + __expf(-u));
                  du2[hlf] = dh * v * sg * (1.0f + u * (1.0f - sg));
                  dvv2[hlf] = dh * u * sg;
                }
                du_out[w] = pack_bf16x2(du2[0], du2[1]);
                dv_out[w] = pack_bf16x2(dvv2[0], dvv2[1]);
              }
              dup[q] = make_uint4(du_out[0], du_out[1], du_out[2], du_out[3]);
              dvp[q] = make_uint4(dv_out[0], dv_out[1], dv_out[2], dv_out[3]);
            }
          }
        }
      } else if (p.mode == kEpiF32) {
        const int col0 = n_blk * NM;
#pragma unroll 1
        for (int c = 0; c < NM; c += 32) {
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
          if (valid && p.aux_out) {
            __nv_bfloat16* arow = p.aux_out + size_t(out_row0 + r) * p.ld_aux + n_blk * BN + c;
            uint4* ug = reinterpret_cast<uint4*>(arow);
            uint4* vg = reinterpret_cast<uint4*>(arow + BN / 2);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              ug[q] = make_uint4(pack_bf16x2(__uint_as_float(gv[8 * q]), __uint_as_float(gv[8 * q + 1])),
                                 pack_bf16x2(__uint_as_float(gv[8 * q + 2]), __uint_as_float(gv[8 * q + 3])),
                                 pack_bf16x2(__uint_as_float(gv[8 * q + 4]), __uint_as_float(gv[8 * q + 5])),
                                 pack_bf16x2(__uint_as_float(gv[8 * q + 6]), __uint_as_float(gv[8 * q + 7])));
              vg[q] = make_uint4(pack_bf16x2(__uint_as_float(uv[8 * q]), __uint_as_float(uv[8 * q + 1])),
                                 pack_bf16x2(__uint_as_float(uv[8 * q + 2]), __uint_as_float(uv[8 * q + 3])),
                                 pack_bf16x2(__uint_as_float(uv[8 * q + 4]), __uint_as_float(uv[8 * q + 5])),
                                 pack_bf16x2(__uint_as_float(uv[8 * q + 6]), __uint_as_float(uv[8 * q + 7])));
            }
          }
          // only valid rows are activated: rows past the segment hold stale
          // accumulators, and activating them anyway made GEMM 1 about 30 %
          // slower on a capacity-padded layer
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
      } else if (p.mode == kEpiCombine) {
        // the row's token and gate: routed rows through the grouped order,
        // the shared expert's rows are the tokens (gate 1)
        int t = -1;
        float gw = 1.0f;
        if (valid) {
          if (g < p.E) {
            const int a = __ldg(p.comb_order + out_row0 + r);
            if (a >= 0) {
              t = a / p.comb_k;
              gw = __ldg(p.comb_gate + a);
            }
          } else {
            t = r;
          }
        }
        const int col0 = n_blk * BN;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t v[32];
          tmem_ld32(taddr + c, v);
          tmem_ld_wait();
          if (t >= 0) {
            __nv_bfloat16* dst = p.comb_y + size_t(t) * p.ld_out + col0 + c;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              if (col0 + c + 8 * i >= p.N) break;
              uint32_t w[4];
#pragma unroll
              for (int q = 0; q < 4; ++q)
                w[q] = pack_bf16x2(gw * __uint_as_float(v[8 * i + 2 * q]),
                                   gw * __uint_as_float(v[8 * i + 2 * q + 1]));
              red_add_bf16x8(dst + 8 * i, w);
            }
          }
        }
      } else if (p.tma_store && !half && m_blk * BM + quarter * 32 + 31 < rows) {
        // all 32 rows of this warp are valid: stage 64 columns at a time in
        // shared memory (128-byte swizzle) and store them with one tensor copy
        const int col0 = n_blk * BN;
        uint8_t* stg = smem + STAGES * STAGE_BYTES + quarter * EPI_STAGE_BYTES;
        const int out_r = out_row0 + m_blk * BM + quarter * 32;
#pragma unroll 1
        for (int c = 0; c < BN && col0 + c < p.N; c += 64) {
          uint32_t v0[32], v1[32];
          tmem_ld32(taddr + c, v0);
          tmem_ld32(taddr + c + 32, v1);
          if (lane == 0) bulk_wait_group_read0();  // the previous store has read the buffer
          __syncwarp();
          tmem_ld_wait();
          uint8_t* row = stg + lane * 128;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint32_t* src = q < 4 ? v0 + 8 * q : v1 + 8 * (q - 4);
            const uint4 w = make_uint4(pack_bf16x2(__uint_as_float(src[0]), __uint_as_float(src[1])),
                                       pack_bf16x2(__uint_as_float(src[2]), __uint_as_float(src[3])),
                                       pack_bf16x2(__uint_as_float(src[4]), __uint_as_float(src[5])),
                                       pack_bf16x2(__uint_as_float(src[6]), __uint_as_float(src[7])));
            *reinterpret_cast<uint4*>(row + ((q ^ (lane & 7)) << 4)) = w;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmOut, stg, col0 + c, out_r);
            bulk_commit_group();
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
    if (p.tma_store && lane == 0) bulk_wait_group0();  // stores complete before the CTA ends
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
bool make_bf16_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols,
                   uint32_t box_rows) {
  if (!get_encoder()) return false;
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
  static PerDeviceOnce once;
  return once.run([] {
    cudaError_t err = cudaFuncSetAttribute(grouped_gemm_kernel<false>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           int(gg::DYN_SMEM));
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(grouped_gemm_kernel<true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, int(gg::DYN_SMEM));
    if (err != cudaSuccess) cudaGetLastError();
    return err == cudaSuccess ? MOE_OK : MOE_E_CUDA;
  });
}

#define MOE_TRY_INTERNAL(expr)      \
  do {                              \
    const int _rc = (expr);         \
    if (_rc != MOE_OK) return _rc;  \
  } while (0)

// One grouped GEMM on at most one CTA per SM and no more CTAs than an upper
// bound on its tiles (rows_ub rows over at most n_seg segments).
static int launch_gg(int64_t rows_ub, int n_seg, const CUtensorMap& a, const CUtensorMap& a_sh,
                     const CUtensorMap& a64, const CUtensorMap& a_sh64, const CUtensorMap& b,
                     const CUtensorMap& out, const GroupedParams& p, cudaStream_t st) {
  const int sms = device_sm_count();
  const long long tiles = (rows_ub / gg::BM + n_seg) * ((p.N + gg::BN - 1) / gg::BN);
  const int grid = int(tiles < sms ? tiles : sms);
  grouped_gemm_kernel<false><<<grid, gg::THREADS, gg::DYN_SMEM, st>>>(a, a_sh, a64, a_sh64, b,
                                                                     out, p);
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_E_CUDA;
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
// Fixed-order sum of the router's K-chunk partials, + logit bias, sigmoid if
// asked: out[t][e] = sum over s of part[s][t][e].
__global__ void __launch_bounds__(256) router_split_reduce_kernel(
    const float* __restrict__ part, int S, int T, int E, const float* __restrict__ lbias,
    int sigmoid, float* __restrict__ out) {
  const size_t n = size_t(T) * E;
  for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += size_t(gridDim.x) * blockDim.x) {
    float l = 0.0f;
    for (int s = 0; s < S; ++s) l += __ldg(part + size_t(s) * n + i);
    if (lbias) l += __ldg(lbias + i % E);
    if (sigmoid) l = 1.0f / (1.0f + expf(-l));
    out[i] = l;
  }
}

int launch_router_tc(const moe_cfg& c, const void* x, const void* W_split, const float* lbias,
                     float* out, int* status, float* part, cudaStream_t st) {
  using namespace gg;
  if (!get_encoder()) return MOE_E_CUDA;
  if (set_smem_attr() != MOE_OK) return MOE_E_CUDA;
  // MMA width: the experts rounded up to 16 (at most 256 per tile)
  const int nm = c.E >= BN ? BN : ((c.E + 15) & ~15);
  CUtensorMap mA, mA64, mB;
  if (!make_bf16_map(&mA, x, uint64_t(c.T), c.d, BM)) return MOE_E_CUDA;
  if (!make_bf16_map(&mA64, x, uint64_t(c.T), c.d, BM / 2)) return MOE_E_CUDA;
  if (!make_bf16_map(&mB, W_split, uint64_t(3) * c.E, c.d, uint32_t(nm))) return MOE_E_CUDA;
  const int sms = sm_count();
  if (sms <= 0) return MOE_E_CUDA;
  GroupedParams p{};
  p.counts = nullptr;
  p.dense_rows = c.T;
  p.K = c.d;
  p.k_passes = 3;
  p.b_pass_rows = c.E;
  // the three B boxes of a k-block fit the stage's B slot together up to 80
  // columns: then A is read once instead of once per term
  p.merge_passes = 3u * uint32_t(nm) * BK * 2 <= B_BYTES ? 1 : 0;
  p.N = c.E;
  p.mode = kEpiF32;
  p.out_f32 = out;
  p.col_bias = lbias;
  p.sigmoid = c.score_fn == MOE_SIGMOID;
  p.ld_out = c.E;
  p.status = status;
  p.n_mma = nm;
  // split K when the output tiles are few (and a partial buffer is given)
  const int ks = part ? router_k_split(c) : 1;
  if (ks > 1) {
    p.k_split = ks;
    p.K = c.d / ks;
    p.out_f32 = part;
    p.col_bias = nullptr;
    p.sigmoid = 0;
  }
  const long long tiles = (long long)((c.T + BM - 1) / BM) * ((c.E + BN - 1) / BN) * ks;
  const int grid = int(tiles < sms ? tiles : sms);
  if (p.merge_passes)
    grouped_gemm_kernel<true><<<grid, THREADS, DYN_SMEM, st>>>(mA, mA, mA64, mA64, mB, mB, p);
  else
    grouped_gemm_kernel<false><<<grid, THREADS, DYN_SMEM, st>>>(mA, mA, mA64, mA64, mB, mB, p);
  note_launches(1);
  if (ks > 1) {
    const long long n = (long long)c.T * c.E;
    const int blocks = int((n + 255) / 256 < 4 * sms ? (n + 255) / 256 : 4 * sms);
    router_split_reduce_kernel<<<blocks, 256, 0, st>>>(part, ks, c.T, c.E, lbias,
                                                       c.score_fn == MOE_SIGMOID, out);
    note_launches(1);
  }
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

// Which tiles run the forward FFN.  The pair tiles (grouped_pair.cu) stage a
// third fewer bytes per MMA but stream a weight block once per 256-token
// block; the one-SM 128-row tiles of this file keep more weight bytes in
// flight.  Measured on B300, the pair tiles win when an expert holds about a
// thousand rows (Mixtral-shaped layer, FFN 1.94 against 1.99 ms) and lose at
// 256 rows per expert (DeepSeek-V3-shaped layer, 6.59 against 6.31 ms), at
// the skewed layer's capacity of 640 and at decode sizes.  So the pair tiles
// take layers whose expected rows per expert, T*k/E (at most the capacity),
// reach 768.  The environment variable MOE_FFN_TILES = "pair" or "single"
// overrides the choice (read at every call).  The gathered and training forms
// always take the one-SM tiles.
bool use_pair_tiles(const moe_cfg& c) {
  const char* v = getenv("MOE_FFN_TILES");
  if (v && strcmp(v, "pair") == 0) return true;
  if (v && strcmp(v, "single") == 0) return false;
  long long rows = (long long)c.T * c.k / c.E;
  if (c.capacity && rows > c.capacity) rows = c.capacity;
  return rows >= 768;
}

namespace {
// GEMM 2 adding its rows straight into the token-order output (kEpiCombine)
struct CombineOut {
  const int32_t* order;
  const float* gate;
  void* y;
};
}  // namespace

static int launch_grouped_ffn_impl(const moe_cfg& c, const void* x_sorted, const void* x,
                                   const int32_t* gather_order, const int32_t* counts,
                                   const int32_t* offsets, const void* W13, const void* W2,
                                   void* h, void* y_sorted, void* g1, void* ws, cudaStream_t st,
                                   const CombineOut* comb) {
  using namespace gg;
  if (!get_encoder()) return MOE_E_CUDA;
  const WsLayout L = ws_layout(c);
  if (gather_order == nullptr && g1 == nullptr && comb == nullptr && use_pair_tiles(c))
    return launch_grouped_ffn_pair(c, x_sorted, x, counts, offsets, W13, W2, h, y_sorted,
                                   ws_ptr<int>(ws, L.status), st);
  if (set_smem_attr() != MOE_OK) return MOE_E_CUDA;
  const int R = c.capacity ? c.E * c.capacity : c.T * c.k;
  const int n_exp = c.E + c.has_shared;
  const uint64_t rows_h = uint64_t(R) + (c.has_shared ? c.T : 0);

  CUtensorMap mA1, mA1s, mA1h, mA1sh, mB1, mA2, mA2h, mB2;
  // the shared expert's rows (or, with no shared expert, any valid map: unused)
  const bool a1s_x = c.has_shared || x_sorted == nullptr;
  const void* a1s = a1s_x ? x : x_sorted;
  const uint64_t a1s_rows = a1s_x ? uint64_t(c.T) : uint64_t(R);
  if (gather_order) {
    // routed rows gathered from the token rows: a map whose box is one row high
    if (!make_bf16_map(&mA1, x, uint64_t(c.T), c.d, 1)) return MOE_E_CUDA;
    mA1h = mA1;
  } else {
    if (!make_bf16_map(&mA1, x_sorted, uint64_t(R), c.d, BM)) return MOE_E_CUDA;
    if (!make_bf16_map(&mA1h, x_sorted, uint64_t(R), c.d, BM / 2)) return MOE_E_CUDA;
  }
  if (!make_bf16_map(&mA1s, a1s, a1s_rows, c.d, BM)) return MOE_E_CUDA;
  if (!make_bf16_map(&mA1sh, a1s, a1s_rows, c.d, BM / 2)) return MOE_E_CUDA;
  if (!make_bf16_map(&mB1, W13, uint64_t(n_exp) * 2 * c.f, c.d, BN)) return MOE_E_CUDA;
  if (!make_bf16_map(&mA2, h, rows_h, c.f, BM)) return MOE_E_CUDA;
  if (!make_bf16_map(&mA2h, h, rows_h, c.f, BM / 2)) return MOE_E_CUDA;
  if (!make_bf16_map(&mB2, W2, uint64_t(n_exp) * c.d, c.f, BN)) return MOE_E_CUDA;

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
  p1.gather_order = gather_order;
  p1.gather_k = c.k;
  p1.aux_out = static_cast<__nv_bfloat16*>(g1);
  p1.ld_aux = 2 * c.f;

  const long long t1 = mt_ub * ((p1.N + BN - 1) / BN);
  const int grid1 = int(t1 < sms ? t1 : sms);
  grouped_gemm_kernel<false><<<grid1, THREADS, DYN_SMEM, st>>>(mA1, mA1s, mA1h, mA1sh, mB1, mB1,
                                                               p1);

  GroupedParams p2 = p1;
  p2.gather_order = nullptr;
  p2.aux_out = nullptr;
  p2.K = c.f;
  p2.N = c.d;
  p2.mode = kEpiBf16;
  p2.shared_a_separate = 0;
  p2.out = static_cast<__nv_bfloat16*>(y_sorted);
  p2.ld_out = c.d;
  const long long t2 = mt_ub * ((p2.N + BN - 1) / BN);
  const int grid2 = int(t2 < sms ? t2 : sms);
  CUtensorMap mOut2 = mB2;  // unused without the tensor-store epilogue
  if (comb) {
    p2.mode = kEpiCombine;
    p2.out = nullptr;
    p2.comb_order = comb->order;
    p2.comb_gate = comb->gate;
    p2.comb_k = c.k;
    p2.comb_y = static_cast<__nv_bfloat16*>(comb->y);
  } else {
    if (!make_bf16_map(&mOut2, y_sorted, rows_h, c.d, 32)) return MOE_E_CUDA;
    p2.tma_store = 1;
  }
  grouped_gemm_kernel<false><<<grid2, THREADS, DYN_SMEM, st>>>(mA2, mA2, mA2h, mA2h, mB2, mOut2, p2);
  note_launches(2);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_E_CUDA;
}

int launch_grouped_ffn(const moe_cfg& c, const void* x_sorted, const void* x,
                       const int32_t* gather_order, const int32_t* counts, const int32_t* offsets,
                       const void* W13, const void* W2, void* h, void* y_sorted, void* g1,
                       void* ws, cudaStream_t st) {
  return launch_grouped_ffn_impl(c, x_sorted, x, gather_order, counts, offsets, W13, W2, h,
                                 y_sorted, g1, ws, st, nullptr);
}

int launch_grouped_ffn_combine(const moe_cfg& c, const void* x_sorted, const void* x,
                               const int32_t* counts, const int32_t* offsets, const void* W13,
                               const void* W2, void* h, const int32_t* order, const float* gate,
                               void* y, void* ws, cudaStream_t st) {
  if (cudaMemsetAsync(y, 0, size_t(c.T) * c.d * 2, st) != cudaSuccess) {
    cudaGetLastError();
    return MOE_E_CUDA;
  }
  const CombineOut comb{order, gate, y};
  return launch_grouped_ffn_impl(c, x_sorted, x, nullptr, counts, offsets, W13, W2, h, nullptr,
                                 nullptr, ws, st, &comb);
}

}  // namespace moe

namespace moe {

// Rows of the transposed-operand buffers of the weight gradients: an upper
// bound on the padded reduction length, sum over segments of roundup(kept, 64).
size_t backward_kpad_bound(const moe_cfg& c) {
  const size_t R = c.capacity ? size_t(c.E) * c.capacity : size_t(c.T) * c.k;
  const size_t ub = R + size_t(c.E) * 64 + (c.has_shared ? ((size_t(c.T) + 63) & ~size_t(63)) : 0);
  return (ub + 63) & ~size_t(63);
}

// Backward workspace: g1 and dg1 [R + T, 2f] bf16, the padded segment offsets,
// and one region reused for the transposed operands of both weight gradients.
BwdLayout backward_layout(const moe_cfg& c) {
  BwdLayout L;
  const size_t rows = (c.capacity ? size_t(c.E) * c.capacity : size_t(c.T) * c.k) +
                      (c.has_shared ? size_t(c.T) : 0);
  const size_t kub = backward_kpad_bound(c);
  size_t off = 0;
  L.g1 = off;   off += align256(rows * 2 * c.f * 2);
  L.dg1 = off;  off += align256(rows * 2 * c.f * 2);
  L.kpad = off; off += align256(size_t(c.E + 2) * 4);
  L.tr = off;
  const size_t w2 = size_t(c.d + c.f), w13 = size_t(2 * c.f + c.d);
  off += align256((w2 > w13 ? w2 : w13) * kub * 2);
  L.total = off;
  L.kub = kub;
  return L;
}

int launch_grouped_ffn_backward(const moe_cfg& c, const void* x_sorted, const void* x,
                                const int32_t* counts, const int32_t* offsets, const void* W13,
                                const void* W13t, const void* W2t, const void* h, const void* g1_saved,
                                const void* d_o, void* dx_sorted, void* dW13, void* dW2,
                                void* bws, void* ws, cudaStream_t st) {
  using namespace gg;
  if (!get_encoder()) return MOE_E_CUDA;
  if (set_smem_attr() != MOE_OK) return MOE_E_CUDA;
  const WsLayout L = ws_layout(c);
  const BwdLayout B = backward_layout(c);
  const int R = c.capacity ? c.E * c.capacity : c.T * c.k;
  const int n_exp = c.E + c.has_shared;
  const uint64_t rows_h = uint64_t(R) + (c.has_shared ? c.T : 0);
  char* bw = static_cast<char*>(bws);
  const __nv_bfloat16* g1 = g1_saved ? static_cast<const __nv_bfloat16*>(g1_saved)
                                     : reinterpret_cast<const __nv_bfloat16*>(bw + B.g1);
  __nv_bfloat16* dg1 = reinterpret_cast<__nv_bfloat16*>(bw + B.dg1);
  int32_t* kpad = reinterpret_cast<int32_t*>(bw + B.kpad);
  __nv_bfloat16* trA = reinterpret_cast<__nv_bfloat16*>(bw + B.tr);
  const size_t kub = B.kub;

  GroupedParams base{};
  base.counts = counts;
  base.offsets = offsets;
  base.E = c.E;
  base.capacity = c.capacity;
  base.has_shared = c.has_shared;
  base.T = c.T;
  base.R = R;
  base.k_passes = 1;
  base.status = ws_ptr<int>(ws, L.status);

  // 1. g1 = x W13^T (recomputed unless the forward kept it; routed rows from
  //    x_sorted, shared rows from x)
  if (!g1_saved) {
    CUtensorMap mA, mAh, mAs, mAsh, mB;
    const bool sx = c.has_shared;
    if (!make_bf16_map(&mA, x_sorted, uint64_t(R), c.d, BM)) return MOE_E_CUDA;
    if (!make_bf16_map(&mAh, x_sorted, uint64_t(R), c.d, BM / 2)) return MOE_E_CUDA;
    if (!make_bf16_map(&mAs, sx ? x : x_sorted, sx ? uint64_t(c.T) : uint64_t(R), c.d, BM))
      return MOE_E_CUDA;
    if (!make_bf16_map(&mAsh, sx ? x : x_sorted, sx ? uint64_t(c.T) : uint64_t(R), c.d, BM / 2))
      return MOE_E_CUDA;
    if (!make_bf16_map(&mB, W13, uint64_t(n_exp) * 2 * c.f, c.d, BN)) return MOE_E_CUDA;
    GroupedParams p = base;
    p.K = c.d;
    p.N = 2 * c.f;
    p.mode = kEpiBf16;
    p.shared_a_separate = 1;
    __nv_bfloat16* g1w = reinterpret_cast<__nv_bfloat16*>(bw + B.g1);
    p.out = g1w;
    p.ld_out = 2 * c.f;
    CUtensorMap mO;
    if (!make_bf16_map(&mO, g1w, rows_h, 2 * c.f, 32)) return MOE_E_CUDA;
    p.tma_store = 1;
    MOE_TRY_INTERNAL(launch_gg(rows_h, n_exp, mA, mAs, mAh, mAsh, mB, mO, p, st));
  }
  // 2. dh = d_o W2 (B = W2^T per expert, N = f, K = d); the epilogue applies the
  //    SwiGLU derivative with g1 and writes dg1 (packed like W13)
  {
    CUtensorMap mA, mAh, mB;
    if (!make_bf16_map(&mA, d_o, rows_h, c.d, BM)) return MOE_E_CUDA;
    if (!make_bf16_map(&mAh, d_o, rows_h, c.d, BM / 2)) return MOE_E_CUDA;
    if (!make_bf16_map(&mB, W2t, uint64_t(n_exp) * c.f, c.d, BN)) return MOE_E_CUDA;
    GroupedParams p = base;
    p.K = c.d;
    p.N = c.f;
    p.mode = kEpiSwigluBwd;
    p.shared_a_separate = 0;
    p.aux = g1;
    p.ld_aux = 2 * c.f;
    p.out = dg1;
    p.ld_out = 2 * c.f;
    MOE_TRY_INTERNAL(launch_gg(rows_h, n_exp, mA, mA, mAh, mAh, mB, mB, p, st));
  }
  // 3. dx_sorted = dg1 W13 (B = W13^T per expert, N = d, K = 2f)
  {
    CUtensorMap mA, mAh, mB;
    if (!make_bf16_map(&mA, dg1, rows_h, 2 * c.f, BM)) return MOE_E_CUDA;
    if (!make_bf16_map(&mAh, dg1, rows_h, 2 * c.f, BM / 2)) return MOE_E_CUDA;
    if (!make_bf16_map(&mB, W13t, uint64_t(n_exp) * c.d, 2 * c.f, BN)) return MOE_E_CUDA;
    GroupedParams p = base;
    p.K = 2 * c.f;
    p.N = c.d;
    p.mode = kEpiBf16;
    p.shared_a_separate = 0;
    p.out = static_cast<__nv_bfloat16*>(dx_sorted);
    p.ld_out = c.d;
    CUtensorMap mO;
    if (!make_bf16_map(&mO, dx_sorted, rows_h, c.d, 32)) return MOE_E_CUDA;
    p.tma_store = 1;
    MOE_TRY_INTERNAL(launch_gg(rows_h, n_exp, mA, mA, mAh, mAh, mB, mO, p, st));
  }
  // 4. weight gradients, each over its expert's rows
  MOE_TRY_INTERNAL(launch_kpad_offsets(c, counts, kpad, st));
  const __nv_bfloat16* hb = static_cast<const __nv_bfloat16*>(h);
  const __nv_bfloat16* dob = static_cast<const __nv_bfloat16*>(d_o);
  __nv_bfloat16* trB = trA + size_t(c.d) * kub;  // after d_o^T [d, kub]
  MOE_TRY_INTERNAL(launch_transpose_segments(c, d_o, dob + size_t(R) * c.d, c.d, offsets, counts,
                                             kpad, trA, kub, st));
  MOE_TRY_INTERNAL(launch_transpose_segments(c, h, hb + size_t(R) * c.f, c.f, offsets, counts,
                                             kpad, trB, kub, st));
  {
    // dW2[g] = d_o^T h: [d, f] per segment
    CUtensorMap mA, mAh, mB;
    if (!make_bf16_map(&mA, trA, uint64_t(c.d), kub, BM)) return MOE_E_CUDA;
    if (!make_bf16_map(&mAh, trA, uint64_t(c.d), kub, BM / 2)) return MOE_E_CUDA;
    if (!make_bf16_map(&mB, trB, uint64_t(c.f), kub, BN)) return MOE_E_CUDA;
    GroupedParams p = base;
    p.K = BK;
    p.N = c.f;
    p.mode = kEpiBf16;
    p.kpad_off = kpad;
    p.m_out = c.d;
    p.out = static_cast<__nv_bfloat16*>(dW2);
    p.ld_out = c.f;
    CUtensorMap mO;
    if (!make_bf16_map(&mO, dW2, uint64_t(n_exp) * c.d, c.f, 32)) return MOE_E_CUDA;
    p.tma_store = 1;
    MOE_TRY_INTERNAL(launch_gg(int64_t(n_exp) * c.d, n_exp, mA, mA, mAh, mAh, mB, mO, p, st));
  }
  __nv_bfloat16* trC = trA + size_t(2 * c.f) * kub;  // after dg1^T [2f, kub]
  MOE_TRY_INTERNAL(launch_transpose_segments(c, dg1, dg1 + size_t(R) * 2 * c.f, 2 * c.f, offsets,
                                             counts, kpad, trA, kub, st));
  MOE_TRY_INTERNAL(launch_transpose_segments(c, x_sorted, c.has_shared ? x : x_sorted, c.d,
                                             offsets, counts, kpad, trC, kub, st));
  {
    // dW13[g] = dg1^T x: [2f, d] per segment (rows packed like W13)
    CUtensorMap mA, mAh, mB;
    if (!make_bf16_map(&mA, trA, uint64_t(2 * c.f), kub, BM)) return MOE_E_CUDA;
    if (!make_bf16_map(&mAh, trA, uint64_t(2 * c.f), kub, BM / 2)) return MOE_E_CUDA;
    if (!make_bf16_map(&mB, trC, uint64_t(c.d), kub, BN)) return MOE_E_CUDA;
    GroupedParams p = base;
    p.K = BK;
    p.N = c.d;
    p.mode = kEpiBf16;
    p.kpad_off = kpad;
    p.m_out = 2 * c.f;
    p.out = static_cast<__nv_bfloat16*>(dW13);
    p.ld_out = c.d;
    CUtensorMap mO;
    if (!make_bf16_map(&mO, dW13, uint64_t(n_exp) * 2 * c.f, c.d, 32)) return MOE_E_CUDA;
    p.tma_store = 1;
    MOE_TRY_INTERNAL(launch_gg(int64_t(n_exp) * 2 * c.f, n_exp, mA, mA, mAh, mAh, mB, mO, p,
                               st));
  }
  return MOE_OK;
}

}  // namespace moe
