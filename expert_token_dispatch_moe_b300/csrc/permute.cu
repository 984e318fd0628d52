// Step 2 of the MoE layer: stable grouping of the T*k assignments into
// per-expert segments, plus the simulated expert-parallel send layout.
//
// "Token permutation and grouped GEMMs" (Expert parallelism page): order is
// the stable argsort of the expert ids and inv[order] = arange.  The stable
// rank of an assignment inside its expert comes from histograms and prefix
// sums, never from the order of atomics, so every output is deterministic.
// Three paths: up to 4096 assignments (and 256 experts), one CTA computes the
// indices; up to 256 experts, one cooperative launch does everything
// (perm_fused_kernel, below); otherwise:
//   1. hist:  per 2048-assignment chunk, a histogram over experts (shared-memory
//             atomics: only counts, not order, depend on them); counts per
//             (source rank, expert) for the layout.  The CTA that finishes
//             last then scans: per expert, the exclusive prefix over chunks
//             (chunk bases) and totals, and the exclusive prefix over experts
//             (segment offsets).
//   2. rank:  per chunk, warp-ordered match/popc ranks, giving each
//             assignment its row; writes inv and order.
//   3. move:  one warp per token reads x[t] once (16-byte vectors) and writes
//             its k copies.
// Capacity mode keeps rank < cap at row e*cap + rank and zero-fills the rest
// of each segment (one warp per row, over the whole grouped buffer).
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace moe {

constexpr int kPermThreads = 256;
constexpr int kPermPerThread = kPermChunk / kPermThreads;  // 8

// ---------------------------------------------------------------------------
// 1. histogram, then (last CTA) the scans
// ---------------------------------------------------------------------------
// Exclusive prefix over the E per-expert totals in tot[] (shared memory),
// in place, by the whole CTA (kPermThreads threads, E <= 4 * kPermThreads).
// Returns the sum of all totals.
__device__ int block_exclusive_scan(int32_t* tot, int E) {
  __shared__ int32_t warp_sum[kPermThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int e0 = threadIdx.x * 4;
  int v[4], local = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[i] = (e0 + i < E) ? tot[e0 + i] : 0;
    local += v[i];
  }
  int incl = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  int before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kPermThreads / 32; ++w) {
    if (w < warp) before += warp_sum[w];
    all += warp_sum[w];
  }
  int run = before + incl - local;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (e0 + i < E) tot[e0 + i] = run;
    run += v[i];
  }
  __syncthreads();
  return all;
}

__global__ void __launch_bounds__(kPermThreads) perm_hist_kernel(
    const int32_t* __restrict__ idx, int A, int E, int k, int T_loc, int capacity,
    int32_t* __restrict__ chunk_hist, int32_t* __restrict__ src_cnt, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int* status, unsigned int* done_ctas) {
  extern __shared__ int32_t h[];  // [E]; reused by the last CTA for totals
  __shared__ bool last;
  for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int base = blockIdx.x * kPermChunk;
#pragma unroll
  for (int i = 0; i < kPermPerThread; ++i) {
    const int a = base + i * kPermThreads + threadIdx.x;
    int key = -1;
    if (a < A) {
      const int e = __ldg(idx + a);
      if (e >= 0 && e < E) {
        atomicAdd(&h[e], 1);
        key = ((a / k) / T_loc) * E + e;
      } else {
        report_status(status, MOE_E_DEVICE_DATA);
      }
    }
    // one global atomic per distinct (source rank, expert) in the warp
    const uint32_t peers = __match_any_sync(0xffffffffu, key);
    if (key >= 0 && (peers & ((1u << lane) - 1u)) == 0) atomicAdd(src_cnt + key, __popc(peers));
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_hist[size_t(blockIdx.x) * E + e] = h[e];

  // The last CTA to finish turns the chunk histograms into chunk bases.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(done_ctas, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  const int n_chunks = gridDim.x;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int total = 0;
    int c = 0;
    for (; c + 4 <= n_chunks; c += 4) {
      int v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = __ldcg(chunk_hist + size_t(c + u) * E + e);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        chunk_hist[size_t(c + u) * E + e] = total;  // becomes the chunk base
        total += v[u];
      }
    }
    for (; c < n_chunks; ++c) {
      const int v = __ldcg(chunk_hist + size_t(c) * E + e);
      chunk_hist[size_t(c) * E + e] = total;
      total += v;
    }
    counts[e] = total;
    h[e] = total;
  }
  __syncthreads();
  const int all = block_exclusive_scan(h, E);
  for (int e = threadIdx.x; e < E; e += blockDim.x) offsets[e] = capacity ? e * capacity : h[e];
  if (threadIdx.x == 0) {
    offsets[E] = capacity ? E * capacity : all;
    *done_ctas = 0u;  // ready for the next call
  }
}

// ---------------------------------------------------------------------------
// 2. stable ranks -> rows
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kPermThreads) perm_rank_kernel(
    const int32_t* __restrict__ idx, int A, int E, int capacity,
    const int32_t* __restrict__ chunk_base, const int32_t* __restrict__ offsets,
    int32_t* __restrict__ inv, int32_t* __restrict__ order) {
  extern __shared__ int32_t wcnt[];  // [8 warps][E]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < 8 * E; i += blockDim.x) wcnt[i] = 0;
  __syncthreads();
  const int base = blockIdx.x * kPermChunk + warp * (kPermChunk / 8);
  const uint32_t lt_mask = (1u << lane) - 1u;
  int my_e[kPermPerThread], my_r[kPermPerThread];
#pragma unroll
  for (int r = 0; r < kPermPerThread; ++r) {
    const int a = base + r * 32 + lane;
    int e = -1;
    if (a < A) {
      e = __ldg(idx + a);
      if (e < 0 || e >= E) e = -1;
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    const int lrank = __popc(peers & lt_mask);
    int prior = 0;
    if (e >= 0) prior = wcnt[warp * E + e];
    __syncwarp();
    if (e >= 0 && lrank == 0) wcnt[warp * E + e] = prior + __popc(peers);
    __syncwarp();
    my_e[r] = e;
    my_r[r] = prior + lrank;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = chunk_base[size_t(blockIdx.x) * E + e];
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const int v = wcnt[w * E + e];
      wcnt[w * E + e] = run;
      run += v;
    }
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < kPermPerThread; ++r) {
    const int a = base + r * 32 + lane;
    if (a >= A) continue;
    const int e = my_e[r];
    int row = -1;
    if (e >= 0) {
      const int rank = wcnt[warp * E + e] + my_r[r];
      if (capacity) row = (rank < capacity) ? e * capacity + rank : -1;
      else row = __ldg(offsets + e) + rank;
    }
    inv[a] = row;
    if (row >= 0) order[row] = a;
  }
}

// ---------------------------------------------------------------------------
// 1+2 in one CTA, for small batches (A <= kPermSmallMaxA, E <= kPermSmallMaxE):
// no chunk tables, no cross-CTA hand-off, one launch.  Pass 1 counts experts
// (and (source rank, expert) pairs) and scans them into offsets; pass 2 walks
// the assignments in rounds of 1024 in index order: warp match/popc ranks
// within a warp, then per expert an exclusive scan over the 32 warps (one
// warp per expert, a lane per warp) on top of the expert's count from earlier
// rounds.  Per-warp counts are tagged with the round, so the table never needs
// clearing.
// ---------------------------------------------------------------------------
constexpr int kPermSmallThreads = 1024;
constexpr int kPermSmallMaxA = 4096;
constexpr int kPermSmallMaxE = 256;

__global__ void __launch_bounds__(kPermSmallThreads, 1) perm_index_small_kernel(
    const int32_t* __restrict__ idx, int A, int E, int k, int T_loc, int n_ep, int capacity,
    int32_t* __restrict__ src_cnt, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ inv, int32_t* __restrict__ order, int* status) {
  extern __shared__ int32_t sm_small[];
  const int ld = E + 1;                  // row pitch of the warp tables (odd: no bank conflicts)
  int32_t* tab = sm_small;               // [32][ld]: (round << 16) | count of e in warp w
  int32_t* pre = sm_small + 32 * ld;     // [32][ld]: rank base of e for warp w this round
  int32_t* base = sm_small + 64 * ld;    // [E]: first row of e (dropless)
  int32_t* seen = base + E;              // [E]: assignments of e in earlier rounds
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t lt = (1u << lane) - 1u;
  for (int i = tid; i < 32 * ld; i += blockDim.x) tab[i] = -1;  // tag -1: no round
  for (int e = tid; e < E; e += blockDim.x) { base[e] = 0; seen[e] = 0; }
  for (int i = tid; i < n_ep * E; i += blockDim.x) src_cnt[i] = 0;
  // every expert id this thread will touch, loaded at once (assignment
  // r * 1024 + tid in round r); -1 past the end or for an invalid id
  constexpr int ROUNDS = kPermSmallMaxA / kPermSmallThreads;
  int ev[ROUNDS];
#pragma unroll
  for (int r = 0; r < ROUNDS; ++r) {
    const int a = r * kPermSmallThreads + tid;
    ev[r] = a < A ? __ldg(idx + a) : -1;
  }
#pragma unroll
  for (int r = 0; r < ROUNDS; ++r) {
    const int a = r * kPermSmallThreads + tid;
    if (a < A && (ev[r] < 0 || ev[r] >= E)) {
      report_status(status, MOE_E_DEVICE_DATA);
      ev[r] = -1;
    }
  }
  __syncthreads();

  // pass 1: expert totals and per-(source rank, expert) counts
#pragma unroll
  for (int r = 0; r < ROUNDS; ++r) {
    if (r * kPermSmallThreads >= A) break;
    const int a = r * kPermSmallThreads + tid;
    const int e = ev[r];
    const int key = e >= 0 ? ((a / k) / T_loc) * E + e : -1;
    const uint32_t pe = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && (pe & lt) == 0) atomicAdd(&base[e], __popc(pe));
    const uint32_t pk = __match_any_sync(0xffffffffu, key);
    if (key >= 0 && (pk & lt) == 0) atomicAdd(src_cnt + key, __popc(pk));
  }
  __syncthreads();
  // counts and offsets: warp 0 scans the totals (8 experts per lane at most)
  if (warp == 0) {
    constexpr int PER = kPermSmallMaxE / 32;
    int v[PER], local = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane * PER + i;
      v[i] = e < E ? base[e] : 0;
      local += v[i];
    }
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    int run = incl - local;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane * PER + i;
      if (e < E) {
        counts[e] = v[i];
        offsets[e] = capacity ? e * capacity : run;
        base[e] = run;
      }
      run += v[i];
    }
    if (lane == 31) offsets[E] = capacity ? E * capacity : run;
  }
  __syncthreads();

  // pass 2: stable ranks, 1024 assignments per round in index order
#pragma unroll
  for (int r = 0; r < ROUNDS; ++r) {
    if (r * kPermSmallThreads >= A) break;
    const int a = r * kPermSmallThreads + tid;
    const int e = ev[r];
    const uint32_t pe = __match_any_sync(0xffffffffu, e);
    const int lrank = __popc(pe & lt);
    if (e >= 0 && lrank == 0) tab[warp * ld + e] = (r << 16) | __popc(pe);
    __syncthreads();
    // warp w scans experts w, w + 32, ...: lane l holds warp l's count
    for (int e2 = warp; e2 < E; e2 += 32) {
      const int tv = tab[lane * ld + e2];
      const int c = (tv >> 16) == r ? (tv & 0xffff) : 0;
      int incl = c;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      const int before = seen[e2];
      pre[lane * ld + e2] = before + incl - c;
      __syncwarp();
      if (lane == 31) seen[e2] = before + incl;
    }
    __syncthreads();
    if (a < A) {
      int row = -1;
      if (e >= 0) {
        const int rank = pre[warp * ld + e] + lrank;
        if (capacity) row = rank < capacity ? e * capacity + rank : -1;
        else row = base[e] + rank;
      }
      inv[a] = row;
      if (row >= 0) order[row] = a;
    }
  }
}

// ---------------------------------------------------------------------------
// Row moves.  A warp copies one token row of vec 16-byte vectors to up to k
// destination rows (lane j < k holds destination row j, or -1): it loads
// 32*V vectors (V per lane) before storing any, so a row of up to 32*V
// vectors costs one memory round trip.
// ---------------------------------------------------------------------------
template <int V>
__device__ __forceinline__ void move_row(const uint4* __restrict__ src, int vec, int my_row,
                                         int k, uint4* __restrict__ dst, int lane) {
  for (int v0 = 0; v0 < vec; v0 += 32 * V) {
    uint4 buf[V];
#pragma unroll
    for (int u = 0; u < V; ++u) {
      const int v = v0 + u * 32 + lane;
      if (v < vec) buf[u] = __ldg(src + v);
    }
    for (int j = 0; j < k; ++j) {
      const int row = __shfl_sync(0xffffffffu, my_row, j);
      if (row < 0) continue;
      uint4* d = dst + size_t(row) * vec;
#pragma unroll
      for (int u = 0; u < V; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < vec) d[v] = buf[u];
      }
    }
  }
}

// The FP8 form of move_row: the row's absmax (warp reduction), then its e4m3
// codes (8 per 16-byte vector of bf16) and the row's scale written to each
// destination row.  scale = absmax / 448 and the factor 448 / absmax are one
// correctly rounded division each (1 for an all-zero row); each code is one
// fp32 product and one conversion.  A row of up to 32*V vectors stays in
// registers between the two passes; a longer one is read twice (the second
// time from L1/L2).
template <int V>
__device__ __forceinline__ void quantize_row(const uint4* __restrict__ src, int vec, int my_row,
                                             int k, uint2* __restrict__ dst_codes,
                                             float* __restrict__ dst_scale, int lane) {
  uint4 buf[V];
  float amax = 0.0f;
  for (int v0 = 0; v0 < vec; v0 += 32 * V) {
#pragma unroll
    for (int u = 0; u < V; ++u) {
      const int v = v0 + u * 32 + lane;
      buf[u] = v < vec ? __ldg(src + v) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < V; ++u) {
      const uint32_t w[4] = {buf[u].x, buf[u].y, buf[u].z, buf[u].w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        amax = fmaxf(amax, fmaxf(fabsf(bf16lo(w[i])), fabsf(bf16hi(w[i]))));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float scale = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  const float inv = amax > 0.0f ? __fdiv_rn(448.0f, amax) : 1.0f;
  if (lane < k && my_row >= 0) dst_scale[my_row] = scale;
  const bool one_pass = vec <= 32 * V;
  for (int v0 = 0; v0 < vec; v0 += 32 * V) {
    if (!one_pass) {
#pragma unroll
      for (int u = 0; u < V; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < vec) buf[u] = __ldg(src + v);
      }
    }
    uint2 code[V];
#pragma unroll
    for (int u = 0; u < V; ++u) {
      const uint4 w = buf[u];
      code[u].x = fp8x4(__fmul_rn(bf16lo(w.x), inv), __fmul_rn(bf16hi(w.x), inv),
                        __fmul_rn(bf16lo(w.y), inv), __fmul_rn(bf16hi(w.y), inv));
      code[u].y = fp8x4(__fmul_rn(bf16lo(w.z), inv), __fmul_rn(bf16hi(w.z), inv),
                        __fmul_rn(bf16lo(w.w), inv), __fmul_rn(bf16hi(w.w), inv));
    }
    for (int j = 0; j < k; ++j) {
      const int row = __shfl_sync(0xffffffffu, my_row, j);
      if (row < 0) continue;
      uint2* d = dst_codes + size_t(row) * vec;
#pragma unroll
      for (int u = 0; u < V; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < vec) d[v] = code[u];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// 3. row move: one warp per token, x[t] read once, written to its k rows.
// ---------------------------------------------------------------------------
template <int V>
__global__ void __launch_bounds__(256) row_scatter_kernel(const uint4* __restrict__ x, int T,
                                                          int vec_per_row, int k,
                                                          const int32_t* __restrict__ rows,
                                                          uint4* __restrict__ dst) {
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  const int my_row = (lane < k) ? __ldg(rows + size_t(t) * k + lane) : -1;
  move_row<V>(x + size_t(t) * vec_per_row, vec_per_row, my_row, k, dst, lane);
}

// Capacity mode: set the order entry of the grouped buffer's padding rows to
// -1 and zero the rows (when the buffer is given).  Row r belongs to expert e = r / cap and is padding when
// r - e*cap >= min(counts[e], cap).  One warp per row, grid-stride.
__global__ void __launch_bounds__(256) perm_pad_kernel(const int32_t* __restrict__ counts,
                                                       int capacity, int R, int vec_per_row,
                                                       int32_t* __restrict__ order,
                                                       uint4* __restrict__ x_sorted) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < R; r += warps) {
    const int e = r / capacity;
    if (r - e * capacity < min(__ldg(counts + e), capacity)) continue;
    if (lane == 0) order[r] = -1;
    if (x_sorted == nullptr) continue;
    uint4* row = x_sorted + size_t(r) * vec_per_row;
    for (int v = lane; v < vec_per_row; v += 32) row[v] = make_uint4(0, 0, 0, 0);
  }
}

// ---------------------------------------------------------------------------
// Expert-parallel layout
// ---------------------------------------------------------------------------
// One CTA per source rank s.  With before[e] = assignments to e from ranks
// < s (kept rows of a rank are a prefix of its ranks in the expert):
//   kept[e]      = c[s][e], or clamp(cap - before[e], 0, c[s][e]) with a capacity
//   sbase[s][e]  = s*T_loc*k + sum_{e'<e} kept[e'] - before[e], so that
//                  slot(a) = sbase[s][e] + rank(a)
//   C[s][q]      = sum of kept[e] over q's experts [q*G, (q+1)*G), G = E/n_ep
//   send_off[s][q] = sum_{e<q*G} kept[e]
//   recv_off[q][s] = rows q received from ranks < s
//                  = sum over q's experts of before[e] (or min(before[e], cap)).
//
// CTA (s, j) computes the tables of source rank s (every CTA of the rank
// recomputes them; CTA (s, 0) writes them out) and then takes the rank's
// assignments j*apc .. (j+1)*apc - 1 (apc a multiple of k, so whole tokens):
// slot(a) = sbase[s][e] + rank(a) for each kept assignment a (send_pos[a], -1
// when dropped; send_idx[slot] = a), marks the slots of that range past the
// rank's kept rows empty (send_idx = -1), and, with a send buffer, moves its
// tokens' rows to their slots (one warp per token, x[t] read once) and zeroes
// the empty slots' rows.
constexpr int kEpMaxPerCta = 2048;  // assignments placed per CTA at most

template <int V, bool FP8>
__global__ void __launch_bounds__(kPermThreads) ep_layout_kernel(
    const int32_t* __restrict__ src_cnt, const int32_t* __restrict__ idx,
    const int32_t* __restrict__ inv, const int32_t* __restrict__ offsets, int n_ep, int E, int k,
    int T_loc, int capacity, int apc, int32_t* __restrict__ C, int32_t* __restrict__ send_off,
    int32_t* __restrict__ recv_off, int32_t* __restrict__ send_idx,
    int32_t* __restrict__ send_pos, const uint4* __restrict__ x, int vec_per_row,
    uint4* __restrict__ send_buf, uint2* __restrict__ send_fp8,
    float* __restrict__ send_scale) {
  extern __shared__ int32_t sm[];
  int32_t* kept = sm;              // [E + 1] -> exclusive prefix
  int32_t* recv = sm + E + 1;      // [E + 1] -> exclusive prefix
  int32_t* bef = sm + 2 * (E + 1); // [E]
  int32_t* slot_s = sm + 3 * E + 2;  // [apc]: slot of each assignment of the range
  const int s = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int b = 0, sp = 0;
    for (; sp + 4 <= s; sp += 4) {
      int v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = __ldg(src_cnt + size_t(sp + u) * E + e);
      b += v[0] + v[1] + v[2] + v[3];
    }
    for (; sp < s; ++sp) b += __ldg(src_cnt + size_t(sp) * E + e);
    const int c = __ldg(src_cnt + size_t(s) * E + e);
    kept[e] = capacity ? max(0, min(capacity - b, c)) : c;
    recv[e] = capacity ? min(b, capacity) : b;
    bef[e] = b;
  }
  __syncthreads();
  const int kept_all = block_exclusive_scan(kept, E);
  const int recv_all = block_exclusive_scan(recv, E);
  if (threadIdx.x == 0) {
    kept[E] = kept_all;
    recv[E] = recv_all;
  }
  __syncthreads();
  const int G = E / n_ep;
  if (blockIdx.y == 0) {
    for (int q = threadIdx.x; q < n_ep; q += blockDim.x) {
      C[size_t(s) * n_ep + q] = kept[(q + 1) * G] - kept[q * G];
      send_off[size_t(s) * n_ep + q] = kept[q * G];
      recv_off[size_t(q) * n_ep + s] = recv[(q + 1) * G] - recv[q * G];
    }
  }
  const int rpr = T_loc * k;
  const int base = s * rpr;
  for (int j = blockIdx.y; j * apc < rpr; j += gridDim.y) {
    const int i0 = j * apc, i_end = min(rpr, i0 + apc);
    for (int i = i0 + threadIdx.x; i < i_end; i += blockDim.x) {
      const int a = base + i;
      const int e = __ldg(idx + a);
      const int row = __ldg(inv + a);
      int p = -1;
      if (row >= 0 && e >= 0 && e < E) {
        p = base + kept[e] + (row - __ldg(offsets + e)) - bef[e];
        send_idx[p] = a;
      }
      send_pos[a] = p;
      slot_s[i - i0] = p;
      if (i >= kept_all) send_idx[a] = -1;  // slot a is past the rank's kept rows
    }
    if (x == nullptr) continue;
    __syncthreads();
    // the range's token rows to their slots (bf16, or e4m3 codes and a scale)
    for (int t = (base + i0) / k + warp; t < (base + i_end) / k; t += kPermThreads / 32) {
      const int my_slot = lane < k ? slot_s[t * k - base - i0 + lane] : -1;
      if (FP8)
        quantize_row<V>(x + size_t(t) * vec_per_row, vec_per_row, my_slot, k, send_fp8,
                        send_scale, lane);
      else
        move_row<V>(x + size_t(t) * vec_per_row, vec_per_row, my_slot, k, send_buf, lane);
    }
    // empty slots of the range (past the rank's kept rows): zero rows (codes
    // and scale 0 in FP8)
    for (int i = max(i0, kept_all) + warp; i < i_end; i += kPermThreads / 32) {
      if (FP8) {
        if (lane == 0) send_scale[base + i] = 0.0f;
        uint2* d = send_fp8 + size_t(base + i) * vec_per_row;
        for (int v = lane; v < vec_per_row; v += 32) d[v] = make_uint2(0, 0);
      } else {
        uint4* d = send_buf + size_t(base + i) * vec_per_row;
        for (int v = lane; v < vec_per_row; v += 32) d[v] = make_uint4(0, 0, 0, 0);
      }
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// The whole permute in one cooperative launch, for layers with few experts
// (E <= kFusedMaxE) and more assignments than the one-CTA path takes.  CTA c
// owns tokens [c*tpc, (c+1)*tpc) and their assignments:
//   1. it loads its expert ids, counts its slice per expert into
//      slice_hist[c] (CTA 0 also clears the per-(rank, expert) counts), and
//      meets the other CTAs at a grid barrier; when the table (E x CTAs) is
//      large it also adds the counts into its group's sums (groups of
//      kFusedGroupCtas CTAs);
//   2. its slice's base in each expert (the sum over earlier CTAs) and the
//      expert totals: read from the whole table when it is small, else from
//      the earlier groups' sums plus the counts of the earlier CTAs of its own
//      group (totals: all groups' sums); then the totals are scanned into the
//      segment offsets (CTA 0 writes them);
//   3. stable ranks inside the slice in index order (warp match/popc, then a
//      scan over the 8 warps), giving inv and order; per-(rank, expert)
//      counts by warp-aggregated atomics; then each warp starts loading its
//      first rows (registers);
//   4. capacity padding rows: order -1 and zero rows (grid-stride);
//   5. its tokens' rows: one warp per token, x[t] written to its k rows, in
//      4 KB chunks through two register buffers (load the next, store this).
// The grid barriers are bounded: after 1 s one records MOE_E_DEVICE_TIMEOUT and
// lets the CTA continue (outputs then unreliable, never a hang).
// ---------------------------------------------------------------------------
constexpr int kFusedThreads = 256;
constexpr int kFusedRounds = 8;        // 2048 assignments per CTA at most
constexpr int kFusedChunk = 8;         // 16-byte vectors per lane in each row buffer
constexpr int kFusedDirectWords = 16 * kFusedThreads;  // slice tables read whole up to this size

__device__ __forceinline__ unsigned int ld_volatile_u32(const unsigned int* p) {
  return *reinterpret_cast<const volatile unsigned int*>(p);
}

// The CTA's last thread arrives and waits; its fence waits for that thread's
// own outstanding memory operations, so it must have no slow loads in flight.
__device__ void grid_barrier(unsigned int* count, unsigned int* gen, int* status) {
  __syncthreads();
  if (threadIdx.x == blockDim.x - 1) {
    const unsigned int g = ld_volatile_u32(gen);
    __threadfence();
    if (atomicAdd(count, 1u) == gridDim.x - 1) {
      atomicExch(count, 0u);
      __threadfence();
      atomicAdd(gen, 1u);
    } else {
      const uint64_t t0 = global_ns();
      while (ld_volatile_u32(gen) == g) {
        if (global_ns() - t0 > 1000000000ull) {
          report_status(status, MOE_E_DEVICE_TIMEOUT);
          break;
        }
      }
    }
    __threadfence();
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kFusedThreads) perm_fused_kernel(
    const int32_t* __restrict__ idx, const uint4* __restrict__ x, int T, int E, int k, int T_loc,
    int n_ep, int capacity, int tpc, int vec_per_row, int32_t* __restrict__ slice_hist,
    int32_t* __restrict__ src_cnt, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ inv, int32_t* __restrict__ order, uint4* __restrict__ x_sorted,
    int* status, unsigned int* bar_count, unsigned int* bar_gen, unsigned int* seq_word,
    int32_t* __restrict__ grp_sums) {
  __shared__ int32_t h[kFusedMaxE];          // slice histogram, then running rank base
  __shared__ int32_t tot[kFusedMaxE];        // expert totals
  __shared__ int32_t seg[kFusedMaxE + 1];    // segment offsets (dropless)
  __shared__ int32_t wcnt[kFusedThreads / 32][kFusedMaxE];
  __shared__ int32_t rows_s[kFusedRounds * kFusedThreads];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t lt = (1u << lane) - 1u;
  const int c = blockIdx.x;
  const int t0 = c * tpc, t1 = min(T, t0 + tpc);
  const int n_a = t1 > t0 ? (t1 - t0) * k : 0;
  const int a0 = t0 * k;
  // every CTA reads the sequence number before the barrier, CTA 0 advances it
  // after: this launch adds into buffer seq & 1 (zero on entry) and clears the
  // other buffer for the next launch
  const unsigned int seq = ld_volatile_u32(seq_word);
  constexpr int kGrpBuf = kFusedMaxE * kFusedMaxGroups;
  int32_t* gsum = grp_sums + (seq & 1u) * kGrpBuf;
  const int q = c / kFusedGroupCtas;  // the CTA's group

  // 1. ids, the slice histogram and the group sums
  for (int e = tid; e < E; e += kFusedThreads) h[e] = 0;
  if (c == 0)
    for (int i = tid; i < n_ep * E; i += kFusedThreads) src_cnt[i] = 0;
  int ev[kFusedRounds];
#pragma unroll
  for (int r = 0; r < kFusedRounds; ++r) {
    const int i = r * kFusedThreads + tid;
    ev[r] = i < n_a ? __ldg(idx + a0 + i) : -1;
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < kFusedRounds; ++r) {
    if (r * kFusedThreads >= n_a) break;
    const int i = r * kFusedThreads + tid;
    int e = ev[r];
    if (i < n_a && (e < 0 || e >= E)) {
      report_status(status, MOE_E_DEVICE_DATA);
      e = -1;
    }
    ev[r] = e;
    const uint32_t pe = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && (pe & lt) == 0) atomicAdd(&h[e], __popc(pe));
  }
  __syncthreads();
  // expert-major table [E][kFusedMaxCtas], so that step 2 reads each
  // expert's words as contiguous, 16-byte aligned runs; with a large table
  // the counts also go into the group sums [E][kFusedMaxGroups]
  const bool direct = E * int(gridDim.x) <= kFusedDirectWords;  // the same in every CTA
  for (int e = tid; e < E; e += kFusedThreads) {
    const int v = h[e];
    slice_hist[e * kFusedMaxCtas + c] = v;
    if (!direct && v) atomicAdd(gsum + e * kFusedMaxGroups + q, v);
  }
  // the row loads go out only now, behind the id loads and the histogram, so
  // that they overlap the barrier and steps 2-3 rather than delay them
  // The warp's rows move as a sequence of items of up to 32 * kFusedChunk
  // vectors (its tokens t0 + warp, t0 + warp + 8, ..., each cut into cpr
  // chunks), through two register buffers: the next item loads while the
  // current one is stored.
  uint4 buf_a[kFusedChunk], buf_b[kFusedChunk];
  const int cpr = (vec_per_row + 32 * kFusedChunk - 1) / (32 * kFusedChunk);
  const int my_tokens = t1 > t0 + warp ? (t1 - t0 - warp + kFusedThreads / 32 - 1) /
                                             (kFusedThreads / 32) : 0;
  const int n_items = x_sorted != nullptr ? my_tokens * cpr : 0;
  auto load_item = [&](uint4 (&b)[kFusedChunk], int it) {
    const int t = t0 + warp + (it / cpr) * (kFusedThreads / 32);
    const int v0 = (it % cpr) * 32 * kFusedChunk;
    const uint4* src = x + size_t(t) * vec_per_row + v0;
#pragma unroll
    for (int u = 0; u < kFusedChunk; ++u)
      if (v0 + u * 32 + lane < vec_per_row) b[u] = __ldg(src + u * 32 + lane);
  };
  grid_barrier(bar_count, bar_gen, status);

  if (c == 0 && !direct) {
    if (tid == 0) *seq_word = seq + 1u;
    int32_t* other = grp_sums + ((seq + 1u) & 1u) * kGrpBuf;
    for (int i = tid; i < kGrpBuf / 4; i += kFusedThreads)
      reinterpret_cast<int4*>(other)[i] = make_int4(0, 0, 0, 0);
  }

  // 2. the slice's base in each expert and the expert totals, read by P
  // threads per expert in one round of loads: from the whole table when it
  // is small (16-byte loads), else from the sums of the earlier groups plus
  // the counts of the group's earlier CTAs (at most kFusedMaxGroups +
  // kFusedGroupCtas words per expert; the totals are the sums of all groups)
  {
    int P = 32;  // threads per expert (a power of two, P * E <= kFusedThreads)
    while (P > 1 && P * E > kFusedThreads) P >>= 1;
    const int e = tid / P, p = tid - e * P;
    int before = 0, total = 0;
    if (direct) {
      // E * gridDim.x <= kFusedDirectWords and P > kFusedThreads / (2E) bound
      // the 16-byte words per thread by kDirectMax
      constexpr int kDirectMax = kFusedDirectWords / (4 * (kFusedThreads / 2));
      const int n4 = (int(gridDim.x) + 3) / 4;
      int4 v[kDirectMax];
      if (e < E) {
        const int4* row = reinterpret_cast<const int4*>(slice_hist + e * kFusedMaxCtas);
#pragma unroll
        for (int i = 0; i < kDirectMax; ++i) {
          const int j = p + i * P;
          v[i] = j < n4 ? __ldcg(row + j) : make_int4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < kDirectMax; ++i) {
          const int w = 4 * (p + i * P);  // first CTA of the word
          const int g = int(gridDim.x);
          const int x0 = w < g ? v[i].x : 0, x1 = w + 1 < g ? v[i].y : 0;
          const int x2 = w + 2 < g ? v[i].z : 0, x3 = w + 3 < g ? v[i].w : 0;
          total += x0 + x1 + x2 + x3;
          before += (w < c ? x0 : 0) + (w + 1 < c ? x1 : 0) + (w + 2 < c ? x2 : 0) +
                    (w + 3 < c ? x3 : 0);
        }
      }
    } else {
      // 16-byte words of the expert's rows: kG4 of group sums (word j holds
      // groups 4j..4j+3), then kS4 of its group's slice counts (CTAs c_first +
      // 4j'..); the P threads of the expert take words p, p + P, ...
      const int nq = (int(gridDim.x) + kFusedGroupCtas - 1) / kFusedGroupCtas;
      const int c_first = q * kFusedGroupCtas;
      constexpr int kG4 = kFusedMaxGroups / 4, kS4 = kFusedGroupCtas / 4;
      constexpr int kW4 = kG4 + kS4;
      int4 v[kW4];
      if (e < E) {
        const int4* gs = reinterpret_cast<const int4*>(gsum + e * kFusedMaxGroups);
        const int4* hs = reinterpret_cast<const int4*>(slice_hist + e * kFusedMaxCtas + c_first);
#pragma unroll
        for (int i = 0; i < kW4; ++i) {
          const int j = p + i * P;
          const bool load = j < kG4 ? 4 * j < nq : (j < kW4 && c_first + 4 * (j - kG4) < c);
          v[i] = load ? __ldcg(j < kG4 ? gs + j : hs + (j - kG4)) : make_int4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < kW4; ++i) {
          const int j = p + i * P;
          const int x4[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (j < kG4) {
              const int gq = 4 * j + u;  // group
              if (gq < nq) total += x4[u];
              if (gq < q) before += x4[u];
            } else if (j < kW4) {
              if (c_first + 4 * (j - kG4) + u < c) before += x4[u];
            }
          }
        }
      }
    }
    for (int off = P >> 1; off > 0; off >>= 1) {
      before += __shfl_xor_sync(0xffffffffu, before, off);
      total += __shfl_xor_sync(0xffffffffu, total, off);
    }
    if (e < E && p == 0) {
      h[e] = before;
      tot[e] = total;
      if (c == 0) counts[e] = total;
    }
  }
  __syncthreads();
  if (warp == 0) {
    // lane L scans experts kPer*L .. kPer*L + kPer - 1
    constexpr int kPer = kFusedMaxE / 32;
    int loc[kPer];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = lane * kPer + i;
      loc[i] = e < E ? tot[e] : 0;
      sum += loc[i];
    }
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    int run = incl - sum;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = lane * kPer + i;
      if (e < E) seg[e] = run;
      run += loc[i];
    }
    if (lane == 31) seg[E] = incl;
  }
  __syncthreads();
  if (c == 0) {
    for (int e = tid; e < E; e += kFusedThreads) offsets[e] = capacity ? e * capacity : seg[e];
    if (tid == 0) offsets[E] = capacity ? E * capacity : seg[E];
  }

  // 3. stable ranks inside the slice, rows, per-(rank, expert) counts
#pragma unroll
  for (int r = 0; r < kFusedRounds; ++r) {
    if (r * kFusedThreads >= n_a) break;
    const int i = r * kFusedThreads + tid;
    const int a = a0 + i;
    const int e = ev[r];
    for (int q = tid; q < (kFusedThreads / 32) * E; q += kFusedThreads) wcnt[q / E][q % E] = 0;
    __syncthreads();
    const uint32_t pe = __match_any_sync(0xffffffffu, e);
    const int lrank = __popc(pe & lt);
    if (e >= 0 && lrank == 0) wcnt[warp][e] = __popc(pe);
    __syncthreads();
    if (tid < E) {
      int run = h[tid];
#pragma unroll
      for (int w = 0; w < kFusedThreads / 32; ++w) {
        const int v = wcnt[w][tid];
        wcnt[w][tid] = run;
        run += v;
      }
      h[tid] = run;
    }
    __syncthreads();
    int row = -1;
    if (e >= 0) {
      const int rank = wcnt[warp][e] + lrank;
      if (capacity) row = rank < capacity ? e * capacity + rank : -1;
      else row = seg[e] + rank;
    }
    if (i < n_a) {
      inv[a] = row;
      if (row >= 0) order[row] = a;
      rows_s[i] = row;
    }
    const int key = e >= 0 ? ((a / k) / T_loc) * E + e : -1;
    const uint32_t pk = __match_any_sync(0xffffffffu, key);
    if (key >= 0 && (pk & lt) == 0) atomicAdd(src_cnt + key, __popc(pk));
    __syncthreads();
  }

  // the first two row items load now, behind the small loads and stores of
  // steps 1-3 (which queue behind row loads issued earlier: a timestamp probe
  // put steps 2 and 3 at 4 us each with the loads in flight)
  if (n_items > 0) load_item(buf_a, 0);
  if (n_items > 1) load_item(buf_b, 1);

  // 4. capacity padding rows
  if (capacity) {
    const int R = E * capacity;
    const int gw = (c * kFusedThreads + tid) >> 5, nw = (gridDim.x * kFusedThreads) >> 5;
    for (int rr = gw; rr < R; rr += nw) {
      const int e = rr / capacity;
      if (rr - e * capacity < min(tot[e], capacity)) continue;
      if (lane == 0) order[rr] = -1;
      if (x_sorted == nullptr) continue;
      uint4* dst = x_sorted + size_t(rr) * vec_per_row;
      for (int v = lane; v < vec_per_row; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
    }
  }

  // 5. the slice's token rows, one warp per token, item by item
  if (x_sorted == nullptr) return;
  auto store_item = [&](const uint4 (&b)[kFusedChunk], int it) {
    const int t = t0 + warp + (it / cpr) * (kFusedThreads / 32);
    const int v0 = (it % cpr) * 32 * kFusedChunk;
    const int my_row = lane < k ? rows_s[(t - t0) * k + lane] : -1;
    for (int j = 0; j < k; ++j) {
      const int row = __shfl_sync(0xffffffffu, my_row, j);
      if (row < 0) continue;
      uint4* d = x_sorted + size_t(row) * vec_per_row + v0;
#pragma unroll
      for (int u = 0; u < kFusedChunk; ++u)
        if (v0 + u * 32 + lane < vec_per_row) d[u * 32 + lane] = b[u];
    }
  };
  for (int it = 0; it < n_items; it += 2) {
    store_item(buf_a, it);
    if (it + 2 < n_items) load_item(buf_a, it + 2);
    if (it + 1 < n_items) {
      store_item(buf_b, it + 1);
      if (it + 3 < n_items) load_item(buf_b, it + 3);
    }
  }
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
// Blocks of 256 threads for a grid-stride pass with one warp per row.
static int row_grid(long long rows) {
  const long long want = (rows + 7) / 8;
  const long long cap = 8LL * device_sm_count();
  return int(want < cap ? (want > 0 ? want : 1) : cap);
}

int launch_row_scatter(const void* x, int T, int d, int k, const int32_t* rows, void* dst,
                       cudaStream_t st) {
  const int vec = d / 8;  // 16-byte vectors per row
  // vectors per lane loaded before any store: rows of up to 256 vectors fit 8
  // (fewer registers, more warps per SM); longer rows take 16 at a time
  if (vec <= 256)
    row_scatter_kernel<8><<<(T + 7) / 8, 256, 0, st>>>(static_cast<const uint4*>(x), T, vec, k,
                                                      rows, static_cast<uint4*>(dst));
  else
    row_scatter_kernel<16><<<(T + 7) / 8, 256, 0, st>>>(static_cast<const uint4*>(x), T, vec, k,
                                                       rows, static_cast<uint4*>(dst));
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_E_CUDA;
}

// CTAs of perm_fused_kernel that fit on the device at once (cached per device).
static int fused_resident_ctas() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 0;
  }
  if (cache[dev] == 0) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, perm_fused_kernel,
                                                      kFusedThreads, 0) != cudaSuccess) {
      cudaGetLastError();
      per_sm = 0;
    }
    int coop = 0;
    if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess) {
      cudaGetLastError();
      coop = 0;
    }
    cache[dev] = coop ? per_sm * device_sm_count() : -1;
  }
  return cache[dev];
}

// The one-launch permute; MOE_E_SHAPE when the batch needs more than one wave of
// CTAs (the caller then takes the multi-launch path).
static int launch_permute_fused(const moe_cfg& c, const void* x, const int32_t* idx,
                                int32_t* counts, int32_t* offsets, int32_t* order, int32_t* inv,
                                void* x_sorted, void* ws, cudaStream_t st) {
  const int resident = fused_resident_ctas();
  if (resident <= 0) return MOE_E_SHAPE;
  // at most two CTAs per SM: more CTAs cost more in the barrier and in step 2
  // than they add to the row moves (measured: Mixtral-shaped permute 23 against
  // 26 us with three per SM)
  int g_max = resident < 2 * device_sm_count() ? resident : 2 * device_sm_count();
  if (g_max > kFusedMaxCtas) g_max = kFusedMaxCtas;
  int tpc = (c.T + g_max - 1) / g_max;
  if (tpc * c.k > kFusedRounds * kFusedThreads) return MOE_E_SHAPE;
  int grid = (c.T + tpc - 1) / tpc;
  const WsLayout L = ws_layout(c);
  const int32_t* idx_p = idx;
  const uint4* x_p = static_cast<const uint4*>(x);
  int T = c.T, E = c.E, k = c.k, T_loc = c.T / c.n_ep, n_ep = c.n_ep, cap = c.capacity;
  int vec = c.d / 8;
  int32_t* slice_hist = ws_ptr<int32_t>(ws, L.slice_hist);
  int32_t* src_cnt = ws_ptr<int32_t>(ws, L.src_cnt);
  uint4* xs = static_cast<uint4*>(x_sorted);
  int* status = ws_ptr<int>(ws, L.status);
  unsigned int* bar_count = ws_ptr<unsigned int>(ws, L.bar_count);
  unsigned int* bar_gen = ws_ptr<unsigned int>(ws, L.bar_gen);
  unsigned int* seq = ws_ptr<unsigned int>(ws, L.perm_seq);
  int32_t* grp = ws_ptr<int32_t>(ws, L.grp_sums);
  void* args[] = {&idx_p, &x_p, &T, &E, &k, &T_loc, &n_ep, &cap, &tpc, &vec, &slice_hist,
                  &src_cnt, &counts, &offsets, &inv, &order, &xs, &status, &bar_count,
                  &bar_gen, &seq, &grp};
  const cudaError_t e = cudaLaunchCooperativeKernel(
      reinterpret_cast<const void*>(perm_fused_kernel), dim3(grid), dim3(kFusedThreads), args,
      0, st);
  note_launches(1);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MOE_E_CUDA;
  }
  return MOE_OK;
}

int launch_permute(const moe_cfg& c, const void* x, const int32_t* idx, int32_t* counts,
                   int32_t* offsets, int32_t* order, int32_t* inv, void* x_sorted, void* ws,
                   cudaStream_t st) {
  const WsLayout L = ws_layout(c);
  const int A = c.T * c.k;
  int32_t* status = ws_ptr<int32_t>(ws, L.status);
  unsigned int* done = ws_ptr<unsigned int>(ws, L.done_ctas);
  int32_t* src_cnt = ws_ptr<int32_t>(ws, L.src_cnt);
  int32_t* chunk_hist = ws_ptr<int32_t>(ws, L.chunk_hist);
  if (A > kPermSmallMaxA && c.E <= kFusedMaxE && c.k <= 32) {
    const int rc = launch_permute_fused(c, x, idx, counts, offsets, order, inv, x_sorted, ws, st);
    if (rc != MOE_E_SHAPE) return rc;   // MOE_E_SHAPE: the batch does not fit one wave
  }
  if (A <= kPermSmallMaxA && c.E <= kPermSmallMaxE) {
    // one CTA does the histogram, the scans and the ranks
    static PerDeviceOnce once;
    const int attr_rc = once.run([] {
      const cudaError_t e = cudaFuncSetAttribute(
          perm_index_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
          int((64 * (kPermSmallMaxE + 1) + 2 * kPermSmallMaxE) * 4));
      if (e != cudaSuccess) cudaGetLastError();
      return e == cudaSuccess ? MOE_OK : MOE_E_CUDA;
    });
    if (attr_rc != MOE_OK) return attr_rc;
    const size_t smem = size_t(64 * (c.E + 1) + 2 * c.E) * 4;
    perm_index_small_kernel<<<1, kPermSmallThreads, smem, st>>>(
        idx, A, c.E, c.k, c.T / c.n_ep, c.n_ep, c.capacity, src_cnt, counts, offsets, inv, order,
        status);
    note_launches(1);
  } else {
    if (cudaMemsetAsync(src_cnt, 0, size_t(c.n_ep) * c.E * 4, st) != cudaSuccess)
      return MOE_E_CUDA;
    perm_hist_kernel<<<L.n_chunks, kPermThreads, c.E * 4, st>>>(
        idx, A, c.E, c.k, c.T / c.n_ep, c.capacity, chunk_hist, src_cnt, counts, offsets, status,
        done);
    perm_rank_kernel<<<L.n_chunks, kPermThreads, 8 * c.E * 4, st>>>(
        idx, A, c.E, c.capacity, chunk_hist, offsets, inv, order);
    note_launches(2);
  }
  if (c.capacity) {
    const int R = c.E * c.capacity;
    perm_pad_kernel<<<row_grid(R), 256, 0, st>>>(counts, c.capacity, R, c.d / 8, order,
                                                 static_cast<uint4*>(x_sorted));
    note_launches(1);
  }
  if (cudaGetLastError() != cudaSuccess) return MOE_E_CUDA;
  if (x_sorted == nullptr) return MOE_OK;  // indices only: the rows are gathered later
  return launch_row_scatter(x, c.T, c.d, c.k, inv, x_sorted, st);
}

int launch_ep_layout(const moe_cfg& c, const int32_t* idx, const int32_t* offsets,
                     const int32_t* inv, int32_t* C, int32_t* send_off, int32_t* recv_off,
                     int32_t* send_idx, const void* x, void* send_buf, void* ws, cudaStream_t st,
                     void* send_fp8, float* send_scale) {
  const WsLayout L = ws_layout(c);
  const int T_loc = c.T / c.n_ep;
  int32_t* src_cnt = ws_ptr<int32_t>(ws, L.src_cnt);
  int32_t* send_pos = ws_ptr<int32_t>(ws, L.send_pos);
  const bool fp8 = x && send_fp8 && send_scale;
  const bool rows = fp8 || (x && send_buf);
  // assignments per CTA: whole tokens; when rows move, one token per warp (as
  // many rows in flight as a plain scatter), else up to kEpMaxPerCta.  (A grid
  // of the CTAs that fit at once, each taking more tokens, measured slower:
  // the skewed layer 41 against 37.5 us, DS-V3 211 against 197 us; with
  // several waves one CTA's tables overlap another's row moves.)
  int tok_per_cta = rows ? kPermThreads / 32 : kEpMaxPerCta / c.k;
  if (tok_per_cta < 1) tok_per_cta = 1;
  const int apc = tok_per_cta * c.k;
  const int per_rank = (T_loc * c.k + apc - 1) / apc;
  const size_t smem = size_t(3 * c.E + 2 + apc) * 4;
  const dim3 grid(c.n_ep, per_rank < 65535 ? per_rank : 65535);
  const uint4* xr = static_cast<const uint4*>(rows ? x : nullptr);
  uint4* sb = static_cast<uint4*>(rows && !fp8 ? send_buf : nullptr);
  uint2* sf = static_cast<uint2*>(fp8 ? send_fp8 : nullptr);
  float* ss = fp8 ? send_scale : nullptr;
  const int vec = c.d / 8;
#define MOE_EP_LAYOUT(V_, F_)                                                                   \
  ep_layout_kernel<V_, F_><<<grid, kPermThreads, smem, st>>>(                                 \
      src_cnt, idx, inv, offsets, c.n_ep, c.E, c.k, T_loc, c.capacity, apc, C, send_off,       \
      recv_off, send_idx, send_pos, xr, vec, sb, sf, ss)
  // vectors per lane held at once: rows of up to 256 vectors take 8 (62
  // registers, four CTAs per SM); longer rows take 16 (one memory round trip
  // for a 4096-wide row: the Mixtral-shaped layout ran 22 against 24 us, in
  // spite of fewer warps per SM)
  if (fp8) {
    if (vec <= 256) MOE_EP_LAYOUT(8, true);
    else MOE_EP_LAYOUT(16, true);
  } else {
    if (vec <= 256) MOE_EP_LAYOUT(8, false);
    else MOE_EP_LAYOUT(16, false);
  }
#undef MOE_EP_LAYOUT
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_E_CUDA;
}

}  // namespace moe
