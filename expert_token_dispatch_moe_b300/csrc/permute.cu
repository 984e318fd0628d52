// Step 2 of the MoE layer: stable grouping of the T*k assignments into
// per-expert segments, plus the simulated expert-parallel send layout.
//
// "Token permutation and grouped GEMMs" (Expert parallelism page): order is
// the stable argsort of the expert ids and inv[order] = arange.  The stable
// rank of an assignment inside its expert comes from histograms and prefix
// sums, never from the order of atomics, so every output is deterministic:
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
// 3. row move: one warp per token, x[t] read once, written to its k rows.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) row_scatter_kernel(const uint4* __restrict__ x, int T,
                                                          int vec_per_row, int k,
                                                          const int32_t* __restrict__ rows,
                                                          uint4* __restrict__ dst) {
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  const int my_row = (lane < k) ? __ldg(rows + size_t(t) * k + lane) : -1;
  const uint4* src = x + size_t(t) * vec_per_row;
  // warp-uniform trip count: every lane takes part in the row broadcasts
  for (int v0 = 0; v0 < vec_per_row; v0 += 32 * 4) {
    uint4 buf[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int v = v0 + u * 32 + lane;
      if (v < vec_per_row) buf[u] = __ldg(src + v);
    }
    for (int j = 0; j < k; ++j) {
      const int row = __shfl_sync(0xffffffffu, my_row, j);
      if (row < 0) continue;
      uint4* d = dst + size_t(row) * vec_per_row;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < vec_per_row) d[v] = buf[u];
      }
    }
  }
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
// recomputes them; CTA (s, 0) writes them out) and then places the rank's
// assignments j*kEpPerCta .. (j+1)*kEpPerCta - 1: slot(a) = sbase[s][e] +
// rank(a) for each kept assignment a (send_pos[a], -1 when dropped;
// send_idx[slot] = a), and marks the rank's slots past its kept rows empty
// (send_idx = -1).
constexpr int kEpPerCta = 1024;  // assignments placed per CTA

__global__ void __launch_bounds__(kPermThreads) ep_layout_kernel(
    const int32_t* __restrict__ src_cnt, const int32_t* __restrict__ idx,
    const int32_t* __restrict__ inv, const int32_t* __restrict__ offsets, int n_ep, int E, int k,
    int T_loc, int capacity, int32_t* __restrict__ C, int32_t* __restrict__ send_off,
    int32_t* __restrict__ recv_off, int32_t* __restrict__ send_idx,
    int32_t* __restrict__ send_pos) {
  extern __shared__ int32_t sm[];
  int32_t* kept = sm;              // [E + 1] -> exclusive prefix
  int32_t* recv = sm + E + 1;      // [E + 1] -> exclusive prefix
  int32_t* bef = sm + 2 * (E + 1); // [E]
  const int s = blockIdx.x;
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
  for (int j = blockIdx.y; j * kEpPerCta < rpr; j += gridDim.y) {
    const int i_end = min(rpr, (j + 1) * kEpPerCta);
    for (int i = j * kEpPerCta + threadIdx.x; i < i_end; i += blockDim.x) {
      const int a = base + i;
      const int e = __ldg(idx + a);
      const int row = __ldg(inv + a);
      int p = -1;
      if (row >= 0 && e >= 0 && e < E) {
        p = base + kept[e] + (row - __ldg(offsets + e)) - bef[e];
        send_idx[p] = a;
      }
      send_pos[a] = p;
      if (i >= kept_all) send_idx[a] = -1;  // slot a is past the rank's kept rows
    }
  }
}

// Zero the send-buffer rows past each rank's kept rows (slot p of rank
// s = p / rows_per_rank is empty when p - s*rows_per_rank >= its kept rows).
// One warp per row, grid-stride.
__global__ void __launch_bounds__(256) ep_pad_kernel(const int32_t* __restrict__ C,
                                                     const int32_t* __restrict__ send_off,
                                                     int n_ep, int rows_per_rank, int A,
                                                     int vec_per_row,
                                                     uint4* __restrict__ send_buf) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int p = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; p < A; p += warps) {
    const int s = p / rows_per_rank;
    const size_t last = size_t(s) * n_ep + n_ep - 1;
    if (p - s * rows_per_rank < __ldg(send_off + last) + __ldg(C + last)) continue;
    uint4* row = send_buf + size_t(p) * vec_per_row;
    for (int v = lane; v < vec_per_row; v += 32) row[v] = make_uint4(0, 0, 0, 0);
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
  row_scatter_kernel<<<(T + 7) / 8, 256, 0, st>>>(static_cast<const uint4*>(x), T, vec, k, rows,
                                                 static_cast<uint4*>(dst));
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_E_CUDA;
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
                     int32_t* send_idx, const void* x, void* send_buf, void* ws,
                     cudaStream_t st) {
  const WsLayout L = ws_layout(c);
  const int A = c.T * c.k;
  const int T_loc = c.T / c.n_ep;
  int32_t* src_cnt = ws_ptr<int32_t>(ws, L.src_cnt);
  int32_t* send_pos = ws_ptr<int32_t>(ws, L.send_pos);
  const size_t smem = size_t(3 * c.E + 2) * 4;
  const int per_rank = (T_loc * c.k + kEpPerCta - 1) / kEpPerCta;
  const dim3 grid(c.n_ep, per_rank < 65535 ? per_rank : 65535);
  ep_layout_kernel<<<grid, kPermThreads, smem, st>>>(src_cnt, idx, inv, offsets, c.n_ep, c.E,
                                                       c.k, T_loc, c.capacity, C, send_off,
                                                       recv_off, send_idx, send_pos);
  note_launches(1);
  if (cudaGetLastError() != cudaSuccess) return MOE_E_CUDA;
  if (x && send_buf) {
    if (c.capacity) {
      ep_pad_kernel<<<row_grid(A), 256, 0, st>>>(C, send_off, c.n_ep, T_loc * c.k, A, c.d / 8,
                                                 static_cast<uint4*>(send_buf));
      note_launches(1);
    }
    return launch_row_scatter(x, c.T, c.d, c.k, send_pos, send_buf, st);
  }
  return MOE_OK;
}

}  // namespace moe
