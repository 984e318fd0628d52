// Step 2 of the MoE layer: stable grouping of the T*k assignments into
// per-expert segments, plus the simulated expert-parallel send layout.
//
// "Token permutation and grouped GEMMs" (Expert parallelism page): order is
// the stable argsort of the expert ids and inv[order] = arange.  The stable
// rank of an assignment inside its expert comes from histograms and prefix
// sums, never from the order of atomics, so every output is deterministic:
//   1. hist:  per 2048-assignment chunk, a histogram over experts (shared-memory
//             atomics: only counts, not order, depend on them); counts per
//             (source rank, expert) for the layout.
//   2. scan:  per expert, exclusive prefix over chunks (chunk bases), totals,
//             and the exclusive prefix over experts (segment offsets).
//   3. rank:  per chunk, warp-ordered match/popc ranks, giving each
//             assignment its row; writes inv and order.
//   4. move:  one warp per token reads x[t] once (16-byte vectors) and writes
//             its k copies.
// Capacity mode keeps rank < cap at row e*cap + rank and zero-fills the rest
// of each segment.
#include "common.cuh"
#include "launch.h"

namespace moe {

constexpr int kPermThreads = 256;
constexpr int kPermPerThread = kPermChunk / kPermThreads;  // 8

// ---------------------------------------------------------------------------
// 1. histogram
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kPermThreads) perm_hist_kernel(
    const int32_t* __restrict__ idx, int A, int E, int k, int T_loc, int32_t* __restrict__ chunk_hist,
    int32_t* __restrict__ src_cnt, int* status) {
  extern __shared__ int32_t h[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
  __syncthreads();
  const int base = blockIdx.x * kPermChunk;
#pragma unroll
  for (int i = 0; i < kPermPerThread; ++i) {
    const int a = base + i * kPermThreads + threadIdx.x;
    if (a < A) {
      const int e = __ldg(idx + a);
      if (e >= 0 && e < E) {
        atomicAdd(&h[e], 1);
        const int s = (a / k) / T_loc;
        atomicAdd(&src_cnt[size_t(s) * E + e], 1);
      } else {
        report_status(status, MOE_E_DEVICE_DATA);
      }
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_hist[size_t(blockIdx.x) * E + e] = h[e];
}

// ---------------------------------------------------------------------------
// 2. scan (one CTA of 1024 threads; E <= 1024)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) perm_scan_kernel(int32_t* __restrict__ chunk_hist,
                                                         int n_chunks, int E, int capacity,
                                                         int32_t* __restrict__ counts,
                                                         int32_t* __restrict__ offsets) {
  __shared__ int32_t warp_tot[32];
  const int e = threadIdx.x;
  int total = 0;
  if (e < E) {
    for (int c = 0; c < n_chunks; ++c) {
      const int v = chunk_hist[size_t(c) * E + e];
      chunk_hist[size_t(c) * E + e] = total;  // becomes the chunk base
      total += v;
    }
    counts[e] = total;
  }
  // exclusive block scan of totals over experts
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = total;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_tot[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += o;
    }
    warp_tot[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int excl = incl - total + (warp > 0 ? warp_tot[warp - 1] : 0);
  if (e < E) offsets[e] = capacity ? e * capacity : excl;
  if (e == E - 1) offsets[E] = capacity ? E * capacity : excl + total;
}

// ---------------------------------------------------------------------------
// 3. stable ranks -> rows
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
// 4. row move: one warp per token, x[t] read once, written to its k rows.
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

// Capacity mode: zero the unfilled rows of each expert segment, order = -1.
__global__ void __launch_bounds__(256) perm_pad_kernel(const int32_t* __restrict__ counts,
                                                       int capacity, int vec_per_row,
                                                       int32_t* __restrict__ order,
                                                       uint4* __restrict__ x_sorted) {
  const int e = blockIdx.x;
  const int kept = min(__ldg(counts + e), capacity);
  const int r0 = e * capacity + kept, r1 = (e + 1) * capacity;
  for (int r = r0 + threadIdx.x; r < r1; r += blockDim.x) order[r] = -1;
  const size_t n = size_t(r1 - r0) * vec_per_row;
  uint4* base = x_sorted + size_t(r0) * vec_per_row;
  for (size_t i = threadIdx.x; i < n; i += blockDim.x) base[i] = make_uint4(0, 0, 0, 0);
}

// ---------------------------------------------------------------------------
// Expert-parallel layout
// ---------------------------------------------------------------------------
// One CTA: kept rows per (source s, expert e), C, send/recv offsets and the
// send-slot base of each (s, e):  slot(a) = s*T_loc*k + sum_{e'<e} kept[s][e']
//                                          + rank(a) - before[s][e]
// where rank(a) is the assignment's stable rank in its expert and before[s][e]
// the assignments to e from ranks < s (kept rows of a rank are a prefix of its
// ranks in the expert).
__global__ void __launch_bounds__(1024) ep_tables_kernel(
    const int32_t* __restrict__ src_cnt, int n_ep, int E, int k, int T_loc, int capacity,
    int32_t* __restrict__ before, int32_t* __restrict__ sbase, int32_t* __restrict__ C,
    int32_t* __restrict__ send_off, int32_t* __restrict__ recv_off) {
  // pass 1: per expert, over sources
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int s = 0; s < n_ep; ++s) {
      const int c = src_cnt[size_t(s) * E + e];
      before[size_t(s) * E + e] = run;
      int kept = c;
      if (capacity) kept = max(0, min(capacity - run, c));
      sbase[size_t(s) * E + e] = kept;  // temporarily: kept count
      run += c;
    }
  }
  __syncthreads();
  // pass 2: per source, over experts (destination = e * n_ep / E, monotone in e)
  for (int s = threadIdx.x; s < n_ep; s += blockDim.x) {
    int run = 0;
    for (int q = 0; q < n_ep; ++q) C[size_t(s) * n_ep + q] = 0;
    for (int e = 0; e < E; ++e) {
      const int kept = sbase[size_t(s) * E + e];
      sbase[size_t(s) * E + e] = s * T_loc * k + run - before[size_t(s) * E + e];
      C[size_t(s) * n_ep + (e * n_ep) / E] += kept;
      run += kept;
    }
    int o = 0;
    for (int q = 0; q < n_ep; ++q) {
      send_off[size_t(s) * n_ep + q] = o;
      o += C[size_t(s) * n_ep + q];
    }
  }
  __syncthreads();
  for (int q = threadIdx.x; q < n_ep; q += blockDim.x) {
    int o = 0;
    for (int s = 0; s < n_ep; ++s) {
      recv_off[size_t(q) * n_ep + s] = o;
      o += C[size_t(s) * n_ep + q];
    }
  }
}

__global__ void __launch_bounds__(256) ep_scatter_kernel(
    const int32_t* __restrict__ idx, const int32_t* __restrict__ inv,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ sbase, int A, int E, int k,
    int T_loc, int32_t* __restrict__ send_idx, int32_t* __restrict__ send_pos) {
  const int a = blockIdx.x * blockDim.x + threadIdx.x;
  if (a >= A) return;
  const int e = __ldg(idx + a);
  const int row = __ldg(inv + a);
  int p = -1;
  if (row >= 0 && e >= 0 && e < E) {
    const int rank = row - __ldg(offsets + e);
    const int s = (a / k) / T_loc;
    p = __ldg(sbase + size_t(s) * E + e) + rank;
    send_idx[p] = a;
  }
  send_pos[a] = p;
}

// Capacity mode: zero the send-buffer rows past each rank's kept rows.
__global__ void __launch_bounds__(256) ep_pad_kernel(const int32_t* __restrict__ C, int n_ep,
                                                     int rows_per_rank, int vec_per_row,
                                                     uint4* __restrict__ send_buf) {
  const int s = blockIdx.x;
  int used = 0;
  for (int q = 0; q < n_ep; ++q) used += __ldg(C + size_t(s) * n_ep + q);
  const size_t n = size_t(rows_per_rank - used) * vec_per_row;
  uint4* base = send_buf + (size_t(s) * rows_per_rank + used) * vec_per_row;
  for (size_t i = threadIdx.x; i < n; i += blockDim.x) base[i] = make_uint4(0, 0, 0, 0);
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
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
  int32_t* src_cnt = ws_ptr<int32_t>(ws, L.src_cnt);
  int32_t* chunk_hist = ws_ptr<int32_t>(ws, L.chunk_hist);
  if (cudaMemsetAsync(src_cnt, 0, size_t(c.n_ep) * c.E * 4, st) != cudaSuccess) return MOE_E_CUDA;
  perm_hist_kernel<<<L.n_chunks, kPermThreads, c.E * 4, st>>>(idx, A, c.E, c.k, c.T / c.n_ep,
                                                              chunk_hist, src_cnt, status);
  perm_scan_kernel<<<1, 1024, 0, st>>>(chunk_hist, L.n_chunks, c.E, c.capacity, counts, offsets);
  perm_rank_kernel<<<L.n_chunks, kPermThreads, 8 * c.E * 4, st>>>(idx, A, c.E, c.capacity,
                                                                  chunk_hist, offsets, inv, order);
  note_launches(3);
  if (c.capacity) {
    perm_pad_kernel<<<c.E, 256, 0, st>>>(counts, c.capacity, c.d / 8, order,
                                         static_cast<uint4*>(x_sorted));
    note_launches(1);
  }
  if (cudaGetLastError() != cudaSuccess) return MOE_E_CUDA;
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
  int32_t* before = ws_ptr<int32_t>(ws, L.ep_before);
  int32_t* sbase = ws_ptr<int32_t>(ws, L.ep_sbase);
  int32_t* send_pos = ws_ptr<int32_t>(ws, L.send_pos);
  if (c.capacity && cudaMemsetAsync(send_idx, 0xff, size_t(A) * 4, st) != cudaSuccess)
    return MOE_E_CUDA;
  ep_tables_kernel<<<1, 1024, 0, st>>>(src_cnt, c.n_ep, c.E, c.k, T_loc, c.capacity, before,
                                       sbase, C, send_off, recv_off);
  ep_scatter_kernel<<<(A + 255) / 256, 256, 0, st>>>(idx, inv, offsets, sbase, A, c.E, c.k, T_loc,
                                                     send_idx, send_pos);
  note_launches(2);
  if (cudaGetLastError() != cudaSuccess) return MOE_E_CUDA;
  if (x && send_buf) {
    if (c.capacity) {
      ep_pad_kernel<<<c.n_ep, 256, 0, st>>>(C, c.n_ep, T_loc * c.k, c.d / 8,
                                            static_cast<uint4*>(send_buf));
      note_launches(1);
    }
    return launch_row_scatter(x, c.T, c.d, c.k, send_pos, send_buf, st);
  }
  return MOE_OK;
}

}  // namespace moe
