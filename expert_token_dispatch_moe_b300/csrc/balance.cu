// Load balancing around the MoE layer.
//
// bias_update: the auxiliary-loss-free control loop ("05 - Expert Parallelism
//   (MoE)", "Load balancing" (b)): after a step, bias[i] += lr * (average load
//   - load[i]); the bias only enters the selection (moe_route), never a gate.
// eplb_plan: redundant experts by replicate-then-pack ("Expert parallelism",
//   "Load imbalance becomes idle time"): spare slots go one at a time to the
//   expert with the largest load per copy; copies, longest first, go to the
//   least-loaded rank that still has a free slot.
// eplb_dispatch: each expert's kept assignments, in their stable order, split
//   evenly over its copies; the rank of every assignment and the resulting
//   source x destination count matrix.
//
// Every decision is exact: load-per-copy ratios are compared by 64-bit cross
// multiplication, and rank loads are fp64 sums of c/q (correctly rounded
// division and addition) accumulated in placement order, so equal inputs give
// equal plans on any IEEE machine.
#include "common.cuh"
#include "launch.h"

namespace moe {

// ---------------------------------------------------------------------------
// bias update (one CTA; E <= 1024)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) bias_update_kernel(const int32_t* __restrict__ counts,
                                                           int E, float lr,
                                                           float* __restrict__ bias) {
  __shared__ long long warp_sum[32];
  const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
  const long long c = e < E ? __ldg(counts + e) : 0;
  long long s = c;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) warp_sum[warp] = s;
  __syncthreads();
  long long total = 0;
  for (int w = 0; w < (E + 31) / 32; ++w) total += warp_sum[w];
  if (e < E) {
    const double avg = double(total) / double(E);
    bias[e] = float(double(bias[e]) + double(lr) * (avg - double(c)));
  }
}

// ---------------------------------------------------------------------------
// replicate-then-pack plan (one CTA of 1024 threads)
// ---------------------------------------------------------------------------

// Does expert i (load ci, qi copies) come before expert j in the order "larger
// load per copy first, equal ratios: lower index first"?
__device__ __forceinline__ bool per_copy_before(long long ci, long long qi, int i, long long cj,
                                                long long qj, int j) {
  const long long a = ci * qj, b = cj * qi;
  return a > b || (a == b && i < j);
}

__global__ void __launch_bounds__(1024) eplb_plan_kernel(
    const int32_t* __restrict__ loads, int E, int n_ranks, int slots,
    int32_t* __restrict__ copies, int32_t* __restrict__ copy_offset,
    int32_t* __restrict__ copy_rank, int32_t* __restrict__ slot_expert,
    double* __restrict__ rank_load) {
  __shared__ int c_sm[1024], q_sm[1024], sorted_sm[1024], off_sm[1024];
  __shared__ int used_sm[1024];
  __shared__ double load_sm[1024], per_sm[1024];
  __shared__ int warp_tot[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < E; i += blockDim.x) {
    c_sm[i] = __ldg(loads + i);
    q_sm[i] = 1;
  }
  for (int r = tid; r < n_ranks; r += blockDim.x) {
    used_sm[r] = 0;
    load_sm[r] = 0.0;
  }
  for (int s = tid; s < n_ranks * slots; s += blockDim.x) slot_expert[s] = -1;
  __syncthreads();

  // 1. Replicate: one warp, one spare slot per round.
  if (warp == 0) {
    const int spare = n_ranks * slots - E;
    for (int round = 0; round < spare; ++round) {
      int bi = -1;
      long long bc = 0, bq = 1;
      for (int i = lane; i < E; i += 32) {
        const long long ci = c_sm[i], qi = q_sm[i];
        if (bi < 0 || per_copy_before(ci, qi, i, bc, bq, bi)) { bi = i; bc = ci; bq = qi; }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        const long long oc = __shfl_xor_sync(0xffffffffu, bc, off);
        const long long oq = __shfl_xor_sync(0xffffffffu, bq, off);
        if (oi >= 0 && (bi < 0 || per_copy_before(oc, oq, oi, bc, bq, bi))) {
          bi = oi; bc = oc; bq = oq;
        }
      }
      if (lane == 0) q_sm[bi] += 1;
      __syncwarp();
    }
  }
  __syncthreads();

  // 2a. Order of the experts by load per copy: position = number of experts
  // that come before it.
  for (int i = tid; i < E; i += blockDim.x) {
    const long long ci = c_sm[i], qi = q_sm[i];
    int pos = 0;
    for (int j = 0; j < E; ++j)
      pos += (j != i && per_copy_before(c_sm[j], q_sm[j], j, ci, qi, i)) ? 1 : 0;
    sorted_sm[pos] = i;
  }
  // 2b. Copy offsets: exclusive prefix of q over expert index (E <= 1024).
  {
    const int v = tid < E ? q_sm[tid] : 0;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w) before += warp_tot[w];
    if (tid < E) {
      off_sm[tid] = before + incl - v;
      copies[tid] = v;
      copy_offset[tid] = before + incl - v;
    }
  }
  __syncthreads();

  // 2c. Pack: one warp places the copies in order.  Each copy's load (one
  // fp64 division per expert) is computed up front, in parallel; rank loads
  // are sums of non-negative doubles, so their order is the order of their
  // bit patterns as integers (no fp64 compares on the critical path).
  for (int i = tid; i < E; i += blockDim.x) per_sm[i] = double(c_sm[i]) / double(q_sm[i]);
  __syncthreads();
  if (warp == 0) {
    for (int p = 0; p < E; ++p) {
      const int i = sorted_sm[p];
      const double per = per_sm[i];
      for (int j = 0; j < q_sm[i]; ++j) {
        int br = -1;
        long long bl = 0;
        for (int r = lane; r < n_ranks; r += 32) {
          if (used_sm[r] >= slots) continue;
          const long long l = __double_as_longlong(load_sm[r]);
          if (br < 0 || l < bl) { br = r; bl = l; }   // ranks ascend per lane
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          const int orr = __shfl_xor_sync(0xffffffffu, br, off);
          const long long ol = __shfl_xor_sync(0xffffffffu, bl, off);
          if (orr >= 0 && (br < 0 || ol < bl || (ol == bl && orr < br))) { br = orr; bl = ol; }
        }
        if (lane == 0) {
          copy_rank[off_sm[i] + j] = br;
          slot_expert[br * slots + used_sm[br]] = i;
          used_sm[br] += 1;
          load_sm[br] = load_sm[br] + per;
        }
        __syncwarp();
      }
    }
  }
  __syncthreads();
  for (int r = tid; r < n_ranks; r += blockDim.x) rank_load[r] = load_sm[r];
}

// ---------------------------------------------------------------------------
// dispatch over the copies
// ---------------------------------------------------------------------------
// Copy j of an expert with m kept assignments and q copies holds its ranks
// [floor(j*m/q), floor((j+1)*m/q)); rank r therefore sits in copy
// ceil((r+1)*q/m) - 1 = floor(((r+1)*q - 1)/m).
__global__ void __launch_bounds__(256) eplb_dispatch_kernel(
    const int32_t* __restrict__ idx, const int32_t* __restrict__ inv,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ counts, int capacity,
    const int32_t* __restrict__ copies, const int32_t* __restrict__ copy_offset,
    const int32_t* __restrict__ copy_rank, int A, int E, int k, int T_loc, int n_ranks,
    int32_t* __restrict__ dest, int32_t* __restrict__ C) {
  const int a = blockIdx.x * blockDim.x + threadIdx.x;
  const int lane = threadIdx.x & 31;
  int key = -1;
  if (a < A) {
    const int e = __ldg(idx + a);
    const int row = __ldg(inv + a);
    int g = -1;
    if (row >= 0 && e >= 0 && e < E) {
      const long long r = row - __ldg(offsets + e);
      const int c = __ldg(counts + e);
      const long long m = capacity ? min(c, capacity) : c;
      const long long q = __ldg(copies + e);
      const int j = int(((r + 1) * q - 1) / m);
      g = __ldg(copy_rank + __ldg(copy_offset + e) + j);
      key = ((a / k) / T_loc) * n_ranks + g;
    }
    dest[a] = g;
  }
  // one atomic per distinct (source, destination) in the warp
  const uint32_t peers = __match_any_sync(0xffffffffu, key);
  if (key >= 0 && (peers & ((1u << lane) - 1u)) == 0) atomicAdd(C + key, int(__popc(peers)));
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
int launch_bias_update(const moe_cfg& c, const int32_t* counts, float lr, float* bias,
                       cudaStream_t st) {
  bias_update_kernel<<<1, 1024, 0, st>>>(counts, c.E, lr, bias);
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_E_CUDA;
}

int launch_eplb_plan(const moe_cfg& c, const int32_t* loads, int slots, int32_t* copies,
                     int32_t* copy_offset, int32_t* copy_rank, int32_t* slot_expert,
                     double* rank_load, cudaStream_t st) {
  eplb_plan_kernel<<<1, 1024, 0, st>>>(loads, c.E, c.n_ep, slots, copies, copy_offset, copy_rank,
                                       slot_expert, rank_load);
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_E_CUDA;
}

int launch_eplb_dispatch(const moe_cfg& c, const int32_t* idx, const int32_t* inv,
                         const int32_t* offsets, const int32_t* counts, const int32_t* copies,
                         const int32_t* copy_offset, const int32_t* copy_rank, int32_t* dest,
                         int32_t* C, cudaStream_t st) {
  const int A = c.T * c.k;
  if (cudaMemsetAsync(C, 0, size_t(c.n_ep) * c.n_ep * 4, st) != cudaSuccess) return MOE_E_CUDA;
  eplb_dispatch_kernel<<<(A + 255) / 256, 256, 0, st>>>(idx, inv, offsets, counts, c.capacity,
                                                        copies, copy_offset, copy_rank, A, c.E,
                                                        c.k, c.T / c.n_ep, c.n_ep, dest, C);
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_E_CUDA;
}

}  // namespace moe
