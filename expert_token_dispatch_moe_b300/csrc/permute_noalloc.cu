// moe_permute_noalloc: the permute step for callers that cannot allocate
// device memory.
//
// moe_permute needs a caller-allocated workspace for its histogram, chunk
// bases and status word.  Some callers cannot provide one: a plugin inside
// an inference runtime that is handed only its input and output tensors and
// has no allocator hook, or a serving loop that must not call cudaMalloc
// because the call can synchronise the device.  This variant keeps that
// scratch in a fixed, file-scope device array instead, so the caller passes
// only inputs and outputs.
//
// The array is kNoallocScratchBytes (1 MiB) and lives in every GPU that loads
// the library, until the process exits.  A configuration needing more scratch
// than that is rejected on the host with MOE_E_SCRATCH_LIMIT.  All calls share
// the one array: calls that overlap on the GPU (different streams, or
// different host threads without ordering) race on it.  The array keeps the
// previous call's contents; each call clears its status word and counters
// itself before use.
#include <mutex>

#include "common.cuh"
#include "launch.h"

#define MOE_API extern "C" __attribute__((visibility("default")))

namespace moe {

constexpr size_t kNoallocScratchBytes = size_t(1) << 20;

static __device__ __align__(256) unsigned char g_permute_scratch[kNoallocScratchBytes];

// Host-side address of g_permute_scratch on each device, looked up once per
// device with that device current (the symbol's host-side name is only a
// stand-in and must never be passed to a kernel).
static void* scratch_address(int dev, int* err) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_permute_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      *err = MOE_E_CUDA;
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace moe

using namespace moe;

MOE_API int moe_permute_noalloc(const moe_cfg* c, const moe_bf16* x, const int32_t* topk_idx,
                                int32_t* counts, int32_t* offsets, int32_t* order, int32_t* inv,
                                moe_bf16* x_sorted, void* stream) {
  reset_launches();
  int rc = moe_validate_cfg(c);
  if (rc != MOE_OK) return rc;
  for (const void* p : {static_cast<const void*>(topk_idx), static_cast<const void*>(counts),
                        static_cast<const void*>(offsets), static_cast<const void*>(order),
                        static_cast<const void*>(inv)}) {
    if (!p) return MOE_E_NULL;
    if (reinterpret_cast<uintptr_t>(p) & 15u) return MOE_E_ALIGN;
  }
  // as in moe_permute: x and x_sorted both NULL computes the indices only; one
  // of them alone is an error
  for (const void* p : {static_cast<const void*>(x), static_cast<const void*>(x_sorted)})
    if (reinterpret_cast<uintptr_t>(p) & 15u) return MOE_E_ALIGN;
  if ((x == nullptr) != (x_sorted == nullptr)) return MOE_E_NULL;
  // The permute touches the status word and histogram counter, the per-(rank,
  // expert) counts and the per-chunk histograms: the workspace regions that
  // precede the EP tables.
  const WsLayout L = ws_layout(*c);
  if (L.ep_sbase > kNoallocScratchBytes) return MOE_E_SCRATCH_LIMIT;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return MOE_E_DEVICE;
  }
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return MOE_E_DEVICE;
  }
  if (major != 10 || minor != 3) return MOE_E_DEVICE;
  int err = MOE_OK;
  void* ws = scratch_address(dev, &err);
  if (!ws) return err;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the status word, the histogram's finished-CTA counter and the one-launch
  // permute's group sums must start at zero (the per-(rank, expert) counts are
  // cleared by the permute)
  if (cudaMemsetAsync(ws, 0, kWsHeadBytes, st) != cudaSuccess) return MOE_E_CUDA;
  return launch_permute(*c, x, topk_idx, counts, offsets, order, inv, x_sorted, ws, st);
}
