// C ABI of libmoe: argument validation on the host, then asynchronous
// launches on the caller's stream.  Declarations and the contract of every
// entry point are in include/moe.h.
#include <mutex>

#include "common.cuh"
#include "launch.h"

#define MOE_API extern "C" __attribute__((visibility("default")))

namespace moe {

static thread_local int g_launches = 0;
void reset_launches() { g_launches = 0; }
void note_launches(int n) { g_launches += n; }

int device_sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 148;
  }
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = 148;
    }
    cache[dev] = n;
  }
  return cache[dev];
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int64_t rows_R(const moe_cfg& c) {
  return c.capacity ? int64_t(c.E) * c.capacity : int64_t(c.T) * c.k;
}

// Is the current device an sm_103 part?  Cached per device ordinal.
int device_ok() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return MOE_E_DEVICE;
  }
  static int cache[64] = {0};  // 0 unknown, 1 ok, -1 not ok
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  if (cache[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      cudaGetLastError();
      return MOE_E_DEVICE;
    }
    cache[dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  return cache[dev] == 1 ? MOE_OK : MOE_E_DEVICE;
}

static int check_ptrs(std::initializer_list<const void*> ps) {
  for (const void* p : ps) {
    if (!p) return MOE_E_NULL;
    if (!aligned16(p)) return MOE_E_ALIGN;
  }
  return MOE_OK;
}
static int check_opt(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (p && !aligned16(p)) return MOE_E_ALIGN;
  return MOE_OK;
}

}  // namespace moe

using namespace moe;

#define MOE_TRY(expr)          \
  do {                         \
    const int _rc = (expr);    \
    if (_rc != MOE_OK) return _rc; \
  } while (0)

MOE_API int moe_validate_cfg(const moe_cfg* c) {
  if (!c) return MOE_E_NULL;
  if (c->T < 1 || c->E < 1 || c->E > 1024 || c->k < 1 || c->k > 32 || c->k > c->E)
    return MOE_E_SHAPE;
  if (c->d < 64 || c->d > 65536 || c->d % 64) return MOE_E_SHAPE;
  if (c->f < 0) return MOE_E_SHAPE;
  if (c->n_ep < 1 || c->E % c->n_ep || c->T % c->n_ep) return MOE_E_SHAPE;
  if (c->n_groups < 1 || c->n_groups > 32 || c->E % c->n_groups) return MOE_E_SHAPE;
  if (c->n_groups > 1 && c->E / c->n_groups < 2) return MOE_E_SHAPE;
  if (c->topk_groups < 1 || c->topk_groups > c->n_groups) return MOE_E_SHAPE;
  if (int64_t(c->topk_groups) * (c->E / c->n_groups) < c->k) return MOE_E_SHAPE;
  if (c->capacity < 0 || (c->has_shared != 0 && c->has_shared != 1)) return MOE_E_SHAPE;
  if (c->score_fn != MOE_SOFTMAX && c->score_fn != MOE_SIGMOID) return MOE_E_SHAPE;
  if (c->norm_topk != 0 && c->norm_topk != 1) return MOE_E_SHAPE;
  const int64_t A = int64_t(c->T) * c->k;
  const int64_t R = c->capacity ? int64_t(c->E) * c->capacity : A;
  if (A >= (int64_t(1) << 31) || R + c->T >= (int64_t(1) << 31)) return MOE_E_SHAPE;
  return MOE_OK;
}

MOE_API int64_t moe_grouped_rows(const moe_cfg* c) {
  if (moe_validate_cfg(c) != MOE_OK) return -1;
  return rows_R(*c) + (c->has_shared ? c->T : 0);
}

MOE_API size_t moe_workspace_bytes(const moe_cfg* c) {
  if (moe_validate_cfg(c) != MOE_OK) return 0;
  return ws_layout(*c).total;
}

static int check_ws(const moe_cfg* c, const void* ws, size_t ws_bytes) {
  if (!ws) return MOE_E_WORKSPACE;
  if (!aligned16(ws)) return MOE_E_ALIGN;
  if (ws_bytes < ws_layout(*c).total) return MOE_E_WORKSPACE;
  return MOE_OK;
}

MOE_API int moe_workspace_init(const moe_cfg* c, void* ws, size_t ws_bytes, void* stream) {
  reset_launches();
  MOE_TRY(moe_validate_cfg(c));
  MOE_TRY(check_ws(c, ws, ws_bytes));
  MOE_TRY(device_ok());
  if (cudaMemsetAsync(ws, 0, kWsHeadBytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MOE_E_CUDA;
  return MOE_OK;
}

MOE_API int moe_pack_router(const moe_cfg* c, const float* W_r, moe_bf16* W_r_split,
                            void* stream) {
  reset_launches();
  MOE_TRY(moe_validate_cfg(c));
  MOE_TRY(check_ptrs({W_r, W_r_split}));
  MOE_TRY(device_ok());
  return launch_pack_router(*c, W_r, W_r_split, static_cast<cudaStream_t>(stream));
}

MOE_API int moe_router_logits(const moe_cfg* c, const moe_bf16* x, const float* W_r,
                              const moe_bf16* W_r_split, const float* logit_bias, float* scores,
                              void* ws, size_t ws_bytes, void* stream) {
  reset_launches();
  MOE_TRY(moe_validate_cfg(c));
  MOE_TRY(check_ptrs({x, scores}));
  MOE_TRY(check_opt({W_r, W_r_split, logit_bias}));
  if (!W_r && !W_r_split) return MOE_E_NULL;
  if (ws) MOE_TRY(check_ws(c, ws, ws_bytes));
  MOE_TRY(device_ok());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* status = ws ? ws_ptr<int>(ws, ws_layout(*c).status) : nullptr;
  float* part = ws ? ws_ptr<float>(ws, ws_layout(*c).router_part) : nullptr;
  if (W_r_split) return launch_router_tc(*c, x, W_r_split, logit_bias, scores, status, part, st);
  return launch_router_logits(*c, x, W_r, logit_bias, scores, status, st);
}

MOE_API int moe_route(const moe_cfg* c, const float* scores, const float* bias, int32_t* topk_idx,
                      float* topk_gate, void* stream) {
  reset_launches();
  MOE_TRY(moe_validate_cfg(c));
  MOE_TRY(check_ptrs({scores, topk_idx, topk_gate}));
  MOE_TRY(check_opt({bias}));
  MOE_TRY(device_ok());
  return launch_route(*c, scores, bias, topk_idx, topk_gate, static_cast<cudaStream_t>(stream));
}

MOE_API int moe_permute(const moe_cfg* c, const moe_bf16* x, const int32_t* topk_idx,
                        int32_t* counts, int32_t* offsets, int32_t* order, int32_t* inv,
                        moe_bf16* x_sorted, void* ws, size_t ws_bytes, void* stream) {
  reset_launches();
  MOE_TRY(moe_validate_cfg(c));
  MOE_TRY(check_ptrs({topk_idx, counts, offsets, order, inv}));
  MOE_TRY(check_opt({x, x_sorted}));
  if ((x == nullptr) != (x_sorted == nullptr)) return MOE_E_NULL;
  MOE_TRY(check_ws(c, ws, ws_bytes));
  MOE_TRY(device_ok());
  return launch_permute(*c, x, topk_idx, counts, offsets, order, inv, x_sorted, ws,
                        static_cast<cudaStream_t>(stream));
}

MOE_API int moe_ep_layout(const moe_cfg* c, const int32_t* topk_idx, const int32_t* offsets,
                          const int32_t* inv, int32_t* count_mat, int32_t* send_off,
                          int32_t* recv_off, int32_t* send_idx, const moe_bf16* x,
                          moe_bf16* send_buf, void* ws, size_t ws_bytes, void* stream) {
  reset_launches();
  MOE_TRY(moe_validate_cfg(c));
  MOE_TRY(check_ptrs({topk_idx, offsets, inv, count_mat, send_off, recv_off, send_idx}));
  MOE_TRY(check_opt({x, send_buf}));
  if ((x == nullptr) != (send_buf == nullptr)) return MOE_E_NULL;
  if (c->n_ep > 1024) return MOE_E_SHAPE;
  MOE_TRY(check_ws(c, ws, ws_bytes));
  MOE_TRY(device_ok());
  return launch_ep_layout(*c, topk_idx, offsets, inv, count_mat, send_off, recv_off, send_idx, x,
                          send_buf, ws, static_cast<cudaStream_t>(stream));
}

MOE_API int moe_ep_layout_fp8(const moe_cfg* c, const int32_t* topk_idx, const int32_t* offsets,
                              const int32_t* inv, int32_t* count_mat, int32_t* send_off,
                              int32_t* recv_off, int32_t* send_idx, const moe_bf16* x,
                              uint8_t* send_fp8, float* send_scale, void* ws, size_t ws_bytes,
                              void* stream) {
  reset_launches();
  MOE_TRY(moe_validate_cfg(c));
  MOE_TRY(check_ptrs({topk_idx, offsets, inv, count_mat, send_off, recv_off, send_idx, x,
                      send_fp8, send_scale}));
  if (c->n_ep > 1024) return MOE_E_SHAPE;
  MOE_TRY(check_ws(c, ws, ws_bytes));
  MOE_TRY(device_ok());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return launch_ep_layout(*c, topk_idx, offsets, inv, count_mat, send_off, recv_off, send_idx, x,
                          nullptr, ws, st, send_fp8, send_scale);
}

MOE_API int moe_dispatch_recv_fp8(const moe_cfg* c, const uint8_t* send_fp8,
                                  const float* send_scale, const int32_t* send_idx,
                                  const int32_t* inv, moe_bf16* x_sorted, void* stream) {
  reset_launches();
  MOE_TRY(moe_validate_cfg(c));
  MOE_TRY(check_ptrs({send_fp8, send_scale, send_idx, inv, x_sorted}));
  MOE_TRY(device_ok());
  return launch_fp8_recv(*c, send_fp8, send_scale, send_idx, inv, x_sorted,
                         static_cast<cudaStream_t>(stream));
}

MOE_API int moe_pack_w13(const moe_cfg* c, const moe_bf16* W1, const moe_bf16* W3, moe_bf16* W13,
                         void* stream) {
  reset_launches();
  MOE_TRY(moe_validate_cfg(c));
  if (c->f < 128 || c->f % 128) return MOE_E_SHAPE;
  MOE_TRY(check_ptrs({W1, W3, W13}));
  MOE_TRY(device_ok());
  return launch_pack_w13(*c, W1, W3, W13, static_cast<cudaStream_t>(stream));
}

MOE_API int moe_ffn_pair_tiles(const moe_cfg* c) {
  MOE_TRY(moe_validate_cfg(c));
  return use_pair_tiles(*c) ? 1 : 0;
}

MOE_API int moe_grouped_ffn(const moe_cfg* c, const moe_bf16* x_sorted, const moe_bf16* x,
                            const int32_t* counts, const int32_t* offsets, const moe_bf16* W13,
                            const moe_bf16* W2, moe_bf16* h, moe_bf16* y_sorted, void* ws,
                            size_t ws_bytes, void* stream) {
  reset_launches();
  MOE_TRY(moe_validate_cfg(c));
  if (c->f < 128 || c->f % 128) return MOE_E_SHAPE;
  if (c->E + c->has_shared > 1025) return MOE_E_SHAPE;
  MOE_TRY(check_ptrs({x_sorted, counts, offsets, W13, W2, h, y_sorted}));
  if (c->has_shared) MOE_TRY(check_ptrs({x}));
  else MOE_TRY(check_opt({x}));
  MOE_TRY(check_ws(c, ws, ws_bytes));
  MOE_TRY(device_ok());
  return launch_grouped_ffn(*c, x_sorted, x, nullptr, counts, offsets, W13, W2, h, y_sorted,
                            nullptr, ws,
                            static_cast<cudaStream_t>(stream));
}

MOE_API int moe_grouped_ffn_combine(const moe_cfg* c, const moe_bf16* x_sorted, const moe_bf16* x,
                                    const int32_t* counts, const int32_t* offsets,
                                    const moe_bf16* W13, const moe_bf16* W2, moe_bf16* h,
                                    const int32_t* order, const float* topk_gate, moe_bf16* y,
                                    void* ws, size_t ws_bytes, void* stream) {
  reset_launches();
  MOE_TRY(moe_validate_cfg(c));
  if (c->f < 128 || c->f % 128) return MOE_E_SHAPE;
  if (c->E + c->has_shared > 1025) return MOE_E_SHAPE;
  MOE_TRY(check_ptrs({x_sorted, counts, offsets, W13, W2, h, order, topk_gate, y}));
  if (c->has_shared) MOE_TRY(check_ptrs({x}));
  else MOE_TRY(check_opt({x}));
  MOE_TRY(check_ws(c, ws, ws_bytes));
  MOE_TRY(device_ok());
  return launch_grouped_ffn_combine(*c, x_sorted, x, counts, offsets, W13, W2, h, order, topk_gate,
                                    y, ws, static_cast<cudaStream_t>(stream));
}

MOE_API int moe_grouped_ffn_gather(const moe_cfg* c, const moe_bf16* x, const int32_t* order,
                                   const int32_t* counts, const int32_t* offsets,
                                   const moe_bf16* W13, const moe_bf16* W2, moe_bf16* h,
                                   moe_bf16* y_sorted, void* ws, size_t ws_bytes, void* stream) {
  reset_launches();
  MOE_TRY(moe_validate_cfg(c));
  if (c->f < 128 || c->f % 128) return MOE_E_SHAPE;
  if (c->E + c->has_shared > 1025) return MOE_E_SHAPE;
  MOE_TRY(check_ptrs({x, order, counts, offsets, W13, W2, h, y_sorted}));
  MOE_TRY(check_ws(c, ws, ws_bytes));
  MOE_TRY(device_ok());
  return launch_grouped_ffn(*c, nullptr, x, order, counts, offsets, W13, W2, h, y_sorted, nullptr,
                            ws, static_cast<cudaStream_t>(stream));
}

MOE_API int moe_grouped_ffn_train(const moe_cfg* c, const moe_bf16* x_sorted, const moe_bf16* x,
                                  const int32_t* counts, const int32_t* offsets,
                                  const moe_bf16* W13, const moe_bf16* W2, moe_bf16* h,
                                  moe_bf16* y_sorted, moe_bf16* g1, void* ws, size_t ws_bytes,
                                  void* stream) {
  reset_launches();
  MOE_TRY(moe_validate_cfg(c));
  if (c->f < 128 || c->f % 128) return MOE_E_SHAPE;
  if (c->E + c->has_shared > 1025) return MOE_E_SHAPE;
  MOE_TRY(check_ptrs({x_sorted, counts, offsets, W13, W2, h, y_sorted, g1}));
  if (c->has_shared) MOE_TRY(check_ptrs({x}));
  else MOE_TRY(check_opt({x}));
  MOE_TRY(check_ws(c, ws, ws_bytes));
  MOE_TRY(device_ok());
  return launch_grouped_ffn(*c, x_sorted, x, nullptr, counts, offsets, W13, W2, h, y_sorted, g1,
                            ws, static_cast<cudaStream_t>(stream));
}

MOE_API int moe_combine(const moe_cfg* c, const moe_bf16* y_sorted, const int32_t* inv,
                        const float* topk_gate, moe_bf16* y, void* stream) {
  reset_launches();
  MOE_TRY(moe_validate_cfg(c));
  MOE_TRY(check_ptrs({y_sorted, inv, topk_gate, y}));
  MOE_TRY(device_ok());
  return launch_combine(*c, y_sorted, inv, topk_gate, y, static_cast<cudaStream_t>(stream));
}

MOE_API int moe_bias_update(const moe_cfg* c, const int32_t* counts, float lr, float* bias,
                            void* stream) {
  reset_launches();
  MOE_TRY(moe_validate_cfg(c));
  MOE_TRY(check_ptrs({counts, bias}));
  MOE_TRY(device_ok());
  return launch_bias_update(*c, counts, lr, bias, static_cast<cudaStream_t>(stream));
}

MOE_API int moe_eplb_plan(const moe_cfg* c, const int32_t* loads, int32_t slots_per_rank,
                          int32_t* copies, int32_t* copy_offset, int32_t* copy_rank,
                          int32_t* slot_expert, double* rank_load, void* stream) {
  reset_launches();
  MOE_TRY(moe_validate_cfg(c));
  if (slots_per_rank < 1 || int64_t(c->n_ep) * slots_per_rank < c->E ||
      int64_t(c->n_ep) * slots_per_rank > 8192)
    return MOE_E_SHAPE;
  MOE_TRY(check_ptrs({loads, copies, copy_offset, copy_rank, slot_expert, rank_load}));
  MOE_TRY(device_ok());
  return launch_eplb_plan(*c, loads, slots_per_rank, copies, copy_offset, copy_rank, slot_expert,
                          rank_load, static_cast<cudaStream_t>(stream));
}

MOE_API int moe_eplb_dispatch(const moe_cfg* c, const int32_t* topk_idx, const int32_t* counts,
                              const int32_t* offsets, const int32_t* inv, const int32_t* copies,
                              const int32_t* copy_offset, const int32_t* copy_rank,
                              int32_t* dest_rank, int32_t* count_mat, void* stream) {
  reset_launches();
  MOE_TRY(moe_validate_cfg(c));
  MOE_TRY(check_ptrs({topk_idx, counts, offsets, inv, copies, copy_offset, copy_rank, dest_rank,
                      count_mat}));
  MOE_TRY(device_ok());
  return launch_eplb_dispatch(*c, topk_idx, inv, offsets, counts, copies, copy_offset, copy_rank,
                              dest_rank, count_mat, static_cast<cudaStream_t>(stream));
}

MOE_API int moe_pack_backward(const moe_cfg* c, const moe_bf16* W13, const moe_bf16* W2,
                              moe_bf16* W13t, moe_bf16* W2t, void* stream) {
  reset_launches();
  MOE_TRY(moe_validate_cfg(c));
  if (c->f < 128 || c->f % 128) return MOE_E_SHAPE;
  MOE_TRY(check_ptrs({W13, W2, W13t, W2t}));
  MOE_TRY(device_ok());
  return launch_pack_backward(*c, W13, W2, W13t, W2t, static_cast<cudaStream_t>(stream));
}

MOE_API int moe_combine_backward(const moe_cfg* c, const moe_bf16* dy, const moe_bf16* y_sorted,
                                 const int32_t* inv, const float* topk_gate, moe_bf16* d_o,
                                 float* dgate, void* stream) {
  reset_launches();
  MOE_TRY(moe_validate_cfg(c));
  MOE_TRY(check_ptrs({dy, y_sorted, inv, topk_gate, d_o, dgate}));
  MOE_TRY(device_ok());
  return launch_combine_backward(*c, dy, y_sorted, inv, topk_gate, d_o, dgate,
                                 static_cast<cudaStream_t>(stream));
}

MOE_API size_t moe_backward_workspace_bytes(const moe_cfg* c) {
  if (moe_validate_cfg(c) != MOE_OK || c->f < 128 || c->f % 128) return 0;
  return backward_layout(*c).total;
}

MOE_API int moe_grouped_ffn_backward(const moe_cfg* c, const moe_bf16* x_sorted, const moe_bf16* x,
                                     const int32_t* counts, const int32_t* offsets,
                                     const moe_bf16* W13, const moe_bf16* W13t,
                                     const moe_bf16* W2t, const moe_bf16* h,
                                     const moe_bf16* g1, const moe_bf16* d_o,
                                     moe_bf16* dx_sorted, moe_bf16* dW13,
                                     moe_bf16* dW2, void* bws, size_t bws_bytes, void* ws,
                                     size_t ws_bytes, void* stream) {
  reset_launches();
  MOE_TRY(moe_validate_cfg(c));
  if (c->f < 128 || c->f % 128) return MOE_E_SHAPE;
  if (c->E + c->has_shared > 1025) return MOE_E_SHAPE;
  MOE_TRY(check_ptrs({x_sorted, counts, offsets, W13, W13t, W2t, h, d_o, dx_sorted, dW13, dW2}));
  MOE_TRY(check_opt({g1}));
  if (c->has_shared) MOE_TRY(check_ptrs({x}));
  else MOE_TRY(check_opt({x}));
  if (!bws) return MOE_E_WORKSPACE;
  if (!aligned16(bws)) return MOE_E_ALIGN;
  if (bws_bytes < backward_layout(*c).total) return MOE_E_WORKSPACE;
  MOE_TRY(check_ws(c, ws, ws_bytes));
  MOE_TRY(device_ok());
  return launch_grouped_ffn_backward(*c, x_sorted, x, counts, offsets, W13, W13t, W2t, h, g1, d_o,
                                     dx_sorted, dW13, dW2, bws, ws,
                                     static_cast<cudaStream_t>(stream));
}

MOE_API int moe_permute_backward(const moe_cfg* c, const moe_bf16* dx_sorted, const int32_t* inv,
                                 moe_bf16* dx, void* stream) {
  reset_launches();
  MOE_TRY(moe_validate_cfg(c));
  MOE_TRY(check_ptrs({dx_sorted, inv, dx}));
  MOE_TRY(device_ok());
  return launch_combine(*c, dx_sorted, inv, nullptr, dx, static_cast<cudaStream_t>(stream));
}

// One CTA waits on an mbarrier whose phase never completes; the bounded wait
// gives up after limit_ns and the kernel reports the time-out and returns.
__global__ void wait_timeout_selftest_kernel(int* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait_bounded(&bar, 0, limit_ns))
    report_status(status, MOE_E_DEVICE_TIMEOUT);
}

MOE_API int moe_selftest_wait_timeout(void* ws, uint64_t limit_ns, void* stream) {
  reset_launches();
  if (!ws) return MOE_E_WORKSPACE;
  if (!aligned16(ws)) return MOE_E_ALIGN;
  if (limit_ns < 1000ull || limit_ns > 1000000000ull) return MOE_E_SHAPE;
  MOE_TRY(device_ok());
  wait_timeout_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<int*>(ws), limit_ns);
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_E_CUDA;
}

MOE_API int moe_get_device_status(void* ws, void* stream) {
  reset_launches();
  if (!ws) return MOE_E_WORKSPACE;
  if (!aligned16(ws)) return MOE_E_ALIGN;
  MOE_TRY(device_ok());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t status = 0;
  if (cudaMemcpyAsync(&status, ws, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess) return MOE_E_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_E_CUDA;
  if (status != 0) {
    if (cudaMemsetAsync(ws, 0, 4, st) != cudaSuccess) return MOE_E_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_E_CUDA;
  }
  return status;
}

MOE_API const char* moe_strerror(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_E_NULL: return "a required pointer is NULL";
    case MOE_E_SHAPE: return "sizes outside the supported limits";
    case MOE_E_ALIGN: return "a pointer is not 16-byte aligned";
    case MOE_E_WORKSPACE: return "workspace missing or too small";
    case MOE_E_CUDA: return "a CUDA call or kernel launch failed";
    case MOE_E_DEVICE: return "the current device is not an sm_103 GPU";
    case MOE_E_DEVICE_DATA: return "an expert id outside [0, E) was found on the device";
    case MOE_E_DEVICE_TIMEOUT: return "a device-side wait timed out";
    case MOE_E_SCRATCH_LIMIT:
      return "moe_permute_noalloc: configuration needs more than its fixed 1 MiB device scratch";
    default: return "unknown error";
  }
}

MOE_API int moe_last_launch_count(void) { return g_launches; }
