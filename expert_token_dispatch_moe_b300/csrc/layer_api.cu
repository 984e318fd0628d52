// The whole layer forward as two C entry points: on device tokens
// (moe_layer_forward), and on a sequence of batches in pinned host memory with
// the copies overlapping compute (moe_layer_forward_host).  Both only sequence
// the step calls of include/moe.h; every step runs in the library's kernels.
#include "common.cuh"
#include "launch.h"

#define MOE_API extern "C" __attribute__((visibility("default")))

using namespace moe;

#define MOE_STEP(call)                        \
  do {                                        \
    const int _rc = (call);                   \
    if (_rc != MOE_OK) return _rc;            \
    total += moe_last_launch_count();         \
  } while (0)

MOE_API int moe_layer_forward(const moe_cfg* c, const moe_layer* L, const moe_bf16* x,
                              moe_bf16* y, void* stream) {
  if (!c || !L) return MOE_E_NULL;
  if (L->gather && L->combine_in_epilogue) return MOE_E_SHAPE;
  int total = 0;
  if (L->W_r || L->W_r_split)
    MOE_STEP(moe_router_logits(c, x, L->W_r_split ? nullptr : L->W_r, L->W_r_split,
                               L->logit_bias, L->scores, L->ws, L->ws_bytes, stream));
  MOE_STEP(moe_route(c, L->scores, L->selection_bias, L->topk_idx, L->topk_gate, stream));
  // the gathered form moves no rows here: GEMM 1 reads them from x
  MOE_STEP(moe_permute(c, L->gather ? nullptr : x, L->topk_idx, L->counts, L->offsets, L->order,
                       L->inv, L->gather ? nullptr : L->x_sorted, L->ws, L->ws_bytes, stream));
  MOE_STEP(moe_ep_layout(c, L->topk_idx, L->offsets, L->inv, L->count_mat, L->send_off,
                         L->recv_off, L->send_idx, L->send_buf ? x : nullptr, L->send_buf, L->ws,
                         L->ws_bytes, stream));
  if (L->combine_in_epilogue) {
    MOE_STEP(moe_grouped_ffn_combine(c, L->x_sorted, c->has_shared ? x : nullptr, L->counts,
                                     L->offsets, L->W13, L->W2, L->h, L->order, L->topk_gate, y,
                                     L->ws, L->ws_bytes, stream));
  } else {
    if (L->gather)
      MOE_STEP(moe_grouped_ffn_gather(c, x, L->order, L->counts, L->offsets, L->W13, L->W2, L->h,
                                      L->y_sorted, L->ws, L->ws_bytes, stream));
    else
      MOE_STEP(moe_grouped_ffn(c, L->x_sorted, c->has_shared ? x : nullptr, L->counts,
                               L->offsets, L->W13, L->W2, L->h, L->y_sorted, L->ws, L->ws_bytes,
                               stream));
    MOE_STEP(moe_combine(c, L->y_sorted, L->inv, L->topk_gate, y, stream));
  }
  reset_launches();
  note_launches(total);
  return MOE_OK;
}

namespace {
// Events of one moe_layer_forward_host call, destroyed when it returns (an
// event destroyed while still pending is released once it completes).
struct Events {
  cudaEvent_t e[7] = {};
  int n = 0;
  int create() {
    for (n = 0; n < 7; ++n)
      if (cudaEventCreateWithFlags(&e[n], cudaEventDisableTiming) != cudaSuccess) {
        cudaGetLastError();
        return MOE_E_CUDA;
      }
    return MOE_OK;
  }
  ~Events() {
    for (int i = 0; i < n; ++i) cudaEventDestroy(e[i]);
  }
};
}  // namespace

#define MOE_CU(call)                                 \
  do {                                               \
    if ((call) != cudaSuccess) {                     \
      cudaGetLastError();                            \
      return MOE_E_CUDA;                             \
    }                                                \
  } while (0)

MOE_API int moe_layer_forward_host(const moe_cfg* c, const moe_layer* L, int n_batches,
                                   const moe_bf16* const* x_host, moe_bf16* const* y_host,
                                   moe_bf16* const* x_dev, moe_bf16* const* y_dev,
                                   void* compute_stream, void* copy_in_stream,
                                   void* copy_out_stream) {
  if (!c || !L || !x_host || !y_host || !x_dev || !y_dev) return MOE_E_NULL;
  const int rc = moe_validate_cfg(c);
  if (rc != MOE_OK) return rc;
  if (n_batches < 0) return MOE_E_SHAPE;
  for (int b = 0; b < 2; ++b) {
    if (!x_dev[b] || !y_dev[b]) return MOE_E_NULL;
    if ((reinterpret_cast<uintptr_t>(x_dev[b]) | reinterpret_cast<uintptr_t>(y_dev[b])) & 15u)
      return MOE_E_ALIGN;
  }
  for (int i = 0; i < n_batches; ++i)
    if (!x_host[i] || !y_host[i]) return MOE_E_NULL;
  if (n_batches == 0) return MOE_OK;
  const int dev_rc = device_ok();
  if (dev_rc != MOE_OK) return dev_rc;
  cudaStream_t comp = static_cast<cudaStream_t>(compute_stream);
  cudaStream_t s_in = static_cast<cudaStream_t>(copy_in_stream);
  cudaStream_t s_out = copy_out_stream ? static_cast<cudaStream_t>(copy_out_stream) : s_in;
  const size_t bytes = size_t(c->T) * c->d * sizeof(moe_bf16);
  Events ev;
  if (ev.create() != MOE_OK) return MOE_E_CUDA;
  cudaEvent_t start = ev.e[0];
  cudaEvent_t* in_done = ev.e + 1;
  cudaEvent_t* comp_done = ev.e + 3;
  cudaEvent_t* out_done = ev.e + 5;
  int total = 0;
  // the first copies wait for the compute stream's earlier work
  MOE_CU(cudaEventRecord(start, comp));
  MOE_CU(cudaStreamWaitEvent(s_in, start, 0));
  if (s_out != s_in) MOE_CU(cudaStreamWaitEvent(s_out, start, 0));
  for (int i = 0; i < n_batches; ++i) {
    const int b = i & 1;
    // batch i-2 has finished reading x_dev[b]
    if (i >= 2) MOE_CU(cudaStreamWaitEvent(s_in, comp_done[b], 0));
    MOE_CU(cudaMemcpyAsync(x_dev[b], x_host[i], bytes, cudaMemcpyHostToDevice, s_in));
    MOE_CU(cudaEventRecord(in_done[b], s_in));
    MOE_CU(cudaStreamWaitEvent(comp, in_done[b], 0));
    // batch i-2's result has left y_dev[b]
    if (i >= 2) MOE_CU(cudaStreamWaitEvent(comp, out_done[b], 0));
    const int frc = moe_layer_forward(c, L, x_dev[b], y_dev[b], compute_stream);
    if (frc != MOE_OK) return frc;
    total += moe_last_launch_count();
    MOE_CU(cudaEventRecord(comp_done[b], comp));
    MOE_CU(cudaStreamWaitEvent(s_out, comp_done[b], 0));
    MOE_CU(cudaMemcpyAsync(y_host[i], y_dev[b], bytes, cudaMemcpyDeviceToHost, s_out));
    MOE_CU(cudaEventRecord(out_done[b], s_out));
  }
  // the compute stream completes after the last result reaches the host
  for (int b = 0; b < (n_batches < 2 ? n_batches : 2); ++b)
    MOE_CU(cudaStreamWaitEvent(comp, out_done[b], 0));
  reset_launches();
  note_launches(total);
  return MOE_OK;
}
