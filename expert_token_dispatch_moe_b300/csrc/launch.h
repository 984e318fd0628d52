// Internal launcher declarations of libmoe (host side).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/moe.h"
#include "common.cuh"

namespace moe {

// Launch accounting for moe_last_launch_count (per host thread).
void reset_launches();
void note_launches(int n);

// Multiprocessors of the current device (cached per device; 148 if unknown).
int device_sm_count();

// MOE_OK when the current device is an sm_103 part, else MOE_E_DEVICE.
int device_ok();

// A set-up step whose effect belongs to one device, such as a kernel's opt-in
// to more than 48 KB of dynamic shared memory (cudaFuncSetAttribute applies to
// the current device only): run(step) calls step() with the caller's device
// current the first time that device is seen, and again on a later call if
// step() failed.  step returns MOE_OK or an error code, which run returns.
class PerDeviceOnce {
 public:
  template <typename F>
  int run(F&& step) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
      cudaGetLastError();
      return MOE_E_DEVICE;
    }
    if (done_[dev].load(std::memory_order_acquire)) return MOE_OK;
    std::lock_guard<std::mutex> lk(mu_);
    if (done_[dev].load(std::memory_order_relaxed)) return MOE_OK;
    const int rc = step();
    if (rc == MOE_OK) done_[dev].store(true, std::memory_order_release);
    return rc;
  }

 private:
  static constexpr int kMaxDevices = 64;
  std::mutex mu_;
  std::atomic<bool> done_[kMaxDevices] = {};
};

int launch_router_logits(const moe_cfg& c, const void* x, const float* W, const float* lbias,
                         float* out, int* status, cudaStream_t st);
int launch_router_tc(const moe_cfg& c, const void* x, const void* W_split, const float* lbias,
                     float* out, int* status, float* part, cudaStream_t st);
int launch_pack_router(const moe_cfg& c, const float* W, void* out, cudaStream_t st);
int launch_route(const moe_cfg& c, const float* scores, const float* bias, int32_t* idx,
                 float* gate, cudaStream_t st);
int launch_permute(const moe_cfg& c, const void* x, const int32_t* idx, int32_t* counts,
                   int32_t* offsets, int32_t* order, int32_t* inv, void* x_sorted, void* ws,
                   cudaStream_t st);
// The EP layout; with x and send_buf, the bf16 send rows; with x, send_fp8 and
// send_scale (send_buf NULL), the e4m3 send rows and their scales.
int launch_ep_layout(const moe_cfg& c, const int32_t* idx, const int32_t* offsets,
                     const int32_t* inv, int32_t* C, int32_t* send_off, int32_t* recv_off,
                     int32_t* send_idx, const void* x, void* send_buf, void* ws, cudaStream_t st,
                     void* send_fp8 = nullptr, float* send_scale = nullptr);
int launch_pack_w13(const moe_cfg& c, const void* W1, const void* W3, void* W13, cudaStream_t st);
int launch_grouped_ffn(const moe_cfg& c, const void* x_sorted, const void* x,
                       const int32_t* gather_order, const int32_t* counts, const int32_t* offsets,
                       const void* W13, const void* W2, void* h, void* y_sorted, void* g1,
                       void* ws, cudaStream_t st);
// The forward FFN on SM pairs (two-CTA clusters, transposed tiles).
// The grouped FFN's choice of SM-pair tiles for this configuration (the shape
// rule, or MOE_FFN_TILES when set).
bool use_pair_tiles(const moe_cfg& c);

// The grouped FFN whose GEMM 2 adds gate * row into the token-order y (zeroed
// first) instead of writing y_sorted: the combine in GEMM 2's epilogue.
int launch_grouped_ffn_combine(const moe_cfg& c, const void* x_sorted, const void* x,
                               const int32_t* counts, const int32_t* offsets, const void* W13,
                               const void* W2, void* h, const int32_t* order, const float* gate,
                               void* y, void* ws, cudaStream_t st);

int launch_grouped_ffn_pair(const moe_cfg& c, const void* x_sorted, const void* x,
                            const int32_t* counts, const int32_t* offsets, const void* W13,
                            const void* W2, void* h, void* y_sorted, int* status,
                            cudaStream_t st);
// 2-D bf16 row-major [rows, cols] tensor map, box = 64 columns x box_rows rows,
// 128-byte swizzle, out-of-bounds elements read as zero (false on failure).
bool make_bf16_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols,
                   uint32_t box_rows);
int launch_combine(const moe_cfg& c, const void* y_sorted, const int32_t* inv, const float* gate,
                   void* y, cudaStream_t st);

int launch_bias_update(const moe_cfg& c, const int32_t* counts, float lr, float* bias,
                       cudaStream_t st);
int launch_eplb_plan(const moe_cfg& c, const int32_t* loads, int slots, int32_t* copies,
                     int32_t* copy_offset, int32_t* copy_rank, int32_t* slot_expert,
                     double* rank_load, cudaStream_t st);
int launch_eplb_dispatch(const moe_cfg& c, const int32_t* idx, const int32_t* inv,
                         const int32_t* offsets, const int32_t* counts, const int32_t* copies,
                         const int32_t* copy_offset, const int32_t* copy_rank, int32_t* dest,
                         int32_t* C, cudaStream_t st);

int launch_fp8_recv(const moe_cfg& c, const void* send_fp8, const float* send_scale,
                    const int32_t* send_idx, const int32_t* inv, void* x_sorted, cudaStream_t st);

// Backward of the layer (routing held fixed).
size_t backward_kpad_bound(const moe_cfg& c);
BwdLayout backward_layout(const moe_cfg& c);
int launch_combine_backward(const moe_cfg& c, const void* dy, const void* y_sorted,
                            const int32_t* inv, const float* gate, void* d_o, float* dgate,
                            cudaStream_t st);
int launch_pack_backward(const moe_cfg& c, const void* W13, const void* W2, void* W13t, void* W2t,
                         cudaStream_t st);
int launch_kpad_offsets(const moe_cfg& c, const int32_t* counts, int32_t* kpad_off,
                        cudaStream_t st);
int launch_transpose_segments(const moe_cfg& c, const void* src, const void* src_shared, int C,
                              const int32_t* offsets, const int32_t* counts,
                              const int32_t* kpad_off, void* dst, size_t ld_dst, cudaStream_t st);
int launch_grouped_ffn_backward(const moe_cfg& c, const void* x_sorted, const void* x,
                                const int32_t* counts, const int32_t* offsets, const void* W13,
                                const void* W13t, const void* W2t, const void* h,
                                const void* g1_saved, const void* d_o, void* dx_sorted,
                                void* dW13, void* dW2, void* bws, void* ws, cudaStream_t st);

// Row move shared by the permute and the send-buffer fill: for each token t
// and slot j, copy x[t] to dst[rows[t*k + j]] when that row is >= 0.
int launch_row_scatter(const void* x, int T, int d, int k, const int32_t* rows, void* dst,
                       cudaStream_t st);

}  // namespace moe
