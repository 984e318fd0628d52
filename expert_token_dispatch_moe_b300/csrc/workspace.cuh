// Workspace layout of libmoe's calls (moe_workspace_bytes) and of the layer's
// backward (moe_backward_workspace_bytes): offsets of every region, computed on
// the host from the configuration alone.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// ---------------------------------------------------------------------------
// Workspace layout (all regions 256-byte aligned)
//   [0, 256)       status word (int32 at 0), finished-CTA counter of the
//                  permute histogram (uint32 at 8, back to 0 after each call),
//                  grid barrier of the one-launch permute: arrival count
//                  (uint32 at 16, back to 0 after each barrier) and generation
//                  (uint32 at 24, only grows); launch sequence number of
//                  the one-launch permute (uint32 at 32, only grows)
//   grp_sums       int32 [2][kFusedMaxE][kFusedMaxGroups] at a fixed offset
//                  (256): the one-launch permute's per-group slice counts, one
//                  buffer per launch parity; each launch clears the other one
//   src_cnt        int32 [n_ep][E]   assignments per (source rank, expert)
//   chunk_hist     int32 [n_chunks][E] per-chunk histogram, then chunk bases
//   slice_hist     int32 [E][kFusedMaxCtas] per-CTA histograms of the
//                  one-launch permute (E <= kFusedMaxE only)
//   ep_sbase       int32 [n_ep][E]   (unused: the layout kernel keeps these bases in shared memory)
//   send_pos       int32 [A]         send slot of each assignment (-1 dropped)
//   router_part    fp32 [S][T][E]    partial logits of the tensor-core router when it
//                                    splits K into S > 1 chunks (router_k_split)
// ---------------------------------------------------------------------------
constexpr int kPermChunk = 2048;   // assignments per histogram/rank CTA
constexpr int kFusedMaxE = 256;    // the one-launch permute's largest expert count
constexpr int kFusedMaxCtas = 512; // and its most CTAs
constexpr int kFusedGroupCtas = 16; // CTAs per group of its slice-count sums
constexpr int kFusedMaxGroups = kFusedMaxCtas / kFusedGroupCtas;
constexpr size_t kWsHeadBytes = 256 + size_t(2) * kFusedMaxE * kFusedMaxGroups * 4;  // cleared by init

struct WsLayout {
  size_t status, done_ctas, bar_count, bar_gen, perm_seq, grp_sums, src_cnt, chunk_hist,
      slice_hist, ep_sbase, send_pos, router_part, total;
  int n_chunks;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// K chunks of the tensor-core router.  Its 128 x 256 output tiles are few when
// T is small (one tile for a 128-token decode batch), so K is split into S
// chunks reduced afterwards in a fixed order: S is the largest divisor of d/64
// that keeps at least 8 k-blocks per chunk and at most 148 tiles in all (one
// wave on a B300).  A rule of the shape alone, so the workspace size is too.
inline int router_k_split(const moe_cfg& c) {
  const long long tiles = (long long)((c.T + 127) / 128) * ((c.E + 255) / 256);
  const int kb = c.d / 64;
  int best = 1;
  for (int s = 2; s <= kb / 8; ++s)
    if (kb % s == 0 && tiles * s <= 148) best = s;
  return best;
}

inline WsLayout ws_layout(const moe_cfg& c) {
  WsLayout L;
  size_t A = size_t(c.T) * c.k;
  L.n_chunks = int((A + kPermChunk - 1) / kPermChunk);
  size_t off = 0;
  L.status = off;     L.done_ctas = off + 8;
  L.bar_count = off + 16;  L.bar_gen = off + 24;  L.perm_seq = off + 32;  off += 256;
  L.grp_sums = off;   off = kWsHeadBytes;
  L.src_cnt = off;    off += align256(size_t(c.n_ep) * c.E * 4);
  L.chunk_hist = off; off += align256(size_t(L.n_chunks) * c.E * 4);
  L.slice_hist = off;
  if (c.E <= kFusedMaxE) off += align256(size_t(kFusedMaxCtas) * c.E * 4);
  L.ep_sbase = off;   off += align256(size_t(c.n_ep) * c.E * 4);
  L.send_pos = off;   off += align256(A * 4);
  const int ks = router_k_split(c);
  L.router_part = off;
  if (ks > 1) off += align256(size_t(ks) * c.T * c.E * 4);
  L.total = off;
  return L;
}

// Workspace of the layer's backward (moe_backward_workspace_bytes).
struct BwdLayout {
  size_t g1, dg1, kpad, tr, total;
  size_t kub;  // columns of the transposed operands (upper bound on the padded rows)
};

template <typename T>
inline T* ws_ptr(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

}  // namespace moe
