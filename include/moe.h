/*
 * moe.h -- C ABI of the single-device MoE layer hot path for NVIDIA B300
 * (sm_103a): route, permute (with a simulated expert-parallel send layout),
 * grouped SwiGLU expert FFN, and unpermute + gate + combine.
 *
 * The calls follow the seven-step forward pass of an expert-parallel MoE
 * layer described in "Expert parallelism" (zerotofrontier.app, MoE chapter,
 * section "Expert parallelism", steps 1-7).  On one device the exchange steps
 * (3 counts, 4 dispatch, 6 combine) move nothing; moe_ep_layout produces the
 * buffers, counts and offsets those exchanges would take.
 *
 * Conventions shared by every call
 *  - Symbols: T tokens, d hidden size, E routed experts, k experts per token,
 *    f expert FFN width, n_ep simulated expert-parallel ranks, T_loc = T/n_ep.
 *    An assignment is one (token t, slot j) pair, flat index a = t*k + j, with
 *    j the rank of the expert in the token's top-k order; A = T*k.
 *    R = rows of the expert-grouped buffer: A when dropless, E*capacity with a
 *    capacity.  Rows R .. R+T-1 of the FFN buffers belong to the shared expert
 *    when cfg->has_shared.
 *  - Every pointer argument is a DEVICE pointer unless stated otherwise, and
 *    must be 16-byte aligned.  Matrices are dense and row-major.  bf16 values
 *    are passed as their 16-bit patterns (moe_bf16).
 *  - Ownership: the caller allocates and frees every buffer, including the
 *    workspace.  The library allocates no device memory and never frees any.
 *  - Every call is asynchronous on the caller's stream (cudaStream_t passed as
 *    void*, NULL = legacy default stream) and never synchronises the host,
 *    except moe_get_device_status.
 *  - Errors: 0 on success; a negative MOE_E_* code otherwise.  Argument
 *    errors are detected on the host before anything is launched.  Invalid
 *    data found on the device (an expert id outside [0, E)) does not trap:
 *    the kernel records MOE_E_DEVICE_DATA in the workspace status word, treats
 *    the assignment as dropped, and moe_get_device_status reports it.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16;  /* bf16 bit pattern */

enum { MOE_SOFTMAX = 0, MOE_SIGMOID = 1 };

enum {
  MOE_OK = 0,
  MOE_E_NULL = -1,           /* a required pointer is NULL */
  MOE_E_SHAPE = -2,          /* sizes violate the limits stated at moe_validate_cfg */
  MOE_E_ALIGN = -3,          /* a pointer is not 16-byte aligned */
  MOE_E_WORKSPACE = -4,      /* workspace NULL or smaller than moe_workspace_bytes */
  MOE_E_CUDA = -5,           /* a CUDA runtime/driver call or a launch failed */
  MOE_E_DEVICE = -6,         /* no sm_103 device is current */
  MOE_E_DEVICE_DATA = -7,    /* device found an expert id outside [0, E) */
  MOE_E_DEVICE_TIMEOUT = -8, /* a device-side wait gave up (kernel returned early) */
  MOE_E_SCRATCH_LIMIT = -9   /* moe_permute_noalloc: the configuration needs more scratch
                                than the library's fixed 1 MiB device array holds */
};

/* Layer configuration (plain data, passed by host pointer). */
typedef struct moe_cfg {
  int32_t T, d, E, k, f;       /* tokens, hidden, routed experts, top-k, FFN width */
  int32_t n_ep;                /* simulated expert-parallel ranks */
  int32_t score_fn;            /* MOE_SOFTMAX: scores are logits, gates = softmax over
                                  all E; MOE_SIGMOID: scores are affinities, gates = s */
  int32_t norm_topk;           /* 1: the k gates are divided by their sum */
  int32_t n_groups;            /* group-limited routing over contiguous expert groups; */
  int32_t topk_groups;         /*   (1, 1) = plain top-k                               */
  int32_t capacity;            /* 0 = dropless; else rows kept per expert (pad to it) */
  int32_t has_shared;          /* 1: one always-on shared expert of width f           */
} moe_cfg;

/* Host-only check of a configuration.  Limits:
 *   T >= 1; 1 <= k <= min(E, 32); 1 <= E <= 1024; d % 64 == 0, 64 <= d <= 65536;
 *   f % 128 == 0 (moe_grouped_ffn only; f >= 128);
 *   n_ep >= 1, E % n_ep == 0, T % n_ep == 0;
 *   n_groups >= 1, E % n_groups == 0, n_groups <= 32, E/n_groups >= 2 when n_groups > 1,
 *   1 <= topk_groups <= n_groups, topk_groups*(E/n_groups) >= k;
 *   capacity >= 0; has_shared in {0, 1}; score_fn in {MOE_SOFTMAX, MOE_SIGMOID};
 *   T*k and R+T each below 2^31.
 * Returns MOE_OK or MOE_E_SHAPE / MOE_E_NULL. */
int moe_validate_cfg(const moe_cfg* cfg);

/* Rows of the expert-grouped buffers: R (+T with a shared expert).  Host only. */
int64_t moe_grouped_rows(const moe_cfg* cfg);

/* Bytes of workspace the calls below need for this configuration (0 on an
 * invalid configuration).  Host only. */
size_t moe_workspace_bytes(const moe_cfg* cfg);

/* Zero the workspace's header: the device status word, the counters of the
 * permute's grid barrier and the one-launch permute's per-group sums (the
 * first 65,792 bytes, at fixed offsets for every configuration; the calls keep
 * them consistent from then on).  Call once after allocating the workspace.
 * ws_bytes is the size of the caller's workspace allocation; every
 * call taking a workspace returns MOE_E_WORKSPACE when ws is NULL or ws_bytes <
 * moe_workspace_bytes(cfg). */
int moe_workspace_init(const moe_cfg* cfg, void* ws, size_t ws_bytes, void* stream);

/* One-time split of the fp32 router weights for the tensor-core router path:
 *   W_r        fp32 [d, E]
 *   W_r_split  bf16 [3, E, d] out: W_r[i][e] = hi + mid + lo exactly, with
 *              hi = bf16(w), mid = bf16(w - hi), lo = bf16(w - hi - mid), stored
 *              transposed (K-major) as W_r_split[0|1|2][e][i]. */
int moe_pack_router(const moe_cfg* cfg, const float* W_r, moe_bf16* W_r_split, void* stream);

/* Step 1, the router ("Expert parallelism", step 1 "Route": compute the
 * router for the local tokens).
 *   x          bf16 [T, d]
 *   W_r        fp32 [d, E], used when W_r_split is NULL: fp32 SIMT dot products
 *              (E <= 16: W_r in registers, x streamed through a shared-memory
 *              ring; larger E: 64 x 64 output tiles)
 *   W_r_split  bf16 [3, E, d] from moe_pack_router, or NULL.  When given, the
 *              logits come from the tensor cores: x times each of the three
 *              bf16 terms (every product exact in fp32), accumulated in fp32.
 *   logit_bias fp32 [E] or NULL: added to every token's logits
 *   scores     fp32 [T, E] out: logits l = x W_r (+ logit_bias), fp32
 *              accumulation; with MOE_SIGMOID the affinity 1/(1+exp(-l)).
 *   ws         workspace or NULL.  With a workspace, the tensor-core path splits
 *              K into chunks when its 128 x 256 output tiles are few (small T)
 *              and keeps the partial logits there, summed afterwards in a fixed
 *              order.  It receives MOE_E_DEVICE_TIMEOUT if a bounded wait
 *              (tensor-core path, or the E <= 16 ring) gives up; the block that
 *              gave up writes no scores. */
int moe_router_logits(const moe_cfg* cfg, const moe_bf16* x, const float* W_r,
                      const moe_bf16* W_r_split, const float* logit_bias, float* scores,
                      void* ws, size_t ws_bytes, void* stream);

/* Step 1, top-k choice and gates ("Expert parallelism", step 1; node-limited
 * routing in "What DeepSeek-V3 did about it"; the selection bias of "05 -
 * Expert Parallelism (MoE)", "Load balancing" (b): chosen = TopK(logits + bias)).
 *   scores    fp32 [T, E]
 *   bias      fp32 [E] or NULL: selection bias, one fp32 add, never in gates
 *   topk_idx  int32 [T, k] out: experts in rank order.  Order: larger
 *             (score + bias) first, equal values -> lower expert index, -0.0 ==
 *             +0.0, NaN below -inf.  Group-limited: a group's score is the fp32
 *             sum of its two highest values; the topk_groups best groups (same
 *             order rule) are kept and the k experts chosen among them.
 *   topk_gate fp32 [T, k] out: softmax over all E scores (MOE_SOFTMAX) or the
 *             score itself (MOE_SIGMOID); divided by the k gates' sum when
 *             norm_topk. */
int moe_route(const moe_cfg* cfg, const float* scores, const float* bias,
              int32_t* topk_idx, float* topk_gate, void* stream);

/* Step 2, permute ("Expert parallelism", step 2; "Token permutation and
 * grouped GEMMs": order = stable argsort of expert ids, inv[order] = arange).
 *   x         bf16 [T, d]
 *   topk_idx  int32 [T, k]
 *   counts    int32 [E] out: assignments routed to each expert (before drops)
 *   offsets   int32 [E+1] out: first row of each expert's segment (dropless:
 *             exclusive prefix sum of counts, offsets[E] = A; capacity: e*cap)
 *   order     int32 [R] out: row -> assignment a (-1 for a padding row)
 *   inv       int32 [A] out: assignment -> row (-1 when dropped)
 *   x_sorted  bf16 [R, d] out: x_sorted[inv[a]] = x[a / k]; padding rows zero.
 *             x and x_sorted may both be NULL: the indices are computed and no
 *             row moves (for moe_grouped_ffn_gather, which reads rows from x).
 *   ws        workspace; keeps the per-(source rank, expert) histogram that
 *             moe_ep_layout reads
 * Capacity: expert e keeps its first `capacity` assignments in increasing a.
 * Layers with up to 256 experts and more than 4096 assignments run as one
 * cooperative launch whose grid barrier keeps its state in the workspace
 * header (moe_workspace_init once; calls on one workspace must not overlap on
 * the GPU).  A barrier wait that exceeds one second records
 * MOE_E_DEVICE_TIMEOUT; the outputs are then unreliable. */
int moe_permute(const moe_cfg* cfg, const moe_bf16* x, const int32_t* topk_idx,
                int32_t* counts, int32_t* offsets, int32_t* order, int32_t* inv,
                moe_bf16* x_sorted, void* ws, size_t ws_bytes, void* stream);

/* Steps 2-4 as a layout: per-destination send buffers, the s->q count matrix
 * and offsets ("Expert parallelism", step 2 "sort by destination GPU and
 * count", step 3, step 4; "A dispatch you can check by hand").  Expert e lives
 * on rank floor(e*n_ep/E); token t belongs to rank floor(t/T_loc).  Inside a
 * rank's buffer rows are ordered by (destination, expert, a).
 *   topk_idx, offsets, inv: as written by moe_route / moe_permute
 *   ws        the workspace the preceding moe_permute wrote (same stream)
 *   count_mat int32 [n_ep, n_ep] out: C[s][q] kept rows rank s sends to rank q
 *   send_off  int32 [n_ep, n_ep] out: start of q's block in s's buffer
 *   recv_off  int32 [n_ep, n_ep] out: recv_off[q][s] = start of s's block in
 *             q's receive buffer
 *   send_idx  int32 [A] out: rank s's buffer is rows [s*T_loc*k, (s+1)*T_loc*k);
 *             entry p = the assignment sent from slot p, -1 past the kept rows
 *   x         bf16 [T, d] or NULL
 *   send_buf  bf16 [A, d] or NULL: when both are given, send_buf[p] =
 *             x[send_idx[p] / k], zero where send_idx[p] == -1; giving only one
 *             of the two is MOE_E_NULL.  n_ep <= 1024. */
int moe_ep_layout(const moe_cfg* cfg, const int32_t* topk_idx, const int32_t* offsets,
                  const int32_t* inv, int32_t* count_mat, int32_t* send_off,
                  int32_t* recv_off, int32_t* send_idx, const moe_bf16* x,
                  moe_bf16* send_buf, void* ws, size_t ws_bytes, void* stream);

/* Steps 2-4 with an FP8 send buffer ("Expert parallelism", "A worked example at
 * DeepSeek-V3's shape": dispatch in FP8, s = 1 byte, combine in BF16; "Lower
 * precision on the wire").  The same count matrix, offsets and slots as
 * moe_ep_layout; the send buffer holds e4m3 codes with one fp32 scale per row:
 *   scale = absmax(x[t]) / 448 (1 for an all-zero row),
 *   code  = e4m3(x * (448 / absmax)), rounded to nearest even, saturated at 448.
 * The format and the per-row granularity are this library's reading (the
 * description fixes only the byte width).
 *   send_fp8   uint8 [A, d] out: codes of slot p's token row; zero in empty slots
 *   send_scale fp32 [A] out: the row's scale; 0 in empty slots
 *   other arguments as for moe_ep_layout (x is required). */
int moe_ep_layout_fp8(const moe_cfg* cfg, const int32_t* topk_idx, const int32_t* offsets,
                      const int32_t* inv, int32_t* count_mat, int32_t* send_off,
                      int32_t* recv_off, int32_t* send_idx, const moe_bf16* x,
                      uint8_t* send_fp8, float* send_scale, void* ws, size_t ws_bytes,
                      void* stream);

/* The receiving side of an FP8 dispatch: slot p carries assignment
 * a = send_idx[p] (skipped when -1), whose row in the expert-grouped buffer
 * is inv[a]; x_sorted[inv[a]] = bf16(code * scale) element by element (one
 * fp32 product, rounded to nearest even).  Rows no slot maps to (capacity
 * padding) are not written.
 *   send_fp8, send_scale, send_idx  from moe_ep_layout_fp8
 *   inv                              from moe_permute
 *   x_sorted   bf16 [R, d] out */
int moe_dispatch_recv_fp8(const moe_cfg* cfg, const uint8_t* send_fp8, const float* send_scale,
                          const int32_t* send_idx, const int32_t* inv, moe_bf16* x_sorted,
                          void* stream);

/* moe_permute without a workspace argument, for callers that cannot allocate
 * device memory.  The pages have no counterpart to this entry point; it exists
 * for integration.  Some callers are handed only their input and output tensors
 * (for example a plugin inside an inference runtime with no allocator hook), and
 * some must not call cudaMalloc on a serving path, because it can synchronise
 * the device.  Such callers cannot provide the workspace that moe_permute needs.
 *
 * Outputs, arguments and results are those of moe_permute.  The scratch lives in
 * a fixed 1 MiB array in device memory that the library holds on every GPU that
 * loads it, until the process exits.
 *  - A configuration whose permute scratch (the workspace header: status word,
 *    counters, the one-launch permute's barrier words and group sums; then the
 *    per-(rank, expert) counts, per-2048-assignment histograms and, with E <= 256,
 *    per-CTA slice histograms) exceeds 1 MiB is rejected on the host with
 *    MOE_E_SCRATCH_LIMIT.
 *  - The first call on a device looks up the array's device address.  Make that
 *    first call before any stream capture on that device.
 *  - Every call shares the one array.  Calls that overlap on the GPU (on
 *    different streams, or from host threads without ordering) race on it.
 *  - Each call clears the workspace header (status word, counters, group sums).  Bad expert ids are
 *    treated as dropped (inv = -1) as in moe_permute, but the status word is not
 *    readable from outside: such ids are dropped silently.
 *  - The per-(source rank, expert) histogram stays in the hidden array, so
 *    moe_ep_layout and moe_ep_layout_fp8, which read it from the workspace of
 *    the preceding moe_permute, cannot follow this call; run moe_permute with a
 *    workspace when the layout is needed.
 *  - The call allocates and frees nothing. */
int moe_permute_noalloc(const moe_cfg* cfg, const moe_bf16* x, const int32_t* topk_idx,
                        int32_t* counts, int32_t* offsets, int32_t* order, int32_t* inv,
                        moe_bf16* x_sorted, void* stream);

/* One-time weight packing for moe_grouped_ffn (not part of a layer step).
 *   W1, W3    bf16 [E + has_shared, f, d]  (out, in)
 *   W13       bf16 [E + has_shared, 2f, d] out: for each block b of 128 rows,
 *             rows [256b, 256b+128) = W1 rows [128b, 128b+128) and rows
 *             [256b+128, 256b+256) = W3 rows [128b, 128b+128), so that a
 *             256-column accumulator tile holds matching gate and up columns. */
int moe_pack_w13(const moe_cfg* cfg, const moe_bf16* W1, const moe_bf16* W3,
                 moe_bf16* W13, void* stream);

/* Step 5, the experts as one grouped product ("Expert parallelism", step 5;
 * "Token permutation and grouped GEMMs", grouped GEMM; SwiGLU expert with
 * 6*d*f FLOPs per row, "A worked example at DeepSeek-V3's shape").
 *   x_sorted  bf16 [R, d]         (moe_permute)
 *   x         bf16 [T, d] or NULL (needed when has_shared)
 *   counts, offsets               (moe_permute); expert e's rows are
 *             [offsets[e], offsets[e] + min(counts[e], capacity or inf))
 *   W13       bf16 [E + has_shared, 2f, d]  (moe_pack_w13)
 *   W2        bf16 [E + has_shared, d, f]   (out, in)
 *   h         bf16 [R + has_shared*T, f] out: silu(x W1^T) * (x W3^T), fp32
 *             accumulation, rounded to bf16; shared expert rows at R + t
 *   y_sorted  bf16 [R + has_shared*T, d] out: h W2^T, fp32 accumulation
 * Rows outside the experts' kept rows are not written.  E + has_shared <= 1025.
 * The kernels are persistent (one CTA per SM, or one two-CTA cluster per SM
 * pair); a device-side wait that exceeds one second records
 * MOE_E_DEVICE_TIMEOUT in the workspace status word and the kernel returns
 * early (outputs then incomplete).
 * Tiles: layers whose expected rows per expert T*k/E (at most the capacity)
 * reach 768 run on SM pairs (256 weight rows by up to 256 tokens per tile,
 * tcgen05 cta_group::2); others on one-SM 128-row tiles.  The environment
 * variable MOE_FFN_TILES = "pair" or "single" overrides the choice; it is read
 * at every call.  Both give results within the layer's tolerance; they are not
 * bit-identical to each other. */
int moe_grouped_ffn(const moe_cfg* cfg, const moe_bf16* x_sorted, const moe_bf16* x,
                    const int32_t* counts, const int32_t* offsets,
                    const moe_bf16* W13, const moe_bf16* W2, moe_bf16* h,
                    moe_bf16* y_sorted, void* ws, size_t ws_bytes, void* stream);

/* moe_grouped_ffn with the combine (step 7) in GEMM 2's epilogue ("Token
 * permutation and grouped GEMMs": production kernels fuse the permutation into
 * the GEMM's loads and the combine into its epilogue).  GEMM 1 is that of
 * moe_grouped_ffn; GEMM 2 does not write y_sorted: each routed row of
 * assignment a adds bf16(topk_gate[a] * row) into y[a / k], each shared-expert
 * row t adds its row into y[t], by 16-byte bf16 reductions in L2.
 *   order      int32 [R]: the grouped rows' assignments (moe_permute's order)
 *   topk_gate  fp32 [T, k]
 *   y          bf16 [T, d] out: zeroed by the call, then accumulated
 * Every add rounds to bf16, and the adds of one token arrive in no fixed order:
 * with more than two contributions per token (k > 2, or k = 2 with a shared
 * expert) y is not bit-reproducible from run to run; it stays within the
 * layer's tolerance.  Runs on one-SM tiles whatever the layer's shape.  Other
 * arguments and errors as for moe_grouped_ffn. */
int moe_grouped_ffn_combine(const moe_cfg* cfg, const moe_bf16* x_sorted, const moe_bf16* x,
                            const int32_t* counts, const int32_t* offsets,
                            const moe_bf16* W13, const moe_bf16* W2, moe_bf16* h,
                            const int32_t* order, const float* topk_gate, moe_bf16* y,
                            void* ws, size_t ws_bytes, void* stream);

/* The tiles moe_grouped_ffn takes for this configuration now (the rule above,
 * MOE_FFN_TILES read at this call): 1 for SM pairs (grouped_pair_kernel), 0 for
 * one-SM tiles (grouped_gemm_kernel), or a negative error code for an invalid
 * configuration.  Host only; no device is touched. */
int moe_ffn_pair_tiles(const moe_cfg* cfg);

/* moe_grouped_ffn with the permute's row move fused into GEMM 1's operand
 * loads ("Token permutation and grouped GEMMs": production kernels fuse the
 * permutation into the grouped GEMM's loads, saving a full read and write of
 * the (T*k, d) tensor).  Row r of expert e's segment is gathered from token
 * order[r] / k of x by four-row tensor-memory-access copies; no x_sorted
 * buffer is read.
 *   x       bf16 [T, d] (also the shared expert's rows)
 *   order   int32 [R] from moe_permute (row -> assignment)
 *   other arguments and outputs as for moe_grouped_ffn. */
int moe_grouped_ffn_gather(const moe_cfg* cfg, const moe_bf16* x, const int32_t* order,
                           const int32_t* counts, const int32_t* offsets, const moe_bf16* W13,
                           const moe_bf16* W2, moe_bf16* h, moe_bf16* y_sorted, void* ws,
                           size_t ws_bytes, void* stream);

/* Step 7, unpermute and weight ("Expert parallelism", step 7: undo the sort
 * and scatter-add each row into its token with its gate).  Computed as a
 * per-token gather in slot order j = 0..k-1 with fp32 accumulation (the same
 * sum, deterministic):
 *   y[t] = sum_{j: inv[t*k+j] >= 0} topk_gate[t*k+j] * y_sorted[inv[t*k+j]]
 *          (+ y_sorted[R + t] when has_shared), rounded to bf16.
 *   y_sorted bf16 [R + has_shared*T, d]; inv int32 [A]; topk_gate fp32 [T, k]
 *   y        bf16 [T, d] out */
int moe_combine(const moe_cfg* cfg, const moe_bf16* y_sorted, const int32_t* inv,
                const float* topk_gate, moe_bf16* y, void* stream);

/* ------------------------------------------------------------------------
 * The whole forward in one call (the seven steps of "Expert parallelism" in
 * order, as the step calls above run them).
 * ------------------------------------------------------------------------ */

/* The layer's weights and step buffers, all device pointers, each as the step
 * call that takes it states. */
typedef struct moe_layer {
  const float* W_r;              /* fp32 [d, E]; NULL with W_r_split NULL: no router
                                    step, `scores` already holds the scores */
  const moe_bf16* W_r_split;     /* bf16 [3, E, d] (moe_pack_router) or NULL */
  const float* logit_bias;       /* fp32 [E] or NULL */
  const float* selection_bias;   /* fp32 [E] or NULL */
  const moe_bf16* W13;           /* moe_pack_w13 */
  const moe_bf16* W2;
  float* scores;
  int32_t* topk_idx;
  float* topk_gate;
  int32_t* counts;
  int32_t* offsets;
  int32_t* order;
  int32_t* inv;
  moe_bf16* x_sorted;
  int32_t* count_mat;
  int32_t* send_off;
  int32_t* recv_off;
  int32_t* send_idx;
  moe_bf16* send_buf;            /* or NULL: the layout without the packed rows */
  moe_bf16* h;
  moe_bf16* y_sorted;
  void* ws;                      /* workspace of moe_workspace_bytes(cfg) bytes */
  size_t ws_bytes;
  int32_t combine_in_epilogue;   /* 1: moe_grouped_ffn_combine replaces moe_grouped_ffn +
                                    moe_combine (y_sorted unused; see its notes) */
  int32_t gather;                /* 1: moe_permute computes the indices only and
                                    moe_grouped_ffn_gather reads GEMM 1's rows from x
                                    (x_sorted unused); not with combine_in_epilogue */
} moe_layer;

/* The forward on device tokens x (bf16 [T, d]) into y (bf16 [T, d]):
 * moe_router_logits (when L has router weights) -> moe_route -> moe_permute ->
 * moe_ep_layout -> moe_grouped_ffn -> moe_combine (or, with
 * L->combine_in_epilogue, moe_grouped_ffn_combine for the last two; with
 * L->gather, moe_permute without the row move and moe_grouped_ffn_gather in
 * place of moe_grouped_ffn), on `stream`.  Both flags set is MOE_E_SHAPE.
 * Returns the first error of a step (nothing after it is launched). */
int moe_layer_forward(const moe_cfg* cfg, const moe_layer* L, const moe_bf16* x, moe_bf16* y,
                      void* stream);

/* The forward on n_batches batches held in host memory:
 *   x_host[i], y_host[i]  HOST pointers, bf16 [T, d] each, page-locked (for
 *                         example cudaHostAlloc) so that the copies overlap
 *   x_dev[0..1], y_dev[0..1]  two device buffers per side, bf16 [T, d]
 * Batch i's host-to-device copy (one cudaMemcpyAsync on copy_in_stream) runs
 * while batch i-1 computes on compute_stream, and batch i-1's device-to-host
 * copy (one cudaMemcpyAsync on copy_out_stream, or copy_in_stream when NULL)
 * while batch i computes; events order each buffer's reuse.  Returns once
 * everything is enqueued: compute_stream completes after the last result has
 * reached y_host.  The call creates and destroys its own events and allocates
 * no memory.  n_batches = 0 does nothing; a negative n_batches is MOE_E_SHAPE. */
int moe_layer_forward_host(const moe_cfg* cfg, const moe_layer* L, int n_batches,
                           const moe_bf16* const* x_host, moe_bf16* const* y_host,
                           moe_bf16* const* x_dev, moe_bf16* const* y_dev, void* compute_stream,
                           void* copy_in_stream, void* copy_out_stream);

/* ------------------------------------------------------------------------
 * Backward of the layer with the routing held fixed ("Expert parallelism":
 * the dispatch and combine run twice more in the backward pass).  Order:
 *   moe_combine_backward -> moe_grouped_ffn_backward -> moe_permute_backward.
 * Gradients are bf16 with fp32 accumulation.  The gradient with respect to
 * the router scores (through the gates) is left to the caller: dgate is
 * returned.
 * ------------------------------------------------------------------------ */

/* One-time transposed copies of the expert weights for the backward:
 *   W13  bf16 [E + has_shared, 2f, d] (moe_pack_w13) -> W13t [E + has_shared, d, 2f]
 *   W2   bf16 [E + has_shared, d, f]                 -> W2t  [E + has_shared, f, d] */
int moe_pack_backward(const moe_cfg* cfg, const moe_bf16* W13, const moe_bf16* W2,
                      moe_bf16* W13t, moe_bf16* W2t, void* stream);

/* Step 7 backward: the combine's gradient is a dispatch of dy.
 *   dy        bf16 [T, d]: gradient of the layer output
 *   y_sorted  bf16 [R + has_shared*T, d]: the forward's expert outputs
 *   inv, topk_gate: the forward's (moe_permute, moe_route)
 *   d_o       bf16 [R + has_shared*T, d] out: kept row of assignment a =
 *             topk_gate[a] * dy[a / k]; shared row R + t = dy[t]; padding rows
 *             are not written
 *   dgate     fp32 [T, k] out: <dy[t], y_sorted[inv[a]]> (fp32 accumulation),
 *             0 for dropped assignments */
int moe_combine_backward(const moe_cfg* cfg, const moe_bf16* dy, const moe_bf16* y_sorted,
                         const int32_t* inv, const float* topk_gate, moe_bf16* d_o,
                         float* dgate, void* stream);

/* Bytes of the backward workspace of moe_grouped_ffn_backward (0 on an
 * invalid configuration).  Host only. */
size_t moe_backward_workspace_bytes(const moe_cfg* cfg);

/* Step 5 for training: moe_grouped_ffn that also keeps GEMM 1's output before
 * the SwiGLU, for moe_grouped_ffn_backward (which then need not recompute it).
 *   g1  bf16 [R + has_shared*T, 2f] out: x W13^T rounded to bf16, columns packed
 *       like W13 rows (each 256-column block: 128 gate then 128 up columns);
 *       rows of the kept assignments and the shared expert
 *   other arguments and outputs as for moe_grouped_ffn. */
int moe_grouped_ffn_train(const moe_cfg* cfg, const moe_bf16* x_sorted, const moe_bf16* x,
                          const int32_t* counts, const int32_t* offsets, const moe_bf16* W13,
                          const moe_bf16* W2, moe_bf16* h, moe_bf16* y_sorted, moe_bf16* g1,
                          void* ws, size_t ws_bytes, void* stream);

/* Step 5 backward, on the tensor cores:
 *   g1 = x W13^T (the forward's, from moe_grouped_ffn_train, or recomputed into
 *        the backward workspace when g1 is NULL),
 *   dg1 = SwiGLU'(g1) applied to d_o W2 (fused into that product's epilogue;
 *         du = dh v s (1 + u (1 - s)), dv = dh u s, s = sigmoid(u)),
 *   dx_sorted = dg1 W13,
 *   dW2[e] = d_o^T h and dW13[e] = dg1^T x over expert e's kept rows (the
 *   operands transposed into the workspace, each expert's rows starting on a
 *   64-column boundary, zero-padded).
 *   x_sorted, x, counts, offsets, W13 as for moe_grouped_ffn; W13t, W2t from
 *   moe_pack_backward; h the forward's [R + has_shared*T, f]; g1 from
 *   moe_grouped_ffn_train or NULL; d_o from moe_combine_backward.
 *   dx_sorted bf16 [R + has_shared*T, d] out (kept and shared rows)
 *   dW13      bf16 [E + has_shared, 2f, d] out, rows packed like W13
 *   dW2       bf16 [E + has_shared, d, f] out (zero for an expert with no rows)
 *   bws       backward workspace of moe_backward_workspace_bytes(cfg) bytes
 *   ws        the layer workspace (status word). */
int moe_grouped_ffn_backward(const moe_cfg* cfg, const moe_bf16* x_sorted, const moe_bf16* x,
                             const int32_t* counts, const int32_t* offsets,
                             const moe_bf16* W13, const moe_bf16* W13t, const moe_bf16* W2t,
                             const moe_bf16* h, const moe_bf16* g1, const moe_bf16* d_o,
                             moe_bf16* dx_sorted, moe_bf16* dW13, moe_bf16* dW2, void* bws,
                             size_t bws_bytes, void* ws, size_t ws_bytes, void* stream);

/* Step 2 backward: the permute's gradient is a combine with unit gates,
 *   dx[t] = sum over kept j of dx_sorted[inv[t*k+j]] (+ dx_sorted[R + t] with a
 *   shared expert), fp32 accumulation in slot order, rounded to bf16. */
int moe_permute_backward(const moe_cfg* cfg, const moe_bf16* dx_sorted, const int32_t* inv,
                         moe_bf16* dx, void* stream);

/* Load balancing, step 1: the auxiliary-loss-free bias update ("05 - Expert
 * Parallelism (MoE)", "Load balancing" (b)).  After a step, with the tokens
 * each expert received:
 *   bias[e] += lr * (avg_load - counts[e]),  avg_load = sum(counts) / E,
 * computed in fp64 and rounded once to fp32.  The bias is the selection bias
 * of moe_route (it changes which experts are chosen, never the gates).
 *   counts  int32 [E] (moe_permute's counts, or any per-expert load)
 *   bias    fp32 [E], updated in place
 * One CTA; asynchronous on `stream`. */
int moe_bias_update(const moe_cfg* cfg, const int32_t* counts, float lr, float* bias,
                    void* stream);

/* Load balancing, step 2: redundant experts placed by replicate-then-pack
 * ("Expert parallelism", "Load imbalance becomes idle time").  The n_ep ranks
 * have slots_per_rank expert slots each (n_ep * slots_per_rank >= E, at most
 * 8192 slots in all).
 *   Replicate: the spare slots go one at a time to the expert with the largest
 *   load per copy loads[e] / copies[e] (equal ratios: the lower expert).
 *   Pack: the copies, by load per copy (largest first; equal: lower expert,
 *   then lower copy), each go to the rank with the smallest load so far among
 *   those with a free slot (equal loads: the lower rank).
 * Ratios are compared exactly (64-bit cross products); rank loads are fp64 sums
 * of loads[e] / copies[e] in placement order.
 *   loads       int32 [E] >= 0 (for example moe_permute's counts)
 *   copies      int32 [E] out: copies of each expert (>= 1)
 *   copy_offset int32 [E] out: exclusive prefix sum of copies
 *   copy_rank   int32 [n_ep * slots_per_rank] out: entry copy_offset[e] + j is
 *               the rank holding copy j of expert e (entries past the total
 *               number of copies are not written)
 *   slot_expert int32 [n_ep, slots_per_rank] out: expert in each filled slot in
 *               fill order, -1 in empty slots
 *   rank_load   fp64 [n_ep] out: planned load of each rank
 * One CTA; asynchronous on `stream`.  MOE_E_SHAPE when the slots do not fit. */
int moe_eplb_plan(const moe_cfg* cfg, const int32_t* loads, int32_t slots_per_rank,
                  int32_t* copies, int32_t* copy_offset, int32_t* copy_rank,
                  int32_t* slot_expert, double* rank_load, void* stream);

/* Load balancing, step 3: dispatch over the copies of a plan.  Expert e's kept
 * assignments, in their stable order (rank r = inv[a] - offsets[e] among m
 * kept), are split evenly over its q copies: copy j takes ranks
 * [floor(j*m/q), floor((j+1)*m/q)).
 *   topk_idx, counts, offsets, inv      as written by moe_route / moe_permute
 *   copies, copy_offset, copy_rank      as written by moe_eplb_plan
 *   dest_rank  int32 [A] out: rank holding the copy that processes assignment a
 *              (-1 when dropped)
 *   count_mat  int32 [n_ep, n_ep] out: C[s][g] = assignments of source rank s
 *              (tokens [s*T_loc, (s+1)*T_loc)) processed on rank g
 * Asynchronous on `stream`. */
int moe_eplb_dispatch(const moe_cfg* cfg, const int32_t* topk_idx, const int32_t* counts,
                      const int32_t* offsets, const int32_t* inv, const int32_t* copies,
                      const int32_t* copy_offset, const int32_t* copy_rank, int32_t* dest_rank,
                      int32_t* count_mat, void* stream);

/* Self-test of the device-side time-out path that every kernel with a wait
 * uses.  Launches one small CTA that waits, through the same bounded
 * mbarrier wait, on a barrier that nothing ever completes; after limit_ns it
 * gives up, records MOE_E_DEVICE_TIMEOUT in the workspace status word and
 * returns, leaving the context usable.  No fault, trap or hang is involved.
 *   ws         workspace of at least moe_workspace_bytes(cfg) for any cfg
 *              (only the status word at offset 0 is touched), 16-byte aligned
 *   limit_ns   how long the wait lasts, 1000 .. 1000000000 (else MOE_E_SHAPE)
 * Asynchronous on `stream`; read the result with moe_get_device_status. */
int moe_selftest_wait_timeout(void* ws, uint64_t limit_ns, void* stream);

/* Synchronises `stream`, then returns and clears the workspace status word:
 * MOE_OK, MOE_E_DEVICE_DATA or MOE_E_DEVICE_TIMEOUT (or MOE_E_CUDA). */
int moe_get_device_status(void* ws, void* stream);

/* Static description of an error code. */
const char* moe_strerror(int code);

/* Number of kernels the most recent successful call on this host thread
 * launched (for launch accounting).  Host only. */
int moe_last_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_B300_H */
