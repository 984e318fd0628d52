/*
 * Per-token loop oracle for the single-device MoE layer, in plain C, fp64.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code with
 * the CUDA library, and it shares no code with the numpy oracle beside it
 * either: it restates the same definitions a second way (one token at a time,
 * counting sorts instead of argsorts), so that the two can check each other.
 *
 * Sources (page titles as published):
 *   [EP]   "Expert parallelism" (zerotofrontier.app, MoE chapter)
 *   [EPS]  "Expert Parallelism at Scale"
 *   [EPM]  "05 - Expert Parallelism (MoE)"
 *
 * Conventions: T tokens, d hidden, E routed experts, k experts per token, f
 * expert width, n_ep simulated expert-parallel ranks, T_loc = T / n_ep.  An
 * assignment is one (token, slot) pair with flat index a = t*k + j, j the slot
 * in rank order.  Floating-point inputs arrive as fp32 arrays holding the exact
 * values the layer sees (bf16 activations and weights are exactly representable
 * in fp32); every product and sum below is formed in fp64.  Selection follows
 * fp32 rules: a bias is added with one fp32 addition, a group score is one fp32
 * addition, and comparisons are on fp32 values.  Build without -ffast-math and
 * without FMA contraction (-ffp-contract=off) so that those fp32 additions stay
 * single, correctly rounded operations.
 *
 * Every entry point returns 0, or -1 on an argument it cannot use (an expert id
 * outside [0, E), sizes that do not divide).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define LOOP_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------------- */
/* Step 1: route ([EP] "Expert parallelism", step 1)                          */
/* ------------------------------------------------------------------------- */

/* Router logits l[t, e] = sum_i x[t, i] * W_r[i, e] (+ logit_bias[e]).  x is
 * [T, d], W_r is [d, E] (fp32), out is [T, E] fp64.  The router is a linear map
 * of the token's hidden vector; the sum runs over i in increasing order. */
LOOP_API int loop_router_logits(int T, int d, int E, const float* x, const float* W_r,
                                const float* logit_bias, double* out) {
  if (T < 0 || d <= 0 || E <= 0) return -1;
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int i = 0; i < d; ++i) acc += (double)x[(size_t)t * d + i] * (double)W_r[(size_t)i * E + e];
      if (logit_bias) acc += (double)logit_bias[e];
      out[(size_t)t * E + e] = acc;
    }
  }
  return 0;
}

/* The selection order on fp32 values: larger first; equal values (including
 * -0.0 against +0.0) in increasing index; a NaN after every number.  Returns
 * nonzero when (va, ia) comes before (vb, ib). */
static int ahead(float va, int ia, float vb, int ib) {
  const int na = isnan(va), nb = isnan(vb);
  if (na || nb) {
    if (na && nb) return ia < ib;
    return nb;  /* the number comes first */
  }
  if (va > vb) return 1;
  if (va < vb) return 0;
  return ia < ib;
}

/* Top-k expert choice for every token ([EP] step 1; group limit from [EP] "What
 * DeepSeek-V3 did about it" and [EPS] "Failure modes": the node limit applies
 * before the final top-k).
 *   scores  fp32 [T, E]  logits (softmax routing) or sigmoid affinities
 *   bias    fp32 [E] or NULL: the selection bias of [EPM] "Load balancing" (b),
 *           added to the score by one fp32 addition; it never enters the gates
 *   groups  with n_groups > 1 the experts form n_groups contiguous groups; a
 *           group's score is the fp32 sum of its two best biased values; the
 *           topk_groups best groups stay eligible, and the k experts come from
 *           them (were k larger than their experts, the rest would follow in
 *           the same order among the excluded experts)
 *   idx     int32 [T, k] out, in rank order
 * One token at a time: the group scores by a scan of each group, then k passes
 * over the experts, each taking the best expert not yet taken. */
LOOP_API int loop_select(int T, int E, int k, const float* scores, const float* bias,
                         int n_groups, int topk_groups, int32_t* idx) {
  if (T < 0 || E <= 0 || k <= 0 || k > E || n_groups <= 0 || E % n_groups) return -1;
  if (topk_groups <= 0 || topk_groups > n_groups) return -1;
  const int gs = E / n_groups;
  if (n_groups > 1 && gs < 2) return -1;
  float* v = (float*)malloc(sizeof(float) * (size_t)E);
  float* gscore = (float*)malloc(sizeof(float) * (size_t)n_groups);
  unsigned char* eligible = (unsigned char*)malloc((size_t)E);
  unsigned char* taken = (unsigned char*)malloc((size_t)(E > n_groups ? E : n_groups));
  if (!v || !gscore || !eligible || !taken) {
    free(v); free(gscore); free(eligible); free(taken);
    return -1;
  }
  for (int t = 0; t < T; ++t) {
    const float* s = scores + (size_t)t * E;
    for (int e = 0; e < E; ++e) {
      volatile float sum = bias ? s[e] + bias[e] : s[e];  /* one fp32 addition */
      v[e] = sum;
    }
    if (n_groups > 1) {
      for (int g = 0; g < n_groups; ++g) {
        /* the group's best and second best values in the selection order */
        int b1 = -1, b2 = -1;
        for (int e = g * gs; e < (g + 1) * gs; ++e) {
          if (b1 < 0 || ahead(v[e], e, v[b1], b1)) {
            b2 = b1;
            b1 = e;
          } else if (b2 < 0 || ahead(v[e], e, v[b2], b2)) {
            b2 = e;
          }
        }
        volatile float gsum = v[b1] + v[b2];  /* one fp32 addition */
        gscore[g] = gsum;
      }
      memset(taken, 0, (size_t)n_groups);
      memset(eligible, 0, (size_t)E);
      for (int r = 0; r < topk_groups; ++r) {
        int best = -1;
        for (int g = 0; g < n_groups; ++g)
          if (!taken[g] && (best < 0 || ahead(gscore[g], g, gscore[best], best))) best = g;
        taken[best] = 1;
        for (int e = best * gs; e < (best + 1) * gs; ++e) eligible[e] = 1;
      }
    } else {
      memset(eligible, 1, (size_t)E);
    }
    memset(taken, 0, (size_t)E);
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0) { best = e; continue; }
        if (eligible[e] != eligible[best]) {
          if (eligible[e]) best = e;
          continue;
        }
        if (ahead(v[e], e, v[best], best)) best = e;
      }
      taken[best] = 1;
      idx[(size_t)t * k + j] = best;
    }
  }
  free(v); free(gscore); free(eligible); free(taken);
  return 0;
}

/* Gate of each chosen expert, fp64 [T, k].
 *   score_fn 0 (softmax): g = exp(l_e - m) / sum over all E of exp(l_e' - m), the
 *     router probability of [EPM] "Load balancing" (a), m the row's largest logit;
 *   score_fn 1 (sigmoid): g = s_e, the affinity itself;
 *   norm_topk: the k gates are divided by their sum (DeepSeek-V3's normalised
 *     gates).  The selection bias never enters ([EPM] "Load balancing" (b)). */
LOOP_API int loop_gates(int T, int E, int k, const float* scores, const int32_t* idx,
                        int score_fn, int norm_topk, double* gates) {
  if (T < 0 || E <= 0 || k <= 0 || (score_fn != 0 && score_fn != 1)) return -1;
  for (int t = 0; t < T; ++t) {
    const float* s = scores + (size_t)t * E;
    double m = 0.0, z = 0.0;
    if (score_fn == 0) {
      m = (double)s[0];
      for (int e = 1; e < E; ++e)
        if ((double)s[e] > m) m = (double)s[e];
      for (int e = 0; e < E; ++e) z += exp((double)s[e] - m);
    }
    double sum = 0.0;
    for (int j = 0; j < k; ++j) {
      const int e = idx[(size_t)t * k + j];
      if (e < 0 || e >= E) return -1;
      const double g = score_fn == 0 ? exp((double)s[e] - m) / z : (double)s[e];
      gates[(size_t)t * k + j] = g;
      sum += g;
    }
    if (norm_topk)
      for (int j = 0; j < k; ++j) gates[(size_t)t * k + j] /= sum;
  }
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Step 2: permute ([EP] step 2; "Token permutation and grouped GEMMs")       */
/* ------------------------------------------------------------------------- */

/* Grouping of the A = T*k assignments into per-expert segments, as a counting
 * sort: one pass counts each expert's assignments, the segment starts follow,
 * and a second pass in increasing a hands each assignment the next row of its
 * expert's segment, so rows inside a segment keep the order of a (the stable
 * grouping the pages build with a stable argsort).
 *   counts  int32 [E]    assignments routed to each expert, before any drop
 *   offsets int32 [E+1]  first row of each segment: dropless, the running sum
 *                        of counts; with a capacity, e*capacity
 *   order   int32 [R]    row -> assignment (-1 on a padding row)
 *   inv     int32 [A]    assignment -> row (-1 when dropped)
 *   kept    int32 [E]    rows holding data in each segment
 * With capacity > 0 ([EP] "Load imbalance becomes idle time": every expert
 * capped at a multiple of its fair share) an expert keeps its first `capacity`
 * assignments in increasing a and its segment has exactly `capacity` rows, R =
 * E*capacity; dropless, R = A. */
LOOP_API int loop_permute(int T, int k, int E, int capacity, const int32_t* idx, int32_t* counts,
                          int32_t* offsets, int32_t* order, int32_t* inv, int32_t* kept) {
  if (T < 0 || k <= 0 || E <= 0 || capacity < 0) return -1;
  const long A = (long)T * k;
  const long R = capacity ? (long)E * capacity : A;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (long a = 0; a < A; ++a) {
    if (idx[a] < 0 || idx[a] >= E) return -1;
    counts[idx[a]] += 1;
  }
  long run = 0;
  for (int e = 0; e < E; ++e) {
    offsets[e] = capacity ? e * capacity : (int32_t)run;
    run += counts[e];
    kept[e] = capacity && counts[e] > capacity ? capacity : counts[e];
  }
  offsets[E] = capacity ? E * capacity : (int32_t)run;
  for (long r = 0; r < R; ++r) order[r] = -1;
  int32_t* fill = (int32_t*)calloc((size_t)E, sizeof(int32_t));
  if (!fill) return -1;
  for (long a = 0; a < A; ++a) {
    const int e = idx[a];
    const int rank = fill[e]++;
    if (capacity && rank >= capacity) {
      inv[a] = -1;
      continue;
    }
    const int32_t row = offsets[e] + rank;
    inv[a] = row;
    order[row] = (int32_t)a;
  }
  free(fill);
  return 0;
}

/* Simulated expert-parallel send layout ([EP] steps 2-4 and "A dispatch you
 * can check by hand").  Expert e lives on rank floor(e*n_ep/E); token t comes
 * from rank floor(t/T_loc).  Source rank s lists its kept assignments by
 * destination rank, inside a destination by expert, inside an expert by a,
 * literally: for each destination q, for each expert e of q, for each of s's
 * assignments a in increasing order.
 *   C        int32 [n_ep, n_ep]  C[s][q] = rows s sends to q
 *   send_off int32 [n_ep, n_ep]  start of q's block in s's send buffer
 *   recv_off int32 [n_ep, n_ep]  recv_off[q][s] = start of s's block in q's
 *                                receive buffer
 *   send_idx int32 [A]           s's buffer is [s*T_loc*k, (s+1)*T_loc*k); slot
 *                                p holds the assignment sent from it, -1 past
 *                                the last kept one */
LOOP_API int loop_ep_layout(int T, int k, int E, int n_ep, const int32_t* idx, const int32_t* inv,
                            int32_t* C, int32_t* send_off, int32_t* recv_off, int32_t* send_idx) {
  if (T < 0 || k <= 0 || E <= 0 || n_ep <= 0 || T % n_ep || E % n_ep) return -1;
  const int T_loc = T / n_ep;
  const long per = (long)T_loc * k;
  for (int s = 0; s < n_ep; ++s) {
    long p = s * per;
    for (int q = 0; q < n_ep; ++q) {
      int32_t n = 0;
      for (int e = 0; e < E; ++e) {
        if ((long)e * n_ep / E != q) continue;
        for (long a = s * per; a < (s + 1) * per; ++a) {
          if (idx[a] < 0 || idx[a] >= E) return -1;
          if (idx[a] != e || inv[a] < 0) continue;
          send_idx[p++] = (int32_t)a;
          n += 1;
        }
      }
      C[s * n_ep + q] = n;
    }
    for (; p < (s + 1) * per; ++p) send_idx[p] = -1;
  }
  for (int s = 0; s < n_ep; ++s) {
    int32_t acc = 0;
    for (int q = 0; q < n_ep; ++q) {
      send_off[s * n_ep + q] = acc;
      acc += C[s * n_ep + q];
    }
  }
  for (int q = 0; q < n_ep; ++q) {
    int32_t acc = 0;
    for (int s = 0; s < n_ep; ++s) {
      recv_off[q * n_ep + s] = acc;
      acc += C[s * n_ep + q];
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Steps 5 and 7: experts and combine, token by token                         */
/* ------------------------------------------------------------------------- */

/* One SwiGLU expert on one token ([EP] "How many bytes move": three d-by-d_e
 * matrices per expert, 6*d*d_e FLOPs per token): u = W1 x, v = W3 x,
 * h = silu(u) * v with silu(u) = u / (1 + exp(-u)), o = W2 h.  W1, W3: [f, d];
 * W2: [d, f].  h (length f) is scratch and keeps the hidden activations; o is
 * added into acc with weight g. */
static void swiglu_token(int d, int f, const float* xt, const float* W1, const float* W3,
                         const float* W2, double g, double* h, double* acc) {
  for (int i = 0; i < f; ++i) {
    double u = 0.0, v = 0.0;
    const float* w1 = W1 + (size_t)i * d;
    const float* w3 = W3 + (size_t)i * d;
    for (int c = 0; c < d; ++c) {
      u += (double)w1[c] * (double)xt[c];
      v += (double)w3[c] * (double)xt[c];
    }
    h[i] = u / (1.0 + exp(-u)) * v;
  }
  for (int c = 0; c < d; ++c) {
    double o = 0.0;
    const float* w2 = W2 + (size_t)c * f;
    for (int i = 0; i < f; ++i) o += (double)w2[i] * h[i];
    acc[c] += g * o;
  }
}

/* The layer output of chosen tokens, one token at a time, straight from the
 * token's expert choices ([EP] steps 5 and 7 with the exchanges of steps 3, 4
 * and 6 being identities on one device):
 *   y[t] = sum over j < k, assignment t*k+j kept, of gate[t, j] * expert_{idx[t, j]}(x[t])
 *          (+ shared(x[t]) when has_shared: an always-on expert, [EPM]
 *          "Fine-grained vs coarse experts", added after the routed sum)
 * in slot order.  Whether an assignment is kept is decided here from the ids
 * alone: with capacity > 0, assignment a is kept iff fewer than `capacity`
 * earlier assignments (smaller a) chose the same expert (overflow dropped by
 * token order); dropless, every assignment is kept.
 *   x        fp32 [T, d]
 *   idx      int32 [T, k]; gates fp64 [T, k]
 *   W1, W3   fp32 [E + has_shared, f, d]; W2 fp32 [E + has_shared, d, f]
 *   tokens   int32 [n_tok]: the tokens to compute
 *   y        fp64 [n_tok, d] out, in the order of `tokens`
 *   h        fp64 [n_tok, k + has_shared, f] out or NULL: each slot's hidden
 *            activations (zeros for a dropped slot), the shared expert's last
 * Tokens are independent; with OpenMP they are shared among threads. */
LOOP_API int loop_layer_tokens(int T, int d, int E, int k, int f, int has_shared, int capacity,
                               const float* x, const int32_t* idx, const double* gates,
                               const float* W1, const float* W3, const float* W2, int n_tok,
                               const int32_t* tokens, double* y, double* h) {
  if (T < 0 || d <= 0 || E <= 0 || k <= 0 || f <= 0 || n_tok < 0 || capacity < 0) return -1;
  const long A = (long)T * k;
  unsigned char* keep = (unsigned char*)malloc((size_t)(A > 0 ? A : 1));
  int32_t* seen = (int32_t*)calloc((size_t)E, sizeof(int32_t));
  if (!keep || !seen) {
    free(keep); free(seen);
    return -1;
  }
  for (long a = 0; a < A; ++a) {
    const int e = idx[a];
    if (e < 0 || e >= E) {
      free(keep); free(seen);
      return -1;
    }
    keep[a] = !capacity || seen[e] < capacity;
    seen[e] += 1;
  }
  free(seen);
  for (int n = 0; n < n_tok; ++n)
    if (tokens[n] < 0 || tokens[n] >= T) {
      free(keep);
      return -1;
    }
  const int slots = k + (has_shared ? 1 : 0);
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int n = 0; n < n_tok; ++n) {
    const int t = tokens[n];
    const float* xt = x + (size_t)t * d;
    double* acc = y + (size_t)n * d;
    double* hs = (double*)malloc(sizeof(double) * (size_t)f);
    if (!hs) {
      bad |= 1;
      continue;
    }
    for (int c = 0; c < d; ++c) acc[c] = 0.0;
    for (int j = 0; j < slots; ++j) {
      const int shared = j == k;
      const long a = (long)t * k + j;
      double* hout = h ? h + ((size_t)n * slots + j) * f : NULL;
      if (!shared && !keep[a]) {
        if (hout) memset(hout, 0, sizeof(double) * (size_t)f);
        continue;
      }
      const int e = shared ? E : idx[a];
      const double g = shared ? 1.0 : gates[a];
      swiglu_token(d, f, xt, W1 + (size_t)e * f * d, W3 + (size_t)e * f * d,
                   W2 + (size_t)e * d * f, g, hs, acc);
      if (hout) memcpy(hout, hs, sizeof(double) * (size_t)f);
    }
    free(hs);
  }
  free(keep);
  return bad ? -1 : 0;
}
