"""Plain fp64 restatement of the single-device MoE layer: route, permute (with a
simulated expert-parallel send layout), SwiGLU experts, unpermute + gate +
scatter-add.  TEST INFRASTRUCTURE ONLY (see the package docstring).

Conventions.
  T tokens, d hidden, E routed experts, k experts per token, f expert width,
  n_ep simulated expert-parallel ranks, T_loc = T / n_ep tokens per rank.
  An *assignment* is one (token, slot) pair; its flat index is a = t*k + j, with
  j the slot in rank order of the token's chosen experts.  A = T*k.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "router_logits", "sigmoid", "select_experts", "gate_weights",
    "capacity_rows", "permute", "ep_layout", "swiglu_hidden", "swiglu_expert",
    "expert_outputs", "expert_rows", "combine", "moe_forward", "dense_mask_forward",
    "imbalance_eta", "alltoall_bytes", "dispatch_combine_bytes_per_token",
    "bias_update", "eplb_replicate", "eplb_pack", "eplb_plan", "eplb_dispatch",
    "E4M3_MAX", "e4m3_encode", "e4m3_decode", "quantize_rows_fp8", "dequantize_rows_fp8",
    "ep_layout_fp8", "swiglu_expert_backward", "moe_backward",
]

F64 = np.float64
F32 = np.float32


# ----------------------------------------------------------------------------
# Step 1: route  ([EP] "Expert parallelism", step 1 "Route")
# ----------------------------------------------------------------------------

def router_logits(x, W_r, logit_bias=None):
    """Router logits l[t, e] = sum_i x[t, i] * W_r[i, e] (+ logit_bias[e]), fp64.

    x holds bf16 values (exactly representable in fp64); W_r is fp32.  [EP]
    step 1 computes "the router" on the local tokens; the router is a linear map
    of the token's hidden vector."""
    l = np.asarray(x, F64) @ np.asarray(W_r, F64)
    if logit_bias is not None:
        l = l + np.asarray(logit_bias, F64)[None, :]
    return l


def sigmoid(l):
    """Affinity s = 1 / (1 + exp(-l)) (DeepSeek-V3 style sigmoid scores, [EP]
    "What DeepSeek-V3 did about it", node-limited routing by affinities)."""
    l = np.asarray(l, F64)
    return 1.0 / (1.0 + np.exp(-l))


def _rank_order(values32, mask_out=None):
    """Per row, the column indices sorted by (value descending, index ascending).

    The order is a total order on fp32 values: -0.0 equals +0.0 (so the lower
    index wins), NaN ranks below -inf, equal values keep index order.  numpy's
    stable lexsort on (-value) gives exactly that: negation is exact, sorting
    treats -0.0 == +0.0, and NaN sorts after +inf.  Columns with mask_out=True
    rank after every other column."""
    v = np.asarray(values32, F32)
    n = v.shape[-1]
    cols = np.broadcast_to(np.arange(n), v.shape)
    keys = [cols, -v]
    if mask_out is not None:
        keys.append(np.asarray(mask_out, np.int8))
    return np.lexsort(keys, axis=-1)


def select_experts(scores, k, bias=None, n_groups=1, topk_groups=1):
    """Top-k expert choice per token, int64 [T, k] in rank order.

    scores: fp32 [T, E] (logits for softmax routing, sigmoid affinities for
    sigmoid routing).  bias: optional fp32 [E] selection bias, the auxiliary-
    loss-free balancing bias of [EPM] "Load balancing", (b): chosen =
    TopK(logits + bias); it is added with one fp32 addition and never enters the
    gates.

    Group-limited (node-limited) routing, [EP] "What DeepSeek-V3 did about it":
    experts are split into n_groups contiguous groups; a group's score is the
    sum of the token's two highest (biased) values in it, computed as one fp32
    addition; the topk_groups best groups are kept ("node limits must be applied
    before final top-k", [EPS] "Failure modes"), and the k experts are chosen
    among the kept groups.  Ties break toward the lower expert (or group) index.
    """
    v = np.asarray(scores, F32)
    T, E = v.shape
    if bias is not None:
        v = (v + np.asarray(bias, F32)[None, :]).astype(F32)
    if n_groups > 1:
        gs = E // n_groups
        vg = v.reshape(T, n_groups, gs)
        srt = np.sort(-vg, axis=-1)                     # NaN last, i.e. lowest value
        top1 = (-srt[..., 0]).astype(F32)
        top2 = (-srt[..., 1]).astype(F32)
        gscore = (top1 + top2).astype(F32)              # one fp32 addition
        gorder = _rank_order(gscore)[:, :topk_groups]   # kept groups
        keep = np.zeros((T, n_groups), bool)
        np.put_along_axis(keep, gorder, True, axis=1)
        excluded = ~np.repeat(keep, gs, axis=1)
        order = _rank_order(v, excluded)
    else:
        order = _rank_order(v)
    return order[:, :k].astype(np.int64)


def gate_weights(scores, idx, score_fn, norm_topk):
    """Gate of each chosen expert, fp64 [T, k].

    softmax: g = exp(l_e - m) / sum_{e' < E} exp(l_e' - m) over all E logits
    (router probability, [EPM] "Load balancing" (a): P_i is the router
    probability); sigmoid: g = s_e.  With norm_topk the k gates are divided by
    their sum (DeepSeek-V3's normalised gates).  The selection bias never enters
    the gates ([EPM] "(b) Auxiliary-loss-free")."""
    s = np.asarray(scores, F32).astype(F64)
    idx = np.asarray(idx)
    if score_fn == "softmax":
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        p = p / p.sum(axis=1, keepdims=True)
        g = np.take_along_axis(p, idx, axis=1)
    elif score_fn == "sigmoid":
        g = np.take_along_axis(s, idx, axis=1)
    else:
        raise ValueError(score_fn)
    if norm_topk:
        g = g / g.sum(axis=1, keepdims=True)
    return g


# ----------------------------------------------------------------------------
# Step 2: permute  ([EP] step 2 "Permute"; "Token permutation and grouped GEMMs")
# ----------------------------------------------------------------------------

def capacity_rows(capacity_factor, T, k, E):
    """Rows per expert under a capacity factor: CF times the fair share T*k/E,
    rounded up ([EP] "Load imbalance becomes idle time": capping every expert at
    CF times its fair share)."""
    return int(math.ceil(capacity_factor * T * k / E))


def permute(idx, E, capacity=0):
    """Stable grouping of the T*k assignments into per-expert segments.

    [EP] "Token permutation and grouped GEMMs": order is the stable argsort of
    the expert ids, X[order] puts the rows in expert order, and the inverse
    permutation inv[order] = arange(n) puts them back.

    Returns a dict with
      counts  int64 [E]   assignments routed to each expert (before any drop)
      offsets int64 [E+1] first row of each expert's segment; dropless: the
                          exclusive prefix sum of counts; capacity: e*cap
      order   int64 [R]   row -> assignment a (-1 for a padding row)
      inv     int64 [A]   assignment -> row (-1 for a dropped assignment)
      kept    int64 [E]   rows holding data in each segment
    Capacity mode ([EP] "Token permutation...", pad to capacity and batch): each
    expert keeps its first `capacity` assignments in increasing a (the stable
    order, i.e. dropping overflow by token order) and its segment is padded to
    exactly `capacity` rows; R = E*capacity.  Dropless: R = A."""
    flat = np.asarray(idx).reshape(-1).astype(np.int64)
    A = flat.size
    if A and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert id out of range")
    srt = np.argsort(flat, kind="stable")               # positions in expert order
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    starts = np.zeros(E + 1, np.int64)
    starts[1:] = np.cumsum(counts)                       # exclusive prefix (+ total)
    rank = np.arange(A, dtype=np.int64) - starts[flat[srt]]   # rank within expert
    inv = np.full(A, -1, np.int64)
    if capacity:
        R = E * capacity
        order = np.full(R, -1, np.int64)
        keep = rank < capacity
        rows = flat[srt][keep] * capacity + rank[keep]
        order[rows] = srt[keep]
        inv[srt[keep]] = rows
        offsets = np.arange(E + 1, dtype=np.int64) * capacity
        kept = np.minimum(counts, capacity)
    else:
        order = srt.astype(np.int64)
        inv[srt] = np.arange(A, dtype=np.int64)
        offsets = starts
        kept = counts.copy()
    return {"counts": counts, "offsets": offsets, "order": order, "inv": inv,
            "kept": kept}


def ep_layout(idx, inv, E, n_ep, T):
    """Simulated expert-parallel send layout ([EP] steps 2-4 and "A dispatch you
    can check by hand").

    Expert e lives on rank floor(e*n_ep/E); token t belongs to source rank
    floor(t/T_loc).  Each source rank sorts its (kept) assignments by
    destination rank, and inside a destination by expert and then by a (a
    stable sort, so the receiver's "sort by local expert", step 5, reproduces
    the global per-expert order).  Returns
      C        int64 [n_ep, n_ep]  C[s, q] = rows rank s sends to rank q
      send_off int64 [n_ep, n_ep]  start of q's block in s's send buffer
      recv_off int64 [n_ep, n_ep]  recv_off[q, s]: start of s's block in q's
                                   receive buffer
      send_idx int64 [A]           s's buffer occupies [s*T_loc*k, (s+1)*T_loc*k);
                                   entry p holds the assignment a sent from that
                                   slot, -1 past the last kept row
    Combine sends the same blocks back (the transpose of C, [EP] "A dispatch
    you can check by hand")."""
    idx = np.asarray(idx)
    T_, k = idx.shape
    assert T_ == T
    flat = idx.reshape(-1).astype(np.int64)
    inv = np.asarray(inv)
    T_loc = T // n_ep
    dest = flat * n_ep // E
    C = np.zeros((n_ep, n_ep), np.int64)
    send_idx = np.full(T * k, -1, np.int64)
    for s in range(n_ep):
        a = np.arange(s * T_loc * k, (s + 1) * T_loc * k, dtype=np.int64)
        a = a[inv[a] >= 0]                               # kept assignments only
        o = np.lexsort((a, flat[a], dest[a]))            # by (dest, expert, a)
        send_idx[s * T_loc * k: s * T_loc * k + a.size] = a[o]
        C[s] = np.bincount(dest[a], minlength=n_ep)
    send_off = np.zeros_like(C)
    send_off[:, 1:] = np.cumsum(C, axis=1)[:, :-1]
    recv_off = np.zeros_like(C)
    recv_off[:, 1:] = np.cumsum(C.T, axis=1)[:, :-1]
    return {"C": C, "send_off": send_off, "recv_off": recv_off,
            "send_idx": send_idx}


# ----------------------------------------------------------------------------
# Step 5: expert compute ([EP] step 5; "How many bytes move": SwiGLU expert)
# ----------------------------------------------------------------------------

def swiglu_hidden(X, W1, W3):
    """The SwiGLU expert's hidden activations on rows X (fp64): h = silu(W1 x) *
    (W3 x), with silu(u) = u / (1 + exp(-u)).  W1, W3: [f, d] (out, in).  This is
    the first two of the expert's three d-by-d_e products ([EP] "DeepSeek-V3's
    layout, counted"); the grouped FFN keeps h between its two products."""
    X = np.asarray(X, F64)
    u = X @ np.asarray(W1, F64).T
    v = X @ np.asarray(W3, F64).T
    return (u / (1.0 + np.exp(-u))) * v


def swiglu_expert(X, W1, W3, W2):
    """SwiGLU expert on rows X (fp64): W2 (silu(W1 x) * (W3 x)).  W2: [d, f]
    (out, in).  One expert holds the three d-by-d_e matrices of [EP]
    "DeepSeek-V3's layout, counted" and costs 6*d*d_e FLOPs per row ([EP] "A
    worked example")."""
    return swiglu_hidden(X, W1, W3) @ np.asarray(W2, F64).T


def expert_outputs(x, perm, k, W1, W3, W2, rows=None):
    """Expert output of every row of the expert-grouped buffer (step 5: each
    expert runs on its contiguous segment).  Returns fp64 [R, d]; rows not in
    `rows`, and padding rows, stay zero.  W1/W3/W2 are indexable per expert."""
    order = perm["order"]
    R = order.size
    x = np.asarray(x)
    out = np.zeros((R, x.shape[1]), F64)
    sel = np.ones(R, bool) if rows is None else np.zeros(R, bool)
    if rows is not None:
        sel[np.asarray(rows)] = True
    offsets, kept = perm["offsets"], perm["kept"]
    for e in range(kept.size):
        rr = np.arange(int(offsets[e]), int(offsets[e]) + int(kept[e]))
        rr = rr[sel[rr]]
        if rr.size:
            out[rr] = swiglu_expert(x[order[rr] // k], W1[e], W3[e], W2[e])
    return out


def expert_rows(x, perm, k, W1, W3, W2, rows):
    """Hidden activations and outputs of chosen rows of the expert-grouped
    buffer (step 5, each expert on its contiguous segment), computed expert by
    expert.  rows: row ids in [0, R); a row past its expert's kept rows (capacity
    padding) gives zeros.  Returns (h fp64 [n, f], out fp64 [n, d]) in the order
    of `rows`."""
    rows = np.asarray(rows, np.int64)
    order, offsets, kept = perm["order"], perm["offsets"], perm["kept"]
    x = np.asarray(x)
    f = np.asarray(W1[0]).shape[0]
    h = np.zeros((rows.size, f), F64)
    out = np.zeros((rows.size, x.shape[1]), F64)
    for e in range(kept.size):
        lo, hi = int(offsets[e]), int(offsets[e]) + int(kept[e])
        sel = np.nonzero((rows >= lo) & (rows < hi))[0]
        if sel.size:
            X = x[order[rows[sel]] // k]
            h[sel] = swiglu_hidden(X, W1[e], W3[e])
            out[sel] = h[sel] @ np.asarray(W2[e], F64).T
    return h, out


def combine(out_rows, perm, k, gates, T, shared_out=None):
    """Step 7 ([EP] "Unpermute and weight"): undo the sort and scatter-add each
    row into its token with its gate: y[t] += g[a] * out[row(a)] for every kept
    assignment; dropped assignments add nothing.  A shared expert's output is
    added to every token ([EPM] "Fine-grained vs coarse experts": shared experts
    always active).  fp64."""
    order = perm["order"]
    g = np.asarray(gates, F64).reshape(-1)
    y = np.zeros((T, out_rows.shape[1]), F64)
    rows = np.nonzero(order >= 0)[0]
    a = order[rows]
    np.add.at(y, a // k, g[a][:, None] * out_rows[rows])
    if shared_out is not None:
        y += shared_out
    return y


def moe_forward(x, scores, cfg, W1, W3, W2, bias=None, tokens=None):
    """The whole single-device layer, steps 1-7 of [EP] "Expert parallelism"
    with the exchange steps 3, 4 and 6 being identities on one device.

    x: bf16 values [T, d]; scores: fp32 [T, E] fed to selection; W1/W3/W2
    indexable by expert (index E = the shared expert when cfg.has_shared).
    tokens: optional subset of token ids whose outputs are computed (the other
    rows of y are left zero); routing and permutation always cover all T.
    Returns (y fp64 [T, d], dict of intermediates)."""
    T, E, k = cfg.T, cfg.E, cfg.k
    idx = select_experts(scores, k, bias, cfg.n_groups, cfg.topk_groups)
    gates = gate_weights(scores, idx, cfg.score_fn, cfg.norm_topk)
    perm = permute(idx, E, cfg.capacity)
    rows = None
    if tokens is not None:
        tok = np.zeros(T, bool)
        tok[np.asarray(tokens)] = True
        order = perm["order"]
        rows = np.nonzero((order >= 0) & tok[np.maximum(order, 0) // k])[0]
    out = expert_outputs(x, perm, k, W1, W3, W2, rows)
    shared = None
    if cfg.has_shared:
        shared = np.zeros((T, np.asarray(x).shape[1]), F64)
        tt = np.arange(T) if tokens is None else np.asarray(tokens)
        shared[tt] = swiglu_expert(np.asarray(x)[tt], W1[E], W3[E], W2[E])
    y = combine(out, perm, k, gates, T, shared)
    return y, {"idx": idx, "gates": gates, "perm": perm}


def dense_mask_forward(x, scores, cfg, W1, W3, W2, bias=None):
    """Brute force: run every expert on every token and weight by a dense
    [T, E] gate mask that is zero outside each token's chosen experts.  Same
    layer as `moe_forward` with no permutation at all; pure loops, for tiny
    sizes only."""
    T, E = cfg.T, cfg.E
    idx = select_experts(scores, cfg.k, bias, cfg.n_groups, cfg.topk_groups)
    gates = gate_weights(scores, idx, cfg.score_fn, cfg.norm_topk)
    mask = np.zeros((T, E), F64)
    for t in range(T):
        for j in range(cfg.k):
            mask[t, idx[t, j]] = gates[t, j]
    x = np.asarray(x, F64)
    y = np.zeros_like(x)
    for e in range(E):
        out = swiglu_expert(x, W1[e], W3[e], W2[e])
        y += mask[:, e:e + 1] * out
    if cfg.has_shared:
        y += swiglu_expert(x, W1[E], W3[E], W2[E])
    return y


# ----------------------------------------------------------------------------
# Layout metrics ([EP] "How many bytes move", "Load imbalance becomes idle time")
# ----------------------------------------------------------------------------

def imbalance_eta(C):
    """Fraction of the group's expert compute doing useful work: the mean GPU
    load over the busiest GPU's load, loads being column sums of the dispatch
    matrix ([EP] "Load imbalance becomes idle time": a GPU with 50 % more than
    its share runs the group at two thirds of its speed)."""
    loads = np.asarray(C, F64).sum(axis=0)
    return float(loads.mean() / loads.max())


def alltoall_bytes(C, d, s_disp, s_comb):
    """Bytes leaving each source rank in one dispatch and one combine: only
    off-diagonal rows cross the network ([EP] "How many bytes move").  Returns
    (dispatch_bytes[s], combine_bytes[s]); combine moves C transposed."""
    C = np.asarray(C, np.int64)
    off = C - np.diag(np.diag(C))
    disp = off.sum(axis=1) * d * s_disp
    comb = off.sum(axis=0) * d * s_comb
    return disp, comb


def dispatch_combine_bytes_per_token(k, d, s_disp, s_comb):
    """Every token ships k copies of its d-vector out and gets k results back:
    k*d*(s_disp + s_comb) bytes ([EPM] "The all-to-all pattern": 2 x top_k x
    hidden x bytes)."""
    return k * d * (s_disp + s_comb)


# ----------------------------------------------------------------------------
# Load balancing: the auxiliary-loss-free bias update ([EPM] "Load balancing"
# (b)) and redundant experts placed by replicate-then-pack ([EP] "Load
# imbalance becomes idle time")
# ----------------------------------------------------------------------------

def bias_update(bias, counts, lr):
    """One step of the bias control loop: after a step, count the tokens each
    expert received; an under-loaded expert's selection bias rises and an
    over-loaded one's falls, in proportion to its distance from the average
    load over the experts ([EPM] "Load balancing" (b)).  fp64."""
    c = np.asarray(counts, F64)
    return np.asarray(bias, F64) + float(lr) * (c.mean() - c)


def eplb_replicate(loads, n_slots):
    """Step 1, Replicate: with n_slots expert slots in the group and E experts,
    the n_slots - E spare slots are handed out one at a time, each to the expert
    whose load per copy c_i / q_i is currently the largest (equal ratios: the
    lower expert index).  Ratios are compared exactly as fractions.  Returns
    q, the number of copies of every expert."""
    from fractions import Fraction
    c = [int(v) for v in loads]
    E = len(c)
    if n_slots < E:
        raise ValueError("fewer slots than experts")
    q = [1] * E
    for _ in range(n_slots - E):
        best = max(range(E), key=lambda i: (Fraction(c[i], q[i]), -i))
        q[best] += 1
    return np.array(q, np.int64)


def eplb_pack(loads, q, n_ranks, slots):
    """Step 2, Pack (longest processing time first): every copy of expert i
    carries c_i / q_i; the copies, sorted by that load (largest first; equal
    loads: lower expert index, then lower copy index), are placed one at a time
    on the rank with the smallest load so far among those with a free slot
    (equal loads: the lower rank).  Rank loads are fp64 sums of c_i / q_i in
    placement order.

    Returns (copy_rank, slot_expert, rank_load): copy_rank[off_i + j] = rank of
    copy j of expert i (off = exclusive prefix of q); slot_expert[r][s] = the
    expert in rank r's s-th filled slot, -1 when empty; rank_load[r] fp64."""
    from fractions import Fraction
    c = [int(v) for v in loads]
    q = [int(v) for v in q]
    E = len(c)
    order = sorted(range(E), key=lambda i: (-Fraction(c[i], q[i]), i))
    off = np.concatenate([[0], np.cumsum(q)])[:-1]
    copy_rank = np.full(int(sum(q)), -1, np.int64)
    slot_expert = np.full((n_ranks, slots), -1, np.int64)
    used = [0] * n_ranks
    load = [0.0] * n_ranks
    for i in order:
        per = float(c[i]) / float(q[i])
        for j in range(q[i]):
            free = [r for r in range(n_ranks) if used[r] < slots]
            r = min(free, key=lambda rr: (load[rr], rr))
            copy_rank[off[i] + j] = r
            slot_expert[r][used[r]] = i
            used[r] += 1
            load[r] = load[r] + per
    return copy_rank, slot_expert, np.array(load, F64)


def eplb_plan(loads, n_ranks, slots):
    """Replicate then pack ([EP] "Load imbalance becomes idle time")."""
    q = eplb_replicate(loads, n_ranks * slots)
    copy_rank, slot_expert, rank_load = eplb_pack(loads, q, n_ranks, slots)
    return {"copies": q, "copy_offset": np.concatenate([[0], np.cumsum(q)])[:-1],
            "copy_rank": copy_rank, "slot_expert": slot_expert, "rank_load": rank_load}


def eplb_dispatch(idx, inv, offsets, counts, plan, n_ranks, T, capacity=0):
    """Where every assignment goes once experts have copies: expert e's kept
    assignments, in their stable order (rank r = inv[a] - offsets[e]), are
    split evenly among its q_e copies, copy j taking ranks
    [floor(j*m/q_e), floor((j+1)*m/q_e)) of its m kept assignments.  Returns
    (dest_rank[A], C[s][g]) with s = the source rank of the token (T/n_ranks
    tokens each) and g the rank holding that copy; dropped assignments get -1."""
    idx = np.asarray(idx).reshape(-1)
    inv = np.asarray(inv).reshape(-1)
    A = idx.size
    k = A // T
    T_loc = T // n_ranks
    dest = np.full(A, -1, np.int64)
    C = np.zeros((n_ranks, n_ranks), np.int64)
    for a in range(A):
        if inv[a] < 0:
            continue
        e = int(idx[a])
        r = int(inv[a]) - int(offsets[e])
        m = int(counts[e]) if not capacity else min(int(counts[e]), capacity)
        qe = int(plan["copies"][e])
        j = 0
        while (j + 1) * m // qe <= r:   # copy j holds ranks [j*m//qe, (j+1)*m//qe)
            j += 1
        g = int(plan["copy_rank"][int(plan["copy_offset"][e]) + j])
        dest[a] = g
        C[(a // k) // T_loc, g] += 1
    return dest, C


# ----------------------------------------------------------------------------
# FP8 dispatch ([EP] "A worked example at DeepSeek-V3's shape": DeepSeek-V3
# dispatches in FP8, s = 1 byte, and combines in BF16; "Lower precision on the
# wire": FP8 halves s_disp).  The pages fix neither the FP8 format nor the
# scale granularity: this restatement uses e4m3 (1 sign, 4 exponent bits with
# bias 7, 3 mantissa bits; largest finite value 448) with one fp32 scale per
# dispatched row, scale = absmax(row) / 448, code = e4m3(x * (448 / absmax)),
# rounding to nearest even and saturating at +-448.  Floating-point steps are fp32, as
# on the device, because they decide integer codes.
# ----------------------------------------------------------------------------

E4M3_MAX = 448.0


def e4m3_encode(v):
    """fp32 values -> e4m3 codes (uint8), round to nearest even, saturate to
    the largest finite magnitude 448 (NaN is not expected)."""
    v = np.asarray(v, F32).astype(F64)          # exact
    sign = (np.signbit(v)).astype(np.uint8) << 7
    a = np.abs(v)
    # quantum of the e4m3 grid around |v|: 2^(e-3) for normals (e >= -6), 2^-9 below
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)
    q = np.exp2(e - 3.0)
    g = np.rint(a / q) * q                      # half to even (exact in fp64)
    g = np.minimum(g, E4M3_MAX)
    # encode the grid value g
    code = np.zeros(a.shape, np.uint8)
    sub = g < 2.0 ** -6
    code[sub] = np.rint(g[sub] / 2.0 ** -9).astype(np.uint8)
    nrm = ~sub
    gn = g[nrm]
    en = np.floor(np.log2(gn))
    mant = np.rint((gn / np.exp2(en) - 1.0) * 8.0)
    code[nrm] = ((en + 7).astype(np.int64) << 3 | mant.astype(np.int64)).astype(np.uint8)
    return code | sign


def e4m3_decode(code):
    """e4m3 codes -> fp32 values (the code 0x7F / 0xFF, NaN, is not produced)."""
    c = np.asarray(code, np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    ef = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(ef == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(ef - 7.0))
    return (s * mag).astype(F32)


def quantize_rows_fp8(rows):
    """One fp32 scale per row, scale = absmax / 448 (1 for an all-zero row),
    and the row's e4m3 codes of x * (448 / absmax): one fp32 division per row
    for each of the two factors, one fp32 product per element."""
    r = np.asarray(rows, F32)
    amax = np.abs(r).max(axis=-1)
    nz = amax > 0
    safe = np.where(nz, amax, F32(1.0)).astype(F32)
    scale = np.where(nz, safe / F32(E4M3_MAX), F32(1.0)).astype(F32)
    inv = np.where(nz, F32(E4M3_MAX) / safe, F32(1.0)).astype(F32)
    return e4m3_encode((r * inv[..., None]).astype(F32)), scale


def dequantize_rows_fp8(codes, scale):
    """code value times the row's scale (one fp32 product), rounded to bf16;
    returned as the fp32 value of that bf16."""
    import torch
    v = e4m3_decode(codes) * np.asarray(scale, F32)[..., None]
    return torch.from_numpy(np.ascontiguousarray(v, F32)).to(torch.bfloat16).float().numpy()


def ep_layout_fp8(x, idx, inv, E, n_ep, T):
    """The expert-parallel layout with an FP8 send buffer: the same slots as
    ep_layout; slot p carries the codes and scale of its token's row, empty
    slots carry zero codes and scale 0."""
    lay = ep_layout(idx, inv, E, n_ep, T)
    k = np.asarray(idx).reshape(T, -1).shape[1]
    codes_t, scale_t = quantize_rows_fp8(np.asarray(x, F32))
    sidx = lay["send_idx"]
    d = codes_t.shape[1]
    send = np.zeros((sidx.size, d), np.uint8)
    sc = np.zeros(sidx.size, F32)
    ok = sidx >= 0
    send[ok] = codes_t[sidx[ok] // k]
    sc[ok] = scale_t[sidx[ok] // k]
    lay["send_fp8"] = send
    lay["send_scale"] = sc
    return lay


# ----------------------------------------------------------------------------
# Backward ([EP] "Expert parallelism": the dispatch and combine run "twice
# more in the backward pass"): the gradients of the layer with the routing
# decision held fixed.  Step 7 backward is a dispatch of dy (each kept
# assignment receives gate * dy of its token, and its gate receives <dy, o>);
# step 5 backward runs the experts' transposed products; step 2 backward is a
# combine (each token sums the input gradients of its kept rows).
# ----------------------------------------------------------------------------

def swiglu_expert_backward(X, W1, W3, W2, dO):
    """Gradients of O = W2 (silu(W1 x) * (W3 x)) for rows X given dO (fp64):
    returns (dX, dW1, dW3, dW2) with silu'(u) = s (1 + u (1 - s)), s = 1/(1+e^-u)."""
    X = np.asarray(X, F64)
    W1 = np.asarray(W1, F64)
    W3 = np.asarray(W3, F64)
    W2 = np.asarray(W2, F64)
    dO = np.asarray(dO, F64)
    u = X @ W1.T
    v = X @ W3.T
    s = 1.0 / (1.0 + np.exp(-u))
    h = u * s * v
    dh = dO @ W2
    du = dh * v * s * (1.0 + u * (1.0 - s))
    dv = dh * u * s
    return du @ W1 + dv @ W3, du.T @ X, dv.T @ X, dO.T @ h


def moe_backward(x, scores, cfg, W1, W3, W2, dy, bias=None):
    """Backward of moe_forward for output gradient dy [T, d] (fp64), routing
    (indices and kept rows) fixed: returns dict with dx [T, d], dW1/dW3
    [E(+1), f, d], dW2 [E(+1), d, f] and dgate [T, k] (the gradient with
    respect to the gate values; dropped assignments get 0)."""
    T, E, k = cfg.T, cfg.E, cfg.k
    x = np.asarray(x, F64)
    dy = np.asarray(dy, F64)
    idx = select_experts(scores, k, bias, cfg.n_groups, cfg.topk_groups)
    gates = gate_weights(scores, idx, cfg.score_fn, cfg.norm_topk).reshape(-1)
    perm = permute(idx, E, cfg.capacity)
    n = E + (1 if cfg.has_shared else 0)
    f, d = np.asarray(W1[0]).shape
    dx = np.zeros((T, d), F64)
    dW1 = np.zeros((n, f, d), F64)
    dW3 = np.zeros((n, f, d), F64)
    dW2 = np.zeros((n, d, f), F64)
    dgate = np.zeros(T * k, F64)
    order, offsets, kept = perm["order"], perm["offsets"], perm["kept"]
    for e in range(E):
        rows = np.arange(int(offsets[e]), int(offsets[e]) + int(kept[e]))
        if rows.size == 0:
            continue
        a = order[rows]
        t = a // k
        Xe = x[t]
        o = swiglu_expert(Xe, W1[e], W3[e], W2[e])
        dgate[a] = (dy[t] * o).sum(axis=1)
        dO = gates[a][:, None] * dy[t]
        dXe, dW1[e], dW3[e], dW2[e] = swiglu_expert_backward(Xe, W1[e], W3[e], W2[e], dO)
        np.add.at(dx, t, dXe)
    if cfg.has_shared:
        dXs, dW1[E], dW3[E], dW2[E] = swiglu_expert_backward(x, W1[E], W3[E], W2[E], dy)
        dx += dXs
    return {"dx": dx, "dW1": dW1, "dW3": dW3, "dW2": dW2, "dgate": dgate.reshape(T, k),
            "idx": idx, "gates": gates.reshape(T, k), "perm": perm}
