"""Property checks of the oracle's permutation and expert-parallel layout over
random small configurations (hypothesis).  Each property is checked by direct
counting with plain loops, not by the oracle's own numpy route (argsort,
bincount, lexsort): per expert, the kept assignments are the first ones in
increasing a and sit in consecutive rows from the segment's start; every row
and every send slot is accounted for exactly once; the count matrix's row
and column sums are the rows each rank sends and receives."""
import numpy as np
from hypothesis import given, settings
from hypothesis import strategies as st

import oracle


@st.composite
def routing(draw):
    n_ep = draw(st.sampled_from([1, 2, 4]))
    E = n_ep * draw(st.integers(1, 4))
    k = draw(st.integers(1, min(E, 3)))
    T = n_ep * draw(st.integers(1, 6))
    rows = []
    for _ in range(T):
        rows.append(draw(st.permutations(list(range(E))))[:k])
    cap = draw(st.sampled_from([0, 0, 1, 2, 3]))
    return np.array(rows, dtype=np.int64).reshape(T, k), E, n_ep, cap


@settings(max_examples=150, deadline=None)
@given(routing())
def test_permute_properties(case):
    idx, E, n_ep, cap = case
    T, k = idx.shape
    A = T * k
    flat = [int(v) for v in idx.reshape(-1)]
    p = oracle.permute(idx, E, cap)
    inv, order, counts, offsets = p["inv"], p["order"], p["counts"], p["offsets"]
    R = E * cap if cap else A
    assert order.shape == (R,) and inv.shape == (A,)
    start = 0
    for e in range(E):
        mine = [a for a in range(A) if flat[a] == e]          # increasing a
        assert counts[e] == len(mine)
        seg = e * cap if cap else start
        assert offsets[e] == seg
        kept = mine[:cap] if cap else mine
        for r, a in enumerate(kept):                          # consecutive rows, stable
            assert inv[a] == seg + r and order[seg + r] == a
        for a in mine[len(kept):]:                            # dropped overflow
            assert inv[a] == -1
        if cap:
            for r in range(len(kept), cap):                   # padding rows
                assert order[seg + r] == -1
        start += len(mine)
    assert offsets[E] == (E * cap if cap else A)
    # every row holds at most one assignment and every kept assignment one row
    rows_used = [r for r in range(R) if order[r] >= 0]
    assert sorted(inv[inv >= 0].tolist()) == rows_used


@settings(max_examples=150, deadline=None)
@given(routing())
def test_ep_layout_properties(case):
    idx, E, n_ep, cap = case
    T, k = idx.shape
    A, T_loc = T * k, T // n_ep
    p = oracle.permute(idx, E, cap)
    lay = oracle.ep_layout(idx, p["inv"], E, n_ep, T)
    C, send_off, recv_off, send_idx = lay["C"], lay["send_off"], lay["recv_off"], lay["send_idx"]
    flat = [int(v) for v in idx.reshape(-1)]
    inv = p["inv"]
    rank_of = [e * n_ep // E for e in range(E)]
    for s in range(n_ep):
        lo, hi = s * T_loc * k, (s + 1) * T_loc * k
        kept = [a for a in range(lo, hi) if inv[a] >= 0]
        # the rank's slots: its kept assignments by (destination, expert, a), then -1
        want = sorted(kept, key=lambda a: (rank_of[flat[a]], flat[a], a))
        assert send_idx[lo:lo + len(want)].tolist() == want
        assert (send_idx[lo + len(want):hi] == -1).all()
        run = 0
        for q in range(n_ep):
            c = sum(1 for a in kept if rank_of[flat[a]] == q)
            assert C[s, q] == c
            assert send_off[s, q] == run
            run += c
        assert C[s].sum() == len(kept)                        # row sum: rows s sends
    for q in range(n_ep):
        received = sum(1 for a in range(A) if inv[a] >= 0 and rank_of[flat[a]] == q)
        assert C[:, q].sum() == received                      # column sum: rows q receives
        run = 0
        for s in range(n_ep):
            assert recv_off[q, s] == run
            run += C[s, q]


@st.composite
def selection_case(draw):
    """Random small routing problems on a coarse value grid (many ties, signed
    zeros), with or without groups, a selection bias and a capacity."""
    G = draw(st.sampled_from([1, 1, 2, 3, 4]))
    gs = draw(st.integers(2, 4))
    E = G * gs
    M = draw(st.integers(1, G))
    k = draw(st.integers(1, min(E, M * gs)))
    T = draw(st.integers(1, 8))
    grid = st.sampled_from([-1.0, -0.5, -0.0, 0.0, 0.25, 0.5, 1.0, 2.0])
    scores = np.array(draw(st.lists(grid, min_size=T * E, max_size=T * E)),
                      np.float32).reshape(T, E)
    bias = None
    if draw(st.booleans()):
        bias = np.array(draw(st.lists(st.sampled_from([0.0, 0.25, -0.25, 0.1]), min_size=E,
                                      max_size=E)), np.float32)
    cap = draw(st.sampled_from([0, 0, 1, 2]))
    return scores, bias, E, k, G, M, cap


@settings(max_examples=200, deadline=None)
@given(selection_case())
def test_loop_and_numpy_oracles_agree_on_routing_and_grouping(case):
    """The per-token C loop (repeated best-not-yet-taken passes, counting sort)
    and the numpy statement (lexsorts, stable argsort) pick the same experts in
    the same order and build the same grouping, bit for bit."""
    from oracle import loop
    scores, bias, E, k, G, M, cap = case
    a = loop.select_experts(scores, k, bias, G, M)
    b = oracle.select_experts(scores, k, bias, G, M)
    assert np.array_equal(a, b)
    pa, pb = loop.permute(a, E, cap), oracle.permute(b, E, cap)
    for key in ("counts", "offsets", "order", "inv", "kept"):
        assert np.array_equal(pa[key], pb[key]), key
    ga = loop.gate_weights(scores, a, "softmax", 1)
    gb = oracle.gate_weights(scores, b, "softmax", 1)
    assert np.allclose(ga, gb, rtol=1e-14, atol=0)


@st.composite
def layer_case(draw):
    """Tiny random layers: groups, sigmoid or softmax gates, normalised or not,
    a shared expert, a capacity, and token/hidden/width sizes that are not
    powers of two."""
    G = draw(st.sampled_from([1, 2]))
    E = G * draw(st.integers(2, 4))
    k = draw(st.integers(1, min(3, E)))
    score_fn = draw(st.sampled_from(["softmax", "sigmoid"]))
    cfg = dict(name="h", T=draw(st.integers(1, 9)), d=draw(st.integers(1, 12)), E=E, k=k,
               f=draw(st.integers(1, 10)), n_ep=1, score_fn=score_fn,
               norm_topk=draw(st.sampled_from([0, 1])), n_groups=G,
               topk_groups=G if k > E // G else draw(st.integers(1, G)),
               capacity=draw(st.sampled_from([0, 0, 1, 2])),
               has_shared=draw(st.sampled_from([0, 1])))
    seed = draw(st.integers(0, 2 ** 16))
    return cfg, seed


@settings(max_examples=120, deadline=None)
@given(layer_case())
def test_loop_and_numpy_oracles_agree_on_the_layer(case):
    """The layer's output token by token (per-token C loop: each token's kept
    slots from its own expert choices) equals the numpy statement (grouped
    buffer, expert-wise products, scatter-add) to 1e-12 of the largest value."""
    import synth
    from oracle import loop
    kw, seed = case
    cfg = synth.LayerConfig(**kw)
    rng = np.random.default_rng(seed)
    n_w = cfg.E + cfg.has_shared
    x = rng.standard_normal((cfg.T, cfg.d)).astype(np.float32)
    W1 = rng.standard_normal((n_w, cfg.f, cfg.d)).astype(np.float32)
    W3 = rng.standard_normal((n_w, cfg.f, cfg.d)).astype(np.float32)
    W2 = rng.standard_normal((n_w, cfg.d, cfg.f)).astype(np.float32)
    s = rng.standard_normal((cfg.T, cfg.E)).astype(np.float32)
    if cfg.score_fn == "sigmoid":
        s = (1.0 / (1.0 + np.exp(-s))).astype(np.float32)
    y, idx, g = loop.forward(x, s, cfg, W1, W3, W2)
    y_np, st_np = oracle.moe_forward(x, s, cfg, W1, W3, W2)
    assert np.array_equal(idx, st_np["idx"])
    scale = max(np.abs(y_np).max(), 1e-300)
    assert np.abs(y - y_np).max() <= 1e-12 * scale
