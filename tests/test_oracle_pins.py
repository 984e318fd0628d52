"""Pins for the oracle: values and identities that do not come from the oracle
itself (the pages' worked examples, brute force on tiny inputs, library
routines for the special cases, closed forms).  CPU only."""
import itertools
import json
import math
import os
import types

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

import oracle
from oracle import moe_ref
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


# --------------------------------------------------------------------------
# The pages' hand dispatch ("A dispatch you can check by hand")
# --------------------------------------------------------------------------

def test_hand_dispatch_permutation_and_layout():
    g = _load("hand_dispatch.json")
    idx = np.array(g["topk_idx"])
    p = oracle.permute(idx, g["E"])
    assert p["counts"].tolist() == g["counts"]
    assert p["offsets"].tolist() == g["offsets"]
    assert p["order"].tolist() == g["order"]
    assert p["inv"].tolist() == g["inv"]
    assert (p["order"] // g["k"]).tolist() == g["row_token"]
    lay = oracle.ep_layout(idx, p["inv"], g["E"], g["n_ep"], g["T"])
    assert lay["C"].tolist() == g["C"]
    assert lay["send_idx"].tolist() == g["send_idx"]
    assert lay["send_off"].tolist() == g["send_off"]
    assert lay["recv_off"].tolist() == g["recv_off"]


def test_hand_dispatch_all_tokens_choose_01():
    g = _load("hand_dispatch.json")
    idx = np.tile(np.array([[0, 1]]), (g["T"], 1))
    p = oracle.permute(idx, g["E"])
    lay = oracle.ep_layout(idx, p["inv"], g["E"], g["n_ep"], g["T"])
    assert lay["C"].tolist() == g["all01_C"]
    # GPU 0 processes all 12 rows while GPU 1 idles: eta = 6 / 12
    assert oracle.imbalance_eta(lay["C"]) == pytest.approx(0.5)


def test_random_router_row_sums():
    """The page's random-router cell: four "GPUs", every row sums to k*T_loc
    (20 there); columns are the rows each GPU receives."""
    rng = np.random.default_rng(5)
    T, E, k, n_ep = 40, 8, 2, 4
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
    p = oracle.permute(idx, E)
    lay = oracle.ep_layout(idx, p["inv"], E, n_ep, T)
    C = lay["C"]
    assert (C.sum(axis=1) == 20).all()
    per_gpu = np.array([p["counts"][q * E // n_ep:(q + 1) * E // n_ep].sum() for q in range(n_ep)])
    assert (C.sum(axis=0) == per_gpu).all()
    # inv is the inverse of order; both are bijections on [0, A)
    A = T * k
    assert sorted(p["order"].tolist()) == list(range(A))
    assert (p["inv"][p["order"]] == np.arange(A)).all()
    assert p["counts"].sum() == A
    # send_idx holds every assignment of rank s exactly once, in s's block
    T_loc = T // n_ep
    for s in range(n_ep):
        blk = lay["send_idx"][s * T_loc * k:(s + 1) * T_loc * k]
        assert sorted(blk.tolist()) == list(range(s * T_loc * k, (s + 1) * T_loc * k))
        # the q-block of s's buffer holds exactly the rows bound for q
        for q in range(n_ep):
            o, n = lay["send_off"][s, q], C[s, q]
            assert ((idx.reshape(-1)[blk[o:o + n]] * n_ep // E) == q).all()
    # receiver q's view: blocks from each s, concatenated at recv_off, then a
    # stable sort by local expert gives the global per-expert order
    for q in range(n_ep):
        recv = np.concatenate([lay["send_idx"][s * T_loc * k + lay["send_off"][s, q]:
                                               s * T_loc * k + lay["send_off"][s, q] + C[s, q]]
                               for s in range(n_ep)])
        assert all(lay["recv_off"][q, s] == C[:s, q].sum() for s in range(n_ep))
        e_of = idx.reshape(-1)[recv]
        recv_sorted = recv[np.argsort(e_of, kind="stable")]
        lo, hi = p["offsets"][q * E // n_ep], p["offsets"][(q + 1) * E // n_ep]
        assert (recv_sorted == p["order"][lo:hi]).all()


def test_capacity_hand_fixture():
    """Pad to capacity, drop overflow by token order ("Token permutation and
    grouped GEMMs"; capacity factor of "Load imbalance becomes idle time")."""
    idx = np.array([[0], [0], [1], [0], [0], [1]])
    p = oracle.permute(idx, 2, capacity=2)
    assert p["counts"].tolist() == [4, 2]
    assert p["kept"].tolist() == [2, 2]
    assert p["offsets"].tolist() == [0, 2, 4]
    assert p["order"].tolist() == [0, 1, 2, 5]
    assert p["inv"].tolist() == [0, 1, 2, -1, -1, 3]
    idx = np.array([[1], [1], [1], [1]])
    p = oracle.permute(idx, 3, capacity=3)
    assert p["order"].tolist() == [-1, -1, -1, 0, 1, 2, -1, -1, -1]
    assert p["inv"].tolist() == [3, 4, 5, -1]
    lay = oracle.ep_layout(idx, p["inv"], 3, 1, 4)
    assert lay["C"].tolist() == [[3]]
    assert lay["send_idx"].tolist() == [0, 1, 2, -1]


def test_capacity_rows_closed_form():
    assert oracle.capacity_rows(1.25, 16384, 2, 64) == 640
    assert oracle.capacity_rows(1.0, 10, 1, 3) == 4


# --------------------------------------------------------------------------
# Routing: brute force on tiny inputs
# --------------------------------------------------------------------------

def _beats(vi, i, vj, j):
    """i ranks before j: larger value, then lower index; NaN below everything;
    -0.0 == +0.0."""
    ni, nj = math.isnan(vi), math.isnan(vj)
    if ni or nj:
        return (ni and nj and i < j) or (nj and not ni)
    if vi == vj:
        return i < j
    return vi > vj


def _brute_topk(vals, cands, k):
    best = None
    for S in itertools.combinations(cands, k):
        rest = [c for c in cands if c not in S]
        if all(_beats(vals[s], s, vals[o], o) for s in S for o in rest):
            assert best is None, "top-k set must be unique"
            best = S
    ordered = sorted(best, key=lambda i: sum(_beats(vals[j], j, vals[i], i) for j in best))
    return list(ordered)


def _brute_select(v, k, n_groups, topk_groups):
    E = len(v)
    if n_groups == 1:
        return _brute_topk(v, list(range(E)), k)
    gs = E // n_groups
    gscore = []
    for g in range(n_groups):
        pair_sums = [float(np.float32(np.float32(v[i]) + np.float32(v[j])))
                     for i, j in itertools.combinations(range(g * gs, (g + 1) * gs), 2)]
        gscore.append(max(pair_sums))
    kept = _brute_topk(gscore, list(range(n_groups)), topk_groups)
    cands = [e for g in sorted(kept) for e in range(g * gs, (g + 1) * gs)]
    return _brute_topk(v, cands, k)


@pytest.mark.parametrize("E,k,G,M", [(6, 2, 1, 1), (7, 3, 1, 1), (8, 3, 4, 2), (12, 4, 3, 2), (8, 2, 2, 1)])
def test_select_matches_brute_force(E, k, G, M):
    rng = np.random.default_rng(E * 100 + k)
    for trial in range(60):
        if trial % 3 == 0:
            v = rng.integers(-3, 4, E).astype(np.float32) / 2      # many ties
            v[rng.random(E) < 0.2] = -0.0
        elif trial % 3 == 1:
            v = rng.standard_normal(E).astype(np.float32)
        else:
            v = rng.choice(np.array([-np.inf, -1.0, 0.0, 1.0, np.inf], np.float32), E)
            if G > 1:
                v = np.where(np.isinf(v), np.float32(2.0), v)    # keep group sums finite
        got = oracle.select_experts(v[None, :], k, None, G, M)[0].tolist()
        assert got == _brute_select([float(x) for x in v], k, G, M), v


def test_select_with_nan_ranks_last():
    v = np.array([[np.nan, 1.0, -np.inf, np.nan, 0.5]], np.float32)
    assert oracle.select_experts(v, 5)[0].tolist() == [1, 4, 2, 0, 3]


def test_select_ties_fixture():
    v = np.array([[1.0, 3.0, 3.0, -0.0, 0.0, 3.0]], np.float32)
    assert oracle.select_experts(v, 3)[0].tolist() == [1, 2, 5]
    assert oracle.select_experts(v, 6)[0].tolist() == [1, 2, 5, 0, 3, 4]
    v = np.array([[0.0, -0.0, 0.0, -0.0]], np.float32)
    assert oracle.select_experts(v, 4)[0].tolist() == [0, 1, 2, 3]


def test_selection_bias_moves_choice_not_gate():
    s = np.array([[0.9, 0.8, 0.1, 0.2]], np.float32)
    b = np.array([0.0, 0.0, 1.0, 0.0], np.float32)
    idx = oracle.select_experts(s, 2, b)
    assert idx[0].tolist() == [2, 0]
    g = oracle.gate_weights(s, idx, "sigmoid", 0)
    assert g[0].tolist() == [np.float32(0.1), np.float32(0.9)]


def test_group_limit_one_group_is_plain_topk():
    rng = np.random.default_rng(1)
    v = rng.standard_normal((50, 16)).astype(np.float32)
    assert (oracle.select_experts(v, 4, None, 1, 1) == oracle.select_experts(v, 4)).all()
    # keeping every group is also plain top-k
    assert (oracle.select_experts(v, 4, None, 4, 4) == oracle.select_experts(v, 4)).all()


def test_softmax_selection_equals_probability_selection():
    """Softmax is monotone, so selecting on fp32 logits picks the same experts
    as selecting on probabilities (scipy's softmax, fp64)."""
    rng = np.random.default_rng(2)
    l = rng.standard_normal((200, 8)).astype(np.float32)
    p = scipy.special.softmax(l.astype(np.float64), axis=1)
    ref = np.argsort(-p, axis=1, kind="stable")[:, :2]
    assert (oracle.select_experts(l, 2) == ref).all()


# --------------------------------------------------------------------------
# Gates
# --------------------------------------------------------------------------

def test_softmax_gates_k_equals_E_is_dense_softmax():
    rng = np.random.default_rng(3)
    l = rng.standard_normal((30, 8)).astype(np.float32)
    idx = oracle.select_experts(l, 8)
    g = oracle.gate_weights(l, idx, "softmax", 0)
    dense = scipy.special.softmax(l.astype(np.float64), axis=1)
    assert np.allclose(np.take_along_axis(dense, idx, 1), g, rtol=1e-14, atol=0)
    assert np.allclose(g.sum(1), 1.0, rtol=1e-14)
    g2 = oracle.gate_weights(l, oracle.select_experts(l, 2), "softmax", 1)
    assert np.allclose(g2.sum(1), 1.0, rtol=1e-14)


def test_sigmoid_normalised_gates_sum_to_one():
    rng = np.random.default_rng(4)
    s = rng.random((30, 16)).astype(np.float32)
    idx = oracle.select_experts(s, 4, None, 4, 2)
    g = oracle.gate_weights(s, idx, "sigmoid", 1)
    assert np.allclose(g.sum(1), 1.0, rtol=1e-14)
    assert (g > 0).all()
    assert np.allclose(oracle.sigmoid(np.array([0.0, 2.0])), scipy.special.expit([0.0, 2.0]), rtol=1e-15)


# --------------------------------------------------------------------------
# Expert compute and the whole layer
# --------------------------------------------------------------------------

def _tiny(**kw):
    base = dict(name="t", T=12, d=16, E=4, k=2, f=8, n_ep=2, score_fn="softmax", norm_topk=0)
    base.update(kw)
    return synth.LayerConfig(**base)


def _inputs(cfg, seed=0):
    x = synth.make_x(cfg, seed=seed).float().numpy()
    W1, W3, W2 = (w.float().numpy() for w in synth.make_expert_weights(cfg, seed=seed + 1))
    s = synth.make_scores(cfg, seed=seed + 2).numpy()
    return x, s, W1, W3, W2


def test_single_expert_is_a_swiglu_mlp():
    """E = 1, k = 1: the layer is one SwiGLU MLP with gate 1 (torch.nn.functional
    in fp64 as the independent reference)."""
    cfg = _tiny(E=1, k=1, n_ep=1)
    x, s, W1, W3, W2 = _inputs(cfg)
    y, _ = oracle.moe_forward(x, s, cfg, W1, W3, W2)
    xt = torch.from_numpy(x).double()
    ref = F.linear(F.silu(F.linear(xt, torch.from_numpy(W1[0]).double())) *
                   F.linear(xt, torch.from_numpy(W3[0]).double()), torch.from_numpy(W2[0]).double())
    assert np.allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_swiglu_hidden_against_torch_fp64():
    """h = silu(W1 x) * (W3 x), with torch.nn.functional's silu in fp64 as the
    independent reference, on several experts' weights."""
    cfg = _tiny(E=3, T=10, d=32, f=16)
    x, s, W1, W3, W2 = _inputs(cfg, seed=4)
    xt = torch.from_numpy(x).double()
    for e in range(cfg.E):
        ref = (F.silu(F.linear(xt, torch.from_numpy(W1[e]).double())) *
               F.linear(xt, torch.from_numpy(W3[e]).double()))
        assert np.allclose(oracle.swiglu_hidden(x, W1[e], W3[e]), ref.numpy(), rtol=1e-13,
                           atol=1e-14)


@pytest.mark.parametrize("kw", [dict(E=6, k=2), dict(E=4, k=2, capacity=4),
                                dict(E=8, k=3, score_fn="sigmoid", norm_topk=1, n_groups=4,
                                     topk_groups=2)])
def test_expert_rows_per_row_brute_force(kw):
    """Each requested row of the grouped buffer: its token and expert looked up
    row by row, h and the output recomputed with torch.nn.functional in fp64;
    capacity padding rows are zero."""
    cfg = _tiny(T=16, **kw)
    x, s, W1, W3, W2 = _inputs(cfg, seed=5)
    idx = oracle.select_experts(s, cfg.k, None, cfg.n_groups, cfg.topk_groups)
    perm = oracle.permute(idx, cfg.E, cfg.capacity)
    R = perm["order"].size
    rows = np.array(sorted(set([0, R - 1] + list(range(1, R, 3)))))
    h, out = oracle.expert_rows(x, perm, cfg.k, W1, W3, W2, rows)
    xt = torch.from_numpy(x).double()
    for n, r in enumerate(rows):
        a = perm["order"][r]
        if a < 0:
            assert not h[n].any() and not out[n].any()
            continue
        t, e = a // cfg.k, idx.reshape(-1)[a]
        hr = (F.silu(F.linear(xt[t], torch.from_numpy(W1[e]).double())) *
              F.linear(xt[t], torch.from_numpy(W3[e]).double()))
        orr = F.linear(hr, torch.from_numpy(W2[e]).double())
        assert np.allclose(h[n], hr.numpy(), rtol=1e-12, atol=1e-14)
        assert np.allclose(out[n], orr.numpy(), rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("kw", [
    dict(),
    dict(E=8, k=3, score_fn="sigmoid", norm_topk=1, n_groups=4, topk_groups=2, has_shared=1),
    dict(E=6, k=2, norm_topk=1),
])
def test_dense_mask_equals_routed_layer(kw):
    cfg = _tiny(**kw)
    x, s, W1, W3, W2 = _inputs(cfg, seed=7)
    y, _ = oracle.moe_forward(x, s, cfg, W1, W3, W2)
    yd = oracle.dense_mask_forward(x, s, cfg, W1, W3, W2)
    assert np.abs(y - yd).max() <= 1e-12 * np.abs(yd).max()


def test_token_subset_matches_full_layer():
    cfg = _tiny(E=8, k=3, score_fn="sigmoid", norm_topk=1, n_groups=4, topk_groups=2, has_shared=1)
    x, s, W1, W3, W2 = _inputs(cfg, seed=9)
    y, _ = oracle.moe_forward(x, s, cfg, W1, W3, W2)
    tok = [0, 5, 11]
    ys, _ = oracle.moe_forward(x, s, cfg, W1, W3, W2, tokens=tok)
    assert np.allclose(ys[tok], y[tok], rtol=1e-12, atol=1e-13)
    assert not np.delete(ys, tok, axis=0).any()


def test_capacity_layer_drops_overflow():
    """With capacity, a dropped assignment contributes nothing: the layer equals
    the dense-mask layer with the dropped (token, expert) gates zeroed."""
    cfg = _tiny(T=16, E=4, k=2, capacity=5)
    x, s, W1, W3, W2 = _inputs(cfg, seed=11)
    s[:, 0] += 3.0                                        # hot expert 0
    y, st = oracle.moe_forward(x, s, cfg, W1, W3, W2)
    inv = st["perm"]["inv"].reshape(cfg.T, cfg.k)
    assert (inv < 0).sum() == (st["perm"]["counts"] - 5).clip(0).sum() > 0
    ref = np.zeros_like(y)
    for t in range(cfg.T):
        for j in range(cfg.k):
            if inv[t, j] >= 0:
                e = st["idx"][t, j]
                ref[t] += st["gates"][t, j] * oracle.swiglu_expert(x[t:t + 1], W1[e], W3[e], W2[e])[0]
    assert np.abs(y - ref).max() <= 1e-12 * np.abs(ref).max()


# --------------------------------------------------------------------------
# Byte model and imbalance ("How many bytes move", "Load imbalance ...")
# --------------------------------------------------------------------------

def test_mixtral_bytes_per_token():
    """2 x top_k x hidden x bytes = 32 KB per token per layer for Mixtral
    ("05 - Expert Parallelism (MoE)", "The all-to-all pattern")."""
    assert oracle.dispatch_combine_bytes_per_token(2, 4096, 2, 2) == 32768
    rng = np.random.default_rng(6)
    T, E, k, n_ep, d = 256, 8, 2, 8, 4096
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
    p = oracle.permute(idx, E)
    C = oracle.ep_layout(idx, p["inv"], E, n_ep, T)["C"]
    assert C.sum() * d * 2 * 2 / T == 32768     # every row goes out and comes back


def test_offdiagonal_fraction_uniform_routing():
    """Balanced routing sends a fraction (n_ep - 1)/n_ep of assignments off
    rank; the all-to-all bytes are T_loc*k*d*s*(n_ep-1)/n_ep per rank."""
    rng = np.random.default_rng(8)
    T, E, k, n_ep, d = 8192, 64, 4, 8, 128
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
    p = oracle.permute(idx, E)
    C = oracle.ep_layout(idx, p["inv"], E, n_ep, T)["C"]
    disp, comb = oracle.alltoall_bytes(C, d, 1, 2)
    T_loc = T // n_ep
    expect = T_loc * k * d * (n_ep - 1) / n_ep
    assert np.allclose(disp, expect * 1, rtol=0.05)
    assert np.allclose(comb, expect * 2, rtol=0.05)
    assert disp.sum() * 2 == comb.sum()        # combine is the transpose of dispatch
    assert disp.sum() / n_ep == pytest.approx(expect, rel=0.01)


def test_imbalance_eta_examples():
    g = _load("eplb_example.json")
    for key, eta in (("plain_gpu_loads", "plain_eta"), ("greedy_gpu_loads", "greedy_eta"),
                     ("better_gpu_loads", "better_eta")):
        assert oracle.imbalance_eta(np.array([g[key]])) == pytest.approx(g[eta], abs=0.005)
    # 50 % more than the share -> two thirds
    assert oracle.imbalance_eta(np.array([[15, 5, 10, 10]])) == pytest.approx(2 / 3)


def test_skewed_workload_sends_half_to_expert_zero():
    cfg = synth.CONFIGS["skew"]
    x = synth.make_x(cfg).float().numpy()
    W_r, b = synth.make_router(cfg)
    l = oracle.router_logits(x, W_r.numpy(), b.numpy()).astype(np.float32)
    idx = oracle.select_experts(l, cfg.k)
    share = (idx == 0).sum() / idx.size
    assert 0.49 <= share <= 0.50
    counts = np.bincount(idx.reshape(-1), minlength=cfg.E)
    assert counts[0] > cfg.capacity          # the hot expert overflows its capacity


def test_router_logits_against_torch_fp64():
    cfg = _tiny(d=64, E=8)
    x = synth.make_x(cfg).float()
    W_r, _ = synth.make_router(cfg)
    l = oracle.router_logits(x.numpy(), W_r.numpy())
    assert np.allclose(l, (x.double() @ W_r.double()).numpy(), rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------
# Planted mistakes: the pins above must catch the placeholder bugs the pages
# list (non-stable sort, bincount without minlength, inclusive offsets,
# order returned as inv, node limit ignored).
# --------------------------------------------------------------------------

class _NumpyMutant(types.ModuleType):
    def __init__(self, **overrides):
        super().__init__("numpy_mutant")
        self.__dict__.update({k: getattr(np, k) for k in dir(np) if not k.startswith("__")})
        self.__dict__.update(overrides)


def _fails(fn):
    try:
        fn()
    except (AssertionError, ValueError, IndexError):
        return True
    return False


def test_planted_unstable_sort_is_caught(monkeypatch):
    def unstable_argsort(a, *args, kind=None, **kw):
        o = np.argsort(a, kind="stable", **kw)
        if np.ndim(a) == 1 and o.size > 1:      # reverse each run of equal keys
            a = np.asarray(a)
            out, i = [], 0
            while i < o.size:
                j = i
                while j < o.size and a[o[j]] == a[o[i]]:
                    j += 1
                out.extend(o[i:j][::-1])
                i = j
            o = np.array(out)
        return o
    monkeypatch.setattr(moe_ref, "np", _NumpyMutant(argsort=unstable_argsort))
    assert _fails(test_hand_dispatch_permutation_and_layout)


def test_planted_inclusive_offsets_is_caught(monkeypatch):
    real_cumsum = np.cumsum

    def shifted(a, *args, **kw):
        r = real_cumsum(a, *args, **kw)
        return r + np.asarray(a).reshape(r.shape)   # inclusive-of-next: wrong offsets
    monkeypatch.setattr(moe_ref, "np", _NumpyMutant(cumsum=shifted))
    assert _fails(test_hand_dispatch_permutation_and_layout)


def test_planted_bincount_without_minlength_is_caught(monkeypatch):
    def no_minlength(x, weights=None, minlength=0):
        return np.bincount(x, weights)
    monkeypatch.setattr(moe_ref, "np", _NumpyMutant(bincount=no_minlength))

    def unused_top_expert():
        idx = np.array([[0, 1], [1, 0]])
        p = oracle.permute(idx, 4)
        assert p["counts"].tolist() == [2, 2, 0, 0]
    assert _fails(unused_top_expert)


def test_planted_tie_break_upward_is_caught(monkeypatch):
    def flipped(values32, mask_out=None):
        v = np.asarray(values32, np.float32)
        n = v.shape[-1]
        cols = np.broadcast_to(-np.arange(n), v.shape)
        keys = [cols, -v] + ([np.asarray(mask_out, np.int8)] if mask_out is not None else [])
        return np.lexsort(keys, axis=-1)
    monkeypatch.setattr(moe_ref, "_rank_order", flipped)
    assert _fails(test_select_ties_fixture)


def test_planted_node_limit_ignored_is_caught(monkeypatch):
    real = moe_ref.select_experts

    def ignores_groups(scores, k, bias=None, n_groups=1, topk_groups=1):
        return real(scores, k, bias)
    monkeypatch.setattr(oracle, "select_experts", ignores_groups)
    assert _fails(lambda: test_select_matches_brute_force(8, 3, 4, 2))


def test_planted_group_score_top1_only_is_caught(monkeypatch):
    real_sort = np.sort

    def sort_zero_second(a, axis=-1, **kw):
        r = real_sort(a, axis=axis, **kw)
        if np.ndim(r) == 3:
            r = r.copy()
            r[..., 1] = 0                       # group score becomes top1 only
        return r
    monkeypatch.setattr(moe_ref, "np", _NumpyMutant(sort=sort_zero_second))
    assert _fails(lambda: test_select_matches_brute_force(12, 4, 3, 2))


def test_planted_wrong_expert_in_expert_rows_is_caught(monkeypatch):
    """expert_rows taking the next expert's weights for a segment fails its
    row-by-row brute force."""
    real = moe_ref.swiglu_hidden
    calls = {"n": 0}

    def shifted(X, W1, W3):
        calls["n"] += 1
        return real(X, W3, W1) if calls["n"] % 2 == 0 else real(X, W1, W3)
    monkeypatch.setattr(moe_ref, "swiglu_hidden", shifted)
    assert _fails(lambda: test_expert_rows_per_row_brute_force(dict(E=6, k=2)))


def test_dsv3_worked_example_bytes_and_flops():
    """The pages' worked example at DeepSeek-V3's shape ("Expert parallelism",
    "A worked example at DeepSeek-V3's shape"): 693 MB cross the network per
    GPU per layer (FP8 dispatch plus BF16 combine), and the experts' compute is
    2.9e12 FLOPs.  The bytes are counted from the oracle's layout of a
    uniformly routed batch of n_ep * T_loc tokens; the FLOPs from the benchmark's
    model of 6*d*d_e per assignment."""
    import importlib.util
    g = _load("dsv3_worked_example.json")
    d, k, T_loc, n_ep = g["d"], g["k"], g["T_loc"], g["n_ep"]
    E = 256
    T = T_loc * n_ep
    rng = np.random.default_rng(12)
    # balanced routing: each token's k distinct experts uniformly at random
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :k]
    p = oracle.permute(idx, E)
    C = oracle.ep_layout(idx, p["inv"], E, n_ep, T)["C"]
    disp, comb = oracle.alltoall_bytes(C, d, g["s_dispatch"], g["s_combine"])
    per_gpu = (disp + comb).mean()
    closed = T_loc * k * d * (g["s_dispatch"] + g["s_combine"]) * (n_ep - 1) / n_ep
    assert closed / 1e6 == pytest.approx(g["bytes_mb"], abs=0.7)
    assert per_gpu == pytest.approx(closed, rel=2e-3)
    assert closed / (g["ib_gbs"] * 1e9) * 1e3 == pytest.approx(g["ib_ms"], abs=0.05)
    assert closed / (g["nvlink_gbs"] * 1e9) * 1e3 == pytest.approx(g["nvlink_ms"], abs=0.05)
    spec = importlib.util.spec_from_file_location(
        "bench_mod", os.path.join(os.path.dirname(GOLDEN), "..", "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    cfg = synth.LayerConfig("worked", T=T_loc, d=d, E=E, k=k, f=g["d_e"], n_ep=1,
                            score_fn="sigmoid", norm_topk=1)
    counts = np.full(E, T_loc * k // E)
    flops = b._algorithmic(cfg, counts)["ffn_flops"]
    assert flops == 4096 * 8 * 6 * 7168 * 2048
    assert flops == pytest.approx(g["flops"], rel=0.01)
    assert flops / (g["peak_tflops"] * 1e12) * 1e3 == pytest.approx(g["compute_ms"], abs=0.05)


def test_decode_batch_tokens_per_expert():
    """"flops/sched-expert-parallelism", notes: with 256 experts and top-8 the
    batch per expert is B*8/256 = B/32, so B = 128 gives each expert 4 tokens on
    average.  The decode workload is that batch; the oracle's counts of a routed
    decode batch average exactly 4 per expert (every token keeps k distinct
    experts, dropless)."""
    cfg = synth.CONFIGS["dsv3_decode"]
    assert (cfg.T, cfg.E, cfg.k) == (128, 256, 8) and cfg.T * cfg.k / cfg.E == 4
    s = synth.make_scores(cfg).numpy()
    idx = oracle.select_experts(s, cfg.k, None, cfg.n_groups, cfg.topk_groups)
    counts = oracle.permute(idx, cfg.E)["counts"]
    assert counts.sum() == 128 * 8 and counts.mean() == 4.0
    assert all(len(set(row)) == cfg.k for row in idx.tolist())
