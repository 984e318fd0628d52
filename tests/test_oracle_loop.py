"""Pins for the per-token loop oracle (oracle/moe_loop.c): the pages' hand
dispatch, brute force on tiny inputs, closed forms and library routines for the
special cases, and agreement with the vectorised numpy oracle, which is pinned
on its own (tests/test_oracle_pins.py).  The two oracles state the layer two
ways (token by token with counting sorts; expert by expert with argsorts and
matrix products), so a slip in either shows up as a disagreement.  CPU only."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

import oracle
import synth
from oracle import loop

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


def _cfg(**kw):
    base = dict(name="t", T=12, d=16, E=4, k=2, f=8, n_ep=2, score_fn="softmax", norm_topk=0)
    base.update(kw)
    return synth.LayerConfig(**base)


def _inputs(cfg, seed=0):
    x = synth.make_x(cfg, seed=seed).float().numpy()
    W1, W3, W2 = (w.float().numpy() for w in synth.make_expert_weights(cfg, seed=seed + 1))
    s = synth.make_scores(cfg, seed=seed + 2).numpy()
    return x, s, W1, W3, W2


def test_library_builds_and_exports():
    h = loop.lib()
    for name in ("loop_router_logits", "loop_select", "loop_gates", "loop_permute",
                 "loop_ep_layout", "loop_layer_tokens"):
        assert hasattr(h, name)


# --------------------------------------------------------------------------
# The pages' hand dispatch ("Expert parallelism", "A dispatch you can check by hand")
# --------------------------------------------------------------------------

def test_hand_dispatch():
    g = _golden("hand_dispatch.json")
    idx = np.array(g["topk_idx"])
    p = loop.permute(idx, g["E"])
    assert p["counts"].tolist() == g["counts"]
    assert p["offsets"].tolist() == g["offsets"]
    assert p["order"].tolist() == g["order"]
    assert p["inv"].tolist() == g["inv"]
    assert (p["order"] // g["k"]).tolist() == g["row_token"]
    lay = loop.ep_layout(idx, p["inv"], g["E"], g["n_ep"])
    assert lay["C"].tolist() == g["C"]
    assert lay["send_idx"].tolist() == g["send_idx"]
    assert lay["send_off"].tolist() == g["send_off"]
    assert lay["recv_off"].tolist() == g["recv_off"]
    idx01 = np.tile(np.array([[0, 1]]), (g["T"], 1))
    p01 = loop.permute(idx01, g["E"])
    assert loop.ep_layout(idx01, p01["inv"], g["E"], g["n_ep"])["C"].tolist() == g["all01_C"]


def test_capacity_hand_fixture():
    """Pad to capacity and drop overflow by token order ("Token permutation and
    grouped GEMMs"; the capacity cap of "Load imbalance becomes idle time")."""
    idx = np.array([[0], [0], [1], [0], [0], [1]])
    p = loop.permute(idx, 2, capacity=2)
    assert p["counts"].tolist() == [4, 2]
    assert p["kept"].tolist() == [2, 2]
    assert p["offsets"].tolist() == [0, 2, 4]
    assert p["order"].tolist() == [0, 1, 2, 5]
    assert p["inv"].tolist() == [0, 1, 2, -1, -1, 3]
    idx = np.array([[1], [1], [1], [1]])
    p = loop.permute(idx, 3, capacity=3)
    assert p["order"].tolist() == [-1, -1, -1, 0, 1, 2, -1, -1, -1]
    assert p["inv"].tolist() == [3, 4, 5, -1]
    lay = loop.ep_layout(idx, p["inv"], 3, 1)
    assert lay["C"].tolist() == [[3]]
    assert lay["send_idx"].tolist() == [0, 1, 2, -1]


def test_rejects_expert_ids_out_of_range():
    with pytest.raises(ValueError):
        loop.permute(np.array([[0, 4]]), 4)
    with pytest.raises(ValueError):
        loop.permute(np.array([[-1, 0]]), 4)


# --------------------------------------------------------------------------
# Routing: brute force on tiny inputs, then agreement with the numpy oracle
# --------------------------------------------------------------------------

def _before(vi, i, vj, j):
    """i ranks before j: larger value first, lower index on equal values
    (-0.0 equal to +0.0), NaN after every number."""
    ni, nj = math.isnan(vi), math.isnan(vj)
    if ni or nj:
        return (ni and nj and i < j) or (nj and not ni)
    return vi > vj or (vi == vj and i < j)


def _best_subset(vals, cands, n):
    """The unique n-subset of cands that ranks entirely before the rest, in
    rank order (exhaustive)."""
    found = [S for S in itertools.combinations(cands, n)
             if all(_before(vals[s], s, vals[o], o) for s in S for o in cands if o not in S)]
    assert len(found) == 1
    return sorted(found[0], key=lambda i: sum(_before(vals[j], j, vals[i], i) for j in found[0]))


def _brute(v, k, G, M):
    E = len(v)
    if G == 1:
        return _best_subset(v, list(range(E)), k)
    gs = E // G
    gscore = []
    for g in range(G):
        top = _best_subset(v, list(range(g * gs, (g + 1) * gs)), 2)
        gscore.append(float(np.float32(v[top[0]]) + np.float32(v[top[1]])))
    kept = _best_subset(gscore, list(range(G)), M)
    cands = [e for g in sorted(kept) for e in range(g * gs, (g + 1) * gs)]
    return _best_subset(v, cands, k)


@pytest.mark.parametrize("E,k,G,M", [(6, 2, 1, 1), (7, 3, 1, 1), (8, 3, 4, 2), (12, 4, 3, 2),
                                     (8, 2, 2, 1), (9, 9, 3, 3)])
def test_select_matches_brute_force(E, k, G, M):
    rng = np.random.default_rng(1000 + E * 10 + k)
    rows = []
    for trial in range(60):
        if trial % 3 == 0:
            v = rng.integers(-3, 4, E).astype(np.float32) / 2
            v[rng.random(E) < 0.2] = -0.0
        elif trial % 3 == 1:
            v = rng.standard_normal(E).astype(np.float32)
        else:
            v = rng.choice(np.array([-np.inf, -1.0, 0.0, 1.0, np.inf], np.float32), E)
            if G > 1:
                v = np.where(np.isinf(v), np.float32(2.0), v)
        rows.append(v)
    V = np.stack(rows)
    got = loop.select_experts(V, k, None, G, M)
    for t, v in enumerate(rows):
        assert got[t].tolist() == _brute([float(a) for a in v], k, G, M), v


def test_select_special_values():
    v = np.array([[np.nan, 1.0, -np.inf, np.nan, 0.5]], np.float32)
    assert loop.select_experts(v, 5)[0].tolist() == [1, 4, 2, 0, 3]
    v = np.array([[1.0, 3.0, 3.0, -0.0, 0.0, 3.0]], np.float32)
    assert loop.select_experts(v, 6)[0].tolist() == [1, 2, 5, 0, 3, 4]


def test_selection_bias_is_one_fp32_addition():
    """0.1f + 0.2f rounds to exactly 0.3f in fp32, while the exact sum lies
    below 0.3f.  Expert 0 (score 0.1f, bias 0.2f) against expert 1 (score 0.3f,
    no bias): one fp32 addition makes a tie, which the lower index wins; a sum
    kept in higher precision would rank expert 1 first."""
    s = np.array([[np.float32(0.1), np.float32(0.3)]], np.float32)
    b = np.array([np.float32(0.2), 0.0], np.float32)
    assert np.float32(np.float32(0.1) + np.float32(0.2)) == np.float32(0.3)
    assert float(np.float32(0.1)) + float(np.float32(0.2)) < float(np.float32(0.3))
    assert loop.select_experts(s, 2, b)[0].tolist() == [0, 1]
    assert oracle.select_experts(s, 2, b)[0].tolist() == [0, 1]


@pytest.mark.parametrize("name", ["tiny", "dsv3_decode", "skew"])
@pytest.mark.parametrize("ties", [False, True])
def test_select_agrees_with_numpy_oracle(name, ties):
    cfg = synth.CONFIGS[name]
    s = synth.make_scores(cfg, seed=5, ties=ties).numpy()
    bias = synth.make_selection_bias(cfg).numpy() if name != "skew" else None
    got = loop.select_experts(s, cfg.k, bias, cfg.n_groups, cfg.topk_groups)
    ref = oracle.select_experts(s, cfg.k, bias, cfg.n_groups, cfg.topk_groups)
    assert np.array_equal(got, ref)


# --------------------------------------------------------------------------
# Gates and logits: closed forms and library routines
# --------------------------------------------------------------------------

def test_softmax_gates_with_k_equal_E_are_the_dense_softmax():
    rng = np.random.default_rng(3)
    s = rng.standard_normal((5, 6)).astype(np.float32)
    idx = np.tile(np.arange(6), (5, 1))
    g = loop.gate_weights(s, idx, "softmax", 0)
    assert np.allclose(g, scipy.special.softmax(s.astype(np.float64), axis=1), rtol=1e-14, atol=0)


def test_sigmoid_gates():
    rng = np.random.default_rng(4)
    s = rng.random((7, 16)).astype(np.float32)
    idx = loop.select_experts(s, 4)
    raw = loop.gate_weights(s, idx, "sigmoid", 0)
    assert np.array_equal(raw, np.take_along_axis(s, idx, 1).astype(np.float64))
    norm = loop.gate_weights(s, idx, "sigmoid", 1)
    assert np.allclose(norm.sum(1), 1.0, rtol=0, atol=1e-15)
    assert np.allclose(norm, raw / raw.sum(1, keepdims=True), rtol=1e-15, atol=0)


def test_router_logits_against_fp64_matmul():
    cfg = _cfg(T=9, d=40, E=6)
    x = synth.make_x(cfg).float().numpy()
    W_r, _ = synth.make_router(cfg)
    lb = np.linspace(-1, 1, cfg.E).astype(np.float32)
    got = loop.router_logits(x, W_r.numpy(), lb)
    ref = (torch.from_numpy(x).double() @ W_r.double()).numpy() + lb.astype(np.float64)
    assert np.allclose(got, ref, rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------
# Permutation and layout against the numpy oracle (dropless and capacity)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name,capacity", [("tiny", 0), ("tiny", 200), ("dsv3_decode", 0),
                                           ("skew", 0), ("skew", 640)])
def test_permute_and_layout_agree_with_numpy_oracle(name, capacity):
    cfg = synth.CONFIGS[name]
    s = synth.make_scores(cfg, seed=8).numpy()
    idx = oracle.select_experts(s, cfg.k, None, cfg.n_groups, cfg.topk_groups)
    ref = oracle.permute(idx, cfg.E, capacity)
    got = loop.permute(idx, cfg.E, capacity)
    for key in ("counts", "offsets", "order", "inv", "kept"):
        assert np.array_equal(got[key], ref[key]), key
    lref = oracle.ep_layout(idx, ref["inv"], cfg.E, cfg.n_ep, cfg.T)
    lgot = loop.ep_layout(idx, got["inv"], cfg.E, cfg.n_ep)
    for key in ("C", "send_off", "recv_off", "send_idx"):
        assert np.array_equal(lgot[key], lref[key]), key
    kept = int(got["kept"].sum())
    assert int(lgot["C"].sum()) == kept
    if not capacity:
        assert lgot["C"].sum(1).tolist() == [cfg.T_loc * cfg.k] * cfg.n_ep


# --------------------------------------------------------------------------
# The layer, token by token
# --------------------------------------------------------------------------

def test_single_expert_is_a_swiglu_mlp():
    """E = 1, k = 1: one SwiGLU MLP with gate 1 (torch.nn.functional in fp64)."""
    cfg = _cfg(E=1, k=1, n_ep=1)
    x, s, W1, W3, W2 = _inputs(cfg)
    y, idx, g = loop.forward(x, s, cfg, W1, W3, W2)
    assert idx.tolist() == [[0]] * cfg.T and np.all(g == 1.0)
    xt = torch.from_numpy(x).double()
    ref = F.linear(F.silu(F.linear(xt, torch.from_numpy(W1[0]).double())) *
                   F.linear(xt, torch.from_numpy(W3[0]).double()), torch.from_numpy(W2[0]).double())
    assert np.allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_hidden_activations_against_torch_fp64():
    cfg = _cfg(E=3, k=2, f=24, has_shared=1)
    x, s, W1, W3, W2 = _inputs(cfg, seed=6)
    idx = loop.select_experts(s, cfg.k)
    g = loop.gate_weights(s, idx, "softmax", 0)
    tokens = np.array([0, 5, 11])
    _, h = loop.layer_tokens(x, idx, g, cfg, W1, W3, W2, tokens, with_h=True)
    for n, t in enumerate(tokens):
        xt = torch.from_numpy(x[t]).double()
        for j, e in enumerate(list(idx[t]) + [cfg.E]):
            ref = F.silu(torch.from_numpy(W1[e]).double() @ xt) * (torch.from_numpy(W3[e]).double() @ xt)
            assert np.allclose(h[n, j], ref.numpy(), rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("kw", [
    dict(), dict(E=6, k=3, norm_topk=1), dict(E=8, k=2, n_groups=4, topk_groups=2,
                                              score_fn="sigmoid", norm_topk=1, has_shared=1),
    dict(E=4, k=2, capacity=4), dict(E=5, k=1, T=10, n_ep=1, capacity=1),
])
def test_layer_agrees_with_numpy_oracle_and_dense_mask(kw):
    cfg = _cfg(**kw)
    x, s, W1, W3, W2 = _inputs(cfg, seed=2)
    y, idx, g = loop.forward(x, s, cfg, W1, W3, W2)
    y_np, st = oracle.moe_forward(x, s, cfg, W1, W3, W2)
    assert np.array_equal(idx, st["idx"])
    assert np.allclose(g, st["gates"], rtol=1e-15, atol=0)
    scale = np.abs(y_np).max()
    assert np.abs(y - y_np).max() <= 1e-12 * scale
    if not cfg.capacity:
        y_dense = oracle.dense_mask_forward(x, s, cfg, W1, W3, W2)
        assert np.abs(y - y_dense).max() <= 1e-12 * scale


def _expert_fp64(W1, W3, W2, e, xt):
    xt = torch.from_numpy(xt).double()
    h = F.silu(torch.from_numpy(W1[e]).double() @ xt) * (torch.from_numpy(W3[e]).double() @ xt)
    return (torch.from_numpy(W2[e]).double() @ h).numpy()


def test_capacity_drops_by_token_order():
    """Capacity 2 on three experts: each expert keeps the first two assignments
    that chose it in increasing a and drops the rest ("Token permutation and
    grouped GEMMs": drop overflow by token order); a token's output sums only
    its kept slots (expected values from torch.nn.functional in fp64)."""
    cfg = _cfg(T=6, E=3, k=2, n_ep=1, capacity=2)
    x, _, W1, W3, W2 = _inputs(cfg, seed=9)
    idx = np.array([[0, 1], [0, 2], [0, 1], [1, 0], [2, 1], [0, 2]], np.int32)
    # a -> expert: 0 1 0 2 0 1 1 0 2 1 0 2; kept: a = 0, 2 (e0), 1, 5 (e1), 3, 8 (e2)
    kept = {0, 1, 2, 3, 5, 8}
    g = np.full((cfg.T, cfg.k), 0.5)
    y = loop.layer_tokens(x, idx, g, cfg, W1, W3, W2, np.arange(cfg.T))
    for t in range(cfg.T):
        ref = np.zeros(cfg.d)
        for j in range(cfg.k):
            if t * cfg.k + j in kept:
                ref += 0.5 * _expert_fp64(W1, W3, W2, idx[t, j], x[t])
        assert np.allclose(y[t], ref, rtol=1e-13, atol=1e-15), t
    assert not np.any(y[3]) and not np.any(y[5])
    p = loop.permute(idx, cfg.E, cfg.capacity)
    assert p["inv"].tolist() == [0, 2, 1, 4, -1, 3, -1, -1, 5, -1, -1, -1]
    assert p["order"].tolist() == [0, 2, 1, 5, 3, 8]


# --------------------------------------------------------------------------
# Planted mistakes: a mutated copy of the C source, built here, must fail the
# pins above (the mutation lives only in a temporary copy).  Every mutation
# keeps its memory accesses inside the buffers it is given, since the mutant
# runs inside this test process.
# --------------------------------------------------------------------------

def _planted(tmp_path, old, new):
    import shutil
    import subprocess
    src = open(loop.SRC).read()
    assert src.count(old) == 1, old
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    so = str(tmp_path / "libmutant.so")
    cc = shutil.which("gcc") or shutil.which("cc")
    res = subprocess.run([cc, *loop.CFLAGS, "-o", so, str(path), "-lm"], capture_output=True,
                         text=True)
    assert res.returncode == 0, res.stderr
    return loop.load(so)


def _caught(monkeypatch, mutant, *pins):
    monkeypatch.setattr(loop, "_lib", mutant)
    for pin in pins:
        try:
            pin()
        except AssertionError:
            return True
    return False


PLANTS = {
    "tie break toward the higher index": (
        "  if (va < vb) return 0;\n  return ia < ib;", "  if (va < vb) return 0;\n  return ia > ib;",
        lambda: test_select_matches_brute_force(6, 2, 1, 1)),
    "group score from the best value only": (
        "v[b1] + v[b2];", "v[b1] + v[b1];",
        lambda: test_select_matches_brute_force(8, 3, 4, 2)),
    "group limit ignored": (
        "if (eligible[e] != eligible[best]) {", "if (0) {",
        lambda: test_select_matches_brute_force(12, 4, 3, 2)),
    "rows handed out in decreasing a (an unstable grouping)": (
        "  for (long a = 0; a < A; ++a) {\n    const int e = idx[a];\n    const int rank = fill[e]++;",
        "  for (long a = A - 1; a >= 0; --a) {\n    const int e = idx[a];\n    const int rank = fill[e]++;",
        test_hand_dispatch),
    "capacity keeps one row too many": (
        "keep[a] = !capacity || seen[e] < capacity;", "keep[a] = !capacity || seen[e] <= capacity;",
        test_capacity_drops_by_token_order),
    "rank destination by expert modulo ranks": (
        "if ((long)e * n_ep / E != q) continue;", "if (e % n_ep != q) continue;",
        test_hand_dispatch),
    "silu with the wrong sign": (
        "h[i] = u / (1.0 + exp(-u)) * v;", "h[i] = u / (1.0 + exp(u)) * v;",
        test_single_expert_is_a_swiglu_mlp),
    "down product reading W2 transposed": (
        "const float* w2 = W2 + (size_t)c * f;\n    for (int i = 0; i < f; ++i) o += (double)w2[i] * h[i];",
        "for (int i = 0; i < f; ++i) o += (double)W2[(size_t)i * d + c] * h[i];",
        test_single_expert_is_a_swiglu_mlp),
    "softmax without the shift's partner in the sum": (
        "for (int e = 0; e < E; ++e) z += exp((double)s[e] - m);",
        "for (int e = 0; e < E; ++e) z += exp((double)s[e]);",
        test_softmax_gates_with_k_equal_E_are_the_dense_softmax),
    "shared expert dropped": (
        "const int slots = k + (has_shared ? 1 : 0);", "const int slots = k;",
        lambda: test_layer_agrees_with_numpy_oracle_and_dense_mask(
            dict(E=8, k=2, n_groups=4, topk_groups=2, score_fn="sigmoid", norm_topk=1,
                 has_shared=1))),
}


@pytest.mark.parametrize("name", list(PLANTS))
def test_planted_mistake_is_caught(name, tmp_path, monkeypatch):
    old, new, pin = PLANTS[name]
    assert _caught(monkeypatch, _planted(tmp_path, old, new), pin), name
