"""Pins for the oracle's backward of the layer (routing held fixed): central
finite differences in fp64 on a tiny layer, and PyTorch autograd (a library
routine) through a dense-mask form of the forward on a small one.  CPU only."""
import numpy as np
import pytest
import torch

import oracle
import synth


def _tiny(**kw):
    base = dict(T=12, d=8, E=4, k=2, f=6, n_ep=2)
    base.update(kw)
    return synth.CONFIGS["tiny"].with_(**base)


def _rand(cfg, seed):
    rng = np.random.default_rng(seed)
    n = cfg.E + cfg.has_shared
    x = rng.normal(size=(cfg.T, cfg.d))
    W1 = rng.normal(size=(n, cfg.f, cfg.d)) / np.sqrt(cfg.d)
    W3 = rng.normal(size=(n, cfg.f, cfg.d)) / np.sqrt(cfg.d)
    W2 = rng.normal(size=(n, cfg.d, cfg.f)) / np.sqrt(cfg.f)
    dy = rng.normal(size=(cfg.T, cfg.d))
    scores = rng.normal(size=(cfg.T, cfg.E)).astype(np.float32)
    if cfg.score_fn == "sigmoid":
        scores = (1 / (1 + np.exp(-scores))).astype(np.float32)
    return x, W1, W3, W2, dy, scores


def _loss(cfg, x, scores, W1, W3, W2, dy, gates=None):
    """<dy, y> with the routing of `scores`; optional gate override."""
    if gates is None:
        y, _ = oracle.moe_forward(x, scores, cfg, W1, W3, W2)
        return float((dy * y).sum())
    idx = oracle.select_experts(scores, cfg.k, None, cfg.n_groups, cfg.topk_groups)
    perm = oracle.permute(idx, cfg.E, cfg.capacity)
    out = oracle.expert_outputs(x, perm, cfg.k, W1, W3, W2)
    shared = None
    if cfg.has_shared:
        shared = oracle.swiglu_expert(x, W1[cfg.E], W3[cfg.E], W2[cfg.E])
    y = oracle.combine(out, perm, cfg.k, gates, cfg.T, shared)
    return float((dy * y).sum())


@pytest.mark.parametrize("kw", [dict(), dict(has_shared=1, score_fn="sigmoid", norm_topk=1),
                                dict(capacity=4)])
def test_backward_against_finite_differences(kw):
    cfg = _tiny(**kw)
    x, W1, W3, W2, dy, scores = _rand(cfg, 0)
    g = oracle.moe_backward(x, scores, cfg, W1, W3, W2, dy)
    eps = 1e-6
    rng = np.random.default_rng(1)

    def fd(arr, setter):
        out = []
        for _ in range(6):
            i = tuple(int(rng.integers(0, s)) for s in arr.shape)
            p, m = arr.copy(), arr.copy()
            p[i] += eps
            m[i] -= eps
            out.append((i, (setter(p) - setter(m)) / (2 * eps)))
        return out

    for i, val in fd(x, lambda a: _loss(cfg, a, scores, W1, W3, W2, dy)):
        assert g["dx"][i] == pytest.approx(val, rel=1e-6, abs=1e-8)
    for name, W in (("dW1", W1), ("dW3", W3), ("dW2", W2)):
        def setter(a, name=name):
            ws = {"dW1": W1, "dW3": W3, "dW2": W2}
            ws = {kk: (a if kk == name else vv) for kk, vv in ws.items()}
            return _loss(cfg, x, scores, ws["dW1"], ws["dW3"], ws["dW2"], dy)
        for i, val in fd(W, setter):
            assert g[name][i] == pytest.approx(val, rel=1e-6, abs=1e-8)
    gates = g["gates"]
    for i, val in fd(gates, lambda a: _loss(cfg, x, scores, W1, W3, W2, dy, gates=a)):
        assert g["dgate"][i] == pytest.approx(val, rel=1e-6, abs=1e-8)


def test_backward_against_autograd_dense_mask():
    cfg = _tiny(T=64, d=16, E=8, k=3, f=12, n_ep=4, has_shared=1)
    x, W1, W3, W2, dy, scores = _rand(cfg, 2)
    g = oracle.moe_backward(x, scores, cfg, W1, W3, W2, dy)
    # dense-mask forward in torch fp64: every expert on every token, masked by
    # the (fixed) routing, gates as leaves
    T, E = cfg.T, cfg.E
    mask = np.zeros((T, E))
    gate_dense = np.zeros((T, E))
    for t in range(T):
        for j in range(cfg.k):
            mask[t, g["idx"][t, j]] = 1
    xt = torch.tensor(x, requires_grad=True)
    W1t, W3t, W2t = (torch.tensor(w, requires_grad=True) for w in (W1, W3, W2))
    gt = torch.tensor(g["gates"], requires_grad=True)
    sel = torch.zeros(T, cfg.k, E, dtype=torch.float64)
    for t in range(T):
        for j in range(cfg.k):
            sel[t, j, g["idx"][t, j]] = 1
    gd = torch.einsum("tj,tje->te", gt, sel)
    y = torch.zeros(T, cfg.d, dtype=torch.float64)
    for e in range(E + 1):
        u = xt @ W1t[e].T
        v = xt @ W3t[e].T
        o = (torch.nn.functional.silu(u) * v) @ W2t[e].T
        y = y + (gd[:, e:e + 1] * o if e < E else o)
    (torch.tensor(dy) * y).sum().backward()
    assert np.allclose(g["dx"], xt.grad.numpy(), rtol=1e-10, atol=1e-12)
    assert np.allclose(g["dW1"], W1t.grad.numpy(), rtol=1e-10, atol=1e-12)
    assert np.allclose(g["dW3"], W3t.grad.numpy(), rtol=1e-10, atol=1e-12)
    assert np.allclose(g["dW2"], W2t.grad.numpy(), rtol=1e-10, atol=1e-12)
    assert np.allclose(g["dgate"], gt.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_planted_swiglu_derivative_mistake_is_caught(monkeypatch):
    """silu'(u) replaced by sigmoid(u) (a common slip) must fail the autograd pin."""
    real = oracle.moe_ref.swiglu_expert_backward

    def wrong(X, W1, W3, W2, dO):
        X = np.asarray(X, np.float64)
        u = X @ np.asarray(W1).T
        v = X @ np.asarray(W3).T
        s = 1 / (1 + np.exp(-u))
        h = u * s * v
        dh = np.asarray(dO) @ np.asarray(W2)
        du = dh * v * s                    # missing (1 + u (1 - s))
        dv = dh * u * s
        return du @ W1 + dv @ W3, du.T @ X, dv.T @ X, np.asarray(dO).T @ h
    monkeypatch.setattr(oracle.moe_ref, "swiglu_expert_backward", wrong)
    with pytest.raises(AssertionError):
        test_backward_against_autograd_dense_mask()
    monkeypatch.setattr(oracle.moe_ref, "swiglu_expert_backward", real)
