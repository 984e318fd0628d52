"""Parity of the layer's backward (routing held fixed) with the oracle's fp64
closed form: dx, dW1, dW3, dW2 and the gate gradients, each within
max|g - g_ref| <= 2e-2 max|g_ref| (bf16 operands, fp32 accumulation); the
weight gradients of an expert with no rows are exactly zero."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu_util import npf

pytestmark = pytest.mark.gpu

C = synth.CONFIGS
TOL = 2e-2
SMALL = {
    "tiny": C["tiny"],
    "tiny_ragged": C["tiny"].with_(name="tiny_ragged", T=1000, n_ep=8),
    "ds_small": C["dsv3"].with_(name="ds_small", T=512, d=256, f=256, E=64, n_ep=16),
    "decode_small": C["dsv3"].with_(name="decode_small", T=32, d=512, f=256, n_ep=16),
    "skew_small": C["skew"].with_(name="skew_small", T=2048, d=256, f=256, E=16, n_ep=8,
                                  capacity=oracle.capacity_rows(1.25, 2048, 2, 16)),
    "single_expert": C["tiny"].with_(name="single_expert", T=300, E=1, k=1, n_ep=1, d=128, f=128),
    "k_equals_E": C["tiny"].with_(name="k_equals_E", T=256, E=32, k=32, n_ep=2, d=128, f=128),
    "norm_softmax": C["tiny"].with_(name="norm_softmax", E=12, k=3, n_ep=4, norm_topk=1),
}


@pytest.fixture(scope="module")
def m():
    import expert_token_dispatch_moe_b300 as mod
    return mod


def _close(got, ref, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref).max()
    scale = np.abs(ref).max()
    assert err <= TOL * scale + 1e-30, f"{what}: max err {err:.3g} > {TOL} * {scale:.3g}"


def _dy(cfg, device="cpu"):
    g = torch.Generator(device=device).manual_seed(77)
    return torch.randn(cfg.T, cfg.d, generator=g, device=device).to(torch.bfloat16)


def _run(m, cfg, x, scores, W1, W3, W2, dy):
    layer = m.MoELayer(cfg, W1, W3, W2)
    layer.forward(x, scores=scores)
    layer.backward(x, dy)
    torch.cuda.synchronize()
    assert m.moe_get_device_status(layer.ws) == 0
    return layer


@pytest.mark.parametrize("name", list(SMALL))
def test_backward_parity_small(m, name):
    cfg = SMALL[name]
    x = synth.make_x(cfg)
    scores = synth.make_scores(cfg)
    if name == "skew_small":
        scores[:, 0] += 4.5
    W1, W3, W2 = synth.make_expert_weights(cfg)
    dy = _dy(cfg)
    layer = _run(m, cfg, x.cuda(), scores.cuda(), W1.cuda(), W3.cuda(), W2.cuda(), dy.cuda())
    g = oracle.moe_backward(x.float().numpy(), scores.numpy(), cfg, W1.float().numpy(),
                            W3.float().numpy(), W2.float().numpy(), dy.float().numpy())
    _close(npf(layer.dx), g["dx"], "dx")
    dW1, dW3 = layer.unpacked_dW13()
    _close(npf(dW1), g["dW1"], "dW1")
    _close(npf(dW3), g["dW3"], "dW3")
    _close(npf(layer.dW2), g["dW2"], "dW2")
    _close(layer.dgate.cpu().numpy(), g["dgate"], "dgate")
    kept = g["perm"]["kept"]
    for e in np.nonzero(kept == 0)[0]:
        assert (dW1[e] == 0).all() and (dW3[e] == 0).all() and (layer.dW2[e] == 0).all()
    assert layer.launches_per_backward >= 10


@pytest.mark.parametrize("name", ["mixtral", "dsv3"])
def test_backward_full_size_sampled(m, name):
    """Full-size layers: the gate gradients and dx of 24 sampled
    tokens, and the weight gradients of one routed expert, each against the
    oracle's closed form on exactly those rows."""
    cfg = C[name]
    x = synth.make_x(cfg, device="cuda")
    scores = synth.make_scores(cfg)
    W1, W3, W2 = synth.make_expert_weights(cfg, device="cuda")
    dy = _dy(cfg, "cuda")
    layer = _run(m, cfg, x, scores.cuda(), W1, W3, W2, dy)
    idx = oracle.select_experts(scores.numpy(), cfg.k, None, cfg.n_groups, cfg.topk_groups)
    gates = oracle.gate_weights(scores.numpy(), idx, cfg.score_fn, cfg.norm_topk)
    perm = oracle.permute(idx, cfg.E, cfg.capacity)
    xf = x.float().cpu().numpy()
    dyf = dy.float().cpu().numpy()
    experts = {}

    def ex(e):
        if e not in experts:
            experts[e] = (W1[e].float().cpu().numpy(), W3[e].float().cpu().numpy(),
                          W2[e].float().cpu().numpy())
        return experts[e]

    rng = np.random.default_rng(3)
    toks = rng.choice(cfg.T, size=24, replace=False)
    dx_ref = np.zeros((toks.size, cfg.d))
    dgate_ref = np.zeros((toks.size, cfg.k))
    for i, t in enumerate(toks):
        for j in range(cfg.k):
            e = int(idx[t, j])
            w1, w3, w2 = ex(e)
            o = oracle.swiglu_expert(xf[t:t + 1], w1, w3, w2)
            dgate_ref[i, j] = (dyf[t] * o[0]).sum()
            dX, _, _, _ = oracle.swiglu_expert_backward(xf[t:t + 1], w1, w3, w2,
                                                        gates[t, j] * dyf[t:t + 1])
            dx_ref[i] += dX[0]
        if cfg.has_shared:
            w1, w3, w2 = ex(cfg.E)
            dX, _, _, _ = oracle.swiglu_expert_backward(xf[t:t + 1], w1, w3, w2, dyf[t:t + 1])
            dx_ref[i] += dX[0]
    _close(npf(layer.dx)[toks], dx_ref, "dx (sampled tokens)")
    _close(layer.dgate.cpu().numpy()[toks], dgate_ref, "dgate (sampled tokens)")
    # one routed expert's weight gradients over all of its rows
    e = 1
    rows = np.arange(int(perm["offsets"][e]), int(perm["offsets"][e]) + int(perm["kept"][e]))
    a = perm["order"][rows]
    t = a // cfg.k
    w1, w3, w2 = ex(e)
    dO = gates.reshape(-1)[a][:, None] * dyf[t]
    _, dW1r, dW3r, dW2r = oracle.swiglu_expert_backward(xf[t], w1, w3, w2, dO)
    dW1, dW3 = layer.unpacked_dW13()
    _close(npf(dW1[e]), dW1r, "dW1[e]")
    _close(npf(dW3[e]), dW3r, "dW3[e]")
    _close(npf(layer.dW2[e]), dW2r, "dW2[e]")


@pytest.mark.parametrize("name", ["ds_small", "skew_small", "tiny_ragged"])
def test_backward_with_saved_preactivations_is_identical(m, name):
    """The training forward keeps GEMM 1's output (g1); the backward that reads it
    gives bit-identical gradients to the backward that recomputes it, and the
    training forward's y is the inference forward's."""
    cfg = SMALL[name]
    x = synth.make_x(cfg, device="cuda")
    scores = synth.make_scores(cfg, device="cuda")
    if name == "skew_small":
        scores[:, 0] += 4.5
    W1, W3, W2 = synth.make_expert_weights(cfg, device="cuda")
    dy = _dy(cfg, "cuda")
    a = m.MoELayer(cfg, W1, W3, W2)
    b = m.MoELayer(cfg, W1, W3, W2, train=True)
    a.forward(x, scores=scores)
    b.forward(x, scores=scores)
    assert torch.equal(a.y.view(torch.int16), b.y.view(torch.int16))
    a.backward(x, dy)
    b.backward(x, dy)
    torch.cuda.synchronize()
    for name_ in ("dx", "dW13", "dW2"):
        assert torch.equal(getattr(a, name_).view(torch.int16), getattr(b, name_).view(torch.int16)), name_
    assert torch.equal(a.dgate, b.dgate)
