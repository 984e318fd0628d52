"""Parity at the full workload sizes, in the launch configuration the
benchmark times (the whole MoELayer path on one stream).  Routing, counts,
offsets and permutations are compared in full elsewhere (test_gpu_parity.py
runs them at these sizes); here the layer output is compared on a seeded
sample of tokens that the oracle computes one by one in fp64, and the router
logits on the same sample."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu_util import assert_y_close, npf, npi

pytestmark = pytest.mark.gpu


class StreamedExperts:
    """Device expert weights fetched to the host one expert at a time."""

    def __init__(self, W):
        self.W = W
        self.last = (None, None)

    def __getitem__(self, e):
        e = int(e)
        if self.last[0] != e:
            self.last = (e, self.W[e].float().cpu().numpy())
        return self.last[1]


@pytest.fixture(scope="module")
def m():
    import expert_token_dispatch_moe_b300 as mod
    return mod


@pytest.mark.parametrize("name,n_sample", [("mixtral", 24), ("dsv3", 10), ("dsv3_decode", 8),
                                           ("skew", 48)])
def test_full_size_layer_on_sampled_tokens(m, name, n_sample):
    cfg = synth.CONFIGS[name]
    dev = torch.device("cuda")
    x = synth.make_x(cfg, device=dev)
    scores = synth.make_scores(cfg, device=dev)
    W1, W3, W2 = synth.make_expert_weights(cfg, device=dev)
    layer = m.MoELayer(cfg, W1, W3, W2, device=dev)
    layer.forward(x, scores=scores)
    torch.cuda.synchronize()
    assert m.moe_get_device_status(layer.ws) == 0
    tokens = synth.sample_tokens(cfg, n_sample).numpy()
    s_np = scores.cpu().numpy()
    x_np = x.float().cpu().numpy()
    y_ref, st = oracle.moe_forward(x_np, s_np, cfg, StreamedExperts(W1), StreamedExperts(W3),
                                   StreamedExperts(W2), tokens=tokens)
    # routing and permutation in full, bit-exact
    assert np.array_equal(npi(layer.topk_idx), st["idx"])
    assert np.array_equal(npi(layer.counts), st["perm"]["counts"])
    assert np.array_equal(npi(layer.inv), st["perm"]["inv"])
    lay = oracle.ep_layout(st["idx"], st["perm"]["inv"], cfg.E, cfg.n_ep, cfg.T)
    assert np.array_equal(npi(layer.count_mat), lay["C"])
    assert np.array_equal(npi(layer.send_idx), lay["send_idx"])
    # layer output on the sampled tokens
    assert_y_close(npf(layer.y[torch.from_numpy(tokens).to(dev)]), y_ref[tokens])


@pytest.mark.parametrize("name,tc", [("mixtral", False), ("mixtral", True), ("dsv3", False),
                                     ("dsv3", True), ("skew", True)])
def test_full_size_router_logits_on_sampled_tokens(m, name, tc):
    cfg = synth.CONFIGS[name]
    dev = torch.device("cuda")
    x = synth.make_x(cfg, device=dev)
    W_r, lb = synth.make_router(cfg, device=dev)
    c = m.MoeCfg.from_layer(cfg)
    out = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device=dev)
    split = None
    if tc:
        split = torch.empty(3, cfg.E, cfg.d, dtype=torch.bfloat16, device=dev)
        m.moe_pack_router(c, W_r, split)
    m.moe_router_logits(c, x, None if tc else W_r, split, lb, out)
    torch.cuda.synchronize()
    tokens = synth.sample_tokens(cfg, 256).numpy()
    xs = x[torch.from_numpy(tokens).to(dev)].float().cpu().numpy()
    Wn = W_r.cpu().numpy()
    l_ref = oracle.router_logits(xs, Wn, None if lb is None else lb.cpu().numpy())
    bound = ((3 if tc else 1) * cfg.d * 2.0 ** -24 * (np.abs(xs) @ np.abs(Wn))
             + 2.0 ** -23 * np.abs(l_ref))
    got = npf(out[torch.from_numpy(tokens).to(dev)])
    if cfg.score_fn == "sigmoid":
        assert (np.abs(got - oracle.sigmoid(l_ref)) <= 0.25 * bound + 4e-7).all()
    else:
        assert (np.abs(got - l_ref) <= bound).all()
