"""The CUDA layer against the oracle's per-token C loop (oracle/moe_loop.c):
each token's output computed on its own from its expert choices, with no
permutation, grouped buffer or combine step on the oracle side.  Routing is
compared bit for bit on the same fp32 scores (the GPU router's own, or
synthetic ones); the layer output within max|y - y_ref| <= 2e-2 * max|y_ref|
(bf16 inputs, fp32 accumulation)."""
import numpy as np
import pytest
import torch

import synth
from _gpu_util import assert_y_close, npf, npi
from oracle import loop

pytestmark = pytest.mark.gpu

C = synth.CONFIGS
CASES = {
    # every token of small layers that span several tiles and ragged tails
    "tiny": (C["tiny"], None),
    "ds_small": (C["dsv3"].with_(name="ds_small", T=512, d=256, f=256, E=64, n_ep=16), None),
    "skew_small": (C["skew"].with_(name="skew_small", T=2048, d=256, f=256, E=16, n_ep=8,
                                   capacity=320), None),
    # the Mixtral layer's expert shapes (d = 4096, f = 14336) on 256 tokens, 48 of
    # them recomputed token by token
    "mixtral_256": (C["mixtral"].with_(name="mixtral_256", T=256), 48),
}


@pytest.fixture(scope="module")
def m():
    import expert_token_dispatch_moe_b300 as mod
    return mod


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("router", [False, True])
def test_layer_against_per_token_loop(m, name, router):
    cfg, n_tok = CASES[name]
    dev = torch.device("cuda")
    x = synth.make_x(cfg, device=dev)
    W1, W3, W2 = synth.make_expert_weights(cfg, device=dev)
    if router:
        W_r, lbias = synth.make_router(cfg, device=dev)
        layer = m.MoELayer(cfg, W1, W3, W2, W_r=W_r, logit_bias=lbias, device=dev)
        layer.forward(x)
        scores = layer.scores   # the router's fp32 output, routed on both sides
    else:
        layer = m.MoELayer(cfg, W1, W3, W2, device=dev)
        scores = synth.make_scores(cfg, device=dev)
        layer.forward(x, scores=scores)
    torch.cuda.synchronize()
    assert m.moe_get_device_status(layer.ws) == 0
    s = scores.cpu().numpy()
    idx = loop.select_experts(s, cfg.k, None, cfg.n_groups, cfg.topk_groups)
    assert np.array_equal(npi(layer.topk_idx), idx)
    gates = loop.gate_weights(s, idx, cfg.score_fn, cfg.norm_topk)
    assert np.allclose(layer.topk_gate.cpu().numpy(), gates, rtol=1e-5, atol=1e-7)
    tokens = (np.arange(cfg.T) if n_tok is None
              else synth.sample_tokens(cfg, n_tok).numpy())
    y_ref = loop.layer_tokens(x, idx, gates, cfg, W1, W3, W2, tokens)
    tok = torch.from_numpy(tokens).to(dev)
    assert_y_close(npf(layer.y[tok]), y_ref)
