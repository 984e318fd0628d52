"""The combine in GEMM 2's epilogue (moe_grouped_ffn_combine): each grouped row
adds gate * row into its token's output by bf16 reductions, instead of writing
y_sorted for a separate combine ("Expert parallelism", "Token permutation and
grouped GEMMs": production kernels fuse the combine into the GEMM's epilogue).
Checked against the oracle's layer output on the routing the GPU took, and
against the unfused path."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu_util import assert_y_close, npf, npi, run_path

C = synth.CONFIGS
CASES = {
    "tiny": C["tiny"],                                           # k = 2, softmax: deterministic
    "ds_small": C["dsv3"].with_(name="ds_small", T=512, d=256, f=256, E=64, n_ep=16),  # k = 8 + shared
    "skew_small": C["skew"].with_(name="skew_small", T=2048, d=256, f=256, E=16, n_ep=8,
                                  capacity=oracle.capacity_rows(1.25, 2048, 2, 16)),
    "single_expert": C["tiny"].with_(name="single_expert", T=300, E=1, k=1, n_ep=1, d=128, f=128),
    "wide_rows": C["mixtral"].with_(name="wide_rows", T=512, d=2048, f=256, n_ep=8),
}

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import expert_token_dispatch_moe_b300 as mod
    return mod


def _fused(m, layer, x):
    c = layer.cfg
    y = torch.full_like(layer.y, 3.0)   # the call zeroes y itself
    m.moe_grouped_ffn_combine(c, layer.x_sorted, x if c.has_shared else None, layer.counts,
                              layer.offsets, layer.W13, layer.W2, layer.h, layer.order,
                              layer.topk_gate, y, layer.ws)
    torch.cuda.synchronize()
    assert m.moe_get_device_status(layer.ws) == 0
    return y


@pytest.mark.parametrize("name", list(CASES))
def test_combine_epilogue_matches_oracle(m, name):
    cfg = CASES[name]
    x = synth.make_x(cfg)
    scores = synth.make_scores(cfg)
    W1, W3, W2 = synth.make_expert_weights(cfg)
    x_dev = x.cuda()
    layer = run_path(m, cfg, x_dev, scores.cuda(), W1.cuda(), W3.cuda(), W2.cuda())
    y_ref, st = oracle.moe_forward(x.float().numpy(), scores.numpy(), cfg, W1.float().numpy(),
                                   W3.float().numpy(), W2.float().numpy())
    assert np.array_equal(npi(layer.topk_idx), st["idx"])
    y_unfused = npf(layer.y)
    y = _fused(m, layer, x_dev)
    assert_y_close(npf(y), y_ref)
    # the same layer's unfused output, to the same tolerance
    assert_y_close(npf(y), y_unfused)


def test_combine_epilogue_two_terms_are_reproducible(m):
    """With two contributions per token (k = 2, no shared expert) every output
    element is 0 + a + b in some order: bf16 addition commutes, so the result
    is the same bytes on every call."""
    cfg = CASES["tiny"]
    x = synth.make_x(cfg, device="cuda")
    scores = synth.make_scores(cfg, device="cuda")
    W1, W3, W2 = synth.make_expert_weights(cfg, device="cuda")
    layer = run_path(m, cfg, x, scores, W1, W3, W2)
    y1 = _fused(m, layer, x).clone()
    y2 = _fused(m, layer, x).clone()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_layer_option_uses_the_epilogue(m):
    """MoELayer(combine_in_epilogue=True): the same routing and permutation, the
    output within the layer's tolerance of the default path, and no backward."""
    cfg = CASES["ds_small"]
    x = synth.make_x(cfg, device="cuda")
    scores = synth.make_scores(cfg, device="cuda")
    W1, W3, W2 = synth.make_expert_weights(cfg, device="cuda")
    ref = m.MoELayer(cfg, W1, W3, W2)
    y_ref = ref.forward(x, scores=scores).clone()
    fused = m.MoELayer(cfg, W1, W3, W2, combine_in_epilogue=True)
    y = fused.forward(x, scores=scores)
    torch.cuda.synchronize()
    assert torch.equal(fused.topk_idx, ref.topk_idx) and torch.equal(fused.inv, ref.inv)
    assert_y_close(npf(y), npf(y_ref))
    with pytest.raises(RuntimeError):
        fused.backward(x, torch.zeros_like(y))


@pytest.mark.parametrize("name", ["tiny", "ds_small"])
def test_whole_forward_from_c_takes_the_flag(m, name):
    """moe_layer_forward with combine_in_epilogue set: the same steps from C.
    With two contributions per token (tiny) the bytes equal the Python-issued
    forward's; otherwise the outputs agree within the layer's tolerance."""
    cfg = CASES[name]
    x = synth.make_x(cfg, device="cuda")
    W1, W3, W2 = synth.make_expert_weights(cfg, device="cuda")
    W_r, lbias = synth.make_router(cfg, device="cuda")
    layer = m.MoELayer(cfg, W1, W3, W2, W_r=W_r, logit_bias=lbias, combine_in_epilogue=True)
    y_py = layer.forward(x).clone()
    y_c = layer.forward_c(x, torch.empty_like(y_py))
    torch.cuda.synchronize()
    assert m.moe_get_device_status(layer.ws) == 0
    if cfg.k == 2 and not cfg.has_shared:
        assert torch.equal(y_c.view(torch.int16), y_py.view(torch.int16))
    else:
        assert_y_close(npf(y_c), npf(y_py))
