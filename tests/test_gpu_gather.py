"""The permute's row move fused into GEMM 1's loads (moe_grouped_ffn_gather):
the gathered operand tiles hold the same bf16 values in the same shared-memory
layout as the x_sorted path, so h, y_sorted and y must be bit-identical to it;
the layer output is also checked against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu_util import assert_y_close, npf, npi

pytestmark = pytest.mark.gpu

C = synth.CONFIGS
SMALL = {
    "tiny": C["tiny"],
    "tiny_ragged": C["tiny"].with_(name="tiny_ragged", T=1000, n_ep=8),
    "ds_small": C["dsv3"].with_(name="ds_small", T=512, d=256, f=256, E=64, n_ep=16),
    "decode_small": C["dsv3"].with_(name="decode_small", T=32, d=512, f=256, n_ep=16),
    "skew_small": C["skew"].with_(name="skew_small", T=2048, d=256, f=256, E=16, n_ep=8,
                                  capacity=oracle.capacity_rows(1.25, 2048, 2, 16)),
    "single_expert": C["tiny"].with_(name="single_expert", T=300, E=1, k=1, n_ep=1, d=128, f=128),
    "k_equals_E": C["tiny"].with_(name="k_equals_E", T=256, E=32, k=32, n_ep=2, d=128, f=128),
}


@pytest.fixture(scope="module")
def m():
    import expert_token_dispatch_moe_b300 as mod
    return mod


def _both(m, cfg, x, scores, W1, W3, W2):
    a = m.MoELayer(cfg, W1, W3, W2, gather=False)
    b = m.MoELayer(cfg, W1, W3, W2, gather=True)
    a.forward(x, scores=scores)
    b.h.fill_(7.0)
    b.y_sorted.fill_(7.0)
    b.forward(x, scores=scores)
    torch.cuda.synchronize()
    assert m.moe_get_device_status(a.ws) == 0 and m.moe_get_device_status(b.ws) == 0
    return a, b


def _kept_rows(layer, cfg):
    rows = torch.nonzero(layer.order >= 0).flatten()
    if cfg.has_shared:
        rows = torch.cat([rows, torch.arange(cfg.R, cfg.R + cfg.T, device=rows.device)])
    return rows


@pytest.mark.parametrize("name", list(SMALL))
def test_gather_matches_unfused_and_oracle(m, name):
    cfg = SMALL[name]
    x = synth.make_x(cfg)
    scores = synth.make_scores(cfg)
    W1, W3, W2 = synth.make_expert_weights(cfg)
    a, b = _both(m, cfg, x.cuda(), scores.cuda(), W1.cuda(), W3.cuda(), W2.cuda())
    rows = _kept_rows(a, cfg)
    assert torch.equal(a.order, b.order) and torch.equal(a.inv, b.inv)
    assert torch.equal(a.h[rows].view(torch.int16), b.h[rows].view(torch.int16))
    assert torch.equal(a.y_sorted[rows].view(torch.int16), b.y_sorted[rows].view(torch.int16))
    assert torch.equal(a.y.view(torch.int16), b.y.view(torch.int16))
    y_ref, st = oracle.moe_forward(x.float().numpy(), scores.numpy(), cfg, W1.float().numpy(),
                                   W3.float().numpy(), W2.float().numpy())
    assert np.array_equal(npi(b.topk_idx), st["idx"])
    assert_y_close(npf(b.y), y_ref)


@pytest.mark.parametrize("name", ["mixtral", "dsv3", "skew", "dsv3_decode"])
def test_gather_matches_unfused_full_size(m, name):
    """Full-size workloads: every kept row of h and y_sorted, and y, bit-identical
    to the x_sorted path."""
    cfg = C[name]
    x = synth.make_x(cfg, device="cuda")
    scores = synth.make_scores(cfg, device="cuda")
    if name == "skew":
        scores[:, 0] += 4.5
    W1, W3, W2 = synth.make_expert_weights(cfg, device="cuda")
    a, b = _both(m, cfg, x, scores, W1, W3, W2)
    del W1, W3, W2
    rows = _kept_rows(a, cfg)
    assert torch.equal(a.h[rows].view(torch.int16), b.h[rows].view(torch.int16))
    assert torch.equal(a.y_sorted[rows].view(torch.int16), b.y_sorted[rows].view(torch.int16))
    assert torch.equal(a.y.view(torch.int16), b.y.view(torch.int16))


@pytest.mark.parametrize("name", ["tiny", "ds_small", "skew_small"])
def test_gather_whole_forward_from_c(m, name):
    """moe_layer_forward and moe_layer_forward_host with the gather flag: the
    same steps issued from C (the permute without its row move, GEMM 1 reading
    rows from x) give the bytes of the Python-issued gathered forward, and of
    the rows path."""
    cfg = SMALL[name]
    dev = torch.device("cuda")
    x = synth.make_x(cfg, device=dev)
    W1, W3, W2 = synth.make_expert_weights(cfg, device=dev)
    W_r, lbias = synth.make_router(cfg, device=dev)
    rows = m.MoELayer(cfg, W1, W3, W2, W_r=W_r, logit_bias=lbias, device=dev)
    fused = m.MoELayer(cfg, W1, W3, W2, W_r=W_r, logit_bias=lbias, device=dev, gather=True)
    y_rows = rows.forward(x).clone()
    y_py = fused.forward(x).clone()
    y_c = fused.forward_c(x, torch.empty_like(y_py))
    x_host = x.cpu().pin_memory()
    y_hosts = [torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16).pin_memory() for _ in range(3)]
    fused.forward_host_c([x_host] * 3, y_hosts)
    torch.cuda.synchronize()
    assert m.moe_get_device_status(fused.ws) == 0
    for y in [y_c, y_rows] + [h.to(dev) for h in y_hosts]:
        assert torch.equal(y.view(torch.int16), y_py.view(torch.int16))
