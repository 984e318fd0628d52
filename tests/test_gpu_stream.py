"""The streaming host call: several host batches through
MoELayer.forward_host_stream (copies on their own streams, overlapping
compute, two device buffers per side), with the forward issued call by call
or replayed from CUDA graphs, give, batch for batch, exactly the outputs of
the plain device forward."""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("graphs", [False, True])
@pytest.mark.parametrize("name,n", [("tiny", 5), ("mixtral", 3), ("dsv3_decode", 3), ("skew", 3)])
def test_forward_host_stream_matches_device_forward(name, n, graphs):
    import expert_token_dispatch_moe_b300 as m
    cfg = synth.CONFIGS[name]
    if name == "mixtral":
        cfg = cfg.with_(T=512)   # the full expert shapes, fewer tokens
    if name == "skew":
        # 5120 assignments over 64 experts: the one-launch (cooperative) permute,
        # captured in the graphs too
        cfg = cfg.with_(T=2560, capacity=100)
    W1, W3, W2 = synth.make_expert_weights(cfg, device="cuda")
    W_r, lb = synth.make_router(cfg, device="cuda")
    layer = m.MoELayer(cfg, W1, W3, W2, W_r=W_r, logit_bias=lb)
    if graphs:
        layer.capture_graphs()
    xs = [synth.make_x(cfg, seed=100 + i).pin_memory() for i in range(n)]
    ys = [torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16).pin_memory() for _ in range(n)]
    layer.forward_host_stream(xs, ys)
    torch.cuda.synchronize()
    for i in range(n):
        ref = layer.forward(xs[i].cuda()).cpu()
        torch.cuda.synchronize()
        assert torch.equal(ys[i].view(torch.int16), ref.view(torch.int16)), i
    assert m.moe_get_device_status(layer.ws) == 0


@pytest.mark.parametrize("name,n", [("tiny", 5), ("skew", 3), ("dsv3_decode", 3)])
def test_library_host_forward_matches_device_forward(name, n):
    """moe_layer_forward_host (the library's own call: one copy per direction
    per batch on copy streams, double-buffered device buffers, the forward
    issued from C) and moe_layer_forward give, batch for batch, exactly the
    outputs of MoELayer.forward."""
    import expert_token_dispatch_moe_b300 as m
    cfg = synth.CONFIGS[name]
    if name == "skew":
        cfg = cfg.with_(T=2048, capacity=80)   # the full expert shapes, fewer tokens
    W1, W3, W2 = synth.make_expert_weights(cfg, device="cuda")
    W_r, lb = synth.make_router(cfg, device="cuda")
    layer = m.MoELayer(cfg, W1, W3, W2, W_r=W_r, logit_bias=lb)
    xs = [synth.make_x(cfg, seed=200 + i).pin_memory() for i in range(n)]
    ys = [torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16).pin_memory() for _ in range(n)]
    layer.forward_host_c(xs, ys)
    torch.cuda.synchronize()
    refs = []
    for i in range(n):
        refs.append(layer.forward(xs[i].cuda()).cpu())
        torch.cuda.synchronize()
        assert torch.equal(ys[i].view(torch.int16), refs[i].view(torch.int16)), i
    y_dev = torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16, device="cuda")
    layer.forward_c(xs[0].cuda(), y_dev)
    torch.cuda.synchronize()
    assert torch.equal(y_dev.cpu().view(torch.int16), refs[0].view(torch.int16))
    assert layer.launches_per_forward > 0
    assert m.moe_get_device_status(layer.ws) == 0
