"""Failure detection on the device without a fault: a bounded wait on a
barrier that nothing completes gives up after its limit, the workspace status
word reads MOE_E_DEVICE_TIMEOUT, reading it clears it, and the context stays
usable (a whole layer forward afterwards matches the oracle)."""
import time

import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu_util import assert_y_close, npf, npi

pytestmark = pytest.mark.gpu

MOE_E_DEVICE_TIMEOUT = -8


@pytest.fixture(scope="module")
def m():
    import expert_token_dispatch_moe_b300 as mod
    return mod


@pytest.mark.parametrize("limit_ms", [5, 50])
def test_wait_timeout_reports_and_context_survives(m, limit_ms):
    cfg = synth.CONFIGS["tiny"]
    c = m.MoeCfg.from_layer(cfg)
    ws = torch.zeros(m.moe_workspace_bytes(c), dtype=torch.uint8, device="cuda")
    m.moe_workspace_init(c, ws)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    m.moe_selftest_wait_timeout(ws, limit_ms * 1_000_000)
    assert m.moe_get_device_status(ws) == MOE_E_DEVICE_TIMEOUT
    elapsed = time.perf_counter() - t0
    assert elapsed >= 0.8 * limit_ms / 1000.0      # the wait lasted its limit
    assert m.moe_get_device_status(ws) == 0        # reading the status cleared it

    # the context still runs the layer correctly
    x = synth.make_x(cfg)
    scores = synth.make_scores(cfg)
    W1, W3, W2 = synth.make_expert_weights(cfg)
    layer = m.MoELayer(cfg, W1.cuda(), W3.cuda(), W2.cuda())
    layer.forward(x.cuda(), scores=scores.cuda())
    torch.cuda.synchronize()
    y_ref, st = oracle.moe_forward(x.float().numpy(), scores.numpy(), cfg, W1.float().numpy(),
                                   W3.float().numpy(), W2.float().numpy())
    assert np.array_equal(npi(layer.topk_idx), st["idx"])
    assert_y_close(npf(layer.y), y_ref)
    assert m.moe_get_device_status(layer.ws) == 0
