"""Edge cases at the limits the C ABI states: the largest expert count and
top-k (E = 1024, k = 32, 32 groups), one expert-parallel rank per expert
(n_ep = E), the widest hidden size (d = 65536), a single token, capacity 1,
every token on one expert, and all-tied scores.  Indices and layouts are
compared with the oracle exactly, layer outputs within 2e-2 of max|y_ref|."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu_util import assert_y_close, npf, npi

pytestmark = pytest.mark.gpu

C = synth.CONFIGS


@pytest.fixture(scope="module")
def m():
    import expert_token_dispatch_moe_b300 as mod
    return mod


def _route(m, cfg, s, bias=None):
    c = m.MoeCfg.from_layer(cfg)
    idx = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device="cuda")
    gate = torch.empty(cfg.T, cfg.k, dtype=torch.float32, device="cuda")
    m.moe_route(c, s.cuda(), None if bias is None else bias.cuda(), idx, gate)
    torch.cuda.synchronize()
    return npi(idx), gate.cpu().numpy().astype(np.float64)


def _layout(m, cfg, x_dev, idx_np):
    c = m.MoeCfg.from_layer(cfg)
    i32 = dict(dtype=torch.int32, device="cuda")
    idx = torch.from_numpy(idx_np.astype(np.int32)).cuda()
    o = dict(counts=torch.empty(cfg.E, **i32), offsets=torch.empty(cfg.E + 1, **i32),
             order=torch.empty(cfg.R, **i32), inv=torch.empty(cfg.A, **i32),
             x_sorted=torch.empty(cfg.R, cfg.d, dtype=torch.bfloat16, device="cuda"),
             C=torch.empty(cfg.n_ep, cfg.n_ep, **i32), send_off=torch.empty(cfg.n_ep, cfg.n_ep, **i32),
             recv_off=torch.empty(cfg.n_ep, cfg.n_ep, **i32), send_idx=torch.empty(cfg.A, **i32),
             send_buf=torch.empty(cfg.A, cfg.d, dtype=torch.bfloat16, device="cuda"))
    ws = torch.zeros(m.moe_workspace_bytes(c), dtype=torch.uint8, device="cuda")
    m.moe_workspace_init(c, ws)
    m.moe_permute(c, x_dev, idx, o["counts"], o["offsets"], o["order"], o["inv"], o["x_sorted"], ws)
    m.moe_ep_layout(c, idx, o["offsets"], o["inv"], o["C"], o["send_off"], o["recv_off"],
                    o["send_idx"], x_dev, o["send_buf"], ws)
    assert m.moe_get_device_status(ws) == 0
    ref = oracle.permute(idx_np, cfg.E, cfg.capacity)
    for key in ("counts", "offsets", "order", "inv"):
        assert np.array_equal(npi(o[key]), ref[key]), key
    lay = oracle.ep_layout(idx_np, ref["inv"], cfg.E, cfg.n_ep, cfg.T)
    for key in ("C", "send_off", "recv_off", "send_idx"):
        assert np.array_equal(npi(o[key]), lay[key]), key
    order = torch.from_numpy(ref["order"]).cuda()
    exp = torch.zeros(cfg.R, cfg.d, dtype=torch.bfloat16, device="cuda")
    filled = order >= 0
    exp[filled] = x_dev[order[filled] // cfg.k]
    assert torch.equal(o["x_sorted"].view(torch.int16), exp.view(torch.int16))
    return o


@pytest.mark.parametrize("ties", [False, True])
def test_route_largest_expert_count_and_topk(m, ties):
    """E = 1024 (32 experts per lane), k = 32, 32 groups of 32 keeping 2, with a
    selection bias."""
    cfg = C["dsv3"].with_(T=257, E=1024, k=32, n_groups=32, topk_groups=2, n_ep=1)
    s = synth.make_scores(cfg, ties=ties)
    bias = (torch.randn(cfg.E, generator=torch.Generator().manual_seed(5)) * 0.1).float()
    idx, gate = _route(m, cfg, s, bias)
    ref = oracle.select_experts(s.numpy(), cfg.k, bias.numpy(), cfg.n_groups, cfg.topk_groups)
    assert np.array_equal(idx, ref)
    assert np.allclose(gate, oracle.gate_weights(s.numpy(), ref, cfg.score_fn, cfg.norm_topk),
                       rtol=1e-5, atol=1e-7)
    cfg2 = cfg.with_(n_groups=1, topk_groups=1, score_fn="softmax", norm_topk=0)
    s2 = synth.make_scores(cfg2, ties=ties)
    idx2, _ = _route(m, cfg2, s2)
    assert np.array_equal(idx2, oracle.select_experts(s2.numpy(), cfg2.k))


def test_layout_one_rank_per_expert(m):
    """n_ep = E = 1024: a 1024 x 1024 count matrix."""
    cfg = C["tiny"].with_(T=2048, E=1024, k=4, n_ep=1024, d=64)
    rng = np.random.default_rng(0)
    idx_np = np.stack([rng.choice(cfg.E, size=cfg.k, replace=False) for _ in range(cfg.T)])
    _layout(m, cfg, synth.make_x(cfg, device="cuda"), idx_np)


def test_widest_hidden_size(m):
    """d = 65536 (128 KB rows): permute, layout, FFN and combine on a few tokens."""
    cfg = C["tiny"].with_(T=16, d=65536, E=4, k=2, f=128, n_ep=2)
    x = synth.make_x(cfg)
    scores = synth.make_scores(cfg)
    W1, W3, W2 = synth.make_expert_weights(cfg)
    idx_np = oracle.select_experts(scores.numpy(), cfg.k)
    _layout(m, cfg, x.cuda(), idx_np)
    layer = m.MoELayer(cfg, W1.cuda(), W3.cuda(), W2.cuda())
    layer.forward(x.cuda(), scores=scores.cuda())
    torch.cuda.synchronize()
    y_ref, _ = oracle.moe_forward(x.float().numpy(), scores.numpy(), cfg, W1.float().numpy(),
                                  W3.float().numpy(), W2.float().numpy())
    assert_y_close(npf(layer.y), y_ref)
    assert m.moe_get_device_status(layer.ws) == 0


@pytest.mark.parametrize("case", ["single_token", "capacity_one", "all_to_one_expert",
                                  "all_tied"])
def test_degenerate_layers(m, case):
    base = C["tiny"].with_(d=128, f=128)
    if case == "single_token":
        cfg = base.with_(T=1, n_ep=1, E=16, k=4)
    elif case == "capacity_one":
        cfg = base.with_(T=256, E=8, k=2, n_ep=4, capacity=1)
    elif case == "all_to_one_expert":
        cfg = base.with_(T=512, E=8, k=1, n_ep=4)
    else:
        cfg = base.with_(T=300, E=8, k=3, n_ep=4)
    x = synth.make_x(cfg)
    scores = synth.make_scores(cfg)
    if case == "all_to_one_expert":
        scores[:, 5] += 100.0
    if case == "all_tied":
        scores = torch.zeros_like(scores)      # every expert equal: the lowest indices win
    W1, W3, W2 = synth.make_expert_weights(cfg)
    layer = m.MoELayer(cfg, W1.cuda(), W3.cuda(), W2.cuda())
    layer.forward(x.cuda(), scores=scores.cuda())
    torch.cuda.synchronize()
    y_ref, st = oracle.moe_forward(x.float().numpy(), scores.numpy(), cfg, W1.float().numpy(),
                                   W3.float().numpy(), W2.float().numpy())
    assert np.array_equal(npi(layer.topk_idx), st["idx"])
    assert np.array_equal(npi(layer.inv), st["perm"]["inv"])
    assert_y_close(npf(layer.y), y_ref)
    if case == "all_tied":
        assert (st["idx"] == np.arange(cfg.k)).all()
    if case == "all_to_one_expert":
        assert (npi(layer.counts)[5] == cfg.T) and npi(layer.counts).sum() == cfg.T
    assert m.moe_get_device_status(layer.ws) == 0
