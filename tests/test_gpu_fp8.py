"""Parity of the FP8 dispatch path with the oracle: the e4m3 send buffer and its
per-row scales (bit-exact), the receiver's dequantized expert-grouped rows
(bit-exact bf16), and the whole layer run on FP8-dispatched rows (within
max|y - y_ref| <= 2e-2 max|y_ref| of the oracle on the same dequantized rows)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu_util import assert_y_close, npi

pytestmark = pytest.mark.gpu

C = synth.CONFIGS
CASES = {
    "tiny": C["tiny"],
    "tiny_ragged": C["tiny"].with_(name="tiny_ragged", T=1000, n_ep=8),
    "ds_small": C["dsv3"].with_(name="ds_small", T=512, d=256, f=256, E=64, n_ep=16),
    "skew_small": C["skew"].with_(name="skew_small", T=2048, d=256, f=256, E=16, n_ep=8,
                                  capacity=oracle.capacity_rows(1.25, 2048, 2, 16)),
    "mixtral": C["mixtral"],
    "skew": C["skew"],
}


@pytest.fixture(scope="module")
def m():
    import expert_token_dispatch_moe_b300 as mod
    return mod


def _fp8_path(m, cfg, x_dev, idx_np):
    """route indices given -> permute -> FP8 layout -> receive; returns tensors."""
    c = m.MoeCfg.from_layer(cfg)
    dev = "cuda"
    i32 = dict(dtype=torch.int32, device=dev)
    idx = torch.from_numpy(idx_np.astype(np.int32)).to(dev)
    o = dict(counts=torch.empty(cfg.E, **i32), offsets=torch.empty(cfg.E + 1, **i32),
             order=torch.empty(cfg.R, **i32), inv=torch.empty(cfg.A, **i32),
             x_sorted=torch.empty(cfg.R, cfg.d, dtype=torch.bfloat16, device=dev),
             C=torch.empty(cfg.n_ep, cfg.n_ep, **i32), send_off=torch.empty(cfg.n_ep, cfg.n_ep, **i32),
             recv_off=torch.empty(cfg.n_ep, cfg.n_ep, **i32), send_idx=torch.empty(cfg.A, **i32),
             send_fp8=torch.full((cfg.A, cfg.d), 0x55, dtype=torch.uint8, device=dev),
             send_scale=torch.full((cfg.A,), 7.0, dtype=torch.float32, device=dev))
    ws = torch.zeros(m.moe_workspace_bytes(c), dtype=torch.uint8, device=dev)
    m.moe_workspace_init(c, ws)
    m.moe_permute(c, x_dev, idx, o["counts"], o["offsets"], o["order"], o["inv"], o["x_sorted"], ws)
    m.moe_ep_layout_fp8(c, idx, o["offsets"], o["inv"], o["C"], o["send_off"], o["recv_off"],
                        o["send_idx"], x_dev, o["send_fp8"], o["send_scale"], ws)
    # the receiver overwrites the kept rows of the grouped buffer
    o["x_sorted"][o["order"] >= 0] = torch.tensor(3.0, dtype=torch.bfloat16, device=dev)
    m.moe_dispatch_recv_fp8(c, o["send_fp8"], o["send_scale"], o["send_idx"], o["inv"],
                            o["x_sorted"])
    torch.cuda.synchronize()
    assert m.moe_get_device_status(ws) == 0
    o["ws"] = ws
    return o


@pytest.mark.parametrize("name", list(CASES))
def test_fp8_layout_and_receive_parity(m, name):
    cfg = CASES[name]
    scores = synth.make_scores(cfg)
    if name == "skew_small":
        scores[:, 0] += 4.5
    idx_np = oracle.select_experts(scores.numpy(), cfg.k, None, cfg.n_groups, cfg.topk_groups)
    x_dev = synth.make_x(cfg, device="cuda")
    o = _fp8_path(m, cfg, x_dev, idx_np)
    xf = x_dev.float().cpu().numpy()
    p = oracle.permute(idx_np, cfg.E, cfg.capacity)
    lay = oracle.ep_layout_fp8(xf, idx_np, p["inv"], cfg.E, cfg.n_ep, cfg.T)
    assert np.array_equal(npi(o["C"]), lay["C"])
    assert np.array_equal(npi(o["send_idx"]), lay["send_idx"])
    assert np.array_equal(o["send_fp8"].cpu().numpy(), lay["send_fp8"])
    assert np.array_equal(o["send_scale"].cpu().numpy(), lay["send_scale"])
    # receiver: kept rows are the dequantized token rows, bit for bit
    codes_t, scale_t = oracle.quantize_rows_fp8(xf)
    deq_t = oracle.dequantize_rows_fp8(codes_t, scale_t)
    order = p["order"]
    kept = order >= 0
    got = o["x_sorted"].float().cpu().numpy()
    assert np.array_equal(got[kept], deq_t[order[kept] // cfg.k])
    if cfg.capacity:
        assert (got[~kept] == 0).all()             # padding rows from the permute stay zero


def test_fp8_layout_dsv3_sampled(m):
    """Full DS-V3 shape (470 MB of codes): every index output in full, the codes
    and scales of 512 sampled slots."""
    cfg = C["dsv3"]
    scores = synth.make_scores(cfg)
    idx_np = oracle.select_experts(scores.numpy(), cfg.k, None, cfg.n_groups, cfg.topk_groups)
    x_dev = synth.make_x(cfg, device="cuda")
    o = _fp8_path(m, cfg, x_dev, idx_np)
    p = oracle.permute(idx_np, cfg.E)
    lay = oracle.ep_layout(idx_np, p["inv"], cfg.E, cfg.n_ep, cfg.T)
    sidx = npi(o["send_idx"])
    assert np.array_equal(sidx, lay["send_idx"])
    rng = np.random.default_rng(0)
    slots = rng.choice(cfg.A, size=512, replace=False)
    toks = sidx[slots] // cfg.k
    codes, scale = oracle.quantize_rows_fp8(x_dev[torch.from_numpy(toks).cuda()].float().cpu().numpy())
    assert np.array_equal(o["send_fp8"][torch.from_numpy(slots).cuda()].cpu().numpy(), codes)
    assert np.array_equal(o["send_scale"][torch.from_numpy(slots).cuda()].cpu().numpy(), scale)


@pytest.mark.parametrize("name", ["tiny", "ds_small", "skew_small"])
def test_layer_with_fp8_dispatch(m, name):
    """Route -> permute -> FP8 layout -> receive -> grouped FFN -> combine,
    against the oracle's layer on the same dequantized token rows."""
    cfg = CASES[name]
    x = synth.make_x(cfg)
    scores = synth.make_scores(cfg)
    if name == "skew_small":
        scores[:, 0] += 4.5
    W1, W3, W2 = synth.make_expert_weights(cfg)
    layer = m.MoELayer(cfg, W1.cuda(), W3.cuda(), W2.cuda())
    c = layer.cfg
    x_dev = x.cuda()
    m.moe_route(c, scores.cuda(), None, layer.topk_idx, layer.topk_gate)
    idx_np = npi(layer.topk_idx)
    o = _fp8_path(m, cfg, x_dev, idx_np)
    m.moe_grouped_ffn(c, o["x_sorted"], x_dev if cfg.has_shared else None, o["counts"],
                      o["offsets"], layer.W13, layer.W2, layer.h, layer.y_sorted, o["ws"])
    m.moe_combine(c, layer.y_sorted, o["inv"], layer.topk_gate, layer.y)
    torch.cuda.synchronize()
    xf = x.float().numpy()
    codes, scale = oracle.quantize_rows_fp8(xf)
    x_deq = oracle.dequantize_rows_fp8(codes, scale)
    # routed experts see the dequantized rows; the shared expert (not dispatched) sees x
    y_ref, st = oracle.moe_forward(x_deq, scores.numpy(), cfg, W1.float().numpy(),
                                   W3.float().numpy(), W2.float().numpy())
    if cfg.has_shared:
        y_sh_deq = oracle.swiglu_expert(x_deq, W1[-1].float().numpy(), W3[-1].float().numpy(),
                                        W2[-1].float().numpy())
        y_sh = oracle.swiglu_expert(xf, W1[-1].float().numpy(), W3[-1].float().numpy(),
                                    W2[-1].float().numpy())
        y_ref = y_ref - y_sh_deq + y_sh
    assert np.array_equal(idx_np, st["idx"])
    assert_y_close(layer.y.float().cpu().numpy(), y_ref)
    assert m.moe_get_device_status(o["ws"]) == 0
