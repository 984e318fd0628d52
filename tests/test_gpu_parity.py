"""Parity of the CUDA path with the oracle on small, seeded inputs that span
several tiles, ragged tails, empty experts, drops and the shared expert.
Indices, counts, offsets, permutations and layouts must match bit-exactly;
gates within fp32 rounding; layer outputs within
max|y - y_ref| <= 2e-2 * max|y_ref|."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu_util import LazyExperts, assert_y_close, npf, npi, run_path

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
    "norm_softmax": C["tiny"].with_(name="norm_softmax", E=12, k=3, n_ep=4, norm_topk=1),
}


@pytest.fixture(scope="module")
def m():
    import expert_token_dispatch_moe_b300 as mod
    return mod


def _route_gpu(m, cfg, scores, bias=None):
    c = m.MoeCfg.from_layer(cfg)
    s = scores.cuda()
    idx = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device="cuda")
    gate = torch.empty(cfg.T, cfg.k, dtype=torch.float32, device="cuda")
    m.moe_route(c, s, None if bias is None else bias.cuda(), idx, gate)
    torch.cuda.synchronize()
    return npi(idx), gate.cpu().numpy().astype(np.float64)


# --------------------------------------------------------------------------
# Routing
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", list(SMALL) + ["mixtral", "dsv3", "dsv3_decode", "skew"])
@pytest.mark.parametrize("ties", [False, True])
@pytest.mark.parametrize("with_bias", [False, True])
def test_route_parity(m, name, ties, with_bias):
    cfg = SMALL.get(name) or C[name]
    scores = synth.make_scores(cfg, ties=ties)
    bias = synth.make_selection_bias(cfg) if with_bias else None
    idx, gate = _route_gpu(m, cfg, scores, bias)
    s = scores.numpy()
    ref_idx = oracle.select_experts(s, cfg.k, None if bias is None else bias.numpy(),
                                    cfg.n_groups, cfg.topk_groups)
    assert np.array_equal(idx, ref_idx)
    ref_g = oracle.gate_weights(s, ref_idx, cfg.score_fn, cfg.norm_topk)
    assert np.allclose(gate, ref_g, rtol=1e-5, atol=1e-7)


def test_route_special_values(m):
    """-0.0/+0.0 ties, +-inf and NaN: gates are the selected scores
    themselves (sigmoid, no normalisation), so they compare exactly."""
    cfg = C["tiny"].with_(T=64, E=16, k=6, n_ep=1, score_fn="sigmoid", norm_topk=0)
    g = torch.Generator().manual_seed(3)
    pool = torch.tensor([0.0, -0.0, 1.0, -1.0, float("inf"), float("-inf"), float("nan"), 0.5])
    s = pool[torch.randint(0, len(pool), (cfg.T, cfg.E), generator=g)].contiguous()
    idx, gate = _route_gpu(m, cfg, s)
    ref = oracle.select_experts(s.numpy(), cfg.k)
    assert np.array_equal(idx, ref)
    assert np.array_equal(gate, np.take_along_axis(s.numpy(), ref, 1).astype(np.float64),
                          equal_nan=True)
    # group-limited with finite values and many ties
    cfg = cfg.with_(n_groups=4, topk_groups=2, k=5)
    s = (pool[:4][torch.randint(0, 4, (cfg.T, cfg.E), generator=g)]).contiguous()
    idx, _ = _route_gpu(m, cfg, s)
    assert np.array_equal(idx, oracle.select_experts(s.numpy(), cfg.k, None, 4, 2))


# --------------------------------------------------------------------------
# Permute and expert-parallel layout
# --------------------------------------------------------------------------

def _permute_case(m, cfg, x_dev, idx_np):
    c = m.MoeCfg.from_layer(cfg)
    dev = "cuda"
    i32 = torch.int32
    idx = torch.from_numpy(idx_np.astype(np.int32)).to(dev)
    out = dict(counts=torch.empty(cfg.E, dtype=i32, device=dev),
               offsets=torch.empty(cfg.E + 1, dtype=i32, device=dev),
               order=torch.empty(cfg.R, dtype=i32, device=dev),
               inv=torch.empty(cfg.A, dtype=i32, device=dev),
               x_sorted=torch.full((cfg.R, cfg.d), 7.0, dtype=torch.bfloat16, device=dev))
    ws = torch.zeros(m.moe_workspace_bytes(c), dtype=torch.uint8, device=dev)
    m.moe_workspace_init(c, ws)
    m.moe_permute(c, x_dev, idx, out["counts"], out["offsets"], out["order"], out["inv"],
                  out["x_sorted"], ws)
    lay = dict(C=torch.empty(cfg.n_ep, cfg.n_ep, dtype=i32, device=dev),
               send_off=torch.empty(cfg.n_ep, cfg.n_ep, dtype=i32, device=dev),
               recv_off=torch.empty(cfg.n_ep, cfg.n_ep, dtype=i32, device=dev),
               send_idx=torch.empty(cfg.A, dtype=i32, device=dev),
               send_buf=torch.full((cfg.A, cfg.d), 7.0, dtype=torch.bfloat16, device=dev))
    m.moe_ep_layout(c, idx, out["offsets"], out["inv"], lay["C"], lay["send_off"],
                    lay["recv_off"], lay["send_idx"], x_dev, lay["send_buf"], ws)
    assert m.moe_get_device_status(ws) == 0
    return out, lay


def _check_permute(cfg, x_dev, idx_np, out, lay):
    ref = oracle.permute(idx_np, cfg.E, cfg.capacity)
    for key in ("counts", "offsets", "order", "inv"):
        assert np.array_equal(npi(out[key]), ref[key]), key
    order = torch.from_numpy(ref["order"]).cuda()
    exp = torch.zeros(cfg.R, cfg.d, dtype=torch.bfloat16, device="cuda")
    filled = order >= 0
    exp[filled] = x_dev[order[filled] // cfg.k]
    assert torch.equal(out["x_sorted"].view(torch.int16), exp.view(torch.int16))
    lref = oracle.ep_layout(idx_np, ref["inv"], cfg.E, cfg.n_ep, cfg.T)
    assert np.array_equal(npi(lay["C"]), lref["C"])
    assert np.array_equal(npi(lay["send_off"]), lref["send_off"])
    assert np.array_equal(npi(lay["recv_off"]), lref["recv_off"])
    assert np.array_equal(npi(lay["send_idx"]), lref["send_idx"])
    sidx = torch.from_numpy(lref["send_idx"]).cuda()
    exp = torch.zeros(cfg.A, cfg.d, dtype=torch.bfloat16, device="cuda")
    filled = sidx >= 0
    exp[filled] = x_dev[sidx[filled] // cfg.k]
    assert torch.equal(lay["send_buf"].view(torch.int16), exp.view(torch.int16))
    # the pages' invariants on the count matrix
    Cm = lref["C"]
    if not cfg.capacity:
        assert (Cm.sum(1) == cfg.k * cfg.T_loc).all()


@pytest.mark.parametrize("name", list(SMALL) + ["mixtral", "dsv3", "dsv3_decode", "skew"])
def test_permute_and_layout_parity(m, name):
    cfg = SMALL.get(name) or C[name]
    scores = synth.make_scores(cfg)
    idx_np = oracle.select_experts(scores.numpy(), cfg.k, None, cfg.n_groups, cfg.topk_groups)
    x_dev = synth.make_x(cfg, device="cuda")
    out, lay = _permute_case(m, cfg, x_dev, idx_np)
    _check_permute(cfg, x_dev, idx_np, out, lay)


# Batches that take the one-launch permute (more than 4096 assignments, at
# most 64 experts): ragged slices, expert counts that are not powers of two,
# k up to 8, capacity drops, a single expert, and a batch too large for one
# wave of CTAs (it falls back to the multi-launch path).
ONE_LAUNCH = {
    "e8_ragged": C["tiny"].with_(name="e8_ragged", T=3000, E=8, k=2, n_ep=4, d=256),
    "e48_k3": C["tiny"].with_(name="e48_k3", T=5000, E=48, k=3, n_ep=4, d=128),
    "e64_k8": C["tiny"].with_(name="e64_k8", T=4104, E=64, k=8, n_ep=8, d=64),
    "e16_cap": C["tiny"].with_(name="e16_cap", T=6000, E=16, k=2, n_ep=4, d=192, capacity=600),
    "e1": C["tiny"].with_(name="e1", T=5000, E=1, k=1, n_ep=1, d=64),
    "e128_k4": C["tiny"].with_(name="e128_k4", T=3000, E=128, k=4, n_ep=8, d=128),
    "e256_k8": C["tiny"].with_(name="e256_k8", T=4096, E=256, k=8, n_ep=64, d=64),
    "e256_cap": C["tiny"].with_(name="e256_cap", T=5008, E=256, k=4, n_ep=16, d=64, capacity=70),
    "fallback": C["tiny"].with_(name="fallback", T=80000, E=8, k=8, n_ep=8, d=64),
}


@pytest.mark.parametrize("name", list(ONE_LAUNCH))
def test_permute_one_launch_parity(m, name):
    cfg = ONE_LAUNCH[name]
    scores = synth.make_scores(cfg, seed=31)
    idx_np = oracle.select_experts(scores.numpy(), cfg.k, None, cfg.n_groups, cfg.topk_groups)
    x_dev = synth.make_x(cfg, device="cuda", seed=32)
    for _ in range(2):   # twice in a row: the grid barrier's words return to their start
        out, lay = _permute_case(m, cfg, x_dev, idx_np)
        _check_permute(cfg, x_dev, idx_np, out, lay)


def test_permute_one_launch_shared_workspace(m):
    """One workspace for one-launch permutes of several shapes, back to back.  The
    per-group slice counts alternate between two buffers (each call clears the
    other one), so every call must find its buffer zero whatever ran before."""
    names = ["e48_k3", "e16_cap", "e256_k8", "e8_ragged", "e64_k8", "e128_k4", "e48_k3", "e256_cap",
             "e64_k8", "e16_cap", "e1"]
    cfgs = [ONE_LAUNCH[n] for n in names]
    ws_bytes = max(m.moe_workspace_bytes(m.MoeCfg.from_layer(cfg)) for cfg in cfgs)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    m.moe_workspace_init(m.MoeCfg.from_layer(cfgs[0]), ws)
    i32 = torch.int32
    for i, cfg in enumerate(cfgs):
        c = m.MoeCfg.from_layer(cfg)
        scores = synth.make_scores(cfg, seed=40 + i)
        idx_np = oracle.select_experts(scores.numpy(), cfg.k)
        counts = torch.empty(cfg.E, dtype=i32, device="cuda")
        offsets = torch.empty(cfg.E + 1, dtype=i32, device="cuda")
        order = torch.empty(cfg.R, dtype=i32, device="cuda")
        inv = torch.empty(cfg.A, dtype=i32, device="cuda")
        idx = torch.from_numpy(idx_np.astype(np.int32)).cuda()
        m.moe_permute(c, None, idx, counts, offsets, order, inv, None, ws)
        torch.cuda.synchronize()
        ref = oracle.permute(idx_np, cfg.E, cfg.capacity)
        for key, t in (("counts", counts), ("offsets", offsets), ("order", order), ("inv", inv)):
            assert np.array_equal(npi(t), ref[key]), (names[i], i, key)
    assert m.moe_get_device_status(ws) == 0


def test_permute_one_launch_indices_only(m):
    cfg = ONE_LAUNCH["e16_cap"]
    scores = synth.make_scores(cfg, seed=33)
    idx_np = oracle.select_experts(scores.numpy(), cfg.k)
    c = m.MoeCfg.from_layer(cfg)
    i32 = torch.int32
    counts = torch.empty(cfg.E, dtype=i32, device="cuda")
    offsets = torch.empty(cfg.E + 1, dtype=i32, device="cuda")
    order = torch.empty(cfg.R, dtype=i32, device="cuda")
    inv = torch.empty(cfg.A, dtype=i32, device="cuda")
    ws = torch.zeros(m.moe_workspace_bytes(c), dtype=torch.uint8, device="cuda")
    m.moe_workspace_init(c, ws)
    idx = torch.from_numpy(idx_np.astype(np.int32)).cuda()
    m.moe_permute(c, None, idx, counts, offsets, order, inv, None, ws)
    torch.cuda.synchronize()
    ref = oracle.permute(idx_np, cfg.E, cfg.capacity)
    for key, t in (("counts", counts), ("offsets", offsets), ("order", order), ("inv", inv)):
        assert np.array_equal(npi(t), ref[key]), key
    assert m.moe_get_device_status(ws) == 0


def test_hand_dispatch_on_gpu(m):
    """The pages' two-GPU hand example, run through the CUDA path."""
    import json, os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_dispatch.json")))
    cfg = C["tiny"].with_(T=g["T"], E=g["E"], k=g["k"], n_ep=g["n_ep"], d=64)
    x_dev = synth.make_x(cfg, device="cuda")
    idx_np = np.array(g["topk_idx"])
    out, lay = _permute_case(m, cfg, x_dev, idx_np)
    assert npi(out["order"]).tolist() == g["order"]
    assert npi(out["inv"]).tolist() == g["inv"]
    assert npi(lay["C"]).tolist() == g["C"]
    assert npi(lay["send_idx"]).tolist() == g["send_idx"]
    assert npi(lay["send_off"]).tolist() == g["send_off"]
    assert npi(lay["recv_off"]).tolist() == g["recv_off"]


def test_hot_expert_capacity_drops(m):
    """Every token routed to expert 0 first: drops by token order."""
    cfg = C["tiny"].with_(T=512, E=8, k=2, n_ep=4, d=64, capacity=100)
    rng = np.random.default_rng(0)
    idx_np = np.stack([np.array([0, 1 + rng.integers(0, 7)]) for _ in range(cfg.T)])
    x_dev = synth.make_x(cfg, device="cuda")
    out, lay = _permute_case(m, cfg, x_dev, idx_np)
    _check_permute(cfg, x_dev, idx_np, out, lay)


# T = 64: the one-CTA index kernel; 2500: the one-launch permute; 2500 with
# 80 experts: the multi-launch path
@pytest.mark.parametrize("T,E", [(64, 8), (2500, 8), (2500, 80)])
def test_bad_expert_id_is_reported(m, T, E):
    cfg = C["tiny"].with_(T=T, E=E, k=2, n_ep=2, d=64)
    c = m.MoeCfg.from_layer(cfg)
    idx = torch.zeros(cfg.T, cfg.k, dtype=torch.int32)
    idx[:, 1] = 1
    idx[5, 0] = E
    idx[9, 1] = -1
    x = synth.make_x(cfg, device="cuda")
    i32 = torch.int32
    counts = torch.empty(cfg.E, dtype=i32, device="cuda")
    offsets = torch.empty(cfg.E + 1, dtype=i32, device="cuda")
    order = torch.empty(cfg.A, dtype=i32, device="cuda")
    inv = torch.empty(cfg.A, dtype=i32, device="cuda")
    xs = torch.empty(cfg.A, cfg.d, dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(m.moe_workspace_bytes(c), dtype=torch.uint8, device="cuda")
    m.moe_workspace_init(c, ws)
    m.moe_permute(c, x, idx.cuda(), counts, offsets, order, inv, xs, ws)
    assert m.moe_get_device_status(ws) == -7
    assert m.moe_get_device_status(ws) == 0          # read-and-clear
    inv = npi(inv)
    assert inv[5 * 2 + 0] == -1 and inv[9 * 2 + 1] == -1
    assert npi(counts).sum() == cfg.A - 2


# --------------------------------------------------------------------------
# Grouped FFN and the whole layer (from fp32 scores)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", list(SMALL))
def test_layer_parity_small(m, name):
    cfg = SMALL[name]
    x = synth.make_x(cfg)
    scores = synth.make_scores(cfg)
    W1, W3, W2 = synth.make_expert_weights(cfg)
    layer = run_path(m, cfg, x.cuda(), scores.cuda(), W1.cuda(), W3.cuda(), W2.cuda())
    y_ref, st = oracle.moe_forward(x.float().numpy(), scores.numpy(), cfg, W1.float().numpy(),
                                   W3.float().numpy(), W2.float().numpy())
    assert np.array_equal(npi(layer.topk_idx), st["idx"])
    assert np.array_equal(npi(layer.inv), st["perm"]["inv"])
    # expert outputs row by row (kept rows only)
    out_ref = oracle.expert_outputs(x.float().numpy(), st["perm"], cfg.k, W1.float().numpy(),
                                    W3.float().numpy(), W2.float().numpy())
    kept = np.nonzero(st["perm"]["order"] >= 0)[0]
    # kept rows only: capacity padding rows of y_sorted are never written
    assert_y_close(npf(layer.y_sorted[torch.from_numpy(kept).cuda()]), out_ref[kept])
    assert_y_close(npf(layer.y), y_ref)
    assert m.moe_get_device_status(layer.ws) == 0


def test_layer_is_deterministic(m):
    cfg = SMALL["ds_small"]
    x = synth.make_x(cfg, device="cuda")
    scores = synth.make_scores(cfg, device="cuda")
    W1, W3, W2 = synth.make_expert_weights(cfg, device="cuda")
    layer = m.MoELayer(cfg, W1, W3, W2)
    y1 = layer.forward(x, scores=scores).clone()
    y2 = layer.forward(x, scores=scores).clone()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


# --------------------------------------------------------------------------
# Router logits (step 1) against fp64
# --------------------------------------------------------------------------

def _logit_bound(x, W):
    """Forward error bound of an fp32 dot product of length d: d * u * sum|x_i w_i|."""
    d = x.shape[1]
    return d * 2.0 ** -24 * (np.abs(x) @ np.abs(W))


def _router_split(m, c, W_r_dev):
    split = torch.empty(3, c.E, c.d, dtype=torch.bfloat16, device="cuda")
    m.moe_pack_router(c, W_r_dev, split)
    return split


@pytest.mark.parametrize("name", ["tiny", "ds_small", "skew_small", "k_equals_E", "norm_softmax"])
@pytest.mark.parametrize("tc", [False, True])
def test_router_logits_parity(m, name, tc):
    """fp32 SIMT path: bound d*u*sum|x_i w_i|.  Tensor-core path: 3d exact
    products summed in fp32, bound 3*d*u*sum|x_i w_i|."""
    cfg = SMALL[name]
    x = synth.make_x(cfg)
    W_r, lb = synth.make_router(cfg)
    c = m.MoeCfg.from_layer(cfg)
    out = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device="cuda")
    W_dev = W_r.cuda()
    split = _router_split(m, c, W_dev) if tc else None
    m.moe_router_logits(c, x.cuda(), None if tc else W_dev, split,
                        None if lb is None else lb.cuda(), out)
    torch.cuda.synchronize()
    xf, Wf = x.float().numpy(), W_r.numpy()
    l_ref = oracle.router_logits(xf, Wf, None if lb is None else lb.numpy())
    bound = (3 if tc else 1) * _logit_bound(xf, Wf) + 1e-30
    got = npf(out)
    if cfg.score_fn == "sigmoid":
        s_ref = oracle.sigmoid(l_ref)
        assert (np.abs(got - s_ref) <= 0.25 * bound + 4e-7).all()
    else:
        if lb is not None:
            bound = bound + 2.0 ** -24 * np.abs(l_ref)
        assert (np.abs(got - l_ref) <= bound).all()
        assert np.median(np.abs(got - l_ref)) < 1e-5


@pytest.mark.parametrize("E,d,T,sig", [
    (1, 64, 1, False), (3, 192, 7, True), (4, 1088, 29, False), (5, 8256, 300, True),
    (8, 4160, 1000, False), (8, 8256, 9001, True), (13, 64, 61, False), (16, 2112, 4099, True),
    (16, 8256, 33, False)])
def test_router_logits_simt_shapes(m, E, d, T, sig):
    """The fp32 SIMT router (E <= 16) at the shapes its tiling has edges: d
    smaller than one column tile (idle warps), d over one or two tiles with a
    partial last tile, token counts that leave a ragged last batch and block,
    one token, one expert; with logit bias, and sigmoid scores."""
    g = torch.Generator().manual_seed(E * 100003 + d * 7 + T)
    cfg = C["tiny"].with_(T=T, d=d, E=E, k=1, n_ep=1, score_fn="sigmoid" if sig else "softmax",
                          norm_topk=int(sig))
    x = torch.randn(T, d, generator=g).bfloat16()
    W_r = (torch.randn(d, E, generator=g) / math.sqrt(d)).float()
    lb = (torch.randn(E, generator=g) * 0.5).float()
    c = m.MoeCfg.from_layer(cfg)
    out = torch.full((T, E), float("nan"), dtype=torch.float32, device="cuda")
    m.moe_router_logits(c, x.cuda(), W_r.cuda(), None, lb.cuda(), out)
    torch.cuda.synchronize()
    xf, Wf = x.float().numpy(), W_r.numpy()
    l_ref = oracle.router_logits(xf, Wf, lb.numpy())
    bound = _logit_bound(xf, Wf) + 2.0 ** -24 * np.abs(l_ref) + 1e-30
    got = npf(out)
    assert np.isfinite(got).all()
    if sig:
        assert (np.abs(got - oracle.sigmoid(l_ref)) <= 0.25 * bound + 4e-7).all()
    else:
        assert (np.abs(got - l_ref) <= bound).all()


@pytest.mark.parametrize("E,d,T,sig", [(256, 2048, 64, True), (64, 1024, 300, False),
                                       (256, 7168, 128, True), (32, 4096, 129, False)])
def test_router_tc_split_k(m, E, d, T, sig):
    """The tensor-core router with its K split into chunks (few output tiles:
    decode-sized batches) and the fixed-order reduction of the partials, with
    logit bias and sigmoid; against fp64 within the three-term bound.  The
    same call without a workspace takes the unsplit path; both must agree
    within twice the bound."""
    g = torch.Generator().manual_seed(E + d + T)
    cfg = C["dsv3"].with_(T=T, d=d, E=E, k=8, n_groups=1, topk_groups=1, n_ep=1,
                          score_fn="sigmoid" if sig else "softmax", norm_topk=int(sig),
                          has_shared=0)
    c = m.MoeCfg.from_layer(cfg)
    x = torch.randn(T, d, generator=g).bfloat16()
    W_r = (torch.randn(d, E, generator=g) / math.sqrt(d)).float()
    lb = (torch.randn(E, generator=g) * 0.5).float()
    split = _router_split(m, c, W_r.cuda())
    ws = torch.zeros(m.moe_workspace_bytes(c), dtype=torch.uint8, device="cuda")
    m.moe_workspace_init(c, ws)
    out = torch.full((T, E), float("nan"), dtype=torch.float32, device="cuda")
    out1 = torch.full((T, E), float("nan"), dtype=torch.float32, device="cuda")
    m.moe_router_logits(c, x.cuda(), None, split, lb.cuda(), out, ws)
    m.moe_router_logits(c, x.cuda(), None, split, lb.cuda(), out1)
    torch.cuda.synchronize()
    assert m.moe_get_device_status(ws) == 0
    xf, Wf = x.float().numpy(), W_r.numpy()
    l_ref = oracle.router_logits(xf, Wf, lb.numpy())
    bound = 3 * _logit_bound(xf, Wf) + 2.0 ** -24 * np.abs(l_ref) + 1e-30
    got, got1 = npf(out), npf(out1)
    assert np.isfinite(got).all() and np.isfinite(got1).all()
    ref = oracle.sigmoid(l_ref) if sig else l_ref
    scale = 0.25 if sig else 1.0
    assert (np.abs(got - ref) <= scale * bound + (4e-7 if sig else 0.0)).all()
    assert (np.abs(got - got1) <= 2 * scale * bound + (8e-7 if sig else 0.0)).all()


def test_router_split_is_exact(m):
    """hi + mid + lo reproduces every fp32 router weight exactly."""
    cfg = SMALL["ds_small"]
    W_r, _ = synth.make_router(cfg)
    c = m.MoeCfg.from_layer(cfg)
    split = _router_split(m, c, W_r.cuda()).double().cpu()
    recon = (split[0] + split[1] + split[2]).T.numpy()
    assert np.array_equal(recon, W_r.double().numpy())


def test_layer_from_tokens_with_router(m):
    """The whole path from x (router included).  Tokens whose fp64 top-k
    decision has a margin larger than the logit error bound must route
    exactly as the oracle does; their outputs must match."""
    cfg = SMALL["tiny"]
    x = synth.make_x(cfg)
    W_r, lb = synth.make_router(cfg)
    W1, W3, W2 = synth.make_expert_weights(cfg)
    layer = m.MoELayer(cfg, W1.cuda(), W3.cuda(), W2.cuda(), W_r=W_r.cuda(), logit_bias=None)
    layer.forward(x.cuda())
    torch.cuda.synchronize()
    xf = x.float().numpy()
    l_ref = oracle.router_logits(xf, W_r.numpy())
    srt = np.sort(l_ref, axis=1)[:, ::-1]
    margin = srt[:, cfg.k - 1] - srt[:, cfg.k]
    safe = margin > 4 * _logit_bound(xf, W_r.numpy()).max(1)
    assert safe.mean() > 0.95
    y_ref, st = oracle.moe_forward(xf, l_ref.astype(np.float32), cfg, W1.float().numpy(),
                                   W3.float().numpy(), W2.float().numpy())
    assert np.array_equal(npi(layer.topk_idx)[safe], st["idx"][safe])
    assert_y_close(npf(layer.y), y_ref, rows=np.nonzero(safe)[0])
