"""Parity of the load-balancing kernels with the oracle: the aux-loss-free bias
update, the replicate-then-pack plan and the dispatch over expert copies.
Every output is exact: the bias update is compared bit for bit after the one
fp64 -> fp32 rounding, plans and dispatches element by element."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu_util import npi

pytestmark = pytest.mark.gpu

C = synth.CONFIGS
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def m():
    import expert_token_dispatch_moe_b300 as mod
    return mod


def _i32(a):
    return torch.as_tensor(np.asarray(a, np.int32)).cuda()


def _plan_gpu(m, cfg, loads, slots):
    c = m.MoeCfg.from_layer(cfg)
    i32 = dict(dtype=torch.int32, device="cuda")
    out = dict(copies=torch.empty(cfg.E, **i32), copy_offset=torch.empty(cfg.E, **i32),
               copy_rank=torch.full((cfg.n_ep * slots,), -7, **i32),
               slot_expert=torch.empty(cfg.n_ep, slots, **i32),
               rank_load=torch.empty(cfg.n_ep, dtype=torch.float64, device="cuda"))
    m.moe_eplb_plan(c, _i32(loads), slots, out["copies"], out["copy_offset"], out["copy_rank"],
                    out["slot_expert"], out["rank_load"])
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def _check_plan(got, ref):
    assert got["copies"].tolist() == ref["copies"].tolist()
    assert got["copy_offset"].tolist() == ref["copy_offset"].tolist()
    n = int(ref["copies"].sum())
    assert got["copy_rank"][:n].tolist() == ref["copy_rank"].tolist()
    assert got["slot_expert"].tolist() == ref["slot_expert"].tolist()
    assert np.array_equal(got["rank_load"], ref["rank_load"])     # fp64, bit for bit


# --------------------------------------------------------------------------
# Bias update
# --------------------------------------------------------------------------

def _bias_gpu(m, cfg, counts, bias, lr):
    b = torch.as_tensor(np.asarray(bias, np.float32)).cuda()
    m.moe_bias_update(m.MoeCfg.from_layer(cfg), _i32(counts), lr, b)
    torch.cuda.synchronize()
    return b.cpu().numpy()


def test_bias_update_page_exercise(m):
    cfg = C["tiny"].with_(E=4, k=2, n_ep=4)
    lr = float(np.float32(2.0 ** -10))
    got = _bias_gpu(m, cfg, [100, 50, 200, 50], np.zeros(4), lr)
    assert got.tolist() == [0.0, 50 * lr, -100 * lr, 50 * lr]


@pytest.mark.parametrize("E", [8, 64, 256, 1000])
def test_bias_update_parity(m, E):
    rng = np.random.default_rng(E)
    cfg = C["tiny"].with_(E=E, k=2, n_ep=1)
    counts = rng.integers(0, 5000, size=E)
    bias = rng.normal(size=E).astype(np.float32)
    lr = float(np.float32(1e-3))
    got = _bias_gpu(m, cfg, counts, bias, lr)
    ref = oracle.bias_update(bias.astype(np.float64), counts, lr).astype(np.float32)
    assert np.array_equal(got, ref)


def test_bias_loop_balances_a_hot_expert(m):
    """The control loop on the skewed workload's router scores: route with the
    bias, count, update.  The hot expert's share falls from about half of all
    assignments toward the mean, and every update equals the oracle's."""
    cfg = C["skew"].with_(T=4096, capacity=0)
    c = m.MoeCfg.from_layer(cfg)
    x = synth.make_x(cfg)
    W_r, lb = synth.make_router(cfg)
    s = (oracle.router_logits(x.float().numpy(), W_r.numpy(), lb.numpy())).astype(np.float32)
    scores = torch.from_numpy(s).cuda()
    dev = "cuda"
    idx = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device=dev)
    gate = torch.empty(cfg.T, cfg.k, dtype=torch.float32, device=dev)
    counts = torch.empty(cfg.E, dtype=torch.int32, device=dev)
    offsets = torch.empty(cfg.E + 1, dtype=torch.int32, device=dev)
    order = torch.empty(cfg.A, dtype=torch.int32, device=dev)
    inv = torch.empty(cfg.A, dtype=torch.int32, device=dev)
    xs = torch.empty(cfg.A, cfg.d, dtype=torch.bfloat16, device=dev)
    ws = torch.zeros(m.moe_workspace_bytes(c), dtype=torch.uint8, device=dev)
    m.moe_workspace_init(c, ws)
    bias = torch.zeros(cfg.E, dtype=torch.float32, device=dev)
    x_dev = x.cuda()
    lr = float(np.float32(2.0 ** -12))
    shares = []
    for _ in range(30):
        m.moe_route(c, scores, bias, idx, gate)
        m.moe_permute(c, x_dev, idx, counts, offsets, order, inv, xs, ws)
        cnt = npi(counts)
        shares.append(cnt.max() / cfg.A)
        before = bias.cpu().numpy()
        m.moe_bias_update(c, counts, lr, bias)
        ref = oracle.bias_update(before.astype(np.float64), cnt, lr).astype(np.float32)
        assert np.array_equal(bias.cpu().numpy(), ref)
    assert m.moe_get_device_status(ws) == 0
    assert shares[0] > 0.45
    assert shares[-1] < 0.2 * shares[0]


# --------------------------------------------------------------------------
# Replicate then pack
# --------------------------------------------------------------------------

def test_eplb_plan_page_example(m):
    with open(os.path.join(GOLDEN, "eplb_example.json")) as fh:
        g = json.load(fh)
    cfg = C["tiny"].with_(E=8, k=2, n_ep=4)
    got = _plan_gpu(m, cfg, g["loads"], 3)
    assert got["rank_load"].tolist() == g["greedy_gpu_loads"]
    _check_plan(got, oracle.eplb_plan(g["loads"], 4, 3))


@pytest.mark.parametrize("case", range(8))
def test_eplb_plan_parity(m, case):
    rng = np.random.default_rng(1000 + case)
    E, n = [(8, 4), (64, 8), (256, 64), (256, 64), (32, 32), (1000, 8), (16, 2), (256, 8)][case]
    slots = E // n + [1, 2, 1, 3, 4, 0, 5, 1][case]
    if case in (2, 6):                        # many ties: equal loads and zeros
        loads = rng.integers(0, 4, size=E) * 16
    elif case == 5:
        loads = np.zeros(E, np.int64)
    else:
        loads = rng.integers(0, 600, size=E)
        loads[rng.integers(0, E, size=3)] += 5000
    cfg = C["tiny"].with_(E=E, k=2, n_ep=n)
    _check_plan(_plan_gpu(m, cfg, loads, slots), oracle.eplb_plan(loads, n, slots))


def test_eplb_plan_rejects_too_few_slots(m):
    cfg = C["tiny"].with_(E=8, k=2, n_ep=4)
    with pytest.raises(m.MoeError):
        _plan_gpu(m, cfg, np.ones(8), 1)


# --------------------------------------------------------------------------
# Dispatch over the copies
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["ds_small", "skew_small", "dsv3"])
def test_eplb_dispatch_parity(m, name):
    cfg = {"ds_small": C["dsv3"].with_(name="ds_small", T=512, d=256, f=256, E=64, n_ep=16),
           "skew_small": C["skew"].with_(name="skew_small", T=2048, d=256, f=256, E=16, n_ep=8,
                                         capacity=oracle.capacity_rows(1.25, 2048, 2, 16)),
           "dsv3": C["dsv3"]}[name]
    c = m.MoeCfg.from_layer(cfg)
    scores = synth.make_scores(cfg)
    if name == "skew_small":
        scores[:, 0] += 4.5                   # one hot expert: drops and copies
    idx_np = oracle.select_experts(scores.numpy(), cfg.k, None, cfg.n_groups, cfg.topk_groups)
    p = oracle.permute(idx_np, cfg.E, cfg.capacity)
    kept = np.minimum(p["counts"], cfg.capacity) if cfg.capacity else p["counts"]
    slots = cfg.E // cfg.n_ep + 2
    plan = oracle.eplb_plan(kept, cfg.n_ep, slots)
    dest_ref, C_ref = oracle.eplb_dispatch(idx_np, p["inv"], p["offsets"], p["counts"], plan,
                                           cfg.n_ep, cfg.T, cfg.capacity)
    # the GPU plan from the GPU's own permute counts, then the GPU dispatch
    dev = "cuda"
    x = synth.make_x(cfg, device=dev)
    i32 = dict(dtype=torch.int32, device=dev)
    idx = _i32(idx_np)
    counts, offsets = torch.empty(cfg.E, **i32), torch.empty(cfg.E + 1, **i32)
    order, inv = torch.empty(cfg.R, **i32), torch.empty(cfg.A, **i32)
    xs = torch.empty(cfg.R, cfg.d, dtype=torch.bfloat16, device=dev)
    ws = torch.zeros(m.moe_workspace_bytes(c), dtype=torch.uint8, device=dev)
    m.moe_workspace_init(c, ws)
    m.moe_permute(c, x, idx, counts, offsets, order, inv, xs, ws)
    loads = torch.clamp(counts, max=cfg.capacity) if cfg.capacity else counts
    got = _plan_gpu(m, cfg, loads.cpu().numpy(), slots)
    _check_plan(got, plan)
    dest = torch.empty(cfg.A, **i32)
    Cm = torch.empty(cfg.n_ep, cfg.n_ep, **i32)
    m.moe_eplb_dispatch(c, idx, counts, offsets, inv, _i32(got["copies"]), _i32(got["copy_offset"]),
                        _i32(got["copy_rank"]), dest, Cm)
    torch.cuda.synchronize()
    assert npi(dest).tolist() == dest_ref.tolist()
    assert np.array_equal(npi(Cm), C_ref)
