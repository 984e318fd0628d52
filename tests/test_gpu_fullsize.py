"""Parity at the full workload sizes, in the launch configuration the
benchmark times (the whole MoELayer path on one stream).  Routing, counts,
offsets, permutations and the EP layout are compared in full, bit for bit.
The grouped FFN is compared on rows drawn from every tile it computes: each
(expert, 128-row block) and each segment's last row, its hidden activations h
and outputs y_sorted against the fp64 expert; the layer output on tokens that
own those rows; the router logits on a seeded token sample."""
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


def stratified_rows(perm, seed, block=128):
    """Rows of the expert-grouped buffer that cover every tile: one seeded
    random kept row from every (expert, 128-row block) of each segment, and
    each segment's last kept row (where ragged tails and half tiles sit)."""
    rng = np.random.default_rng(seed)
    rows = []
    for e in range(perm["kept"].size):
        lo, kept = int(perm["offsets"][e]), int(perm["kept"][e])
        for b in range(0, kept, block):
            rows.append(lo + int(rng.integers(b, min(kept, b + block))))
        if kept:
            rows.append(lo + kept - 1)
    return np.unique(np.array(rows, np.int64))


# Rows compared per workload (each expert's segment, every 128-row block):
#   mixtral      8 experts x 8-9 blocks + last rows          ~ 80 rows
#   dsv3         256 experts x 2-3 blocks + last rows        ~ 800 rows (+ 3 shared)
#   dsv3_decode  ~250 non-empty experts x (1 block + last)   ~ 480 rows (+ 3 shared)
#   skew         64 experts x 3-5 blocks (capacity 640)      ~ 230 rows
# The layer output y is compared on up to 48 tokens that own compared rows (the
# first and last token included).
@pytest.mark.parametrize("name", ["mixtral", "dsv3", "dsv3_decode", "skew"])
def test_full_size_every_tile_against_oracle(m, name):
    cfg = synth.CONFIGS[name]
    dev = torch.device("cuda")
    x = synth.make_x(cfg, device=dev)
    scores = synth.make_scores(cfg, device=dev)
    W1, W3, W2 = synth.make_expert_weights(cfg, device=dev)
    layer = m.MoELayer(cfg, W1, W3, W2, device=dev)
    layer.forward(x, scores=scores)
    torch.cuda.synchronize()
    assert m.moe_get_device_status(layer.ws) == 0
    s_np = scores.cpu().numpy()
    x_np = x.float().cpu().numpy()
    # routing and permutation in full, bit-exact
    idx = oracle.select_experts(s_np, cfg.k, None, cfg.n_groups, cfg.topk_groups)
    perm = oracle.permute(idx, cfg.E, cfg.capacity)
    assert np.array_equal(npi(layer.topk_idx), idx)
    assert np.array_equal(npi(layer.counts), perm["counts"])
    assert np.array_equal(npi(layer.offsets), perm["offsets"])
    assert np.array_equal(npi(layer.inv), perm["inv"])
    lay = oracle.ep_layout(idx, perm["inv"], cfg.E, cfg.n_ep, cfg.T)
    assert np.array_equal(npi(layer.count_mat), lay["C"])
    assert np.array_equal(npi(layer.send_idx), lay["send_idx"])

    # every tile's rows: h and y_sorted against the fp64 expert
    rows = stratified_rows(perm, seed=5)
    h_ref, out_ref = oracle.expert_rows(x_np, perm, cfg.k, StreamedExperts(W1),
                                        StreamedExperts(W3), StreamedExperts(W2), rows)
    ridx = torch.from_numpy(rows).to(dev)
    assert_y_close(npf(layer.h[ridx]), h_ref)
    assert_y_close(npf(layer.y_sorted[ridx]), out_ref)
    if cfg.has_shared:
        tt = np.array([0, cfg.T // 2 + 1, cfg.T - 1])
        E = cfg.E
        sidx = torch.from_numpy(cfg.R + tt).to(dev)
        assert_y_close(npf(layer.h[sidx]),
                       oracle.swiglu_hidden(x_np[tt], npf(W1[E]), npf(W3[E])))
        assert_y_close(npf(layer.y_sorted[sidx]),
                       oracle.swiglu_expert(x_np[tt], npf(W1[E]), npf(W3[E]), npf(W2[E])))

    # the layer output on tokens that own compared rows
    owners = np.unique(perm["order"][rows] // cfg.k)
    rng = np.random.default_rng(6)
    tokens = np.unique(np.concatenate([rng.choice(owners, min(46, owners.size), replace=False),
                                       [0, cfg.T - 1]]))
    y_ref, _ = oracle.moe_forward(x_np, s_np, cfg, StreamedExperts(W1), StreamedExperts(W3),
                                  StreamedExperts(W2), tokens=tokens)
    tok = torch.from_numpy(tokens).to(dev)
    assert_y_close(npf(layer.y[tok]), y_ref[tokens])

    # the combine in GEMM 2's epilogue at full size: the same sampled tokens
    # against the oracle, and every token against the default path
    y_f = torch.empty_like(layer.y)
    m.moe_grouped_ffn_combine(layer.cfg, layer.x_sorted, x if cfg.has_shared else None,
                              layer.counts, layer.offsets, layer.W13, layer.W2, layer.h,
                              layer.order, layer.topk_gate, y_f, layer.ws)
    torch.cuda.synchronize()
    assert m.moe_get_device_status(layer.ws) == 0
    assert_y_close(npf(y_f[tok]), y_ref[tokens])
    err = (y_f.float() - layer.y.float()).abs().max().item()
    assert err <= 2e-2 * layer.y.float().abs().max().item()


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
