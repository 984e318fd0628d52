"""The forward grouped FFN on SM pairs: tiles of 256 weight rows by up to 256
tokens, each CTA staging a power of two of the tile's tokens (the MMA's N is
twice that).  Segment lengths
chosen around every boundary of that rounding (0, 1, 15, 16, 17, ... 513 rows)
are routed through the layer and every row of h and y_sorted is compared with
the fp64 expert; the one-SM tiles (the training forward) give the same rows
within the same tolerance."""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu_util import LazyExperts, assert_y_close, npf, npi

pytestmark = pytest.mark.gpu

COUNTS = [0, 1, 15, 16, 17, 31, 33, 127, 128, 129, 240, 255, 256, 257, 272, 300, 383, 511, 513]


@pytest.fixture(scope="module")
def m():
    import expert_token_dispatch_moe_b300 as mod
    return mod


@pytest.fixture(autouse=True)
def pair_tiles(monkeypatch):
    """These layers are small; force the pair tiles (the choice is read at every call)."""
    monkeypatch.setenv("MOE_FFN_TILES", "pair")


def _one_hot_scores(counts, seed):
    """fp32 logits that send exactly counts[e] tokens to expert e (top-1), the
    tokens in a seeded random order."""
    ids = np.repeat(np.arange(len(counts)), counts)
    np.random.default_rng(seed).shuffle(ids)
    s = np.zeros((ids.size, len(counts)), np.float32)
    s[np.arange(ids.size), ids] = 4.0
    return torch.from_numpy(s)


@pytest.mark.parametrize("d,f,shared", [(256, 256, 0), (512, 384, 1), (192, 128, 0)])
def test_pair_tiles_every_tail_length(m, d, f, shared):
    counts = list(COUNTS)
    T = int(sum(counts))
    cfg = synth.LayerConfig("pair", T=T, d=d, E=len(counts), k=1, f=f, n_ep=1,
                            score_fn="softmax", norm_topk=0, has_shared=shared)
    dev = torch.device("cuda")
    x = synth.make_x(cfg, device=dev, seed=3)
    scores = _one_hot_scores(counts, seed=4).to(dev)
    W1, W3, W2 = synth.make_expert_weights(cfg, device=dev, seed=5)
    layer = m.MoELayer(cfg, W1, W3, W2, device=dev)
    layer.forward(x, scores=scores)
    torch.cuda.synchronize()
    assert m.moe_get_device_status(layer.ws) == 0
    assert npi(layer.counts).tolist() == counts
    idx = oracle.select_experts(scores.cpu().numpy(), 1)
    perm = oracle.permute(idx, cfg.E)
    rows = np.arange(cfg.A)
    x_np = x.float().cpu().numpy()
    h_ref, out_ref = oracle.expert_rows(x_np, perm, 1, LazyExperts(W1), LazyExperts(W3),
                                        LazyExperts(W2), rows)
    for e, c in enumerate(counts):   # every segment on its own scale
        lo = int(perm["offsets"][e])
        if c:
            assert_y_close(npf(layer.h[lo:lo + c]), h_ref[lo:lo + c])
            assert_y_close(npf(layer.y_sorted[lo:lo + c]), out_ref[lo:lo + c])
    if shared:
        E = cfg.E
        assert_y_close(npf(layer.h[cfg.R:]),
                       oracle.swiglu_hidden(x_np, npf(W1[E]), npf(W3[E])))
        assert_y_close(npf(layer.y_sorted[cfg.R:]),
                       oracle.swiglu_expert(x_np, npf(W1[E]), npf(W3[E]), npf(W2[E])))

    # the one-SM tiles on the same inputs: the training forward, and the forward
    # with the choice overridden
    os.environ["MOE_FFN_TILES"] = "single"
    h2 = torch.empty_like(layer.h)
    y2 = torch.empty_like(layer.y_sorted)
    m.moe_grouped_ffn(layer.cfg, layer.x_sorted, x if shared else None, layer.counts,
                      layer.offsets, layer.W13, layer.W2, h2, y2, layer.ws)
    os.environ["MOE_FFN_TILES"] = "pair"
    g1 = torch.empty(layer.h.shape[0], 2 * f, dtype=torch.bfloat16, device=dev)
    h1 = torch.empty_like(layer.h)
    y1 = torch.empty_like(layer.y_sorted)
    m.moe_grouped_ffn_train(layer.cfg, layer.x_sorted, x if shared else None, layer.counts,
                            layer.offsets, layer.W13, layer.W2, h1, y1, g1, layer.ws)
    torch.cuda.synchronize()
    assert_y_close(npf(layer.h), npf(h1))
    assert_y_close(npf(layer.y_sorted), npf(y1))
    assert torch.equal(h1.view(torch.int16), h2.view(torch.int16))
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_pair_tiles_leave_rows_outside_segments_untouched(m):
    """Rows past the kept rows (capacity padding) are not written."""
    cfg = synth.LayerConfig("pairpad", T=256, d=256, E=4, k=2, f=256, n_ep=1,
                            score_fn="softmax", norm_topk=0, capacity=100)
    dev = torch.device("cuda")
    x = synth.make_x(cfg, device=dev, seed=7)
    scores = synth.make_scores(cfg, device=dev, seed=8)
    W1, W3, W2 = synth.make_expert_weights(cfg, device=dev, seed=9)
    layer = m.MoELayer(cfg, W1, W3, W2, device=dev)
    layer.h.fill_(7.0)
    layer.y_sorted.fill_(7.0)
    layer.forward(x, scores=scores)
    torch.cuda.synchronize()
    kept = np.minimum(npi(layer.counts), cfg.capacity)
    for e in range(cfg.E):
        lo = e * cfg.capacity
        assert (npf(layer.h[lo + kept[e]:lo + cfg.capacity]) == 7.0).all()
        assert (npf(layer.y_sorted[lo + kept[e]:lo + cfg.capacity]) == 7.0).all()
