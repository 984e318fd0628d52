"""moe_permute_noalloc: the permute step for callers that cannot allocate
device memory (for example a runtime plugin that is handed only its input and
output tensors, or a serving loop where cudaMalloc could synchronise the
device).  It must produce exactly what moe_permute produces with a
caller-allocated workspace, call after call, although every call reuses the
library's one fixed scratch array."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

CASES = {
    "tiny": synth.CONFIGS["tiny"],
    "dsv3": synth.CONFIGS["dsv3"],
    "skew": synth.CONFIGS["skew"],
}


@pytest.fixture(scope="module")
def m():
    import expert_token_dispatch_moe_b300 as mod
    return mod


def _outputs(cfg):
    i32 = torch.int32
    return dict(counts=torch.empty(cfg.E, dtype=i32, device="cuda"),
                offsets=torch.empty(cfg.E + 1, dtype=i32, device="cuda"),
                order=torch.empty(cfg.R, dtype=i32, device="cuda"),
                inv=torch.empty(cfg.A, dtype=i32, device="cuda"),
                x_sorted=torch.empty(cfg.R, cfg.d, dtype=torch.bfloat16, device="cuda"))


def _inputs(cfg, seed):
    x = synth.make_x(cfg, device="cuda", seed=seed)
    scores = synth.make_scores(cfg, seed=100 + seed)
    idx = oracle.select_experts(scores.numpy(), cfg.k, None, cfg.n_groups, cfg.topk_groups)
    return x, torch.from_numpy(idx.astype(np.int32)).cuda()


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_permute_on_consecutive_calls(m, name):
    cfg = CASES[name]
    c = m.MoeCfg.from_layer(cfg)
    ws = torch.zeros(m.moe_workspace_bytes(c), dtype=torch.uint8, device="cuda")
    m.moe_workspace_init(c, ws)
    for seed in (0, 1):   # two calls in a row on different inputs
        x, idx = _inputs(cfg, seed)
        ref = _outputs(cfg)
        m.moe_permute(c, x, idx, ref["counts"], ref["offsets"], ref["order"], ref["inv"],
                      ref["x_sorted"], ws)
        got = _outputs(cfg)
        m.moe_permute_noalloc(c, x, idx, got["counts"], got["offsets"], got["order"],
                              got["inv"], got["x_sorted"])
        torch.cuda.synchronize()
        for key in ("counts", "offsets", "order", "inv"):
            assert torch.equal(got[key], ref[key]), (name, seed, key)
        assert torch.equal(got["x_sorted"].view(torch.int16), ref["x_sorted"].view(torch.int16))


def test_noalloc_rejects_configurations_beyond_its_scratch(m):
    # per-(rank, expert) counts alone need 1024 * 1024 * 4 B = 4 MiB > 1 MiB
    cfg = synth.CONFIGS["tiny"].with_(T=1024, E=1024, k=2, n_ep=1024, d=64)
    c = m.MoeCfg.from_layer(cfg)
    out = _outputs(cfg)
    x = torch.zeros(cfg.T, cfg.d, dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros(cfg.T, cfg.k, dtype=torch.int32, device="cuda")
    with pytest.raises(m.MoeError) as ei:
        m.moe_permute_noalloc(c, x, idx, out["counts"], out["offsets"], out["order"],
                              out["inv"], out["x_sorted"])
    assert ei.value.code == -9


def test_noalloc_indices_only_mode(m):
    """x and x_sorted both NULL: the indices alone, equal to moe_permute's in the
    same mode; one of the two alone is rejected as in moe_permute."""
    cfg = CASES["dsv3"]
    c = m.MoeCfg.from_layer(cfg)
    ws = torch.zeros(m.moe_workspace_bytes(c), dtype=torch.uint8, device="cuda")
    m.moe_workspace_init(c, ws)
    for seed in (2, 3):
        _, idx = _inputs(cfg, seed)
        ref, got = _outputs(cfg), _outputs(cfg)
        m.moe_permute(c, None, idx, ref["counts"], ref["offsets"], ref["order"], ref["inv"],
                      None, ws)
        m.moe_permute_noalloc(c, None, idx, got["counts"], got["offsets"], got["order"],
                              got["inv"], None)
        torch.cuda.synchronize()
        for key in ("counts", "offsets", "order", "inv"):
            assert torch.equal(got[key], ref[key]), (seed, key)
    with pytest.raises(m.MoeError) as ei:
        m.moe_permute_noalloc(c, None, idx, got["counts"], got["offsets"], got["order"],
                              got["inv"], got["x_sorted"])
    assert ei.value.code == -1
