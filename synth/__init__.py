"""Seeded synthetic inputs for the MoE layer hot path.

This module is shared by the CUDA path's tests/benchmark and by the oracle's
tests.  It holds workload shapes and seeded random draws only: no step of the
layer (routing, permutation, expert FFN, combine) is computed here.

Workloads follow the shapes the expert-parallelism pages discuss: a tiny layer at
the scale of the pages' worked example, a Mixtral-8x7B-shaped layer, a
DeepSeek-V3-shaped layer (prefill and decode sizes) and a skewed,
capacity-limited layer.  Trained weights are not available, so every tensor is a
seeded random draw: activations x ~ N(0, 1) in bf16, expert weights ~ N(0, 1/d)
in bf16, router weights W_r ~ N(0, 1/d) in fp32 (so router logits are ~N(0, 1)).
"""
from __future__ import annotations

import dataclasses
import math

import torch

SOFTMAX = "softmax"
SIGMOID = "sigmoid"


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int              # tokens in the batch (all simulated ranks together)
    d: int              # hidden size
    E: int              # routed experts
    k: int              # experts per token
    f: int              # expert FFN width (d_e)
    n_ep: int           # simulated expert-parallel ranks
    score_fn: str       # "softmax" (gates from logits) or "sigmoid" (gates from scores)
    norm_topk: int      # 1: gates renormalised over the k chosen experts
    n_groups: int = 1   # group-limited routing: contiguous expert groups
    topk_groups: int = 1
    capacity: int = 0   # 0 = dropless; else rows kept per expert
    has_shared: int = 0  # one always-on shared expert of width f
    logit_bias_e0: float = 0.0  # constant added to expert 0's router logit

    @property
    def A(self) -> int:
        return self.T * self.k

    @property
    def R(self) -> int:
        """Rows of the expert-grouped buffer (dropless: T*k; capacity: E*cap)."""
        return self.E * self.capacity if self.capacity else self.T * self.k

    @property
    def T_loc(self) -> int:
        return self.T // self.n_ep

    def with_(self, **kw) -> "LayerConfig":
        return dataclasses.replace(self, **kw)


# The five workloads.  Capacity of the skewed layer: ceil(1.25 * 16384 * 2 / 64) = 640
# rows per expert (capacity factor 1.25 times the fair share T*k/E).
CONFIGS = {
    "tiny": LayerConfig("tiny", T=1024, d=256, E=8, k=2, f=512, n_ep=4,
                        score_fn=SOFTMAX, norm_topk=0),
    "mixtral": LayerConfig("mixtral", T=4096, d=4096, E=8, k=2, f=14336, n_ep=8,
                           score_fn=SOFTMAX, norm_topk=0),
    "dsv3": LayerConfig("dsv3", T=8192, d=7168, E=256, k=8, f=2048, n_ep=64,
                        score_fn=SIGMOID, norm_topk=1, n_groups=8, topk_groups=4,
                        has_shared=1),
    "dsv3_decode": LayerConfig("dsv3_decode", T=128, d=7168, E=256, k=8, f=2048, n_ep=64,
                               score_fn=SIGMOID, norm_topk=1, n_groups=8, topk_groups=4,
                               has_shared=1),
    "skew": LayerConfig("skew", T=16384, d=2048, E=64, k=2, f=1408, n_ep=8,
                        score_fn=SOFTMAX, norm_topk=0, capacity=640,
                        logit_bias_e0=4.5),
}

DATA_SEED = 0
WEIGHT_SEED = 1


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_x(cfg: LayerConfig, device="cpu", seed: int = DATA_SEED) -> torch.Tensor:
    """Token activations x, bf16 [T, d], entries ~ N(0, 1)."""
    g = _gen(seed, device)
    return torch.randn(cfg.T, cfg.d, generator=g, device=device,
                       dtype=torch.float32).to(torch.bfloat16)


def make_router(cfg: LayerConfig, device="cpu", seed: int = WEIGHT_SEED):
    """Router weights W_r fp32 [d, E] ~ N(0, 1/d) and the per-expert logit bias
    (fp32 [E]; all zero except expert 0 in the skewed workload), or None."""
    g = _gen(seed + 1000, device)
    W_r = torch.randn(cfg.d, cfg.E, generator=g, device=device,
                      dtype=torch.float32) * (1.0 / math.sqrt(cfg.d))
    bias = None
    if cfg.logit_bias_e0:
        bias = torch.zeros(cfg.E, dtype=torch.float32, device=device)
        bias[0] = cfg.logit_bias_e0
    return W_r, bias


def make_expert_weights(cfg: LayerConfig, device="cpu", seed: int = WEIGHT_SEED,
                        experts=None):
    """Expert weights in the natural (out, in) layout, bf16, entries ~ N(0, 1/d):
    W1, W3: [n, f, d]; W2: [n, d, f], n = E (+1 for the shared expert, stored last).

    `experts` optionally restricts the draw to a list of expert ids; each expert's
    matrices come from their own seeded stream, so a subset equals the
    corresponding slices of the full draw on the same device."""
    n = cfg.E + cfg.has_shared
    ids = list(range(n)) if experts is None else list(experts)
    std = 1.0 / math.sqrt(cfg.d)
    W1 = torch.empty(len(ids), cfg.f, cfg.d, dtype=torch.bfloat16, device=device)
    W3 = torch.empty(len(ids), cfg.f, cfg.d, dtype=torch.bfloat16, device=device)
    W2 = torch.empty(len(ids), cfg.d, cfg.f, dtype=torch.bfloat16, device=device)
    for i, e in enumerate(ids):
        g = _gen(seed * 1_000_003 + 7919 * (e + 1), device)
        W1[i] = (torch.randn(cfg.f, cfg.d, generator=g, device=device) * std).to(torch.bfloat16)
        W3[i] = (torch.randn(cfg.f, cfg.d, generator=g, device=device) * std).to(torch.bfloat16)
        W2[i] = (torch.randn(cfg.d, cfg.f, generator=g, device=device) * std).to(torch.bfloat16)
    return W1, W3, W2


def make_scores(cfg: LayerConfig, device="cpu", seed: int = DATA_SEED + 17,
                ties: bool = False) -> torch.Tensor:
    """Synthetic fp32 router scores [T, E] fed directly to the routing step.

    softmax workloads: logits ~ N(0, 1) (plus the expert-0 bias of the skewed
    workload); sigmoid workloads: affinities ~ U(0, 1).  With ties=True the values
    are drawn from a small grid (multiples of 1/4 or 1/16) so that equal scores,
    and signed zeros, occur often."""
    g = _gen(seed, device)
    if ties:
        if cfg.score_fn == SIGMOID:
            s = torch.randint(0, 17, (cfg.T, cfg.E), generator=g, device=device).float() / 16
        else:
            s = torch.randint(-8, 9, (cfg.T, cfg.E), generator=g, device=device).float() / 4
            sign = torch.randint(0, 2, (cfg.T, cfg.E), generator=g, device=device)
            s = torch.where((s == 0) & (sign == 1), torch.full_like(s, -0.0), s)
        return s.contiguous()
    if cfg.score_fn == SIGMOID:
        s = torch.rand(cfg.T, cfg.E, generator=g, device=device, dtype=torch.float32)
    else:
        s = torch.randn(cfg.T, cfg.E, generator=g, device=device, dtype=torch.float32)
        if cfg.logit_bias_e0:
            s[:, 0] += cfg.logit_bias_e0
    return s.contiguous()


def make_selection_bias(cfg: LayerConfig, device="cpu", seed: int = 23) -> torch.Tensor:
    """A per-expert fp32 selection bias (the auxiliary-loss-free balancing bias),
    drawn ~ 0.1 * N(0, 1)."""
    g = _gen(seed, device)
    return (torch.randn(cfg.E, generator=g, device=device) * 0.1).contiguous()


def sample_tokens(cfg: LayerConfig, n: int, seed: int = 99) -> torch.Tensor:
    """A seeded sorted subset of n token indices (always includes the first and
    last token, so both ends of the buffers are exercised)."""
    g = _gen(seed, "cpu")
    n = min(n, cfg.T)
    perm = torch.randperm(cfg.T, generator=g)[: max(0, n - 2)]
    s = torch.cat([perm, torch.tensor([0, cfg.T - 1])]).unique()
    return s.sort().values
