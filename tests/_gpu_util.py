"""Helpers shared by the GPU parity tests: run the CUDA path step by step
through the C ABI and fetch results as numpy arrays."""
import numpy as np
import torch

import synth

TOL_Y = 2e-2   # max|y - y_ref| <= TOL_Y * max|y_ref| (bf16 inputs, fp32 accumulation)


def npf(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def npi(t):
    return t.detach().cpu().numpy().astype(np.int64)


def dev_weights(cfg, seed=synth.WEIGHT_SEED):
    return synth.make_expert_weights(cfg, device="cuda", seed=seed)


def host_expert(W, e):
    """One expert's matrix as fp32 numpy (the oracle upcasts to fp64 itself)."""
    return W[e].float().cpu().numpy()


class LazyExperts:
    """Indexable view of device expert weights that copies one expert to the
    host on first use (so the oracle touches only the experts it needs)."""

    def __init__(self, W):
        self.W = W
        self.cache = {}

    def __getitem__(self, e):
        e = int(e)
        if e not in self.cache:
            self.cache[e] = host_expert(self.W, e)
        return self.cache[e]


def run_path(m, cfg, x, scores, W1, W3, W2, bias=None, with_send_buf=True):
    """Run route -> permute -> ep_layout -> grouped FFN -> combine on the GPU
    from fp32 scores; returns the MoELayer holding every intermediate."""
    layer = m.MoELayer(cfg, W1, W3, W2, selection_bias=bias, with_send_buf=with_send_buf)
    layer.forward(x, scores=scores)
    torch.cuda.synchronize()
    return layer


def assert_y_close(y, y_ref, rows=None, tol=TOL_Y):
    y = np.asarray(y, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    if rows is not None:
        y, y_ref = y[rows], y_ref[rows]
    err = np.abs(y - y_ref).max()
    scale = np.abs(y_ref).max()
    assert err <= tol * scale, f"max|y-y_ref| = {err:.4g} > {tol} * {scale:.4g}"
    return err / scale
