"""The per-token loop oracle (moe_loop.c) from Python: the layer's definition
restated one token at a time in plain C, fp64, as a second statement beside
the vectorised numpy oracle.  TEST INFRASTRUCTURE ONLY (see the package
docstring): only the tests, the package's smoke check and the benchmark's
CPU-baseline leg may use it.

The C source is compiled with gcc into oracle/_build/ on first use (and by the
repository's build entry point); it is rebuilt when the source is newer than
the library.  Arguments are marshalled here; every step of the arithmetic runs
in the C file.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_loop.c")
LIB = os.path.join(HERE, "_build", "libmoe_loop.so")
# no fast-math, no FMA contraction: the selection's fp32 additions must stay
# single, correctly rounded operations
CFLAGS = ["-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
          "-std=c11", "-Wall", "-Wextra"]

_lock = threading.Lock()
_lib = None

_I32 = ctypes.c_int
_P = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile moe_loop.c into oracle/_build/libmoe_loop.so (skipped when up to date)."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("no C compiler found for the per-token loop oracle")
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    tmp = f"{LIB}.{os.getpid()}.tmp"
    res = subprocess.run([cc, *CFLAGS, "-o", tmp, SRC, "-lm"], capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("gcc failed on moe_loop.c:\n" + res.stderr[-4000:])
    os.replace(tmp, LIB)
    return LIB


_SIGNATURES = {
    "loop_router_logits": [_I32, _I32, _I32, _P, _P, _P, _P],
    "loop_select": [_I32, _I32, _I32, _P, _P, _I32, _I32, _P],
    "loop_gates": [_I32, _I32, _I32, _P, _P, _I32, _I32, _P],
    "loop_permute": [_I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P],
    "loop_ep_layout": [_I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P],
    "loop_layer_tokens": [_I32] * 7 + [_P] * 6 + [_I32, _P, _P, _P],
}


def load(path):
    """A library built from moe_loop.c at `path`, with its argument types set."""
    h = ctypes.CDLL(path)
    for name, args in _SIGNATURES.items():
        fn = getattr(h, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    return h


def lib():
    """The loaded library (built first if needed)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = load(build())
    return _lib


def _c(a, dtype):
    """A C-contiguous array of `dtype` (copied only when needed)."""
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def _p(a):
    return None if a is None else a.ctypes.data


def _ok(rc, what):
    if rc != 0:
        raise ValueError(f"{what}: rejected its arguments")


def router_logits(x, W_r, logit_bias=None):
    """fp64 [T, E] router logits of fp32 x [T, d] (bf16 values) and W_r [d, E]."""
    x, W_r = _c(x, np.float32), _c(W_r, np.float32)
    T, d = x.shape
    E = W_r.shape[1]
    lb = None if logit_bias is None else _c(logit_bias, np.float32)
    out = np.empty((T, E), np.float64)
    _ok(lib().loop_router_logits(T, d, E, _p(x), _p(W_r), _p(lb), _p(out)), "router_logits")
    return out


def select_experts(scores, k, bias=None, n_groups=1, topk_groups=1):
    """int32 [T, k] expert choice per token in rank order (fp32 selection rules)."""
    s = _c(scores, np.float32)
    T, E = s.shape
    b = None if bias is None else _c(bias, np.float32)
    idx = np.empty((T, k), np.int32)
    _ok(lib().loop_select(T, E, k, _p(s), _p(b), n_groups, topk_groups, _p(idx)),
        "select_experts")
    return idx


def gate_weights(scores, idx, score_fn, norm_topk):
    """fp64 [T, k] gates: softmax over all E, or the sigmoid affinity; optionally
    normalised over the k chosen."""
    s = _c(scores, np.float32)
    idx = _c(idx, np.int32)
    T, E = s.shape
    k = idx.shape[1]
    fn = {"softmax": 0, "sigmoid": 1}[score_fn]
    g = np.empty((T, k), np.float64)
    _ok(lib().loop_gates(T, E, k, _p(s), _p(idx), fn, int(norm_topk), _p(g)), "gate_weights")
    return g


def permute(idx, E, capacity=0):
    """Counting-sort grouping: dict of int32 counts [E], offsets [E+1], order [R],
    inv [A], kept [E]."""
    idx = _c(idx, np.int32)
    T, k = idx.shape
    A = T * k
    R = E * capacity if capacity else A
    out = {"counts": np.empty(E, np.int32), "offsets": np.empty(E + 1, np.int32),
           "order": np.empty(R, np.int32), "inv": np.empty(A, np.int32),
           "kept": np.empty(E, np.int32)}
    _ok(lib().loop_permute(T, k, E, capacity, _p(idx), _p(out["counts"]), _p(out["offsets"]),
                           _p(out["order"]), _p(out["inv"]), _p(out["kept"])), "permute")
    return out


def ep_layout(idx, inv, E, n_ep):
    """Send layout by literal (destination, expert, a) loops: dict of int32 C,
    send_off, recv_off [n_ep, n_ep] and send_idx [A]."""
    idx = _c(idx, np.int32)
    inv = _c(inv, np.int32)
    T, k = idx.shape
    out = {"C": np.empty((n_ep, n_ep), np.int32), "send_off": np.empty((n_ep, n_ep), np.int32),
           "recv_off": np.empty((n_ep, n_ep), np.int32), "send_idx": np.empty(T * k, np.int32)}
    _ok(lib().loop_ep_layout(T, k, E, n_ep, _p(idx), _p(inv), _p(out["C"]), _p(out["send_off"]),
                             _p(out["recv_off"]), _p(out["send_idx"])), "ep_layout")
    return out


def layer_tokens(x, idx, gates, cfg, W1, W3, W2, tokens, with_h=False):
    """Layer output of the given tokens, one token at a time: fp64 [n, d] (and,
    with with_h, the hidden activations fp64 [n, k + has_shared, f]).

    W1, W3: [E + has_shared, f, d]; W2: [E + has_shared, d, f]; bf16 values as
    fp32 (numpy arrays, or torch tensors converted here)."""
    x = _c(_np(x), np.float32)
    idx = _c(idx, np.int32)
    gates = _c(gates, np.float64)
    W1, W3, W2 = (_c(_np(w), np.float32) for w in (W1, W3, W2))
    tokens = _c(tokens, np.int32).reshape(-1)
    T, d = x.shape
    E, k, f, sh = cfg.E, cfg.k, cfg.f, int(cfg.has_shared)
    if W1.shape != (E + sh, f, d) or W3.shape != W1.shape or W2.shape != (E + sh, d, f):
        raise ValueError("expert weight shapes do not match the layer")
    y = np.empty((tokens.size, d), np.float64)
    h = np.empty((tokens.size, k + sh, f), np.float64) if with_h else None
    _ok(lib().loop_layer_tokens(T, d, E, k, f, sh, int(cfg.capacity), _p(x), _p(idx), _p(gates),
                                _p(W1), _p(W3), _p(W2), tokens.size, _p(tokens), _p(y), _p(h)),
        "layer_tokens")
    return (y, h) if with_h else y


def _np(a):
    """numpy view of a CPU torch tensor (bf16 upcast to fp32), else the array."""
    if hasattr(a, "detach"):
        t = a.detach()
        if t.device.type != "cpu":
            t = t.cpu()
        return t.float().numpy()
    return a


def forward(x, scores, cfg, W1, W3, W2, bias=None, tokens=None):
    """The layer, token by token: selection on the fp32 scores, gates, and the
    outputs of `tokens` (all tokens when None).  Returns (y fp64 [n, d], idx,
    gates)."""
    idx = select_experts(scores, cfg.k, bias, cfg.n_groups, cfg.topk_groups)
    g = gate_weights(scores, idx, cfg.score_fn, cfg.norm_topk)
    if tokens is None:
        tokens = np.arange(cfg.T)
    y = layer_tokens(x, idx, g, cfg, W1, W3, W2, tokens)
    return y, idx, g
