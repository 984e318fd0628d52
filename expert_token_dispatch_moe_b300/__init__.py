"""B300-native single-device MoE layer hot path.

Python binding of libmoe.so (C ABI, declared in include/moe.h): argument
marshalling only.  Every step of the layer runs in the library's CUDA kernels;
torch supplies device memory and streams.  There is no CPU fallback: importing
this package fails if libmoe.so is missing, and every call raises MoeError when
the library reports an error (including "no sm_103 device").
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python expert_token_dispatch_moe_b300/build.py`"
        " (there is no fallback implementation)")
_lib = ctypes.CDLL(LIB_PATH)

MOE_SOFTMAX, MOE_SIGMOID = 0, 1
ERRORS = {
    0: "MOE_OK", -1: "MOE_E_NULL", -2: "MOE_E_SHAPE", -3: "MOE_E_ALIGN", -4: "MOE_E_WORKSPACE",
    -5: "MOE_E_CUDA", -6: "MOE_E_DEVICE", -7: "MOE_E_DEVICE_DATA", -8: "MOE_E_DEVICE_TIMEOUT",
    -9: "MOE_E_SCRATCH_LIMIT",
}
EXPORTS = ("moe_validate_cfg", "moe_grouped_rows", "moe_workspace_bytes", "moe_workspace_init",
           "moe_pack_router", "moe_router_logits", "moe_route", "moe_permute", "moe_permute_noalloc",
           "moe_ep_layout", "moe_ep_layout_fp8", "moe_dispatch_recv_fp8", "moe_pack_w13",
           "moe_grouped_ffn", "moe_ffn_pair_tiles", "moe_grouped_ffn_combine", "moe_grouped_ffn_gather", "moe_grouped_ffn_train", "moe_combine", "moe_bias_update", "moe_eplb_plan",
           "moe_eplb_dispatch", "moe_pack_backward", "moe_combine_backward",
           "moe_backward_workspace_bytes", "moe_grouped_ffn_backward", "moe_permute_backward",
           "moe_selftest_wait_timeout", "moe_get_device_status", "moe_strerror",
           "moe_last_launch_count", "moe_layer_forward", "moe_layer_forward_host")


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = _lib.moe_strerror(code).decode()
        super().__init__(f"{where}: {ERRORS.get(code, code)} ({msg})")


class MoeCfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("T", "d", "E", "k", "f", "n_ep", "score_fn", "norm_topk", "n_groups",
                 "topk_groups", "capacity", "has_shared")]

    @classmethod
    def from_layer(cls, lc) -> "MoeCfg":
        """From any object with the layer-configuration attributes (T, d, E, k,
        f, n_ep, score_fn as "softmax"/"sigmoid" or 0/1, norm_topk, n_groups,
        topk_groups, capacity, has_shared)."""
        sf = lc.score_fn
        if isinstance(sf, str):
            sf = {"softmax": MOE_SOFTMAX, "sigmoid": MOE_SIGMOID}[sf]
        return cls(lc.T, lc.d, lc.E, lc.k, lc.f, lc.n_ep, sf, lc.norm_topk, lc.n_groups,
                   lc.topk_groups, lc.capacity, lc.has_shared)

    @property
    def A(self):
        return self.T * self.k

    @property
    def R(self):
        return self.E * self.capacity if self.capacity else self.T * self.k


_P = ctypes.c_void_p
_CFG = ctypes.POINTER(MoeCfg)


class MoeLayerBufs(ctypes.Structure):
    """struct moe_layer: the layer's weights and step buffers (device pointers)."""
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("W_r", "W_r_split", "logit_bias", "selection_bias", "W13", "W2", "scores",
                 "topk_idx", "topk_gate", "counts", "offsets", "order", "inv", "x_sorted",
                 "count_mat", "send_off", "recv_off", "send_idx", "send_buf", "h", "y_sorted",
                 "ws")] + [("ws_bytes", ctypes.c_size_t), ("combine_in_epilogue", ctypes.c_int32),
                           ("gather", ctypes.c_int32)]

    @classmethod
    def of(cls, combine_in_epilogue=False, gather=False, **tensors) -> "MoeLayerBufs":
        b = cls()
        for name, _ in cls._fields_[:-3]:
            setattr(b, name, _ptr(tensors.get(name)))
        ws = tensors.get("ws")
        b.ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
        b.combine_in_epilogue = 1 if combine_in_epilogue else 0
        b.gather = 1 if gather else 0
        return b


_LAYER = ctypes.POINTER(MoeLayerBufs)
_SZ = ctypes.c_size_t
_sig = {
    "moe_validate_cfg": (ctypes.c_int, [_CFG]),
    "moe_grouped_rows": (ctypes.c_int64, [_CFG]),
    "moe_workspace_bytes": (_SZ, [_CFG]),
    "moe_workspace_init": (ctypes.c_int, [_CFG, _P, _SZ, _P]),
    "moe_pack_router": (ctypes.c_int, [_CFG, _P, _P, _P]),
    "moe_router_logits": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_route": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P]),
    "moe_permute": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_permute_noalloc": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_ep_layout": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_ep_layout_fp8": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                                         _P]),
    "moe_dispatch_recv_fp8": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P]),
    "moe_pack_w13": (ctypes.c_int, [_CFG, _P, _P, _P, _P]),
    "moe_grouped_ffn": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_ffn_pair_tiles": (ctypes.c_int, [_CFG]),
    "moe_grouped_ffn_combine": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                               _SZ, _P]),
    "moe_grouped_ffn_gather": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                                              _P]),
    "moe_combine": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P]),
    "moe_bias_update": (ctypes.c_int, [_CFG, _P, ctypes.c_float, _P, _P]),
    "moe_eplb_plan": (ctypes.c_int, [_CFG, _P, ctypes.c_int32, _P, _P, _P, _P, _P, _P]),
    "moe_eplb_dispatch": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_pack_backward": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P]),
    "moe_combine_backward": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P]),
    "moe_backward_workspace_bytes": (_SZ, [_CFG]),
    "moe_grouped_ffn_backward": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                                _P, _P, _P, _P, _SZ, _P, _SZ, _P]),
    "moe_grouped_ffn_train": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                                             _P]),
    "moe_permute_backward": (ctypes.c_int, [_CFG, _P, _P, _P, _P]),
    "moe_selftest_wait_timeout": (ctypes.c_int, [_P, ctypes.c_uint64, _P]),
    "moe_get_device_status": (ctypes.c_int, [_P, _P]),
    "moe_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_last_launch_count": (ctypes.c_int, []),
    "moe_layer_forward": (ctypes.c_int, [_CFG, _LAYER, _P, _P, _P]),
    "moe_layer_forward_host": (ctypes.c_int, [_CFG, _LAYER, ctypes.c_int,
                                              ctypes.POINTER(_P), ctypes.POINTER(_P),
                                              ctypes.POINTER(_P), ctypes.POINTER(_P),
                                              _P, _P, _P]),
}
for _name, (_res, _args) in _sig.items():
    _fn = getattr(_lib, _name)
    _fn.restype, _fn.argtypes = _res, _args


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, where: str):
    if rc != 0:
        raise MoeError(rc, where)


def _ws(ws):
    return _ptr(ws), (ws.numel() * ws.element_size() if isinstance(ws, torch.Tensor) else 0)


# ----------------------------------------------------------------------------
# One wrapper per C entry point, same names and argument order.
# ----------------------------------------------------------------------------

def moe_validate_cfg(cfg: MoeCfg) -> int:
    return _lib.moe_validate_cfg(ctypes.byref(cfg))


def moe_grouped_rows(cfg: MoeCfg) -> int:
    return _lib.moe_grouped_rows(ctypes.byref(cfg))


def moe_ffn_pair_tiles(cfg: MoeCfg) -> bool:
    """True when moe_grouped_ffn takes SM-pair tiles for cfg (MOE_FFN_TILES read now)."""
    rc = _lib.moe_ffn_pair_tiles(ctypes.byref(cfg))
    _check(min(rc, 0), "moe_ffn_pair_tiles")
    return rc == 1


def moe_workspace_bytes(cfg: MoeCfg) -> int:
    return _lib.moe_workspace_bytes(ctypes.byref(cfg))


def moe_workspace_init(cfg, ws, stream=None):
    p, n = _ws(ws)
    _check(_lib.moe_workspace_init(ctypes.byref(cfg), p, n, _stream(stream)), "moe_workspace_init")


def moe_pack_router(cfg, W_r, W_r_split, stream=None):
    _check(_lib.moe_pack_router(ctypes.byref(cfg), _ptr(W_r), _ptr(W_r_split), _stream(stream)),
           "moe_pack_router")


def moe_router_logits(cfg, x, W_r, W_r_split, logit_bias, scores, ws=None, stream=None):
    p, n = _ws(ws)
    _check(_lib.moe_router_logits(ctypes.byref(cfg), _ptr(x), _ptr(W_r), _ptr(W_r_split),
                                  _ptr(logit_bias), _ptr(scores), p, n, _stream(stream)),
           "moe_router_logits")


def moe_route(cfg, scores, bias, topk_idx, topk_gate, stream=None):
    _check(_lib.moe_route(ctypes.byref(cfg), _ptr(scores), _ptr(bias), _ptr(topk_idx),
                          _ptr(topk_gate), _stream(stream)), "moe_route")


def moe_permute(cfg, x, topk_idx, counts, offsets, order, inv, x_sorted, ws, stream=None):
    p, n = _ws(ws)
    _check(_lib.moe_permute(ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(counts),
                            _ptr(offsets), _ptr(order), _ptr(inv), _ptr(x_sorted), p, n,
                            _stream(stream)), "moe_permute")


def moe_permute_noalloc(cfg, x, topk_idx, counts, offsets, order, inv, x_sorted, stream=None):
    """moe_permute for callers that cannot allocate: no workspace argument, the
    library's fixed device scratch is used (calls must not overlap on the GPU)."""
    _check(_lib.moe_permute_noalloc(ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(counts),
                                    _ptr(offsets), _ptr(order), _ptr(inv), _ptr(x_sorted),
                                    _stream(stream)), "moe_permute_noalloc")


def moe_ep_layout(cfg, topk_idx, offsets, inv, count_mat, send_off, recv_off, send_idx, x,
                  send_buf, ws, stream=None):
    p, n = _ws(ws)
    _check(_lib.moe_ep_layout(ctypes.byref(cfg), _ptr(topk_idx), _ptr(offsets), _ptr(inv),
                              _ptr(count_mat), _ptr(send_off), _ptr(recv_off), _ptr(send_idx),
                              _ptr(x), _ptr(send_buf), p, n, _stream(stream)), "moe_ep_layout")


def moe_ep_layout_fp8(cfg, topk_idx, offsets, inv, count_mat, send_off, recv_off, send_idx, x,
                      send_fp8, send_scale, ws, stream=None):
    p, n = _ws(ws)
    _check(_lib.moe_ep_layout_fp8(ctypes.byref(cfg), _ptr(topk_idx), _ptr(offsets), _ptr(inv),
                                  _ptr(count_mat), _ptr(send_off), _ptr(recv_off),
                                  _ptr(send_idx), _ptr(x), _ptr(send_fp8), _ptr(send_scale), p, n,
                                  _stream(stream)), "moe_ep_layout_fp8")


def moe_dispatch_recv_fp8(cfg, send_fp8, send_scale, send_idx, inv, x_sorted, stream=None):
    _check(_lib.moe_dispatch_recv_fp8(ctypes.byref(cfg), _ptr(send_fp8), _ptr(send_scale),
                                      _ptr(send_idx), _ptr(inv), _ptr(x_sorted), _stream(stream)),
           "moe_dispatch_recv_fp8")


def moe_pack_w13(cfg, W1, W3, W13, stream=None):
    _check(_lib.moe_pack_w13(ctypes.byref(cfg), _ptr(W1), _ptr(W3), _ptr(W13), _stream(stream)),
           "moe_pack_w13")


def moe_grouped_ffn(cfg, x_sorted, x, counts, offsets, W13, W2, h, y_sorted, ws, stream=None):
    p, n = _ws(ws)
    _check(_lib.moe_grouped_ffn(ctypes.byref(cfg), _ptr(x_sorted), _ptr(x), _ptr(counts),
                                _ptr(offsets), _ptr(W13), _ptr(W2), _ptr(h), _ptr(y_sorted), p, n,
                                _stream(stream)), "moe_grouped_ffn")


def moe_grouped_ffn_gather(cfg, x, order, counts, offsets, W13, W2, h, y_sorted, ws, stream=None):
    p, n = _ws(ws)
    _check(_lib.moe_grouped_ffn_gather(ctypes.byref(cfg), _ptr(x), _ptr(order), _ptr(counts),
                                       _ptr(offsets), _ptr(W13), _ptr(W2), _ptr(h),
                                       _ptr(y_sorted), p, n, _stream(stream)),
           "moe_grouped_ffn_gather")


def moe_grouped_ffn_combine(cfg, x_sorted, x, counts, offsets, W13, W2, h, order, topk_gate, y, ws,
                            stream=None):
    p, n = _ws(ws)
    _check(_lib.moe_grouped_ffn_combine(ctypes.byref(cfg), _ptr(x_sorted), _ptr(x), _ptr(counts),
                                        _ptr(offsets), _ptr(W13), _ptr(W2), _ptr(h), _ptr(order),
                                        _ptr(topk_gate), _ptr(y), p, n, _stream(stream)),
           "moe_grouped_ffn_combine")


def moe_combine(cfg, y_sorted, inv, topk_gate, y, stream=None):
    _check(_lib.moe_combine(ctypes.byref(cfg), _ptr(y_sorted), _ptr(inv), _ptr(topk_gate), _ptr(y),
                            _stream(stream)), "moe_combine")


def moe_bias_update(cfg, counts, lr, bias, stream=None):
    _check(_lib.moe_bias_update(ctypes.byref(cfg), _ptr(counts), float(lr), _ptr(bias),
                                _stream(stream)), "moe_bias_update")


def moe_eplb_plan(cfg, loads, slots_per_rank, copies, copy_offset, copy_rank, slot_expert,
                  rank_load, stream=None):
    _check(_lib.moe_eplb_plan(ctypes.byref(cfg), _ptr(loads), int(slots_per_rank), _ptr(copies),
                              _ptr(copy_offset), _ptr(copy_rank), _ptr(slot_expert),
                              _ptr(rank_load), _stream(stream)), "moe_eplb_plan")


def moe_eplb_dispatch(cfg, topk_idx, counts, offsets, inv, copies, copy_offset, copy_rank,
                      dest_rank, count_mat, stream=None):
    _check(_lib.moe_eplb_dispatch(ctypes.byref(cfg), _ptr(topk_idx), _ptr(counts), _ptr(offsets),
                                  _ptr(inv), _ptr(copies), _ptr(copy_offset), _ptr(copy_rank),
                                  _ptr(dest_rank), _ptr(count_mat), _stream(stream)),
           "moe_eplb_dispatch")


def moe_pack_backward(cfg, W13, W2, W13t, W2t, stream=None):
    _check(_lib.moe_pack_backward(ctypes.byref(cfg), _ptr(W13), _ptr(W2), _ptr(W13t), _ptr(W2t),
                                  _stream(stream)), "moe_pack_backward")


def moe_combine_backward(cfg, dy, y_sorted, inv, topk_gate, d_o, dgate, stream=None):
    _check(_lib.moe_combine_backward(ctypes.byref(cfg), _ptr(dy), _ptr(y_sorted), _ptr(inv),
                                     _ptr(topk_gate), _ptr(d_o), _ptr(dgate), _stream(stream)),
           "moe_combine_backward")


def moe_backward_workspace_bytes(cfg) -> int:
    return _lib.moe_backward_workspace_bytes(ctypes.byref(cfg))


def moe_grouped_ffn_backward(cfg, x_sorted, x, counts, offsets, W13, W13t, W2t, h, g1, d_o,
                             dx_sorted, dW13, dW2, bws, ws, stream=None):
    bp, bn = _ws(bws)
    p, n = _ws(ws)
    _check(_lib.moe_grouped_ffn_backward(ctypes.byref(cfg), _ptr(x_sorted), _ptr(x),
                                         _ptr(counts), _ptr(offsets), _ptr(W13), _ptr(W13t),
                                         _ptr(W2t), _ptr(h), _ptr(g1), _ptr(d_o),
                                         _ptr(dx_sorted), _ptr(dW13), _ptr(dW2), bp, bn, p, n,
                                         _stream(stream)), "moe_grouped_ffn_backward")


def moe_grouped_ffn_train(cfg, x_sorted, x, counts, offsets, W13, W2, h, y_sorted, g1, ws,
                          stream=None):
    p, n = _ws(ws)
    _check(_lib.moe_grouped_ffn_train(ctypes.byref(cfg), _ptr(x_sorted), _ptr(x), _ptr(counts),
                                      _ptr(offsets), _ptr(W13), _ptr(W2), _ptr(h),
                                      _ptr(y_sorted), _ptr(g1), p, n, _stream(stream)),
           "moe_grouped_ffn_train")


def moe_permute_backward(cfg, dx_sorted, inv, dx, stream=None):
    _check(_lib.moe_permute_backward(ctypes.byref(cfg), _ptr(dx_sorted), _ptr(inv), _ptr(dx),
                                     _stream(stream)), "moe_permute_backward")


def moe_selftest_wait_timeout(ws, limit_ns, stream=None):
    _check(_lib.moe_selftest_wait_timeout(_ptr(ws), int(limit_ns), _stream(stream)),
           "moe_selftest_wait_timeout")


def moe_get_device_status(ws, stream=None) -> int:
    return _lib.moe_get_device_status(_ptr(ws), _stream(stream))


def moe_strerror(code) -> str:
    return _lib.moe_strerror(int(code)).decode()


def moe_last_launch_count() -> int:
    return _lib.moe_last_launch_count()




def moe_layer_forward(cfg, bufs, x, y, stream=None):
    """bufs: MoeLayerBufs.  The whole forward on device tokens x into y."""
    _check(_lib.moe_layer_forward(ctypes.byref(cfg), ctypes.byref(bufs), _ptr(x), _ptr(y),
                                  _stream(stream)), "moe_layer_forward")


def moe_layer_forward_host(cfg, bufs, x_hosts, y_hosts, x_devs, y_devs, compute_stream=None,
                           copy_in_stream=None, copy_out_stream=None):
    """The forward over pinned host batches x_hosts -> y_hosts (equal-length
    lists of bf16 [T, d] page-locked CPU tensors), with two device buffers per
    side; returns once enqueued (the compute stream completes after the last
    copy out)."""
    n = len(x_hosts)
    if len(y_hosts) != n or len(x_devs) != 2 or len(y_devs) != 2:
        raise ValueError("x_hosts and y_hosts of equal length, two device buffers per side")
    arr = lambda ts: (_P * max(len(ts), 1))(*[_ptr(t) for t in ts])  # noqa: E731
    _check(_lib.moe_layer_forward_host(
        ctypes.byref(cfg), ctypes.byref(bufs), n, arr(x_hosts), arr(y_hosts), arr(x_devs),
        arr(y_devs), _stream(compute_stream), _stream(copy_in_stream),
        None if copy_out_stream is None else _stream(copy_out_stream)),
        "moe_layer_forward_host")


from .layer import MoELayer  # noqa: E402,F401
