"""Host-side checks of the C ABI: the library loads, exports every entry point
include/moe.h declares, and rejects bad arguments on the host before touching
the device.  No kernel is launched: the calls with fake device addresses that
pass every host check (and would launch on a GPU) are made only where no CUDA
device is visible, where they must fail with MOE_E_DEVICE."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

import synth

# a call whose arguments pass the host checks reaches the device: with fake
# addresses that may only happen on a machine without a GPU
NO_GPU = not torch.cuda.is_available()

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def m():
    import __graft_entry__
    __graft_entry__.build()
    import expert_token_dispatch_moe_b300 as mod
    return mod


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    return set(re.findall(r"^\s*(?:const\s+)?[a-z0-9_]+\**\s+\**(moe_[a-z0-9_]+)\(", src, re.M))


def test_header_declares_what_library_exports(m):
    declared = _declared()
    assert declared == set(m.EXPORTS)
    out = subprocess.run(["nm", "-D", "--defined-only", m.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert exported == declared


def test_every_entry_point_has_a_wrapper(m):
    assert [n for n in m.EXPORTS if not callable(getattr(m, n, None))] == []
    assert m.moe_strerror(-8) == "a device-side wait timed out"


def test_validate_cfg_limits(m):
    ok = m.MoeCfg.from_layer(synth.CONFIGS["dsv3"])
    assert m.moe_validate_cfg(ok) == 0
    for name in synth.CONFIGS:
        assert m.moe_validate_cfg(m.MoeCfg.from_layer(synth.CONFIGS[name])) == 0
    bad = [dict(k=0), dict(k=33), dict(E=1025), dict(d=100), dict(n_ep=3), dict(n_groups=7),
           dict(topk_groups=9), dict(topk_groups=0), dict(capacity=-1), dict(has_shared=2),
           dict(score_fn=5), dict(T=0), dict(n_groups=64, topk_groups=1)]
    for b in bad:
        c = m.MoeCfg.from_layer(synth.CONFIGS["dsv3"].with_(**b))
        assert m.moe_validate_cfg(c) == -2, b
    # too few experts in the kept groups for top-k
    c = m.MoeCfg.from_layer(synth.CONFIGS["dsv3"].with_(topk_groups=1, k=33))
    assert m.moe_validate_cfg(c) == -2
    c = m.MoeCfg.from_layer(synth.CONFIGS["tiny"].with_(n_groups=4, topk_groups=1, k=3))
    assert m.moe_validate_cfg(c) == -2
    assert m._lib.moe_validate_cfg(None) == -1


def test_workspace_and_rows(m):
    c = m.MoeCfg.from_layer(synth.CONFIGS["skew"])
    assert m.moe_grouped_rows(c) == 64 * 640
    c = m.MoeCfg.from_layer(synth.CONFIGS["dsv3"])
    assert m.moe_grouped_rows(c) == 8192 * 8 + 8192
    assert m.moe_workspace_bytes(c) >= 256 + 4 * 8192 * 8
    bad = m.MoeCfg.from_layer(synth.CONFIGS["dsv3"].with_(k=0))
    assert m.moe_workspace_bytes(bad) == 0
    assert m.moe_grouped_rows(bad) == -1


def test_host_argument_errors(m):
    """Null, misaligned and undersized arguments fail on the host; a valid
    call on a machine without an sm_103 GPU fails with MOE_E_DEVICE."""
    lib = m._lib
    c = m.MoeCfg.from_layer(synth.CONFIGS["tiny"])
    P = 1 << 20          # an aligned fake address: never dereferenced on the host
    cfg = ctypes.byref(c)
    assert lib.moe_route(cfg, None, None, P, P, None) == -1
    assert lib.moe_route(cfg, P + 4, None, P, P, None) == -3
    assert lib.moe_route(cfg, P, P + 8, P, P, None) == -3
    ws_need = m.moe_workspace_bytes(c)
    assert lib.moe_permute(cfg, P, P, P, P, P, P, P, None, ws_need, None) == -4
    assert lib.moe_permute(cfg, P, P, P, P, P, P, P, P, ws_need - 1, None) == -4
    assert lib.moe_ep_layout(cfg, P, P, P, P, P, P, P, P, None, P, ws_need, None) == -1
    if NO_GPU:
        assert lib.moe_grouped_ffn(cfg, P, None, P, P, P, P, P, P, P, ws_need, None) == -6
    shared = m.MoeCfg.from_layer(synth.CONFIGS["tiny"].with_(has_shared=1))
    assert lib.moe_grouped_ffn(ctypes.byref(shared), P, None, P, P, P, P, P, P, P,
                               m.moe_workspace_bytes(shared), None) == -1
    odd_f = m.MoeCfg.from_layer(synth.CONFIGS["tiny"].with_(f=200))
    assert lib.moe_grouped_ffn(ctypes.byref(odd_f), P, None, P, P, P, P, P, P, P, ws_need,
                               None) == -2
    assert lib.moe_pack_w13(ctypes.byref(odd_f), P, P, P, None) == -2
    bad = m.MoeCfg.from_layer(synth.CONFIGS["tiny"].with_(E=7))
    assert lib.moe_route(ctypes.byref(bad), P, None, P, P, None) == -2
    if NO_GPU:
        assert lib.moe_route(cfg, P, None, P, P, None) == -6
        assert lib.moe_combine(cfg, P, P, P, P, None) == -6
    assert lib.moe_get_device_status(None, None) == -4
    assert lib.moe_selftest_wait_timeout(None, 10 ** 6, None) == -4
    assert lib.moe_selftest_wait_timeout(P + 4, 10 ** 6, None) == -3
    assert lib.moe_selftest_wait_timeout(P, 999, None) == -2
    assert lib.moe_selftest_wait_timeout(P, 10 ** 9 + 1, None) == -2
    if NO_GPU:
        assert lib.moe_selftest_wait_timeout(P, 10 ** 6, None) == -6
    for code in range(-8, 1):
        assert lib.moe_strerror(code)


def test_layer_entry_points_host_errors(m):
    """moe_layer_forward and moe_layer_forward_host check their arguments on the
    host; without an sm_103 GPU a valid call fails with MOE_E_DEVICE."""
    lib = m._lib
    c = m.MoeCfg.from_layer(synth.CONFIGS["tiny"])
    cfg = ctypes.byref(c)
    P = 1 << 20
    bufs = m.MoeLayerBufs()
    for name, _ in m.MoeLayerBufs._fields_[:-3]:     # the device pointers
        setattr(bufs, name, P)
    bufs.ws_bytes = m.moe_workspace_bytes(c)
    lb = ctypes.byref(bufs)
    # the gathered form and the combine epilogue do not go together
    bufs.gather, bufs.combine_in_epilogue = 1, 1
    assert lib.moe_layer_forward(cfg, lb, P, P, None) == -2
    bufs.gather, bufs.combine_in_epilogue = 0, 0
    arr = (ctypes.c_void_p * 2)(P, P)
    assert lib.moe_layer_forward(cfg, None, P, P, None) == -1
    assert lib.moe_layer_forward_host(cfg, None, 1, arr, arr, arr, arr, None, None, None) == -1
    assert lib.moe_layer_forward_host(cfg, lb, 1, None, arr, arr, arr, None, None, None) == -1
    assert lib.moe_layer_forward_host(cfg, lb, 2, (ctypes.c_void_p * 2)(P, None), arr, arr, arr,
                                      None, None, None) == -1
    assert lib.moe_layer_forward_host(cfg, lb, 1, arr, arr, (ctypes.c_void_p * 2)(P, P + 4),
                                      arr, None, None, None) == -3
    assert lib.moe_layer_forward_host(cfg, lb, -1, arr, arr, arr, arr, None, None, None) == -2
    assert lib.moe_layer_forward_host(cfg, lb, 0, arr, arr, arr, arr, None, None, None) == 0
    bad = m.MoeCfg.from_layer(synth.CONFIGS["tiny"].with_(E=7))
    assert lib.moe_layer_forward_host(ctypes.byref(bad), lb, 1, arr, arr, arr, arr, None, None,
                                      None) == -2
    if NO_GPU:
        assert lib.moe_layer_forward(cfg, lb, P, P, None) == -6
        assert lib.moe_layer_forward_host(cfg, lb, 1, arr, arr, arr, arr, None, None, None) == -6


def _k_split(T, E, d):
    """The router's K-split rule restated: the largest divisor S of d/64 with at
    least 8 k-blocks per chunk and at most 148 output tiles in all."""
    tiles = ((T + 127) // 128) * ((E + 255) // 256)
    kb = d // 64
    return max([s for s in range(1, kb // 8 + 1) if kb % s == 0 and tiles * s <= 148] or [1])


def test_workspace_holds_router_k_split_partials(m):
    """The workspace grows by exactly S*T*E fp32 partial logits (256-byte
    aligned) when the tensor-core router splits K, and not at all otherwise."""
    def align(x):
        return (x + 255) // 256 * 256
    for name, kw in [("dsv3_decode", {}), ("dsv3", {}), ("dsv3", {"T": 64, "d": 2048}),
                     ("mixtral", {}), ("skew", {}), ("tiny", {})]:
        cfg = synth.CONFIGS[name].with_(**kw)
        c = m.MoeCfg.from_layer(cfg)
        S = _k_split(cfg.T, cfg.E, cfg.d)
        base = m.moe_workspace_bytes(m.MoeCfg.from_layer(cfg.with_(d=64)))  # d/64 = 1: never splits
        extra = m.moe_workspace_bytes(c) - base
        assert extra == (align(S * cfg.T * cfg.E * 4) if S > 1 else 0), (name, kw, S)
    assert _k_split(128, 256, 7168) == 14 and _k_split(8192, 256, 7168) == 2



def test_ffn_tile_choice(m, monkeypatch):
    """moe_ffn_pair_tiles reports the grouped FFN's tiles: SM pairs from 768
    expected rows per expert (capped by the capacity), one-SM tiles below, and
    MOE_FFN_TILES overrides either way at the call."""
    monkeypatch.delenv("MOE_FFN_TILES", raising=False)
    pick = {n: m.moe_ffn_pair_tiles(m.MoeCfg.from_layer(synth.CONFIGS[n])) for n in synth.CONFIGS}
    assert pick["mixtral"] is True          # 4096 * 2 / 8 = 1024 rows per expert
    assert pick["dsv3"] is False and pick["dsv3_decode"] is False and pick["tiny"] is False
    assert pick["skew"] is False            # 512 rows per expert, capacity 640
    edge = synth.CONFIGS["tiny"].with_(T=3072, E=8, k=2)   # exactly 768
    assert m.moe_ffn_pair_tiles(m.MoeCfg.from_layer(edge)) is True
    assert m.moe_ffn_pair_tiles(m.MoeCfg.from_layer(edge.with_(T=3064))) is False
    capped = synth.CONFIGS["mixtral"].with_(capacity=700)
    assert m.moe_ffn_pair_tiles(m.MoeCfg.from_layer(capped)) is False
    monkeypatch.setenv("MOE_FFN_TILES", "single")
    assert m.moe_ffn_pair_tiles(m.MoeCfg.from_layer(synth.CONFIGS["mixtral"])) is False
    monkeypatch.setenv("MOE_FFN_TILES", "pair")
    assert m.moe_ffn_pair_tiles(m.MoeCfg.from_layer(synth.CONFIGS["tiny"])) is True
    with pytest.raises(m.MoeError):
        m.moe_ffn_pair_tiles(m.MoeCfg.from_layer(synth.CONFIGS["tiny"].with_(k=0)))


def test_noalloc_permute_host_errors(m):
    """moe_permute_noalloc checks its arguments and its scratch limit on the
    host, before it looks up its scratch array or launches anything: NULL and
    misaligned pointers, one of x / x_sorted without the other, and a
    configuration whose permute scratch exceeds the fixed 1 MiB."""
    lib = m._lib
    c = m.MoeCfg.from_layer(synth.CONFIGS["tiny"])
    cfg = ctypes.byref(c)
    P = 1 << 20
    assert lib.moe_permute_noalloc(cfg, P, None, P, P, P, P, P, None) == -1
    assert lib.moe_permute_noalloc(cfg, P, P + 4, P, P, P, P, P, None) == -3
    assert lib.moe_permute_noalloc(cfg, P + 8, P, P, P, P, P, P, None) == -3
    assert lib.moe_permute_noalloc(cfg, None, P, P, P, P, P, P, None) == -1
    assert lib.moe_permute_noalloc(cfg, P, P, P, P, P, P, None, None) == -1
    # per-(rank, expert) counts alone: 1024 ranks x 1024 experts x 4 B = 4 MiB
    big = m.MoeCfg.from_layer(synth.CONFIGS["tiny"].with_(T=1024, E=1024, k=2, n_ep=1024, d=64))
    assert lib.moe_permute_noalloc(ctypes.byref(big), P, P, P, P, P, P, P, None) == -9
    bad = m.MoeCfg.from_layer(synth.CONFIGS["tiny"].with_(E=7))
    assert lib.moe_permute_noalloc(ctypes.byref(bad), P, P, P, P, P, P, P, None) == -2
    if NO_GPU:
        assert lib.moe_permute_noalloc(cfg, P, P, P, P, P, P, P, None) == -6
