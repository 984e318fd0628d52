"""Pins for the FP8-dispatch part of the oracle ("Expert parallelism": DeepSeek-V3
dispatches in FP8 with s = 1 byte and combines in BF16; "Lower precision on the
wire").  The e4m3 encoder and decoder are checked against PyTorch's own
float8_e4m3fn conversion (a library routine), on every finite code, every
midpoint between neighbouring codes (ties to even), random values and the
subnormal range; the row quantizer against the format's bounds.  CPU only."""
import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _torch_e4m3(v):
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def _finite_grid():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    return codes, vals


def test_decode_matches_library_on_every_finite_code():
    codes, vals = _finite_grid()
    assert np.array_equal(oracle.e4m3_decode(codes), vals)
    assert oracle.e4m3_decode(np.uint8(0x7E)) == 448.0
    assert oracle.e4m3_decode(np.uint8(0x01)) == 2.0 ** -9


def test_encode_matches_library_on_grid_midpoints_and_random():
    codes, vals = _finite_grid()
    pos = np.unique(vals[vals >= 0])
    mids = ((pos[1:].astype(np.float64) + pos[:-1]) / 2).astype(np.float32)
    rng = np.random.default_rng(0)
    rnd = np.concatenate([rng.uniform(-448, 448, 20000), rng.normal(0, 1e-2, 20000),
                          rng.uniform(-2.0 ** -6, 2.0 ** -6, 5000)]).astype(np.float32)
    for v in (vals, mids, -mids, rnd):
        assert np.array_equal(oracle.e4m3_encode(v), _torch_e4m3(v))


def test_encode_saturates_at_the_largest_finite_value():
    big = np.array([448.0, 449.0, 463.9, 464.0, 1e6, -500.0], np.float32)
    assert [int(c) for c in oracle.e4m3_encode(big)] == [0x7E] * 5 + [0xFE]


def test_quantize_rows_bounds():
    rng = np.random.default_rng(1)
    rows = (rng.normal(size=(64, 512)) * rng.uniform(1e-3, 30, size=(64, 1))).astype(np.float32)
    rows = torch.from_numpy(rows).to(torch.bfloat16).float().numpy()    # bf16 activations
    rows[3] = 0.0
    codes, scale = oracle.quantize_rows_fp8(rows)
    amax = np.abs(rows).max(axis=1)
    assert np.array_equal(scale[amax > 0], (amax / np.float32(448.0))[amax > 0])
    assert scale[3] == 1.0 and (codes[3] == 0).all()
    # the largest element lands on +-448
    top = np.abs(rows).argmax(axis=1)
    assert (oracle.e4m3_decode(codes[np.arange(64), top])[amax > 0] ** 2 == 448.0 ** 2).all()
    deq = oracle.dequantize_rows_fp8(codes, scale)
    # 3 mantissa bits: half an ulp is 2^-4 relative (normals); subnormal
    # quantum 2^-9 of the scale; then one bf16 rounding (2^-9 relative)
    err = np.abs(deq - rows)
    bound = (2.0 ** -4 + 2.0 ** -8) * np.abs(rows) + 2.0 ** -10 * scale[:, None] * 1.01
    assert (err <= bound).all()


def test_fp8_layout_hand_dispatch_halves_the_bytes():
    with open(os.path.join(GOLDEN, "hand_dispatch.json")) as fh:
        g = json.load(fh)
    T, E, k, n = g["T"], g["E"], g["k"], g["n_ep"]
    rng = np.random.default_rng(2)
    x = torch.from_numpy(rng.normal(size=(T, 64)).astype(np.float32)).to(torch.bfloat16).float()
    idx = np.array(g["topk_idx"])
    p = oracle.permute(idx, E)
    lay = oracle.ep_layout_fp8(x.numpy(), idx, p["inv"], E, n, T)
    assert lay["send_idx"].tolist() == g["send_idx"]
    codes, scale = oracle.quantize_rows_fp8(x.numpy())
    for slot, a in enumerate(g["send_idx"]):
        assert np.array_equal(lay["send_fp8"][slot], codes[a // k])
        assert lay["send_scale"][slot] == scale[a // k]
    # the pages' byte model: FP8 dispatch moves half the BF16 dispatch bytes
    d1, c1 = oracle.alltoall_bytes(lay["C"], 64, 1, 2)
    d2, c2 = oracle.alltoall_bytes(lay["C"], 64, 2, 2)
    assert (2 * d1 == d2).all() and (c1 == c2).all()
