"""Pins for the oracle's format tables and rounding (CPU only).

Independent anchors: the format landmarks and the E2M1 grid (tests/golden),
PyTorch's float8_e4m3fn and bfloat16 conversions (library routines), and
closed-form tie points.
"""
import math

import numpy as np
import torch

from conftest import read_golden


def test_e4m3_landmarks(orc):
    for code, val in read_golden("e4m3_landmarks.txt"):
        v = orc.e4m3_value(int(code, 16))
        if val == "nan":
            assert math.isnan(v)
        else:
            assert v == float(val) and math.copysign(1.0, v) == math.copysign(1.0, float(val))


def test_e4m3_decode_matches_torch():
    import oracle
    codes = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    table = oracle.e4m3_table()
    for c in range(256):
        if math.isnan(codes[c]):
            assert math.isnan(table[c])
        else:
            assert table[c] == codes[c], c


def test_e4m3_encode_matches_torch_rne_in_range(orc):
    rng = np.random.default_rng(123)
    # random magnitudes over the whole E4M3 range and below, both signs
    mags = np.exp2(rng.uniform(-14, math.log2(464.0), size=20000)).astype(np.float32)
    vals = mags * np.where(rng.random(20000) < 0.5, -1, 1).astype(np.float32)
    # every midpoint between consecutive finite codes (ties), and values next to them
    pos = np.array(sorted(set(orc.e4m3_table()[:127].tolist())), dtype=np.float64)
    mids = ((pos[1:] + pos[:-1]) / 2).astype(np.float32)
    vals = np.concatenate([vals, mids, -mids, np.nextafter(mids, 0), np.nextafter(mids, 1000)])
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(float(v)) for v in vals], dtype=np.uint8)
    np.testing.assert_array_equal(got, ref)


def test_e4m3_satfinite(orc):
    for v in [464.0, 465.0, 480.0, 1e6, float("inf")]:
        assert orc.e4m3_encode(v) == 0x7E
        assert orc.e4m3_encode(-v) == 0xFE


def test_e2m1_grid(orc):
    for code, val in read_golden("e2m1_grid.txt"):
        assert orc.e2m1_value(int(code)) == float(val)
        assert orc.e2m1_value(int(code) | 8) == -float(val) or float(val) == 0.0


def test_e2m1_rne_ties(orc):
    for inp, code in read_golden("e2m1_rne_ties.txt"):
        assert orc.e2m1_encode(float(inp)) == int(code), inp


def test_e2m1_encode_is_nearest_bruteforce(orc):
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float64)
    rng = np.random.default_rng(7)
    for v in rng.uniform(-7, 7, size=4000).astype(np.float32):
        code = orc.e2m1_encode(float(v))
        a = min(abs(float(v)), 6.0)
        d = np.abs(grid - a)
        best = np.flatnonzero(d == d.min())
        assert (code & 7) in best.tolist()
        assert (code >> 3) == (1 if v < 0 else 0)


def test_e8m0(orc):
    assert orc.e8m0_value(127) == 1.0
    assert orc.e8m0_value(0) == 2.0 ** -127
    assert orc.e8m0_value(254) == 2.0 ** 127
    assert math.isnan(orc.e8m0_value(255))


def test_float_to_bf16_matches_torch(orc):
    rng = np.random.default_rng(5)
    vals = np.concatenate([
        rng.standard_normal(5000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),       # FP32 subnormals
        np.array([1.00390625, 1.01171875, -1.00390625, 3.0e38, 1e-45], dtype=np.float32),  # ties
    ])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.float_to_bf16(float(v)) for v in vals], dtype=np.uint16)
    np.testing.assert_array_equal(got, ref)
