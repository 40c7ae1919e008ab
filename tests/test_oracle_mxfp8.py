"""Pins for the oracle's MXFP8 quantizer and dequantizer (CPU only).

MXFP8: 32 E4M3 values share one E8M0 scale (remio.ai "Miles Blackwell RL";
thelatestinai.com 2610.34915 Table 10 F6: E8M0 keeps only the exponent).
Anchors: closed forms for the scale exponent, PyTorch's float8_e4m3fn
rounding of x * 2^-e (a library routine), transposition, idempotence.
"""
import numpy as np
import torch

import synthetic


def _torch_e4m3(v: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def _bf16(vals):
    return synthetic.to_bf16_bits(np.asarray(vals, dtype=np.float32))


def test_amax_448_times_power_of_two(orc):
    for k in [-20, -3, 0, 5, 60]:
        row = np.full(32, 0.75 * 2.0 ** k, dtype=np.float32)
        row[7] = 448.0 * 2.0 ** k
        q, s = orc.mxfp8_quantize_rowwise(_bf16(row)[None, :])
        assert s[0, 0] == k + 127
        assert q[0, 7] == 0x7E


def test_amax_one(orc):
    q, s = orc.mxfp8_quantize_rowwise(_bf16(np.ones(32))[None, :])
    assert s[0, 0] == 127 - 8
    assert (q == 0x78).all()            # 1 * 2^8 = 256


def test_worked_tie_even(orc):
    """Block amax 50: e = floor(log2 50) - 8 = -3; 50 * 8 = 400 is the midpoint of
    384 (mantissa 100) and 416 (mantissa 101): ties go to 384."""
    row = np.zeros(32, dtype=np.float32)
    row[0] = 50.0
    row[1] = -50.0
    q, s = orc.mxfp8_quantize_rowwise(_bf16(row)[None, :])
    assert s[0, 0] == 124
    assert q[0, 0] == 0x7C and q[0, 1] == 0xFC
    assert (q[0, 2:] == 0).all()


def test_zero_and_subnormal_blocks(orc):
    d = synthetic.tiny()
    q, s = orc.mxfp8_quantize_rowwise(d["x"])
    assert s[0, 0] == 0 and (q[0, :32] == 0).all()          # all-zero block: e = -127
    assert s[1, 0] == 0                                        # subnormal-only block clamps to -127
    x1 = orc.bf16_to_f32(d["x"][1, :32]).astype(np.float64) * 2.0 ** 127
    np.testing.assert_array_equal(q[1, :32], _torch_e4m3(x1.astype(np.float32)))


def test_codes_match_library_rounding(orc):
    x = synthetic.tiny()["x"]
    q, s = orc.mxfp8_quantize_rowwise(x)
    xf = orc.bf16_to_f32(x).astype(np.float64).reshape(x.shape[0], -1, 32)
    amax = np.abs(xf).max(axis=2)
    with np.errstate(divide="ignore"):
        e = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1))) - 8, -127)
    e = np.clip(e, -127, 127)
    np.testing.assert_array_equal(s.astype(np.int64), (e + 127).astype(np.int64))
    scaled = xf * np.exp2(-e)[:, :, None]
    assert np.abs(scaled).max() < 512.0
    ref = _torch_e4m3(np.minimum(np.abs(scaled), 448.0) * np.sign(scaled)).reshape(q.shape)
    # torch encodes -0.0 as 0x80 too; exact match everywhere
    np.testing.assert_array_equal(q, ref)


def test_colwise_is_rowwise_of_transpose(orc):
    x = synthetic.random_bf16(11, (96, 64), "student_t")
    qc, sc = orc.mxfp8_quantize_colwise(x)
    qr, sr = orc.mxfp8_quantize_rowwise(np.ascontiguousarray(x.T))
    np.testing.assert_array_equal(qc, qr)
    np.testing.assert_array_equal(sc, sr)


def test_dequant_matches_library_conversion(orc):
    x = synthetic.tiny()["x"]
    q, s = orc.mxfp8_quantize_rowwise(x)
    y = orc.dequant_mxfp8(q, s)
    vals = orc.e4m3_table()[q] * np.exp2(s.astype(np.float64) - 127).repeat(32, axis=1)
    ref = synthetic.to_bf16_bits(vals.astype(np.float32))
    np.testing.assert_array_equal(y, ref)


def test_requantize_idempotent(orc):
    """Q(DQ(Q(x))) == Q(x) whenever every block's exponent is >= -124 (so the
    dequantized values stay representable in BF16)."""
    w = synthetic.random_bf16(3, (128, 256), "normal", 0.02)
    q, s = orc.mxfp8_quantize_rowwise(w)
    assert s.min() >= 3
    q2, s2 = orc.mxfp8_quantize_rowwise(orc.dequant_mxfp8(q, s))
    np.testing.assert_array_equal(q, q2)
    np.testing.assert_array_equal(s, s2)


def test_deterministic(orc):
    x = synthetic.random_bf16(4, (64, 128), "student_t")
    a = orc.mxfp8_quantize_rowwise(x)
    b = orc.mxfp8_quantize_rowwise(x.copy())
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)
