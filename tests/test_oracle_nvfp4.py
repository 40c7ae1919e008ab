"""Pins for the oracle's NVFP4 quantizers and dequantizer (CPU only).

NVFP4: E2M1 values with one E4M3 scale per 16 under a second FP32 scale,
per token (remio.ai "Miles Blackwell RL"; socker-news "NVFP4 RL training",
per-token activation scaling) or per tensor with 16x16 weight tiles (MaxText
NVFP4 page, "NVFP4 pretraining recipe").
Anchors: closed forms at the amax element, brute-force nearest-grid search,
per-token independence under permutation and gather, transposition of 2D
weights, an error bound, and re-quantization idempotence.
"""
import numpy as np

import synthetic

GRID = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float64)


def _nibbles(q: np.ndarray) -> np.ndarray:
    out = np.empty(q.shape[:-1] + (q.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = q & 0xF
    out[..., 1::2] = q >> 4
    return out


def _vals(q):
    n = _nibbles(q)
    return GRID[n & 7] * np.where(n & 8, -1.0, 1.0)


def test_amax_element_gets_448_and_6(orc):
    x = synthetic.random_bf16(21, (32, 256), "student_t")
    q, s, st = orc.nvfp4_quantize_per_token(x)
    xf = orc.bf16_to_f32(x)
    n = _nibbles(q)
    for t in range(x.shape[0]):
        k = int(np.argmax(np.abs(xf[t])))
        assert st[t] == np.float32(np.abs(xf[t]).max()) / np.float32(2688.0)
        assert s[t, k // 16] == 0x7E                           # block scale 448
        assert (n[t, k] & 7) == 7                              # |code| = 6
        assert (n[t, k] >> 3) == (1 if xf[t, k] < 0 else 0)


def test_codes_are_nearest_grid_values(orc):
    x = synthetic.random_bf16(22, (16, 128), "student_t")
    q, s, st = orc.nvfp4_quantize_per_token(x)
    xf = orc.bf16_to_f32(x)
    n = _nibbles(q)
    for t in range(x.shape[0]):
        for b in range(x.shape[1] // 16):
            r = orc._load().orc_nvfp4_block_recip(int(s[t, b]), float(st[t]))
            v = (xf[t, b * 16:(b + 1) * 16] * np.float32(r)).astype(np.float64)
            for i in range(16):
                a = min(abs(v[i]), 6.0)
                d = np.abs(GRID - a)
                assert (n[t, b * 16 + i] & 7) in np.flatnonzero(d == d.min()).tolist()


def test_reconstruction_error_bound(orc):
    """|x - q*bs*S| <= half a grid step (at q's magnitude) times bs*S, up to
    FP32 rounding of r; for saturated blocks the E4M3 rounding of bs can push
    x*r to at most 6*(1+1/16)."""
    x = synthetic.random_bf16(23, (64, 512), "student_t")
    q, s, st = orc.nvfp4_quantize_per_token(x)
    xf = orc.bf16_to_f32(x).astype(np.float64)
    bs = orc.e4m3_table()[s].repeat(16, axis=1)
    d = bs * st.astype(np.float64)[:, None]
    xhat = _vals(q) * d
    step = np.where(np.abs(xhat) < 2 * d, 0.5, np.where(np.abs(xhat) < 4 * d, 1.0, 2.0))
    bound = 0.5 * step * d * (1 + 2.0 ** -20) + 0.0625 * 6 * d
    assert (np.abs(xf - xhat) <= bound).all()
    rel = np.linalg.norm(xf - xhat) / np.linalg.norm(xf)
    assert rel < 0.15


def test_zero_token(orc):
    x = synthetic.random_bf16(24, (4, 64), "normal")
    x[2] = 0
    q, s, st = orc.nvfp4_quantize_per_token(x)
    assert st[2] == 0 and (s[2] == 0).all() and (q[2] == 0).all()
    assert (st[[0, 1, 3]] > 0).all()


def test_per_token_independent_of_batch(orc):
    x = synthetic.random_bf16(25, (48, 128), "student_t")
    q, s, st = orc.nvfp4_quantize_per_token(x)
    perm = np.random.default_rng(0).permutation(48)
    q2, s2, st2 = orc.nvfp4_quantize_per_token(np.ascontiguousarray(x[perm]))
    np.testing.assert_array_equal(q2, q[perm])
    np.testing.assert_array_equal(s2, s[perm])
    np.testing.assert_array_equal(st2, st[perm])
    # gather with repeats (expert routing) commutes with quantization
    idx = np.random.default_rng(1).integers(0, 48, size=100)
    q3, s3, st3 = orc.nvfp4_quantize_per_token(np.ascontiguousarray(x[idx]))
    np.testing.assert_array_equal(q3, q[idx])
    np.testing.assert_array_equal(s3, s[idx])
    # a token's bytes do not depend on the other rows' magnitudes
    y = x.copy()
    y[5] = synthetic.to_bf16_bits(orc.bf16_to_f32(x[5]) * np.float32(1000.0))
    q4, s4, _ = orc.nvfp4_quantize_per_token(y)
    mask = np.arange(48) != 5
    np.testing.assert_array_equal(q4[mask], q[mask])


def test_single_outlier_block(orc):
    row = np.full(64, 0.01, dtype=np.float32)
    row[20] = 100.0
    x = synthetic.to_bf16_bits(row)[None, :]
    q, s, st = orc.nvfp4_quantize_per_token(x)
    n = _nibbles(q)[0]
    assert s[0, 1] == 0x7E and n[20] == 7
    # the outlier's block: 0.01 * r rounds to 0
    assert (n[16:32][np.arange(16) != 4] == 0).all()
    # other blocks keep their own scale: 0.01 is their amax -> code 6
    assert (n[0:16] == 7).all() and (n[32:64] == 7).all()


def test_block_scale_rounding_to_zero(orc):
    """A block whose amax is below 2^-10 * 6 * S has block scale E4M3 0; its
    reciprocal is taken as 0, so every code is a (signed) zero."""
    row = np.full(32, 1e-9, dtype=np.float32)
    row[1::2] *= -1
    row[20] = 100.0
    q, s, st = orc.nvfp4_quantize_per_token(synthetic.to_bf16_bits(row)[None, :])
    n = _nibbles(q)[0]
    assert s[0, 0] == 0
    np.testing.assert_array_equal(n[0:16], np.where(np.arange(16) % 2 == 1, 8, 0))
    assert s[0, 1] == 0x7E and n[20] == 7


def test_weight_2d_transpose_invariance(orc):
    w = synthetic.random_bf16(26, (64, 96), "normal", 0.02)
    qr, qc, st, sw = orc.nvfp4_quantize_weight_2d(w)
    qr2, qc2, st2, sw2 = orc.nvfp4_quantize_weight_2d(np.ascontiguousarray(w.T))
    np.testing.assert_array_equal(qr2, qc)
    np.testing.assert_array_equal(qc2, qr)
    np.testing.assert_array_equal(st2, st.T)
    assert sw == sw2
    # the codes of the transposed copy are the same values, transposed
    np.testing.assert_array_equal(_nibbles(qc), _nibbles(qr).T)


def test_weight_2d_tile_scale_closed_form(orc):
    w = synthetic.random_bf16(27, (32, 32), "normal", 0.02)
    wf = orc.bf16_to_f32(w)
    qr, qc, st, sw = orc.nvfp4_quantize_weight_2d(w)
    assert sw == np.float32(np.abs(wf).max()) / np.float32(2688.0)
    i, j = np.unravel_index(np.argmax(np.abs(wf)), wf.shape)
    assert st[i // 16, j // 16] == 0x7E
    assert (_nibbles(qr)[i, j] & 7) == 7


def test_dequant_matches_library_conversion(orc):
    x = synthetic.random_bf16(28, (32, 128), "student_t")
    q, s, st = orc.nvfp4_quantize_per_token(x)
    y = orc.dequant_nvfp4(q, s, st, per_row=True)
    p = (_vals(q) * orc.e4m3_table()[s].repeat(16, axis=1)).astype(np.float32)   # exact products
    ref = synthetic.to_bf16_bits(p * st[:, None])
    np.testing.assert_array_equal(y, ref)


def test_requantize_idempotent_weights(orc):
    w = synthetic.random_bf16(29, (64, 128), "normal", 0.02)
    qr, qc, st, sw = orc.nvfp4_quantize_weight_2d(w)
    assert (st >= 0x08).all()                      # every tile scale is a normal E4M3 code
    ops = orc.weight_2d_operand_scales(st, "row")
    y = orc.dequant_nvfp4(qr, ops, sw, per_row=False)
    qr2, qc2, st2, sw2 = orc.nvfp4_quantize_weight_2d(y)
    np.testing.assert_array_equal(qr2, qr)
    np.testing.assert_array_equal(st2, st)
    assert sw2 == sw


def test_per_tensor_rowwise_vs_colwise_transpose(orc):
    x = synthetic.random_bf16(30, (64, 48), "student_t")
    qc, sc, Sc = orc.nvfp4_quantize_1x16(x, colwise=True)
    qr, sr, Sr = orc.nvfp4_quantize_1x16(np.ascontiguousarray(x.T), colwise=False)
    np.testing.assert_array_equal(qc, qr)
    np.testing.assert_array_equal(sc, sr)
    assert Sc == Sr == np.float32(np.abs(orc.bf16_to_f32(x)).max()) / np.float32(2688.0)


def test_per_tensor_differs_from_per_token_only_by_second_scale(orc):
    """With one row, per-tensor and per-token scopes coincide."""
    x = synthetic.random_bf16(31, (1, 256), "student_t")
    q1, s1, st = orc.nvfp4_quantize_per_token(x)
    q2, s2, S = orc.nvfp4_quantize_1x16(x, colwise=False)
    np.testing.assert_array_equal(q1, q2)
    np.testing.assert_array_equal(s1, s2)
    assert st[0] == S
