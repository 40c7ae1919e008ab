"""Pins for the oracle's blockwise FP8 (NVIDIA NeMo RL FP8 page, "FP8 nas camadas lineares": E4M3 codes,
weights in [128, 128] blocks, activations and gradients in [1, 128] tiles, one FP32 scale per block;
"Opções avançadas": power-of-two scales instead).  Expected codes come from closed forms worked by hand,
from a brute-force nearest search over every finite E4M3 value built from the format's fields, and from
invariants (transposition, block locality, zero padding, monotonicity of the block maximum)."""
import numpy as np
import pytest

import synthetic


def bf16_bits(values):
    f = np.asarray(values, dtype=np.float32)
    b = f.view(np.uint32)
    assert not (b & 0xFFFF).any(), "test values must be exact in BF16"
    return (b >> 16).astype(np.uint16)


def bits_to_f32(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


def e4m3_table():
    """Values of the 127 non-negative finite E4M3 codes from the field definition (bias 7, 3 mantissa bits,
    subnormals m * 2^-9, S.1111.111 is NaN)."""
    vals = []
    for c in range(0x7F):
        e, m = c >> 3, c & 7
        vals.append(m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    return np.array(vals)


E4M3 = e4m3_table()


def nearest_e4m3(t):
    """Brute force: the nearest finite E4M3 value to t (ties to the even code, saturating at 448)."""
    a = abs(float(t))
    d = np.abs(E4M3 - a)
    best = np.flatnonzero(d == d.min())
    c = int(best[0]) if len(best) == 1 else int([b for b in best if b % 2 == 0][0])
    return c | (0x80 if np.signbit(t) else 0)


def row_with(values, at=0):
    """One 128-value tile holding ``values`` from position ``at``, zeros elsewhere."""
    row = np.zeros(128, dtype=np.float32)
    row[at:at + len(values)] = values
    return row


@pytest.mark.parametrize("amax,k,code", [
    (448.0, 0, 0x7E),                 # 448 * 2^0 reaches the maximum exactly
    (448.0 * 2.0 ** -10, -10, 0x7E),
    (448.0 * 2.0 ** 3, 3, 0x7E),
    (224.0, -1, 0x7E),
    (450.0, 1, 0x76),                 # next BF16 above 448: k = 1, 450 / 2 = 225 -> 224
    (446.0, 0, 0x7E),                 # below 448: k = 0, 446 -> 448 (step 32 in [256, 512))
    (256.0, 0, 0x78),                 # 448 / 2 = 224 < 256, so k = 0 and 256 is exact
    (3.0, -7, 0x7C),                  # 448 / 128 = 3.5 >= 3 > 1.75: 3 * 128 = 384
])
def test_pow2_exponent_closed_forms(orc, amax, k, code):
    x = bf16_bits(row_with([amax, -amax / 2]))[None, :]
    q, s, e8 = orc.fp8_blockwise_1x128(x, pow2=True)
    assert e8[0, 0] == k + 127
    assert s[0, 0] == np.float32(2.0 ** k)
    assert q[0, 0] == code
    assert q[0, 1] == nearest_e4m3(-amax / 2 * 2.0 ** -k)
    assert (q[0, 2:] == 0).all()


def test_fp32_scale_closed_forms(orc):
    # amax 3: s = fp32(3 / 448); 3 / s -> 448, 1.5 / s -> 224, 1 / s = 149.33 -> 144 (step 16), -0.75 / s -> -112
    x = bf16_bits(row_with([3.0, 1.5, 1.0, -0.75]))[None, :]
    q, s, e8 = orc.fp8_blockwise_1x128(x, pow2=False)
    assert s[0, 0] == np.float32(3.0) / np.float32(448.0)
    assert list(q[0, :4]) == [0x7E, 0x76, 0x71, 0xEE]
    assert e8[0, 0] == 0
    # the same tile with a power-of-two scale 2^-7: 384, 192, 128, -96
    q2, s2, e2 = orc.fp8_blockwise_1x128(x, pow2=True)
    assert list(q2[0, :4]) == [0x7C, 0x74, 0x70, 0xEC]
    assert s2[0, 0] == np.float32(2.0 ** -7) and e2[0, 0] == 120


@pytest.mark.parametrize("pow2", [False, True])
def test_zero_tile(orc, pow2):
    vals = np.zeros(256, dtype=np.float32)
    vals[5] = -0.0
    vals[128:130] = [1.0, -2.0]                           # the second tile is not zero
    q, s, e8 = orc.fp8_blockwise_1x128(bf16_bits(vals)[None, :], pow2=pow2)
    assert s[0, 0] == (np.float32(2.0 ** -127) if pow2 else 0.0)
    assert e8[0, 0] == 0                                  # E8M0 code of 2^-127 (power of two), else unused
    assert q[0, 5] == 0x80 and (np.delete(q[0, :128], 5) == 0).all()
    assert q[0, 129] == (0xF8 if pow2 else 0xFE)          # |-2| is that tile's maximum: -256 (2^-7) or -448


@pytest.mark.parametrize("pow2", [False, True])
def test_codes_are_nearest_and_scale_rule(orc, pow2):
    """Every code is the nearest E4M3 value to the scaled input; power-of-two exponents are the smallest
    that fit the tile's maximum in 448; FP32 scales are fp32(amax / 448)."""
    rng = np.random.default_rng(7)
    R, K = 24, 384
    x = bits_to_f32(synthetic.random_bf16(11, (R, K)))
    x *= (2.0 ** rng.integers(-30, 30, size=(R, 1))).astype(np.float32)      # per-row magnitudes
    x[3, :] = x[3, :] * np.float32(2.0 ** -110)                              # BF16 subnormal range
    xb = ((x.view(np.uint32) + 0x8000) >> 16).astype(np.uint16)              # back to BF16 (input only)
    q, s, e8 = orc.fp8_blockwise_1x128(xb, pow2=pow2)
    xf = bits_to_f32(xb)
    for r in range(R):
        for b in range(K // 128):
            tile = xf[r, b * 128:(b + 1) * 128]
            amax = float(np.abs(tile).max())
            if pow2:
                k = int(e8[r, b]) - 127
                assert 448.0 * 2.0 ** k >= amax
                assert k == -127 or 448.0 * 2.0 ** (k - 1) < amax
                scaled = tile.astype(np.float64) * 2.0 ** -k
            else:
                sc = np.float32(amax) / np.float32(448.0)
                assert s[r, b] == sc
                scaled = tile / sc                                            # FP32 division
            for i in range(0, 128, 7):
                assert q[r, b * 128 + i] == nearest_e4m3(scaled[i]), (r, b, i)


@pytest.mark.parametrize("pow2", [False, True])
def test_dequantization_error_bound(orc, pow2):
    """|q * s - x| stays within half an E4M3 step: 2^-4 |x| for normal codes, 2^-10 s below 2^-6."""
    x = synthetic.random_bf16(3, (16, 512))
    q, s, _ = orc.fp8_blockwise_1x128(x, pow2=pow2)
    xf = bits_to_f32(x)
    mag = E4M3[q & 0x7F] * np.where(q & 0x80, -1.0, 1.0)
    deq = mag * np.repeat(s.astype(np.float64), 128, axis=1)
    bound = 2.0 ** -4 * np.abs(xf) * (1 + 2.0 ** -20) + 2.0 ** -10 * np.repeat(s, 128, axis=1)
    assert (np.abs(deq - xf) <= bound).all()


@pytest.mark.parametrize("pow2", [False, True])
def test_weight_blocks_transpose(orc, pow2):
    w = synthetic.random_bf16(5, (200, 300), scale=0.02)
    q_row, q_col, s, e8 = orc.fp8_blockwise_128x128(w, pow2=pow2)
    assert s.shape == (2, 3) and q_row.shape == (200, 300) and q_col.shape == (300, 200)
    assert np.array_equal(q_col, q_row.T)
    t_row, t_col, t_s, t_e8 = orc.fp8_blockwise_128x128(np.ascontiguousarray(w.T), pow2=pow2)
    assert np.array_equal(t_row, q_col) and np.array_equal(t_col, q_row)
    assert np.array_equal(t_s, s.T) and np.array_equal(t_e8, e8.T)


@pytest.mark.parametrize("pow2", [False, True])
def test_weight_block_is_max_of_its_row_tiles(orc, pow2):
    """A [128, 128] block's scale is that of its largest [1, 128] tile (the block maximum is the maximum of
    the tiles' maxima, and both scale rules are monotone); rows holding the block maximum quantize alike."""
    w = synthetic.random_bf16(9, (256, 384), scale=0.05)
    q_row, _, s, e8 = orc.fp8_blockwise_128x128(w, pow2=pow2)
    tq, ts, te8 = orc.fp8_blockwise_1x128(w, pow2=pow2)
    wf = np.abs(bits_to_f32(w))
    for bo in range(2):
        for bh in range(3):
            rows = slice(bo * 128, bo * 128 + 128)
            assert s[bo, bh] == ts[rows, bh].max()
            assert e8[bo, bh] == te8[rows, bh].max()
            blk = wf[rows, bh * 128:(bh + 1) * 128]
            r = bo * 128 + int(np.unravel_index(blk.argmax(), blk.shape)[0])
            assert np.array_equal(q_row[r, bh * 128:(bh + 1) * 128], tq[r, bh * 128:(bh + 1) * 128])


@pytest.mark.parametrize("pow2", [False, True])
def test_weight_block_extent_ragged(orc, pow2):
    """Blocks cover rows/columns [128 b, 128 b + 128) and stop at the matrix edge: zero padding to whole
    blocks changes nothing, and a large value changes the scale of its own block only."""
    w = synthetic.random_bf16(13, (200, 300), scale=0.02)
    q_row, _, s, e8 = orc.fp8_blockwise_128x128(w, pow2=pow2)
    pad = np.zeros((256, 384), dtype=np.uint16)
    pad[:200, :300] = w
    p_row, _, p_s, p_e8 = orc.fp8_blockwise_128x128(pad, pow2=pow2)
    assert np.array_equal(p_row[:200, :300], q_row) and np.array_equal(p_s, s) and np.array_equal(p_e8, e8)
    for (i, j) in [(199, 299), (127, 255), (128, 0), (0, 256)]:
        w2 = w.copy()
        w2[i, j] = bf16_bits([64.0])[0]
        _, _, s2, _ = orc.fp8_blockwise_128x128(w2, pow2=pow2)
        changed = np.argwhere(s2 != s)
        assert changed.tolist() == [[i // 128, j // 128]], (i, j)


def test_pow2_scales_feed_the_mxfp8_layout(orc):
    """Power-of-two blockwise codes decode identically through MXFP8 with each E8M0 code repeated over its
    four 32-element sub-blocks (the form the MXFP8 tensor-core GEMM consumes)."""
    x = synthetic.random_bf16(17, (64, 512))
    q, s, e8 = orc.fp8_blockwise_1x128(x, pow2=True)
    mx = orc.fp8_blockwise_e8m0_rowwise(e8, 128)
    assert mx.shape == (64, 16)
    direct = E4M3[q & 0x7F] * np.where(q & 0x80, -1.0, 1.0) * np.repeat(s.astype(np.float64), 128, axis=1)
    assert np.array_equal(orc.decode_mxfp8_f64(q, mx), direct)
    w = synthetic.random_bf16(19, (256, 384), scale=0.02)
    q_row, q_col, ws, we8 = orc.fp8_blockwise_128x128(w, pow2=True)
    row_mx = orc.fp8_blockwise_e8m0_weight(we8, 256, 384, "row")
    col_mx = orc.fp8_blockwise_e8m0_weight(we8, 256, 384, "col")
    assert row_mx.shape == (256, 12) and col_mx.shape == (384, 8)
    wd = orc.decode_mxfp8_f64(q_row, row_mx)
    assert np.array_equal(orc.decode_mxfp8_f64(q_col, col_mx), wd.T)
    assert np.array_equal(wd, E4M3[q_row & 0x7F] * np.where(q_row & 0x80, -1.0, 1.0)
                          * np.repeat(np.repeat(ws.astype(np.float64), 128, 0), 128, 1))


def test_blockwise_gemm_reference(orc):
    """The FP32-scale blockwise GEMM reference: the exact product of the decoded operands.  Pinned by a
    triple loop over hand-decoded values (code value from the field table times its tile's scale) and by the
    block-scaled MXFP8 reference on the same codes when every scale is a power of two."""
    rng = np.random.default_rng(3)
    M, N, K = 5, 130, 256
    qa = rng.integers(0, 0x7F, size=(M, K), dtype=np.uint8) | (rng.integers(0, 2, size=(M, K), dtype=np.uint8) << 7)
    qb = rng.integers(0, 0x7F, size=(N, K), dtype=np.uint8)
    sa = rng.random((M, K // 128)).astype(np.float32) + np.float32(0.5)
    sb = rng.random(((N + 127) // 128, K // 128)).astype(np.float32)
    ref = orc.gemm_ref_fp8_blockwise(qa, sa, qb, sb)
    val = lambda c: (-1.0 if c & 0x80 else 1.0) * E4M3[c & 0x7F]
    for (m, n) in [(0, 0), (4, 129), (2, 77)]:
        want = sum(val(qa[m, k]) * float(sa[m, k // 128]) * val(qb[n, k]) * float(sb[n // 128, k // 128])
                   for k in range(K))
        assert ref[m, n] == pytest.approx(want, rel=1e-12, abs=1e-300)
    e_a = rng.integers(120, 135, size=(M, K // 128))
    e_b = rng.integers(120, 135, size=((N + 127) // 128, K // 128))
    p2 = orc.gemm_ref_fp8_blockwise(qa, 2.0 ** (e_a - 127.0), qb, 2.0 ** (e_b - 127.0))
    mx_a = orc.fp8_blockwise_e8m0_rowwise(e_a.astype(np.uint8))
    mx_b = np.repeat(np.repeat(e_b.astype(np.uint8), 128, 0)[:N], 4, 1)
    assert np.array_equal(p2, orc.gemm_ref_mxfp8(qa, mx_a, qb, mx_b))


def test_blockwise_wgrad_reference(orc):
    """The weight-gradient form (per-row FP32 scales on both operands): a triple loop over hand-decoded
    values; the forward form on the same codes whenever B's row scales are equal within each 128-row block;
    and the transpose relation ref(A, B) = ref(B, A)^T (both operands are tiled the same way)."""
    rng = np.random.default_rng(4)
    M, N, K = 6, 131, 384
    qa = rng.integers(0, 0x7F, size=(M, K), dtype=np.uint8) | (rng.integers(0, 2, size=(M, K), dtype=np.uint8) << 7)
    qb = rng.integers(0, 0x7F, size=(N, K), dtype=np.uint8) | (rng.integers(0, 2, size=(N, K), dtype=np.uint8) << 7)
    sa = rng.random((M, K // 128)).astype(np.float32) + np.float32(0.25)
    sb = rng.random((N, K // 128)).astype(np.float32) + np.float32(0.25)
    ref = orc.gemm_ref_fp8_blockwise_wgrad(qa, sa, qb, sb)
    val = lambda c: (-1.0 if c & 0x80 else 1.0) * E4M3[c & 0x7F]
    for (m, n) in [(0, 0), (5, 130), (3, 64), (1, 127)]:
        want = sum(val(qa[m, k]) * float(sa[m, k // 128]) * val(qb[n, k]) * float(sb[n, k // 128]) for k in range(K))
        assert ref[m, n] == pytest.approx(want, rel=1e-12, abs=1e-300)
    blocks = rng.random(((N + 127) // 128, K // 128)).astype(np.float32)
    sb_rows = np.repeat(blocks, 128, 0)[:N]
    assert np.array_equal(orc.gemm_ref_fp8_blockwise_wgrad(qa, sa, qb, sb_rows),
                          orc.gemm_ref_fp8_blockwise(qa, sa, qb, blocks))
    assert np.allclose(orc.gemm_ref_fp8_blockwise_wgrad(qb, sb, qa, sa), ref.T, rtol=1e-13, atol=0)
