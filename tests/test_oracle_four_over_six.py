"""Pins for the oracle's Four-over-Six NVFP4 (NVIDIA RL blog, "Four-Over-Six (4/6)": per block, map the
maximum to 4 or to 6 and keep the lower error).  Expected bytes come from closed forms on the E2M1 grid
and from the standard quantizer (pinned elsewhere), never from the 4/6 code itself."""
import numpy as np

import synthetic
from conftest import read_golden

S_EXP = -10                                   # token amax 2.625 = 2688 * 2^-10, so S = 2^-10
GRID = {0.0: 0, 0.5: 1, 1.0: 2, 1.5: 3, 2.0: 4, 3.0: 5, 4.0: 6, 6.0: 7}


def bf16_bits(values):
    f = np.asarray(values, dtype=np.float32)
    b = f.view(np.uint32)
    assert not (b & 0xFFFF).any(), "test values must be exact in BF16"
    return (b >> 16).astype(np.uint16)


def e2m1_code(v):
    return (8 if v < 0 or (v == 0 and np.signbit(v)) else 0) | GRID[abs(float(v))]


def token_with_block(block_units):
    """Row of 32 values: block 0 holds the token amax 2.625 (so S = 2^-10), block 1 holds
    block_units * 2^-10."""
    row = np.zeros(32, dtype=np.float32)
    row[0] = 2.625
    row[16:] = np.asarray(block_units, dtype=np.float32) * np.float32(2.0 ** S_EXP)
    return bf16_bits(row)[None, :]


def codes_of(q_row, b):
    """The 16 codes of block b of a packed row (even index in the low nibble)."""
    out = []
    for k in range(16 * b, 16 * b + 16):
        byte = int(q_row[k // 2])
        out.append((byte >> 4) & 0xF if k & 1 else byte & 0xF)
    return out


def test_block_exact_with_scale_four_takes_four(orc):
    units = [4, 3, 2, 1.5, 1, 0.5, 0, -4, -3, -2, -1.5, -1, -0.5, 0, 3, 2]
    q, s, st = orc.nvfp4_quantize_per_token_46(token_with_block(units))
    assert st[0] == np.float32(2.0 ** S_EXP)
    assert s[0, 1] == 0x38                    # E4M3 1.0: 4 * 2^-10 / 4 / 2^-10
    assert codes_of(q[0], 1) == [e2m1_code(u) for u in units]
    assert s[0, 0] == 0x7E and codes_of(q[0], 0)[0] == 7   # the amax block: 448 and 6 either way
    # the standard quantizer maps the block maximum to 6 and cannot represent it exactly
    _, s6, _ = orc.nvfp4_quantize_per_token(token_with_block(units))
    assert s6[0, 1] != 0x38


def test_block_exact_with_scale_six_keeps_six(orc):
    units = [6, 4, 3, 2, 1.5, 1, 0.5, 0, -6, -4, -3, -2, -1.5, -1, -0.5, 0]
    q, s, _ = orc.nvfp4_quantize_per_token_46(token_with_block(units))
    assert s[0, 1] == 0x38                    # E4M3 1.0: 6 * 2^-10 / 6 / 2^-10; scale-to-4 gives 1.5
    assert codes_of(q[0], 1) == [e2m1_code(u) for u in units]


def test_exact_under_both_scales_keeps_six(orc):
    # 12 * 2^-10: scale to 6 -> bs 2 (grid x 2), scale to 4 -> bs 3 (grid x 3); 12, 6, 3, 0 are exact
    # under both, so the errors tie and the standard 6 stays
    units = [12, 6, 3, 0, -12, -6, -3, 0, 12, 6, 3, 0, -12, -6, -3, 0]
    q, s, _ = orc.nvfp4_quantize_per_token_46(token_with_block(units))
    assert s[0, 1] == 0x40                    # E4M3 2.0 (3.0 would be 0x44)
    assert codes_of(q[0], 1) == [e2m1_code(u / 2) for u in units]


def _block_errors(orc, x_bits, q, s, st):
    """Largest |FP32 DQ - x| per 1x16 block, from the codes with the golden E2M1 grid."""
    rows = sorted((int(c), float(v)) for c, v in read_golden("e2m1_grid.txt"))
    grid = np.array([v for c, v in rows if c < 8], dtype=np.float32)
    assert grid.size == 8
    T, H = x_bits.shape
    x = (x_bits.astype(np.uint32) << 16).view(np.float32)
    lo, hi = q & 0xF, q >> 4
    codes = np.empty((T, H), dtype=np.uint8)
    codes[:, 0::2], codes[:, 1::2] = lo, hi
    val = grid[codes & 7] * np.where(codes & 8, np.float32(-1), np.float32(1))
    bsv = np.array([orc.e4m3_value(int(c)) for c in range(256)], dtype=np.float64).astype(np.float32)[s]
    deq = (val * np.repeat(bsv, 16, axis=1)) * st[:, None]
    return np.abs(deq - x).reshape(T, H // 16, 16).max(axis=2)


def test_never_worse_than_standard_and_only_on_a_strict_gain(orc):
    for seed, kind in [(11, "student_t"), (12, "normal")]:
        x = synthetic.random_bf16(seed, (96, 512), kind=kind)
        q46, s46, st46 = orc.nvfp4_quantize_per_token_46(x)
        q6, s6, st6 = orc.nvfp4_quantize_per_token(x)
        assert np.array_equal(st46, st6)                         # second-level scale unchanged
        e46, e6 = _block_errors(orc, x, q46, s46, st46), _block_errors(orc, x, q6, s6, st6)
        assert (e46 <= e6).all()
        differs = (s46 != s6) | (q46.reshape(96, -1, 8) != q6.reshape(96, -1, 8)).any(axis=2)
        assert np.array_equal(differs, e46 < e6)
        assert differs.mean() > 0.2                              # the option is exercised


def test_scale_four_candidate_is_the_documented_scale(orc):
    x = synthetic.random_bf16(13, (32, 256), kind="student_t")
    q46, s46, st = orc.nvfp4_quantize_per_token_46(x)
    _, s6, _ = orc.nvfp4_quantize_per_token(x)
    xf = (x.astype(np.uint32) << 16).view(np.float32).reshape(32, 16, 16)
    amax_b = np.abs(xf).max(axis=2)
    four = s46 != s6
    t = (amax_b / np.float32(4)) / st[:, None]                   # FP32, in the documented order
    expect = np.vectorize(lambda v: orc.e4m3_encode(float(v)))(t)
    assert np.array_equal(s46[four], expect[four])


def test_weight_2d_four_over_six_transpose_and_gain(orc):
    w = synthetic.random_bf16(14, (64, 96), scale=0.02)
    qr, qc, st, sw = orc.nvfp4_quantize_weight_2d_46(w)
    qrT, qcT, stT, swT = orc.nvfp4_quantize_weight_2d_46(np.ascontiguousarray(w.T))
    assert np.array_equal(st.T, stT) and sw == swT
    assert np.array_equal(qr, qcT) and np.array_equal(qc, qrT)
    _, _, st6, sw6 = orc.nvfp4_quantize_weight_2d(w)
    assert sw == sw6
    assert (st != st6).any()


def test_per_token_permutation_invariance(orc):
    x = synthetic.random_bf16(15, (40, 128), kind="student_t")
    perm = np.random.default_rng(0).permutation(40)
    q, s, st = orc.nvfp4_quantize_per_token_46(x)
    qp, sp, stp = orc.nvfp4_quantize_per_token_46(np.ascontiguousarray(x[perm]))
    assert np.array_equal(q[perm], qp) and np.array_equal(s[perm], sp) and np.array_equal(st[perm], stp)
