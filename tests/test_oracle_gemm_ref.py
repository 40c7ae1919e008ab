"""Pins for the oracle's FP64 GEMM reference on dequantized operands.

MaxText NVFP4 page: the FPROP / DGRAD / WGRAD GEMMs take quantized inputs and
emit BF16; remio.ai "Miles Blackwell RL": MXFP8 forward, data-gradient and
weight-gradient GEMMs.  Anchors: a brute-force triple loop over decoded
values, integer-exact sums, K-block permutation invariance, and the 2D-weight
FPROP/DGRAD consistency DQ(W) = DQ(W^T)^T.
"""
import numpy as np

import synthetic

GRID = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float64)


def test_mxfp8_ref_vs_triple_loop(orc):
    a = synthetic.random_bf16(50, (8, 64), "student_t")
    b = synthetic.random_bf16(51, (6, 64), "normal", 0.02)
    qa, sa = orc.mxfp8_quantize_rowwise(a)
    qb, sb = orc.mxfp8_quantize_rowwise(b)
    ref = orc.gemm_ref_mxfp8(qa, sa, qb, sb)
    t = orc.e4m3_table()
    for m in range(8):
        for n in range(6):
            acc = 0.0
            for k in range(64):
                acc += t[qa[m, k]] * 2.0 ** (int(sa[m, k // 32]) - 127) * t[qb[n, k]] * 2.0 ** (int(sb[n, k // 32]) - 127)
            assert abs(acc - ref[m, n]) <= 1e-12 * max(1.0, abs(acc))


def test_nvfp4_ref_vs_triple_loop_with_alphas(orc):
    a = synthetic.random_bf16(52, (5, 32), "student_t")
    b = synthetic.random_bf16(53, (7, 32), "normal", 0.02)
    qa, sa, sta = orc.nvfp4_quantize_per_token(a)
    qb, sb, Sb = orc.nvfp4_quantize_1x16(b, colwise=False)
    ref = orc.gemm_ref_nvfp4(qa, sa, sta, qb, sb, Sb)
    t = orc.e4m3_table()

    def val(q, r, k):
        byte = q[r, k // 2]
        c = (byte >> 4) if k & 1 else (byte & 0xF)
        return GRID[c & 7] * (-1.0 if c & 8 else 1.0)

    for m in range(5):
        for n in range(7):
            acc = sum(val(qa, m, k) * t[sa[m, k // 16]] * val(qb, n, k) * t[sb[n, k // 16]] for k in range(32))
            acc *= float(sta[m]) * float(Sb)
            assert abs(acc - ref[m, n]) <= 1e-12 * max(1e-30, abs(acc))


def test_integer_exact_case(orc):
    """E8M0 scale 2^0 and small-integer E4M3 codes: the reference equals the
    integer matmul exactly."""
    rng = np.random.default_rng(6)
    ia = rng.integers(-8, 9, size=(16, 128))
    ib = rng.integers(-8, 9, size=(12, 128))
    enc = {v: orc.e4m3_encode(float(v)) for v in range(-8, 9)}
    qa = np.vectorize(enc.get)(ia).astype(np.uint8)
    qb = np.vectorize(enc.get)(ib).astype(np.uint8)
    sa = np.full((16, 4), 127, dtype=np.uint8)
    sb = np.full((12, 4), 127, dtype=np.uint8)
    np.testing.assert_array_equal(orc.gemm_ref_mxfp8(qa, sa, qb, sb), (ia @ ib.T).astype(np.float64))


def test_k_block_permutation_invariance(orc):
    a = synthetic.random_bf16(54, (8, 128), "student_t")
    b = synthetic.random_bf16(55, (8, 128), "student_t")
    qa, sa = orc.mxfp8_quantize_rowwise(a)
    qb, sb = orc.mxfp8_quantize_rowwise(b)
    ref = orc.gemm_ref_mxfp8(qa, sa, qb, sb)
    perm = np.array([2, 0, 3, 1])
    cols = np.concatenate([np.arange(p * 32, p * 32 + 32) for p in perm])
    ref2 = orc.gemm_ref_mxfp8(qa[:, cols].copy(), sa[:, perm].copy(), qb[:, cols].copy(), sb[:, perm].copy())
    np.testing.assert_allclose(ref2, ref, rtol=1e-12, atol=0)


def test_2d_weights_fprop_dgrad_consistency(orc):
    w = synthetic.random_bf16(56, (48, 64), "normal", 0.02)
    qr, qc, st, sw = orc.nvfp4_quantize_weight_2d(w)
    dq_row = orc.decode_nvfp4_f64(qr, orc.weight_2d_operand_scales(st, "row"))
    dq_col = orc.decode_nvfp4_f64(qc, orc.weight_2d_operand_scales(st, "col"))
    np.testing.assert_array_equal(dq_row, dq_col.T)


def test_rel_fro_error(orc):
    ref = np.ones((4, 4))
    assert orc.rel_fro_error(ref * 1.01, ref) == np.float64(0.01).item() or \
        abs(orc.rel_fro_error(ref * 1.01, ref) - 0.01) < 1e-12


def test_dq_backward_ref_matches_block_scaled_ref_when_dequantization_is_exact(orc):
    """The dequantized-backward reference (BF16 A times the BF16 DQ(B)) equals the block-scaled NVFP4
    reference on the same codes when every dequantized value is exact in BF16 (power-of-two second-level
    scales), and a triple loop over hand-decoded values; a transposed or mis-scaled operand fails."""
    rng = np.random.default_rng(21)
    M, N, K = 6, 5, 64
    qa = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    qb = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sa = rng.integers(0x28, 0x48, size=(M, K // 16), dtype=np.uint8)      # E4M3 scales 2^-2 .. 2^1.9
    sb = rng.integers(0x28, 0x48, size=(N, K // 16), dtype=np.uint8)
    Sa, Sb = np.float32(0.125), np.float32(4.0)
    a_bf16 = orc.dequant_nvfp4(qa, sa, Sa, False)                          # exact: <= 6 significant bits
    ref = orc.gemm_ref_bf16_dq_nvfp4(a_bf16, qb, sb, Sb, False)
    assert np.array_equal(ref, orc.gemm_ref_nvfp4(qa, sa, Sa, qb, sb, Sb))
    e2m1 = [0, .5, 1, 1.5, 2, 3, 4, 6]

    def val(q, s, S, r, k):
        c = (int(q[r, k // 2]) >> (4 * (k & 1))) & 0xF
        return (-1 if c & 8 else 1) * e2m1[c & 7] * orc.e4m3_value(int(s[r, k // 16])) * float(S)

    loop = np.array([[sum(val(qa, sa, Sa, m, k) * val(qb, sb, Sb, n, k) for k in range(K)) for n in range(N)]
                     for m in range(M)])
    assert np.array_equal(ref, loop)
    # per-row second-level scales of B and a per-row alpha of A
    Sb_rows = np.float32(2.0) ** rng.integers(-3, 3, size=N).astype(np.float32)
    aa = np.float32(2.0) ** rng.integers(-2, 2, size=M).astype(np.float32)
    ref2 = orc.gemm_ref_bf16_dq_nvfp4(a_bf16, qb, sb, Sb_rows, True, alpha_a=aa)
    assert np.array_equal(ref2, orc.gemm_ref_nvfp4(qa, sa, Sa * aa, qb, sb, Sb_rows))
