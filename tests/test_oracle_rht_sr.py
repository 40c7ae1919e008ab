"""Pins for the oracle's random Hadamard transform and stochastic rounding.

MaxText NVFP4 page, "NVFP4 pretraining recipe": a random Hadamard transform
on the WGRAD GEMM inputs only (it must cancel inside that GEMM), and
stochastic rounding of gradients so the rounding is unbiased.
Anchors: scipy's Sylvester Hadamard matrix (a library routine), exact
orthogonality, FP64 matrix-vector agreement, integer exactness, the WGRAD
cancellation, SR's mean over seeds, and SR's one-step property.
"""
import numpy as np
import scipy.linalg

import synthetic

GRID = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float64)


def _transform_matrix(orc, seed):
    """Columns = transform applied to unit vectors (FP32 path)."""
    cols = [orc.rht16_vec_f32(np.eye(16, dtype=np.float32)[j], seed) for j in range(16)]
    return np.stack(cols, axis=1).astype(np.float64)


def test_rht_matrix_is_scaled_sylvester_hadamard_with_signs(orc):
    for seed in [0, 8, 12345]:
        M = _transform_matrix(orc, seed)
        d = orc.rht16_signs(seed).astype(np.float64)
        np.testing.assert_array_equal(M, 0.25 * scipy.linalg.hadamard(16) @ np.diag(d))
        H = 4 * M @ np.diag(d)
        np.testing.assert_array_equal(H @ H.T, 16 * np.eye(16))
        np.testing.assert_array_equal(M @ M.T, np.eye(16))


def test_rht_butterfly_vs_fp64_matvec(orc):
    rng = np.random.default_rng(3)
    M = 0.25 * scipy.linalg.hadamard(16) @ np.diag(orc.rht16_signs(8).astype(np.float64))
    for _ in range(200):
        x = (rng.standard_t(3, 16)).astype(np.float32)
        y = orc.rht16_vec_f32(x, 8).astype(np.float64)
        ref = M @ x.astype(np.float64)
        # four levels of FP32 additions: |err| <= 4 * 2^-24 * sum|x| / 4 (+ slack)
        assert np.all(np.abs(y - ref) <= 2.0 ** -22 * np.abs(x).sum() * 0.25 * 1.01)


def test_rht_integer_inputs_exact(orc):
    rng = np.random.default_rng(4)
    M = 0.25 * scipy.linalg.hadamard(16) @ np.diag(orc.rht16_signs(5).astype(np.float64))
    for _ in range(50):
        x = rng.integers(-1000, 1000, size=16).astype(np.float32)
        np.testing.assert_array_equal(orc.rht16_vec_f32(x, 5).astype(np.float64), M @ x)


def test_rht_tensor_is_chunked_along_tokens(orc):
    x = synthetic.random_bf16(40, (64, 24), "student_t")
    y = orc.rht16(x, 8)
    M = 0.25 * scipy.linalg.hadamard(16) @ np.diag(orc.rht16_signs(8).astype(np.float64))
    xf = orc.bf16_to_f32(x).astype(np.float64)
    ref = np.concatenate([M @ xf[c * 16:(c + 1) * 16] for c in range(4)], axis=0)
    yf = orc.bf16_to_f32(y).astype(np.float64)
    # one BF16 rounding (2^-9 relative) on top of the FP32 sums
    assert np.all(np.abs(yf - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-30 + 2.0 ** -22 * np.abs(xf).max() * 4)


def test_rht_cancels_in_wgrad(orc):
    """sum_t RHT(dY)[t, o] * RHT(X)[t, h] ~= (dY^T X)[o, h] with the same seed."""
    dy = synthetic.random_bf16(41, (256, 32), "normal", 1.0)
    x = synthetic.random_bf16(42, (256, 48), "student_t")
    ref = orc.bf16_to_f32(dy).astype(np.float64).T @ orc.bf16_to_f32(x).astype(np.float64)
    got = orc.bf16_to_f32(orc.rht16(dy, 8)).astype(np.float64).T @ \
        orc.bf16_to_f32(orc.rht16(x, 8)).astype(np.float64)
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) < 1e-2
    bad = orc.bf16_to_f32(orc.rht16(dy, 8)).astype(np.float64).T @ \
        orc.bf16_to_f32(orc.rht16(x, 9)).astype(np.float64)
    assert np.linalg.norm(bad - ref) / np.linalg.norm(ref) > 0.5


def test_colwise_rht_quantizes_the_transformed_tensor(orc):
    x = synthetic.random_bf16(43, (64, 32), "student_t")
    q1, s1, S1 = orc.nvfp4_quantize_1x16(x, colwise=True, rht=True, rht_seed=8)
    q2, s2, S2 = orc.nvfp4_quantize_1x16(orc.rht16(x, 8), colwise=True)
    np.testing.assert_array_equal(q1, q2)
    np.testing.assert_array_equal(s1, s2)
    assert S1 == S2


def test_sr_on_grid_exact_and_one_step(orc):
    rng = np.random.default_rng(5)
    for g in GRID:
        for k in [0, 1, 32768, 65535]:
            assert orc.e2m1_encode_sr(g, k) == int(np.flatnonzero(GRID == g)[0])
    for v in rng.uniform(-6.5, 6.5, size=3000).astype(np.float32):
        code = orc.e2m1_encode_sr(float(v), int(rng.integers(0, 65536)))
        a = min(abs(float(v)), 6.0)
        lo = GRID[GRID <= a].max()
        hi = GRID[GRID >= a].min()
        assert GRID[code & 7] in (lo, hi)
        assert (code >> 3) == (1 if v < 0 else 0)


def test_sr_mean_converges(orc):
    """Over 10^4 seeds the mean of the rounded value approaches the input."""
    lib = orc._load()
    vals = np.array([0.1, 0.3, 0.74, 1.2, 2.2, 2.9, 3.7, 4.5, 5.5, -1.3], dtype=np.float32)
    for v in vals:
        acc = 0.0
        n = 10000
        for seed in range(n):
            c = lib.orc_e2m1_encode_sr(float(v), lib.orc_sr_bits16(seed, 77))
            acc += GRID[c & 7] * (-1 if c & 8 else 1)
        step = 0.5 if abs(v) < 2 else (1.0 if abs(v) < 4 else 2.0)
        # five standard deviations of a Bernoulli mean, plus the 2^-16 bias bound
        assert abs(acc / n - float(v)) < 5 * 0.5 * step / np.sqrt(n) + step * 2.0 ** -16


def test_sr_quantizer_end_to_end_unbiased(orc):
    """The 1x16 SR quantizer's dequantized values average to the input."""
    x = synthetic.random_bf16(44, (32, 16), "normal", 1.0)
    xf = orc.bf16_to_f32(x).astype(np.float64)
    acc = np.zeros_like(xf)
    n = 400
    for seed in range(n):
        q, s, S = orc.nvfp4_quantize_1x16(x, colwise=True, sr=True, sr_seed=seed)
        y = orc.decode_nvfp4_f64(q, s) * np.float64(S)          # [N, T]
        acc += y.T
    err = np.abs(acc / n - xf)
    assert err.mean() < 0.02 * np.abs(xf).mean() + 2e-3


def test_sr_differs_from_rne_and_depends_on_seed(orc):
    x = synthetic.random_bf16(45, (64, 32), "normal", 1e-3)
    qa, _, _ = orc.nvfp4_quantize_1x16(x, colwise=True, sr=True, sr_seed=9)
    qb, _, _ = orc.nvfp4_quantize_1x16(x, colwise=True, sr=True, sr_seed=10)
    qr, _, _ = orc.nvfp4_quantize_1x16(x, colwise=True, sr=False)
    assert not np.array_equal(qa, qb)
    assert not np.array_equal(qa, qr)
    qa2, _, _ = orc.nvfp4_quantize_1x16(x, colwise=True, sr=True, sr_seed=9)
    np.testing.assert_array_equal(qa, qa2)


def test_sr_bits_follow_the_logical_element(orc):
    """The random bits of element (t, n) do not depend on which copy is made:
    with every 16-block holding exactly one entry of the tensor amax (so all
    block scales are 448 in both orientations), the column-wise and row-wise
    SR quantizers round each element the same way."""
    T = N = 64
    rng = np.random.default_rng(46)
    x = (rng.uniform(0.05, 0.9, size=(T, N)) * np.where(rng.random((T, N)) < 0.5, -1, 1)).astype(np.float32)
    for a in range(T // 16):
        for b in range(N // 16):
            for i in range(16):
                x[a * 16 + i, b * 16 + (i * 5 + a + b) % 16] = 1.0
    xb = synthetic.to_bf16_bits(x)
    qc, sc, Sc = orc.nvfp4_quantize_1x16(xb, colwise=True, sr=True, sr_seed=77)
    qr, sr_, Sr = orc.nvfp4_quantize_1x16(xb, colwise=False, sr=True, sr_seed=77)
    assert (sc == 0x7E).all() and (sr_ == 0x7E).all() and Sc == Sr

    def nib(q):
        out = np.empty((q.shape[0], q.shape[1] * 2), dtype=np.uint8)
        out[:, 0::2] = q & 0xF
        out[:, 1::2] = q >> 4
        return out
    np.testing.assert_array_equal(nib(qc).T, nib(qr))


def test_two_pass_split_over_column_slabs_matches_whole_tensor(orc):
    """Pass 1 max-combined over column slabs and pass 2 per slab (with global SR indices) give the
    whole-tensor result: the transform, the blocks and the random bits are all column-local."""
    x = synthetic.random_bf16(47, (64, 48), "student_t")
    q, s, S = orc.nvfp4_quantize_1x16(x, colwise=True, rht=True, rht_seed=8, sr=True, sr_seed=9)
    slabs = [(0, 16), (16, 40), (40, 48)]
    A = max(orc.nvfp4_1x16_amax(np.ascontiguousarray(x[:, a:b]), rht=True, rht_seed=8) for a, b in slabs)
    assert orc.nvfp4_second_scale(A) == S
    for a, b in slabs:
        qs, ss = orc.nvfp4_1x16_pass2(np.ascontiguousarray(x[:, a:b]), a, 48, S, colwise=True, rht=True, rht_seed=8,
                                      sr=True, sr_seed=9)
        np.testing.assert_array_equal(qs, q[a:b])
        np.testing.assert_array_equal(ss, s[a:b])
