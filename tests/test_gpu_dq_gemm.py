"""GPU parity: the BF16 GEMM with a dequantized-NVFP4 B operand expanded inside the GEMM (the dequantized
backward without a BF16 copy of the weight) against the oracle's FP64 product of A and the oracle's BF16
DQ(B).  Bar: ||D - ref||_F / ||ref||_F <= 1e-2 plus the element-wise diagnostic of the block-scaled GEMM
tests; operands whose every partial sum is exact in FP32 must match the reference bit for bit after BF16
rounding.  Operands are produced by the oracle, so the GEMM is checked independently of the GPU
quantizers; one case also runs the GPU 2D weight quantizer to feed it."""
import numpy as np
import pytest
import torch

import synthetic
from gpu_util import DEV, bf16_dev

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module")
def mx():
    import microscaled_precision_numerics_gb300 as m
    m.lib()
    return m


def dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).to(DEV)


def dev_f32(a):
    return torch.from_numpy(np.ascontiguousarray(np.atleast_1d(a), dtype=np.float32)).to(DEV)


def run(mx, orc, a, qb, sb_compact, sb2, per_row, M, N, K, alpha_a=None):
    d = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    aa = dev_f32(alpha_a) if alpha_a is not None else None
    scope_a = (mx.MX_SCOPE_ROW if np.ndim(alpha_a) else mx.MX_SCOPE_TENSOR) if alpha_a is not None else 0
    mx.mx_gemm_bf16_dq_nvfp4(bf16_dev(a), dev_u8(qb), dev_u8(orc.scales_to_gemm_layout(sb_compact)), dev_f32(sb2),
                             mx.MX_SCOPE_ROW if per_row else mx.MX_SCOPE_TENSOR, M, N, K, d, alpha_a=aa,
                             alpha_a_scope=scope_a)
    torch.cuda.synchronize()
    mx.check_device_status()
    ref = orc.gemm_ref_bf16_dq_nvfp4(a, qb, sb_compact, sb2, per_row, alpha_a=alpha_a)
    A = orc.bf16_to_f32(a).astype(np.float64)
    B = orc.bf16_to_f32(orc.dequant_nvfp4(qb, sb_compact, sb2, per_row)).astype(np.float64)
    absprod = np.abs(A) @ np.abs(B).T
    if alpha_a is not None:
        absprod = absprod * np.abs(np.asarray(alpha_a, dtype=np.float64)).reshape(-1, 1)
    return d.float().cpu().numpy().astype(np.float64), ref, absprod


def check(orc, got, ref, absprod):
    err = orc.rel_fro_error(got, ref)
    assert err <= TOL, f"relative Frobenius error {err}"
    bound = 2.0 ** -7 * np.abs(ref) + 2.0 ** -15 * absprod + 1e-30
    bad = np.abs(got - ref) > bound
    assert not bad.any(), f"{int(bad.sum())} elements outside the element-wise bound; first {np.argwhere(bad)[0]}"


@pytest.mark.parametrize("M,N,K", [(256, 256, 64), (512, 512, 1024), (200, 304, 192), (1, 16, 64),
                                   (640, 1280, 2048), (384, 144, 320)])
def test_dgrad_with_2d_weight(mx, orc, M, N, K):
    """dX = dY DQ(W): A = dY [T, O] (K = O), B = the column-wise codes of W [O, H] quantized in 16x16 tiles
    (N = H), one FP32 scale for the matrix."""
    O, H = K, N
    w = synthetic.random_bf16(M + N + K, (O, H), "normal", 0.02)
    _, q_col, st, s_w = orc.nvfp4_quantize_weight_2d(w)
    dy = synthetic.random_bf16(M * 3 + K, (M, O), "student_t", 1e-3)
    got, ref, absprod = run(mx, orc, dy, q_col, orc.weight_2d_operand_scales(st, "col"), s_w, False, M, N, K)
    check(orc, got, ref, absprod)


def test_per_row_second_level_scale_and_row_alpha(mx, orc):
    """B quantized per row (per-token NVFP4), its S per B row; a per-row alpha on A."""
    M, N, K = 384, 512, 768
    b = synthetic.random_bf16(5, (N, K), "student_t")
    qb, sb, sb2 = orc.nvfp4_quantize_per_token(b)
    a = synthetic.random_bf16(6, (M, K), "normal")
    alpha = (2.0 ** np.random.default_rng(7).integers(-3, 3, size=M)).astype(np.float32)
    got, ref, absprod = run(mx, orc, a, qb, sb, sb2, True, M, N, K, alpha_a=alpha)
    check(orc, got, ref, absprod)


def test_integer_exact(mx, orc):
    """A small integers, B codes under block scale 1.0 (E4M3 0x38) and S = 1: every partial sum is a
    multiple of 0.5 well inside FP32's exact range, so D = BF16(ref) exactly."""
    M, N, K = 256, 512, 1024
    rng = np.random.default_rng(3)
    a_f = rng.integers(-2, 3, size=(M, K)).astype(np.float32)
    a = (a_f.view(np.uint32) >> 16).astype(np.uint16)
    qb = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sb = np.full((N, K // 16), 0x38, dtype=np.uint8)
    got, ref, _ = run(mx, orc, a, qb, sb, np.float32(1.0), False, M, N, K)
    want = orc.bf16_to_f32(np.array([orc.float_to_bf16(float(v)) for v in ref.reshape(-1)], dtype=np.uint16))
    assert np.array_equal(got.reshape(-1), want.astype(np.float64))


def test_fed_by_the_gpu_weight_quantizer(mx, orc):
    """The GPU 2D weight quantizer's column-wise output feeds the GEMM directly (the layout the quantizer
    writes is the one the GEMM reads)."""
    T, O, H = 512, 1024, 768
    w = synthetic.random_bf16(8, (O, H), "normal", 0.02)
    dy = synthetic.random_bf16(9, (T, O), "student_t", 1e-3)
    out = mx.alloc_nvfp4_weight_2d(1, O, H, DEV)
    mx.mx_nvfp4_quantize_weight_2d(bf16_dev(w)[None], out["q_row"], out["s_row"], out["q_col"], out["s_col"],
                                   out["s_w"], out["ws"])
    d = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    mx.mx_gemm_bf16_dq_nvfp4(bf16_dev(dy), out["q_col"][0], out["s_col"], out["s_w"], mx.MX_SCOPE_TENSOR, T, H, O, d)
    torch.cuda.synchronize()
    mx.check_device_status()
    _, q_col, st, s_w = orc.nvfp4_quantize_weight_2d(w)
    ref = orc.gemm_ref_bf16_dq_nvfp4(dy, q_col, orc.weight_2d_operand_scales(st, "col"), s_w, False)
    assert orc.rel_fro_error(d.float().cpu().numpy().astype(np.float64), ref) <= TOL


def run_wgrad(mx, orc, dy, qx, sx_compact, sx2, per_row):
    T, O = dy.shape
    H = qx.shape[1] * 2
    dw = torch.full((O, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    mx.mx_wgrad_bf16_dq_nvfp4(bf16_dev(dy), dev_u8(qx), dev_u8(orc.scales_to_gemm_layout(sx_compact)), dev_f32(sx2),
                              mx.MX_SCOPE_ROW if per_row else mx.MX_SCOPE_TENSOR, dw)
    torch.cuda.synchronize()
    mx.check_device_status()
    Y = orc.bf16_to_f32(dy).astype(np.float64)
    X = orc.bf16_to_f32(orc.dequant_nvfp4(qx, sx_compact, sx2, per_row)).astype(np.float64)
    ref = Y.T @ X                  # the dequantized-backward weight gradient: dY^T DQ(X), FP64
    return dw.float().cpu().numpy().astype(np.float64), ref, np.abs(Y).T @ np.abs(X)


@pytest.mark.parametrize("T,O,H", [(256, 256, 256), (512, 384, 320), (64, 128, 64), (1024, 640, 1024),
                                   (2048, 1536, 768)])
def test_wgrad_per_token_activations(mx, orc, T, O, H):
    """dW = dY^T DQ(X): X quantized per token (1x16 along H, one FP32 scale per token), tokens along K."""
    x = synthetic.random_bf16(T + O + H, (T, H), "student_t")
    qx, sx, sx2 = orc.nvfp4_quantize_per_token(x)
    dy = synthetic.random_bf16(T * 3 + O, (T, O), "normal", 1e-3)
    got, ref, absprod = run_wgrad(mx, orc, dy, qx, sx, sx2, True)
    check(orc, got, ref, absprod)


def test_wgrad_per_tensor_scale(mx, orc):
    T, O, H = 512, 256, 512
    x = synthetic.random_bf16(41, (T, H), "normal")
    qx, sx, S = orc.nvfp4_quantize_1x16(x, colwise=False)
    dy = synthetic.random_bf16(42, (T, O), "normal", 1e-2)
    got, ref, absprod = run_wgrad(mx, orc, dy, qx, sx, S, False)
    check(orc, got, ref, absprod)
