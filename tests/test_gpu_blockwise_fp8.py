"""GPU parity: blockwise FP8 quantizers ([1, 128] activation / gradient tiles, [128, 128] weight blocks;
FP32 and power-of-two scales) against the CPU oracle, bit-exact for every code and FP32 scale and for the
E8M0 bytes written into the MXFP8 GEMM scale layout; then the three GEMMs of a linear layer (forward,
data gradient, weight gradient) on power-of-two blockwise operands through the MXFP8 tensor-core GEMM,
against the oracle's FP64 product of the decoded operands (||D - ref||_F / ||ref||_F <= 1e-2)."""
import numpy as np
import pytest
import torch

import synthetic
from gpu_util import DEV, bf16_dev, first_mismatch, to_np

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module")
def mx():
    import microscaled_precision_numerics_gb300 as m
    m.lib()
    return m


def edge_tensor(seed, shape, scale=1.0):
    """Random values with planted boundary cases: BF16 max, subnormals, signed zeros, 448, 449-ish."""
    rng = np.random.default_rng(seed)
    x = synthetic.random_bf16(seed, shape, "student_t", scale)
    flat = x.reshape(-1)
    idx = rng.choice(flat.size, size=min(flat.size, 64), replace=False)
    specials = np.array([0x7F7F, 0xFF7F, 0x0001, 0x8001, 0x007F, 0x8000, 0x0000, 0x0080, 0x3F80, 0x43E0,
                         0x43E1, 0xC3E0], dtype=np.uint16)
    flat[idx] = specials[np.arange(idx.size) % specials.size]
    return x


def zero_tile_rows(x, rows, c0=0):
    x[rows, c0:c0 + 128] = 0
    return x


def u8(shape):
    return torch.zeros(shape, dtype=torch.uint8, device=DEV)


def f32(shape):
    return torch.full(shape, float("nan"), dtype=torch.float32, device=DEV)


def check_codes(got, want):
    assert np.array_equal(to_np(got), want), first_mismatch(to_np(got), want)


def check_scales(got, want):
    g = to_np(got)
    assert np.array_equal(g.view(np.uint32), np.asarray(want, dtype=np.float32).view(np.uint32)), \
        first_mismatch(g.view(np.uint32), np.asarray(want, dtype=np.float32).view(np.uint32))


# ------------------------------------------------------------------------------------------------
# [1, 128] tiles
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("pow2", [False, True])
@pytest.mark.parametrize("R,K", [(37, 256), (200, 384), (1, 128), (1031, 1024)])
def test_rowwise(mx, orc, pow2, R, K):
    x = zero_tile_rows(edge_tensor(R * 3 + K + pow2, (R, K)), slice(0, 1), 128 if K > 128 else 0)
    q, s = u8((R, K)), f32((R, K // 128))
    sf = u8(mx.scale_bytes(R, K, 32)) if pow2 else None
    mx.mx_fp8_blockwise_quantize_1x128(bf16_dev(x), pow2, q_row=q, s_row=s, sf_row=sf)
    torch.cuda.synchronize()
    wq, ws, we8 = orc.fp8_blockwise_1x128(x, pow2)
    check_codes(q, wq)
    check_scales(s, ws)
    if pow2:
        check_codes(sf, orc.scales_to_gemm_layout(orc.fp8_blockwise_e8m0_rowwise(we8)))


def test_rowwise_strided_input(mx, orc):
    base = edge_tensor(4, (64, 640))
    xt = bf16_dev(base)[:, :512]
    q, s = u8((64, 512)), f32((64, 4))
    mx.mx_fp8_blockwise_quantize_1x128(xt, True, q_row=q, s_row=s)
    wq, ws, _ = orc.fp8_blockwise_1x128(np.ascontiguousarray(base[:, :512]), True)
    check_codes(q, wq)
    check_scales(s, ws)


@pytest.mark.parametrize("pow2", [False, True])
@pytest.mark.parametrize("R,K,row", [(256, 384, True), (384, 1024, True), (128, 208, False), (512, 96, False)])
def test_row_and_col(mx, orc, pow2, R, K, row):
    x = edge_tensor(R + K * 5 + pow2, (R, K))
    x[128:256, 3] = 0                                     # one zero column tile
    q_row = u8((R, K)) if row else None
    s_row = f32((R, K // 128)) if row else None
    sf_row = u8(mx.scale_bytes(R, K, 32)) if (row and pow2) else None
    q_col, s_col = u8((K, R)), f32((K, R // 128))
    sf_col = u8(mx.scale_bytes(K, R, 32)) if pow2 else None
    mx.mx_fp8_blockwise_quantize_1x128(bf16_dev(x), pow2, q_row=q_row, s_row=s_row, sf_row=sf_row,
                                       q_col=q_col, s_col=s_col, sf_col=sf_col)
    torch.cuda.synchronize()
    if row:
        wq, ws, we8 = orc.fp8_blockwise_1x128(x, pow2)
        check_codes(q_row, wq)
        check_scales(s_row, ws)
        if pow2:
            check_codes(sf_row, orc.scales_to_gemm_layout(orc.fp8_blockwise_e8m0_rowwise(we8)))
    cq, cs, ce8 = orc.fp8_blockwise_1x128(np.ascontiguousarray(x.T), pow2)
    check_codes(q_col, cq)
    check_scales(s_col, cs)
    if pow2:
        check_codes(sf_col, orc.scales_to_gemm_layout(orc.fp8_blockwise_e8m0_rowwise(ce8)))


# ------------------------------------------------------------------------------------------------
# [128, 128] weight blocks
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("pow2", [False, True])
@pytest.mark.parametrize("G,O,H", [(1, 256, 384), (3, 208, 304), (2, 16, 16), (1, 1024, 640)])
def test_weight_blocks(mx, orc, pow2, G, O, H):
    w = np.stack([edge_tensor(100 * g + O + H + pow2, (O, H), 0.02) for g in range(G)])
    w[0, :min(O, 128), :min(H, 128)] = 0                 # a zero block
    q_row, q_col = u8((G, O, H)), u8((G, H, O))
    bo, bh = (O + 127) // 128, (H + 127) // 128
    s = f32((G, bo, bh))
    whole = O % 128 == 0 and H % 128 == 0 and pow2
    sf_row = u8(G * mx.scale_bytes(O, H, 32)) if whole else None
    sf_col = u8(G * mx.scale_bytes(H, O, 32)) if whole else None
    mx.mx_fp8_blockwise_quantize_128x128(bf16_dev(w), pow2, q_row, q_col, s, sf_row=sf_row, sf_col=sf_col)
    torch.cuda.synchronize()
    for g in range(G):
        wr, wc, ws, we8 = orc.fp8_blockwise_128x128(w[g], pow2)
        check_codes(q_row[g], wr)
        check_codes(q_col[g], wc)
        check_scales(s[g], ws)
        if whole:
            n_r, n_c = mx.scale_bytes(O, H, 32), mx.scale_bytes(H, O, 32)
            check_codes(sf_row[g * n_r:(g + 1) * n_r],
                        orc.scales_to_gemm_layout(orc.fp8_blockwise_e8m0_weight(we8, O, H, "row")))
            check_codes(sf_col[g * n_c:(g + 1) * n_c],
                        orc.scales_to_gemm_layout(orc.fp8_blockwise_e8m0_weight(we8, O, H, "col")))


# ------------------------------------------------------------------------------------------------
# GEMMs on power-of-two blockwise operands (the MXFP8 tensor-core GEMM reads them unchanged)
# ------------------------------------------------------------------------------------------------
def gemm(mx, a, sa, b, sb, M, N, K):
    d = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    mx.mx_scaled_gemm(mx.MX_FMT_MXFP8, a, sa, None, 0, b, sb, None, 0, M, N, K, d)
    torch.cuda.synchronize()
    mx.check_device_status()
    return d.float().cpu().numpy().astype(np.float64)


def test_linear_layer_gemms_pow2(mx, orc):
    T, H, O = 512, 384, 640
    x = synthetic.random_bf16(1, (T, H), "student_t")
    w = synthetic.random_bf16(2, (O, H), "normal", 0.02)
    dy = synthetic.random_bf16(3, (T, O), "normal", 1e-3)

    def act(t):
        R, C = t.shape
        q_row, s_row, sf_row = u8((R, C)), f32((R, C // 128)), u8(mx.scale_bytes(R, C, 32))
        q_col, s_col, sf_col = u8((C, R)), f32((C, R // 128)), u8(mx.scale_bytes(C, R, 32))
        mx.mx_fp8_blockwise_quantize_1x128(bf16_dev(t), True, q_row=q_row, s_row=s_row, sf_row=sf_row,
                                           q_col=q_col, s_col=s_col, sf_col=sf_col)
        return q_row, s_row, sf_row, q_col, s_col, sf_col

    xq, xs, xsf, xqc, xsc, xsfc = act(x)
    gq, gs, gsf, gqc, gsc, gsfc = act(dy)
    wq_row, wq_col, wsc = u8((1, O, H)), u8((1, H, O)), f32((1, O // 128, H // 128))
    wsf_row, wsf_col = u8(mx.scale_bytes(O, H, 32)), u8(mx.scale_bytes(H, O, 32))
    mx.mx_fp8_blockwise_quantize_128x128(bf16_dev(w[None]), True, wq_row, wq_col, wsc, sf_row=wsf_row,
                                         sf_col=wsf_col)

    # reference: the oracle's quantization of the same inputs, decoded exactly, multiplied in FP64
    def ref_act(t):
        q, _, e8 = orc.fp8_blockwise_1x128(t, True)
        qc, _, e8c = orc.fp8_blockwise_1x128(np.ascontiguousarray(t.T), True)
        return (orc.decode_mxfp8_f64(q, orc.fp8_blockwise_e8m0_rowwise(e8)),
                orc.decode_mxfp8_f64(qc, orc.fp8_blockwise_e8m0_rowwise(e8c)))

    X, Xc = ref_act(x)
    G, Gc = ref_act(dy)
    rq, cq, _, we8 = orc.fp8_blockwise_128x128(w, True)
    W = orc.decode_mxfp8_f64(rq, orc.fp8_blockwise_e8m0_weight(we8, O, H, "row"))
    Wc = orc.decode_mxfp8_f64(cq, orc.fp8_blockwise_e8m0_weight(we8, O, H, "col"))
    y = gemm(mx, xq, xsf, wq_row[0], wsf_row, T, O, H)                   # forward  Y  = X W^T
    assert orc.rel_fro_error(y, X @ W.T) <= TOL
    dx = gemm(mx, gq, gsf, wq_col[0], wsf_col, T, H, O)                 # data     dX = dY W
    assert orc.rel_fro_error(dx, G @ Wc.T) <= TOL
    dw = gemm(mx, gqc, gsfc, xqc, xsfc, O, H, T)                         # weight   dW = dY^T X
    assert orc.rel_fro_error(dw, Gc @ Xc.T) <= TOL
    # and against the unquantized product, loosely (E4M3 operands)
    xf, wf = orc.bf16_to_f32(x).astype(np.float64), orc.bf16_to_f32(w).astype(np.float64)
    assert orc.rel_fro_error(y, xf @ wf.T) <= 0.1


# ------------------------------------------------------------------------------------------------
# FP32-scale blockwise GEMM (scaling around the tensor cores)
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (512, 640, 1024), (200, 296, 384), (1, 8, 128),
                                   (1024, 1280, 4096)])
def test_fp32_scale_gemm(mx, orc, M, N, K):
    """Operands from the oracle quantizers (X [1,128] row-wise, W [128,128]); FPROP D = X W^T."""
    x = synthetic.random_bf16(M + N + K, (M, K), "student_t")
    w = synthetic.random_bf16(M + 2 * N + K, (N, K), "normal", 0.02)
    qx, sx, _ = orc.fp8_blockwise_1x128(x, False)
    qw, _, sw, _ = orc.fp8_blockwise_128x128(w, False)
    d = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    mx.mx_fp8_blockwise_gemm(torch.from_numpy(qx).to(DEV), torch.from_numpy(sx).to(DEV),
                             torch.from_numpy(qw).to(DEV), torch.from_numpy(np.ascontiguousarray(sw)).to(DEV),
                             M, N, K, d)
    torch.cuda.synchronize()
    mx.check_device_status()
    ref = orc.gemm_ref_fp8_blockwise(qx, sx, qw, sw)
    got = d.float().cpu().numpy().astype(np.float64)
    assert orc.rel_fro_error(got, ref) <= TOL
    A = orc.fp8_blockwise_decode_f64(qx, sx, 1, 128)
    B = orc.fp8_blockwise_decode_f64(qw, sw, 128, 128)
    bound = 2.0 ** -7 * np.abs(ref) + 2.0 ** -15 * (np.abs(A) @ np.abs(B).T) + 1e-30
    assert not (np.abs(got - ref) > bound).any()


def test_fp32_scale_gemm_dgrad_with_gpu_quantizers(mx, orc):
    """DGRAD dX = dY W with the GPU quantizers' outputs: dY [1,128] row-wise, W's column-wise codes with the
    transposed block scales."""
    T, O, H = 512, 768, 384
    w = synthetic.random_bf16(51, (O, H), "normal", 0.02)
    dy = synthetic.random_bf16(52, (T, O), "normal", 1e-3)
    q_row, q_col, s = u8((1, O, H)), u8((1, H, O)), f32((1, O // 128, H // 128))
    mx.mx_fp8_blockwise_quantize_128x128(bf16_dev(w[None]), False, q_row, q_col, s)
    qg, sg = u8((T, O)), f32((T, O // 128))
    mx.mx_fp8_blockwise_quantize_1x128(bf16_dev(dy), False, q_row=qg, s_row=sg)
    d = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    mx.mx_fp8_blockwise_gemm(qg, sg, q_col[0], s[0].t().contiguous(), T, H, O, d)
    torch.cuda.synchronize()
    mx.check_device_status()
    rq, rs, _ = orc.fp8_blockwise_1x128(dy, False)
    _, wc, ws, _ = orc.fp8_blockwise_128x128(w, False)
    ref = orc.gemm_ref_fp8_blockwise(rq, rs, wc, np.ascontiguousarray(ws.T))
    assert orc.rel_fro_error(d.float().cpu().numpy().astype(np.float64), ref) <= TOL


@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (384, 640, 1024), (200, 296, 384), (1, 8, 128),
                                   (1024, 1280, 4096), (512, 384, 640)])
def test_fp32_scale_gemm_wgrad(mx, orc, M, N, K):
    """WGRAD dW = dY^T X with both operands the column-wise [1, 128] copies (tiles along tokens = K) and one
    FP32 scale per row and 128-token block; operands from the oracle quantizer (column-wise = row-wise of the
    transpose)."""
    dyT = synthetic.random_bf16(M + N + 7 * K, (M, K), "normal", 1e-3)
    xT = synthetic.random_bf16(M + 3 * N + K, (N, K), "student_t")
    qa, sa, _ = orc.fp8_blockwise_1x128(dyT, False)
    qb, sb, _ = orc.fp8_blockwise_1x128(xT, False)
    d = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    mx.mx_fp8_blockwise_gemm_wgrad(torch.from_numpy(qa).to(DEV), torch.from_numpy(sa).to(DEV),
                                   torch.from_numpy(qb).to(DEV), torch.from_numpy(sb).to(DEV), M, N, K, d)
    torch.cuda.synchronize()
    mx.check_device_status()
    ref = orc.gemm_ref_fp8_blockwise_wgrad(qa, sa, qb, sb)
    got = d.float().cpu().numpy().astype(np.float64)
    assert orc.rel_fro_error(got, ref) <= TOL
    A = orc.fp8_blockwise_decode_f64(qa, sa, 1, 128)
    B = orc.fp8_blockwise_decode_f64(qb, sb, 1, 128)
    bound = 2.0 ** -7 * np.abs(ref) + 2.0 ** -15 * (np.abs(A) @ np.abs(B).T) + 1e-30
    assert not (np.abs(got - ref) > bound).any()


def test_fp32_scale_gemm_wgrad_integer_exact(mx, orc):
    """Small-integer codes with power-of-two FP32 scales: every partial sum and every promoted product is
    exact in FP32, so the GEMM must equal the reference bit for bit after BF16 rounding."""
    rng = np.random.default_rng(21)
    M, N, K = 256, 384, 512
    ints = np.array([0x00, 0x30, 0x38, 0x3C, 0x40, 0x44, 0xB8, 0xC0], dtype=np.uint8)   # 0, +-0.5..3
    qa = ints[rng.integers(0, ints.size, size=(M, K))]
    qb = ints[rng.integers(0, ints.size, size=(N, K))]
    sa = (2.0 ** rng.integers(-2, 3, size=(M, K // 128))).astype(np.float32)
    sb = (2.0 ** rng.integers(-2, 3, size=(N, K // 128))).astype(np.float32)
    d = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    mx.mx_fp8_blockwise_gemm_wgrad(torch.from_numpy(qa).to(DEV), torch.from_numpy(sa).to(DEV),
                                   torch.from_numpy(qb).to(DEV), torch.from_numpy(sb).to(DEV), M, N, K, d)
    torch.cuda.synchronize()
    ref = orc.gemm_ref_fp8_blockwise_wgrad(qa, sa, qb, sb)
    want = torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    got = d.view(torch.int16).cpu().numpy()
    assert np.array_equal(got, want), first_mismatch(got, want)


def test_fp32_scale_gemm_wgrad_with_gpu_quantizers(mx, orc):
    """The weight gradient of a linear layer from the GPU quantizers' column-wise outputs: dY [T, O] and X [T, H]
    quantized in [1, 128] tiles along tokens, dW [O, H] = dY^T X, against the oracle's quantization of the same
    tensors (codes and scales compared bit-exact first)."""
    T, O, H = 1024, 768, 512
    dy = synthetic.random_bf16(61, (T, O), "normal", 1e-3)
    x = synthetic.random_bf16(62, (T, H), "student_t")
    qdy, sdy = u8((O, T)), f32((O, T // 128))
    qx, sx = u8((H, T)), f32((H, T // 128))
    mx.mx_fp8_blockwise_quantize_1x128(bf16_dev(dy), False, q_col=qdy, s_col=sdy)
    mx.mx_fp8_blockwise_quantize_1x128(bf16_dev(x), False, q_col=qx, s_col=sx)
    d = torch.full((O, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    mx.mx_fp8_blockwise_gemm_wgrad(qdy, sdy, qx, sx, O, H, T, d)
    torch.cuda.synchronize()
    mx.check_device_status()
    rq_dy, rs_dy, _ = orc.fp8_blockwise_1x128(np.ascontiguousarray(dy.T), False)
    rq_x, rs_x, _ = orc.fp8_blockwise_1x128(np.ascontiguousarray(x.T), False)
    assert np.array_equal(to_np(qdy), rq_dy) and np.array_equal(to_np(sdy), rs_dy)
    assert np.array_equal(to_np(qx), rq_x) and np.array_equal(to_np(sx), rs_x)
    ref = orc.gemm_ref_fp8_blockwise_wgrad(rq_dy, rs_dy, rq_x, rs_x)
    assert orc.rel_fro_error(d.float().cpu().numpy().astype(np.float64), ref) <= TOL
