"""GPU parity: block-scaled tcgen05 GEMMs (dense MXFP8 / NVFP4, grouped) against the oracle's FP64
reference on exactly decoded operands.

Operands are produced by the CPU oracle, so the GEMM is checked independently of the GPU
quantizers.  Bar: ||D - ref||_F / ||ref||_F <= 1e-2 (BF16 output), plus an element-wise diagnostic
|D - ref| <= 2^-7 |ref| + 2^-15 sum_k |a_k b_k|.  Small-integer operands whose every partial sum is
exact in FP32 must match the reference bit for bit after BF16 rounding.
"""
import numpy as np
import pytest
import torch

import synthetic
from gpu_util import DEV, first_mismatch

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


def check_close(orc, d, ref, absprod):
    got = d.float().cpu().numpy().astype(np.float64)
    err = orc.rel_fro_error(got, ref)
    assert err <= TOL, f"relative Frobenius error {err}"
    bound = 2.0 ** -7 * np.abs(ref) + 2.0 ** -15 * absprod + 1e-30
    bad = np.abs(got - ref) > bound
    assert not bad.any(), f"{int(bad.sum())} elements outside the element-wise bound; first {np.argwhere(bad)[0]}"
    return err


def run_mxfp8(mx, orc, a, b, M, N, K):
    qa, sa = orc.mxfp8_quantize_rowwise(a)
    qb, sb = orc.mxfp8_quantize_rowwise(b)
    d = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    mx.mx_scaled_gemm(mx.MX_FMT_MXFP8, dev_u8(qa), dev_u8(orc.scales_to_gemm_layout(sa)), None, 0,
                      dev_u8(qb), dev_u8(orc.scales_to_gemm_layout(sb)), None, 0, M, N, K, d)
    torch.cuda.synchronize()
    mx.check_device_status()
    A, B = orc.decode_mxfp8_f64(qa, sa), orc.decode_mxfp8_f64(qb, sb)
    return d, A @ B.T, np.abs(A) @ np.abs(B).T


# (4096, 4000, 1024) and (2304, 4096, 128) give every CTA pair several tiles (more than the 76 pairs of
# the GPU run at once), so the accumulator slots rotate and their barriers wrap; one with K beyond the
# 6-stage ring and a ragged N, one with a single K stage.  The last two are wide enough for the
# 256 x 384 tiles (two MMAs per K step, B rows in three 64-row boxes): several tiles per pair, K beyond
# that ring's 5 stages, and a ragged M with a ragged last column tile (12280 = 31 x 384 + 376)
@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (128, 256, 512), (256, 512, 1024), (200, 296, 384),
                                   (1, 8, 128), (640, 1280, 2048), (4096, 4000, 1024), (2304, 4096, 128),
                                   (2304, 12288, 1024), (2000, 12280, 384)])
def test_mxfp8_gemm(mx, orc, M, N, K):
    a = synthetic.random_bf16(M + K, (M, K), "student_t")
    b = synthetic.random_bf16(N + K + 1, (N, K), "normal", 0.02)
    d, ref, absprod = run_mxfp8(mx, orc, a, b, M, N, K)
    check_close(orc, d, ref, absprod)


def test_mxfp8_gemm_tiny_config(mx, orc):
    """The tiny workload: activation 256x1024 (outliers, zero and subnormal blocks) times weight 512x1024."""
    data = synthetic.tiny()
    d, ref, absprod = run_mxfp8(mx, orc, data["x"], data["w"], 256, 512, 1024)
    check_close(orc, d, ref, absprod)


# the second shape runs on the 256 x 384 tiles
@pytest.mark.parametrize("M,N,K", [(256, 512, 256), (2304, 12288, 256)])
def test_mxfp8_gemm_integer_exact(mx, orc, M, N, K):
    rng = np.random.default_rng(0)
    ia = rng.integers(-8, 9, size=(M, K))
    ib = rng.integers(-8, 9, size=(N, K))
    enc = np.array([orc.e4m3_encode(float(v)) for v in range(-8, 9)], dtype=np.uint8)
    qa, qb = enc[ia + 8], enc[ib + 8]
    sa = np.full((M, K // 32), 127, dtype=np.uint8)
    sb = np.full((N, K // 32), 127, dtype=np.uint8)
    d = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    mx.mx_scaled_gemm(mx.MX_FMT_MXFP8, dev_u8(qa), dev_u8(orc.scales_to_gemm_layout(sa)), None, 0,
                      dev_u8(qb), dev_u8(orc.scales_to_gemm_layout(sb)), None, 0, M, N, K, d)
    # integer products summed exactly (|sum| <= 64 K < 2^24) in FP64, then rounded once to BF16
    ref = torch.from_numpy((ia.astype(np.float64) @ ib.T.astype(np.float64)).astype(np.float32)).to(torch.bfloat16)
    got = d.cpu()
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), first_mismatch(got.float().numpy(), ref.float().numpy())


def test_mxfp8_gemm_rejects_wrong_scale_layout(mx, orc):
    """Scales passed in the compact layout instead of the GEMM layout give a large error: the
    parity check catches a stale or un-rearranged scale copy (E2E page, Table 10 F3)."""
    M, N, K = 256, 512, 1024
    a = synthetic.random_bf16(5, (M, K), "student_t")
    b = synthetic.random_bf16(6, (N, K), "normal", 0.02)
    qa, sa = orc.mxfp8_quantize_rowwise(a)
    qb, sb = orc.mxfp8_quantize_rowwise(b)
    wrong_a = np.zeros(orc.scale_layout_bytes(M, K // 32), dtype=np.uint8)
    wrong_a[:sa.size] = sa.reshape(-1)
    d = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    mx.mx_scaled_gemm(mx.MX_FMT_MXFP8, dev_u8(qa), dev_u8(wrong_a), None, 0,
                      dev_u8(qb), dev_u8(orc.scales_to_gemm_layout(sb)), None, 0, M, N, K, d)
    err = orc.rel_fro_error(d.float().cpu().numpy(), orc.gemm_ref_mxfp8(qa, sa, qb, sb))
    assert err > 0.1


# ------------------------------------------------------------------------------------------------
# NVFP4
# ------------------------------------------------------------------------------------------------
# K <= 768 (at most three K stages) writes through 32 x 64-column staged stores, longer K through
# 32 x 16-column ones; the last shape gives every CTA pair several tiles with a ragged M and a ragged
# last 64-column store (4040 = 63 x 64 + 8)
@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (256, 512, 1024), (200, 296, 512), (640, 768, 2048),
                                   (2000, 4040, 768)])
def test_nvfp4_gemm_per_token_times_per_tensor(mx, orc, M, N, K):
    a = synthetic.random_bf16(M * 3 + K, (M, K), "student_t")
    b = synthetic.random_bf16(N * 3 + K, (N, K), "normal", 0.02)
    qa, sa, sta = orc.nvfp4_quantize_per_token(a)
    qb, sb, Sb = orc.nvfp4_quantize_1x16(b, colwise=False)
    d = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    mx.mx_scaled_gemm(mx.MX_FMT_NVFP4, dev_u8(qa), dev_u8(orc.scales_to_gemm_layout(sa)), dev_f32(sta), mx.MX_SCOPE_ROW,
                      dev_u8(qb), dev_u8(orc.scales_to_gemm_layout(sb)), dev_f32(Sb), mx.MX_SCOPE_TENSOR, M, N, K, d)
    torch.cuda.synchronize()
    mx.check_device_status()
    A = orc.decode_nvfp4_f64(qa, sa) * sta.astype(np.float64)[:, None]
    B = orc.decode_nvfp4_f64(qb, sb) * np.float64(Sb)
    check_close(orc, d, A @ B.T, np.abs(A) @ np.abs(B).T)


def test_nvfp4_gemm_integer_exact(mx, orc):
    rng = np.random.default_rng(1)
    M, N, K = 128, 256, 512
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    ca = rng.integers(0, 16, size=(M, K)).astype(np.uint8)
    cb = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    pack = lambda c: (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
    one = orc.e4m3_encode(1.0)
    sa = np.full((M, K // 16), one, dtype=np.uint8)
    sb = np.full((N, K // 16), one, dtype=np.uint8)
    d = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    mx.mx_scaled_gemm(mx.MX_FMT_NVFP4, dev_u8(pack(ca)), dev_u8(orc.scales_to_gemm_layout(sa)), None, 0,
                      dev_u8(pack(cb)), dev_u8(orc.scales_to_gemm_layout(sb)), None, 0, M, N, K, d)
    va = grid[ca & 7] * np.where(ca & 8, -1, 1)
    vb = grid[cb & 7] * np.where(cb & 8, -1, 1)
    ref = torch.from_numpy((va @ vb.T).astype(np.float32)).to(torch.bfloat16)
    assert torch.equal(d.cpu().view(torch.int16), ref.view(torch.int16))


def test_nvfp4_gemm_2d_weights_fprop_dgrad(mx, orc):
    """FPROP with the row-wise 2D weight copy and DGRAD with its transposed copy see the same
    dequantized weight values (MaxText page, 2D weight scaling)."""
    T, O, H = 256, 512, 768
    x = synthetic.random_bf16(7, (T, H), "student_t")
    dy = synthetic.random_bf16(8, (T, O), "normal", 1e-3)
    w = synthetic.random_bf16(9, (O, H), "normal", 0.02)
    qr, qc, st, sw = orc.nvfp4_quantize_weight_2d(w)
    qx, sx, stx = orc.nvfp4_quantize_per_token(x)
    qd, sd, std_ = orc.nvfp4_quantize_per_token(dy)
    # FPROP: Y[T, O] = X . W^T
    y = torch.empty((T, O), dtype=torch.bfloat16, device=DEV)
    mx.mx_scaled_gemm(mx.MX_FMT_NVFP4, dev_u8(qx), dev_u8(orc.scales_to_gemm_layout(sx)), dev_f32(stx), 2,
                      dev_u8(qr), dev_u8(orc.scales_to_gemm_layout(orc.weight_2d_operand_scales(st, "row"))),
                      dev_f32(sw), 1, T, O, H, y)
    # DGRAD: dX[T, H] = dY . W  (B = W^T, rows h, K = o)
    dx = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    mx.mx_scaled_gemm(mx.MX_FMT_NVFP4, dev_u8(qd), dev_u8(orc.scales_to_gemm_layout(sd)), dev_f32(std_), 2,
                      dev_u8(qc), dev_u8(orc.scales_to_gemm_layout(orc.weight_2d_operand_scales(st, "col"))),
                      dev_f32(sw), 1, T, H, O, dx)
    Wd = orc.decode_nvfp4_f64(qr, orc.weight_2d_operand_scales(st, "row")) * np.float64(sw)
    X = orc.decode_nvfp4_f64(qx, sx) * stx.astype(np.float64)[:, None]
    D = orc.decode_nvfp4_f64(qd, sd) * std_.astype(np.float64)[:, None]
    check_close(orc, y, X @ Wd.T, np.abs(X) @ np.abs(Wd).T)
    check_close(orc, dx, D @ Wd, np.abs(D) @ np.abs(Wd))


# ------------------------------------------------------------------------------------------------
# grouped (expert-sorted rows)
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("fmt", [0, 1])
def test_grouped_gemm_ragged(mx, orc, fmt):
    sizes = [0, 130, 7, 300, 128, 1]
    G, N, K = len(sizes), 512, 512
    offs = np.zeros(G + 1, dtype=np.int64)
    offs[1:] = np.cumsum(sizes)
    R = int(offs[-1])
    a = synthetic.random_bf16(11, (R, K), "student_t")
    w = synthetic.random_bf16(12, (G, N, K), "normal", 0.02)
    if fmt == 1:
        qa, sa, sta = orc.nvfp4_quantize_per_token(a)
        qbs, sbs, sws = [], [], []
        for g in range(G):
            q, s, S = orc.nvfp4_quantize_1x16(np.ascontiguousarray(w[g]), colwise=False)
            qbs.append(q); sbs.append(orc.scales_to_gemm_layout(s)); sws.append(S)
        alpha_a, alpha_b = dev_f32(sta), dev_f32(np.array(sws, dtype=np.float32))
        decode = lambda q, s: orc.decode_nvfp4_f64(q, s)
    else:
        qa, sa = orc.mxfp8_quantize_rowwise(a)
        sta = np.ones(R, dtype=np.float32)
        qbs, sbs, sws = [], [], []
        for g in range(G):
            q, s = orc.mxfp8_quantize_rowwise(np.ascontiguousarray(w[g]))
            qbs.append(q); sbs.append(orc.scales_to_gemm_layout(s)); sws.append(1.0)
        alpha_a, alpha_b = None, None
        decode = lambda q, s: orc.decode_mxfp8_f64(q, s)
    d = torch.full((R, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    sa_grouped = orc.scales_to_grouped_layout(sa, offs, mx.grouped_scale_bytes(R, G, K, 32 if fmt == 0 else 16))
    mx.mx_grouped_scaled_gemm(fmt, torch.from_numpy(offs).to(DEV), dev_u8(qa), dev_u8(sa_grouped),
                              alpha_a, dev_u8(np.stack(qbs)), dev_u8(np.concatenate(sbs)), alpha_b, N, K, d)
    torch.cuda.synchronize()
    mx.check_device_status()
    scols = K // (32 if fmt == 0 else 16)
    A = decode(qa, sa) * sta.astype(np.float64)[:, None]
    for g in range(G):
        if sizes[g] == 0:
            continue
        r0, r1 = offs[g], offs[g + 1]
        sb_c = orc.scales_from_gemm_layout(sbs[g], N, scols)
        B = decode(qbs[g], sb_c) * np.float64(sws[g])
        ref = A[r0:r1] @ B.T
        check_close(orc, d[r0:r1], ref, np.abs(A[r0:r1]) @ np.abs(B).T)


def test_nvfp4_gemm_per_column_alpha(mx, orc):
    """Both operands per-token quantized: the B side's FP32 scales are per output column."""
    M, N, K = 384, 520, 512
    a = synthetic.random_bf16(21, (M, K), "student_t")
    b = synthetic.random_bf16(22, (N, K), "student_t")
    qa, sa, sta = orc.nvfp4_quantize_per_token(a)
    qb, sb, stb = orc.nvfp4_quantize_per_token(b)
    d = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    mx.mx_scaled_gemm(mx.MX_FMT_NVFP4, dev_u8(qa), dev_u8(orc.scales_to_gemm_layout(sa)), dev_f32(sta), mx.MX_SCOPE_ROW,
                      dev_u8(qb), dev_u8(orc.scales_to_gemm_layout(sb)), dev_f32(stb), mx.MX_SCOPE_ROW, M, N, K, d)
    A = orc.decode_nvfp4_f64(qa, sa) * sta.astype(np.float64)[:, None]
    B = orc.decode_nvfp4_f64(qb, sb) * stb.astype(np.float64)[:, None]
    check_close(orc, d, A @ B.T, np.abs(A) @ np.abs(B).T)
