"""GPU parity at the workloads' full sizes, in the launch configuration bench.py times, checked on
sampled outputs the oracle computes one by one.

Every quantizer output is per row, per column or per tile, so the oracle recomputes sampled rows,
column slabs or experts from the same BF16 inputs and the device bytes must match exactly; the
per-tensor scale of the WGRAD operands is rebuilt by the oracle over the whole tensor (slab by
slab).  GEMM outputs are checked on sampled row x column blocks against the FP64 reference on the
oracle's own quantization of the sampled operand rows.
"""
import numpy as np
import pytest
import torch

import synthetic
from gpu_util import DEV, bf16_dev, first_mismatch, to_np, to_np_u16

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module")
def mx():
    import microscaled_precision_numerics_gb300 as m
    m.lib()
    return m


def laid_rows(orc, laid, rows_total, scols, rows):
    """Compact scales of the selected rows out of a GEMM-layout scale tensor."""
    full = orc.scales_from_gemm_layout(laid, rows_total, scols)
    return full[rows]


def check_block(orc, got, ref, absprod):
    got = got.astype(np.float64)
    err = orc.rel_fro_error(got, ref)
    assert err <= TOL, f"relative Frobenius error {err}"
    bad = np.abs(got - ref) > 2.0 ** -7 * np.abs(ref) + 2.0 ** -15 * absprod + 1e-30
    assert not bad.any(), f"{int(bad.sum())} sampled elements outside the element-wise bound"


# ------------------------------------------------------------------------------------------------
# dense_mlp: Qwen3-8B MLP linear, MXFP8
# ------------------------------------------------------------------------------------------------
@pytest.fixture(scope="module")
def dense(mx):
    d = synthetic.dense_mlp()
    T, H = d["x"].shape
    F = d["w"].shape[0]
    dev = {k: bf16_dev(v) for k, v in d.items()}
    q = {k: mx.alloc_mxfp8(*dev[k].shape, DEV) for k in dev}
    for k in dev:
        mx.mx_quantize_mxfp8(dev[k], **q[k])
    y = torch.empty((T, F), dtype=torch.bfloat16, device=DEV)
    dx = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    dw = torch.empty((F, H), dtype=torch.bfloat16, device=DEV)
    F8 = mx.MX_FMT_MXFP8
    mx.mx_scaled_gemm(F8, q["x"]["q_row"], q["x"]["s_row"], None, 0, q["w"]["q_row"], q["w"]["s_row"], None, 0, T, F, H, y)
    mx.mx_scaled_gemm(F8, q["dy"]["q_row"], q["dy"]["s_row"], None, 0, q["w"]["q_col"], q["w"]["s_col"], None, 0, T, H, F, dx)
    mx.mx_scaled_gemm(F8, q["dy"]["q_col"], q["dy"]["s_col"], None, 0, q["x"]["q_col"], q["x"]["s_col"], None, 0, F, H, T, dw)
    torch.cuda.synchronize()
    mx.check_device_status()
    return {"data": d, "q": q, "y": y, "dx": dx, "dw": dw, "T": T, "H": H, "F": F}


def test_dense_mlp_quantizers_sampled(orc, dense):
    rng = np.random.default_rng(100)
    for name in ("x", "w", "dy"):
        a = dense["data"][name]
        R, K = a.shape
        q = dense["q"][name]
        rows = np.sort(rng.choice(R, 48, replace=False))
        qr, sr = orc.mxfp8_quantize_rowwise(np.ascontiguousarray(a[rows]))
        assert np.array_equal(to_np(q["q_row"])[rows], qr), name
        assert np.array_equal(laid_rows(orc, to_np(q["s_row"]), R, K // 32, rows), sr), name
        c0 = int(rng.integers(0, K // 64)) * 64
        qc, sc = orc.mxfp8_quantize_colwise(np.ascontiguousarray(a[:, c0:c0 + 64]))
        assert np.array_equal(to_np(q["q_col"][c0:c0 + 64]), qc), name
        assert np.array_equal(laid_rows(orc, to_np(q["s_col"]), K, R // 32, np.arange(c0, c0 + 64)), sc), name


def test_dense_mlp_gemms_sampled(orc, dense):
    rng = np.random.default_rng(101)
    d, T, H, F = dense["data"], dense["T"], dense["H"], dense["F"]
    dec = orc.decode_mxfp8_f64

    def rowq(a, rows):
        return dec(*orc.mxfp8_quantize_rowwise(np.ascontiguousarray(a[rows])))

    def colq(a, cols):
        return dec(*orc.mxfp8_quantize_colwise(np.ascontiguousarray(a[:, cols])))

    m = np.sort(rng.choice(T, 64, replace=False))
    n = np.sort(rng.choice(F, 64, replace=False))
    A, B = rowq(d["x"], m), rowq(d["w"], n)                     # FPROP: Y = X W^T
    check_block(orc, dense["y"].float().cpu().numpy()[np.ix_(m, n)], A @ B.T, np.abs(A) @ np.abs(B).T)
    h = np.sort(rng.choice(H, 64, replace=False))
    A, B = rowq(d["dy"], m), colq(d["w"], h)                     # DGRAD: dX = dY W
    check_block(orc, dense["dx"].float().cpu().numpy()[np.ix_(m, h)], A @ B.T, np.abs(A) @ np.abs(B).T)
    o = np.sort(rng.choice(F, 64, replace=False))
    A, B = colq(d["dy"], o), colq(d["x"], h)                     # WGRAD: dW = dY^T X
    check_block(orc, dense["dw"].float().cpu().numpy()[np.ix_(o, h)], A @ B.T, np.abs(A) @ np.abs(B).T)


def test_dense_mlp_gemms_full(orc, dense):
    """Every output element of the three dense-MLP GEMMs (2.47 TFLOP) against the FP64 products of the
    oracle's own MXFP8 quantization of the whole operands: the relative Frobenius error of each output
    within 1e-2.  The element-wise bound is checked on the sampled blocks above."""
    d, T, H, F = dense["data"], dense["T"], dense["H"], dense["F"]
    dec = orc.decode_mxfp8_f64
    X_r = dec(*orc.mxfp8_quantize_rowwise(d["x"]))
    W_r = dec(*orc.mxfp8_quantize_rowwise(d["w"]))
    err = orc.rel_fro_error(dense["y"].float().cpu().numpy().astype(np.float64), X_r @ W_r.T)     # FPROP
    assert err <= TOL, f"FPROP {err}"
    del W_r
    dY_r = dec(*orc.mxfp8_quantize_rowwise(d["dy"]))
    W_c = dec(*orc.mxfp8_quantize_colwise(d["w"]))
    err = orc.rel_fro_error(dense["dx"].float().cpu().numpy().astype(np.float64), dY_r @ W_c.T)   # DGRAD
    assert err <= TOL, f"DGRAD {err}"
    del dY_r, W_c, X_r
    dY_c = dec(*orc.mxfp8_quantize_colwise(d["dy"]))
    X_c = dec(*orc.mxfp8_quantize_colwise(d["x"]))
    err = orc.rel_fro_error(dense["dw"].float().cpu().numpy().astype(np.float64), dY_c @ X_c.T)   # WGRAD
    assert err <= TOL, f"WGRAD {err}"


def test_dense_mlp_fp32_scale_blockwise_sampled(mx, orc, dense):
    """The dense MLP shapes in blockwise FP8 with FP32 scales (NeMo RL FP8 page, the DeepSeek-V3 recipe), in the
    launch configuration `bench.py --workload dense_fp8_blockwise` times: X row-wise [1, 128] and W [128, 128]
    for FPROP; dY and X column-wise [1, 128] (tiles along tokens) for WGRAD.  Sampled codes and scales are
    compared bit-exact with the oracle, sampled 64 x 64 output blocks within the GEMM tolerance of the FP64
    product of the oracle's own quantization."""
    d, T, H, F = dense["data"], dense["T"], dense["H"], dense["F"]
    u8 = lambda *sh: torch.empty(sh, dtype=torch.uint8, device=DEV)
    f32 = lambda *sh: torch.empty(sh, dtype=torch.float32, device=DEV)
    x, w, dy = bf16_dev(d["x"]), bf16_dev(d["w"]), bf16_dev(d["dy"])
    qx, sx, qxc, sxc = u8(T, H), f32(T, H // 128), u8(H, T), f32(H, T // 128)
    mx.mx_fp8_blockwise_quantize_1x128(x, False, q_row=qx, s_row=sx, q_col=qxc, s_col=sxc)
    qdyc, sdyc = u8(F, T), f32(F, T // 128)
    mx.mx_fp8_blockwise_quantize_1x128(dy, False, q_col=qdyc, s_col=sdyc)
    qw, qwc, sw = u8(1, F, H), u8(1, H, F), f32(1, F // 128, H // 128)
    mx.mx_fp8_blockwise_quantize_128x128(w[None], False, qw, qwc, sw)
    y = torch.empty((T, F), dtype=torch.bfloat16, device=DEV)
    dw = torch.empty((F, H), dtype=torch.bfloat16, device=DEV)
    mx.mx_fp8_blockwise_gemm(qx, sx, qw[0], sw[0], T, F, H, y)
    mx.mx_fp8_blockwise_gemm_wgrad(qdyc, sdyc, qxc, sxc, F, H, T, dw)
    torch.cuda.synchronize()
    mx.check_device_status()
    rng = np.random.default_rng(104)
    dec = orc.fp8_blockwise_decode_f64
    # FPROP: 64 rows of X and a 64-row slab of W inside one 128 x 128 block row
    m = np.sort(rng.choice(T, 64, replace=False))
    rq, rs, _ = orc.fp8_blockwise_1x128(np.ascontiguousarray(d["x"][m]), False)
    assert np.array_equal(to_np(qx)[m], rq) and np.array_equal(to_np(sx)[m], rs)
    fb = int(rng.integers(0, F // 128)) * 128
    wq, _, ws, _ = orc.fp8_blockwise_128x128(np.ascontiguousarray(d["w"][fb:fb + 128]), False)
    assert np.array_equal(to_np(qw[0, fb:fb + 128]), wq) and np.array_equal(to_np(sw[0, fb // 128]), ws[0])
    A, B = dec(rq, rs, 1, 128), dec(wq[:64], ws, 128, 128)
    check_block(orc, y.float().cpu().numpy()[m][:, fb:fb + 64], A @ B.T, np.abs(A) @ np.abs(B).T)
    # WGRAD: 64 columns of dY and of X over all tokens, each column's tiles along the tokens
    o0 = int(rng.integers(0, F // 64)) * 64
    h0 = int(rng.integers(0, H // 64)) * 64
    aq, as_, _ = orc.fp8_blockwise_1x128(np.ascontiguousarray(d["dy"][:, o0:o0 + 64].T), False)
    bq, bs, _ = orc.fp8_blockwise_1x128(np.ascontiguousarray(d["x"][:, h0:h0 + 64].T), False)
    assert np.array_equal(to_np(qdyc[o0:o0 + 64]), aq) and np.array_equal(to_np(sdyc[o0:o0 + 64]), as_)
    assert np.array_equal(to_np(qxc[h0:h0 + 64]), bq) and np.array_equal(to_np(sxc[h0:h0 + 64]), bs)
    A, B = dec(aq, as_, 1, 128), dec(bq, bs, 1, 128)
    check_block(orc, dw.float().cpu().numpy()[o0:o0 + 64, h0:h0 + 64], A @ B.T, np.abs(A) @ np.abs(B).T)


# ------------------------------------------------------------------------------------------------
# moe: Qwen3-30B-A3B expert layer, NVFP4
# ------------------------------------------------------------------------------------------------
@pytest.fixture(scope="module")
def moe(mx):
    d = synthetic.moe()
    rows = int(d["group_offsets"][-1])
    x = bf16_dev(d["x"])
    a = x.index_select(0, torch.from_numpy(d["row_token"]).to(DEV)).contiguous()
    G, O1, H = d["w_gate_up"].shape
    offs = torch.from_numpy(d["group_offsets"]).to(DEV)
    qa = mx.alloc_nvfp4_rows_grouped(rows, G, H, DEV)
    mx.mx_nvfp4_quantize_per_token_grouped(a, offs, qa["q"], qa["s"], qa["s2"])
    qw = mx.alloc_nvfp4_weight_2d(G, O1, H, DEV)
    mx.mx_nvfp4_quantize_weight_2d(bf16_dev(d["w_gate_up"]), qw["q_row"], qw["s_row"], qw["q_col"], qw["s_col"],
                                   qw["s_w"], qw["ws"])
    y = torch.empty((rows, O1), dtype=torch.bfloat16, device=DEV)
    mx.mx_grouped_scaled_gemm(mx.MX_FMT_NVFP4, offs, qa["q"], qa["s"], qa["s2"], qw["q_row"], qw["s_row"], qw["s_w"],
                              O1, H, y)
    dq = torch.empty((G * O1, H), dtype=torch.bfloat16, device=DEV)
    mx.mx_dequantize_bf16(mx.MX_FMT_NVFP4, qw["q_row"], qw["s_row"], qw["s_w"], mx.MX_SCOPE_GROUP, G * O1, H, dq,
                          group_rows=O1)
    torch.cuda.synchronize()
    mx.check_device_status()
    return {"d": d, "qa": qa, "qw": qw, "y": y, "dq": dq, "rows": rows, "G": G, "O1": O1, "H": H}


def test_moe_per_token_sampled(orc, moe):
    d, qa, H, R = moe["d"], moe["qa"], moe["H"], moe["rows"]
    rows = np.sort(np.random.default_rng(102).choice(R, 256, replace=False))
    q, s, st = orc.nvfp4_quantize_per_token(np.ascontiguousarray(d["x"][d["row_token"][rows]]))
    assert np.array_equal(to_np(qa["q"])[rows], q)
    offs = d["group_offsets"]
    laid = orc.scales_from_gemm_layout(to_np(qa["s"]), to_np(qa["s"]).size // 512 * 128 // ((H // 16 + 3) // 4), H // 16)
    # padded row of r: its group's first 128-row tile plus the offset inside the group
    g = np.searchsorted(offs, rows, side="right") - 1
    ptile = np.concatenate([[0], np.cumsum((np.diff(offs) + 127) // 128)])
    assert np.array_equal(laid[ptile[g] * 128 + (rows - offs[g])], s)
    assert np.array_equal(to_np(qa["s2"])[rows], st)


def test_moe_weights_grouped_gemm_and_dq_sampled(orc, moe):
    d, qw, G, O1, H = moe["d"], moe["qw"], moe["G"], moe["O1"], moe["H"]
    offs = d["group_offsets"]
    srb = orc.scale_layout_bytes(O1, H // 16)
    dq = to_np_u16(moe["dq"]).reshape(G, O1, H)
    y = moe["y"].float().cpu().numpy()
    for g in (0, 77, G - 1):
        w = np.ascontiguousarray(d["w_gate_up"][g])
        qr, qc, st, sw = orc.nvfp4_quantize_weight_2d(w)
        assert np.array_equal(to_np(qw["q_row"][g]), qr), g
        assert np.array_equal(to_np(qw["q_col"][g]), qc), g
        assert np.array_equal(to_np(qw["s_row"][g * srb:(g + 1) * srb]),
                              orc.scales_to_gemm_layout(orc.weight_2d_operand_scales(st, "row"))), g
        assert to_np(qw["s_w"])[g] == sw
        sr = orc.weight_2d_operand_scales(st, "row")
        assert np.array_equal(dq[g], orc.dequant_nvfp4(qr, sr, sw, per_row=False)), g
        r0, r1 = int(offs[g]), int(offs[g + 1])
        rows = np.arange(r0, r1)
        qa, sa, sta = orc.nvfp4_quantize_per_token(np.ascontiguousarray(d["x"][d["row_token"][rows]]))
        A = orc.decode_nvfp4_f64(qa, sa) * sta.astype(np.float64)[:, None]
        B = orc.decode_nvfp4_f64(qr, sr) * np.float64(sw)
        cols = np.sort(np.random.default_rng(g).choice(O1, 128, replace=False))
        check_block(orc, y[r0:r1][:, cols], A @ B[cols].T, np.abs(A) @ np.abs(B[cols]).T)


# ------------------------------------------------------------------------------------------------
# moe with MXFP8: the same expert layer, routed rows and expert weights in MXFP8, grouped MXFP8 GEMM
# ------------------------------------------------------------------------------------------------
@pytest.fixture(scope="module")
def moe8(mx):
    d = synthetic.moe()
    rows = int(d["group_offsets"][-1])
    x = bf16_dev(d["x"])
    a = x.index_select(0, torch.from_numpy(d["row_token"]).to(DEV)).contiguous()
    G, O1, H = d["w_gate_up"].shape
    offs = torch.from_numpy(d["group_offsets"]).to(DEV)
    qa = torch.empty((rows, H), dtype=torch.uint8, device=DEV)
    sa = torch.zeros(mx.grouped_scale_bytes(rows, G, H, 32), dtype=torch.uint8, device=DEV)
    mx.mx_quantize_mxfp8_grouped(a, offs, qa, sa)
    qw = mx.alloc_mxfp8(G * O1, H, DEV, rowwise=True, colwise=False)     # the G matrices stacked
    mx.mx_quantize_mxfp8(bf16_dev(d["w_gate_up"].reshape(G * O1, H)), qw["q_row"], qw["s_row"])
    y = torch.empty((rows, O1), dtype=torch.bfloat16, device=DEV)
    mx.mx_grouped_scaled_gemm(mx.MX_FMT_MXFP8, offs, qa, sa, None, qw["q_row"], qw["s_row"], None, O1, H, y)
    torch.cuda.synchronize()
    mx.check_device_status()
    return {"d": d, "qa": qa, "sa": sa, "qw": qw, "y": y, "G": G, "O1": O1, "H": H}


def test_moe_mxfp8_grouped_gemm_sampled(orc, moe8):
    d, G, O1, H = moe8["d"], moe8["G"], moe8["O1"], moe8["H"]
    offs = d["group_offsets"]
    y = moe8["y"].float().cpu().numpy()
    qw, sw_laid = to_np(moe8["qw"]["q_row"]).reshape(G, O1, H), to_np(moe8["qw"]["s_row"])
    srb = orc.scale_layout_bytes(O1, H // 32)
    ptile = np.concatenate([[0], np.cumsum((np.diff(offs) + 127) // 128)])
    sa_laid = orc.scales_from_gemm_layout(to_np(moe8["sa"]), int(ptile[-1]) * 128, H // 32)
    for g in (0, 77, G - 1):
        qb, sb = orc.mxfp8_quantize_rowwise(np.ascontiguousarray(d["w_gate_up"][g]))
        assert np.array_equal(qw[g], qb), g
        assert np.array_equal(sw_laid[g * srb:(g + 1) * srb], orc.scales_to_gemm_layout(sb)), g
        r0, r1 = int(offs[g]), int(offs[g + 1])
        qa, sa = orc.mxfp8_quantize_rowwise(np.ascontiguousarray(d["x"][d["row_token"][r0:r1]]))
        assert np.array_equal(to_np(moe8["qa"])[r0:r1], qa), g
        assert np.array_equal(sa_laid[ptile[g] * 128:ptile[g] * 128 + (r1 - r0)], sa), g
        A, B = orc.decode_mxfp8_f64(qa, sa), orc.decode_mxfp8_f64(qb, sb)
        cols = np.sort(np.random.default_rng(1000 + g).choice(O1, 128, replace=False))
        check_block(orc, y[r0:r1][:, cols], A @ B[cols].T, np.abs(A) @ np.abs(B[cols]).T)


# ------------------------------------------------------------------------------------------------
# wgrad: Llama-3-8B WGRAD, RHT16 + column-wise NVFP4 (SR on dY) + NVFP4 GEMM
# ------------------------------------------------------------------------------------------------
def test_wgrad_fullsize_sampled(mx, orc):
    d = synthetic.wgrad()
    T, H = d["x"].shape
    F = d["dy"].shape[1]
    rs, ss = d["rht_seed"], d["sr_seed"]
    u8 = lambda n: torch.empty(n, dtype=torch.uint8, device=DEV)
    qdy, sdy, Sdy = torch.empty((F, T // 2), dtype=torch.uint8, device=DEV), u8(mx.scale_bytes(F, T, 16)), \
        torch.empty(1, dtype=torch.float32, device=DEV)
    qx, sx, Sx = torch.empty((H, T // 2), dtype=torch.uint8, device=DEV), u8(mx.scale_bytes(H, T, 16)), \
        torch.empty(1, dtype=torch.float32, device=DEV)
    mx.mx_nvfp4_quantize_1x16(bf16_dev(d["dy"]), True, True, rs, True, ss, qdy, sdy, Sdy, u8(16))
    mx.mx_nvfp4_quantize_1x16(bf16_dev(d["x"]), True, True, rs, False, 0, qx, sx, Sx, u8(16))
    dw = torch.empty((F, H), dtype=torch.bfloat16, device=DEV)
    mx.mx_scaled_gemm(mx.MX_FMT_NVFP4, qdy, sdy, Sdy, mx.MX_SCOPE_TENSOR, qx, sx, Sx, mx.MX_SCOPE_TENSOR, F, H, T, dw)
    torch.cuda.synchronize()
    mx.check_device_status()

    # per-tensor scales over the whole transformed tensors, slab by slab (the transform is per column)
    def tensor_scale(a, slab):
        amax = np.float32(0)
        for c0 in range(0, a.shape[1], slab):
            amax = max(amax, orc.nvfp4_1x16_amax(np.ascontiguousarray(a[:, c0:c0 + slab]), rht=True, rht_seed=rs))
        return orc.nvfp4_second_scale(amax)

    S_dy, S_x = tensor_scale(d["dy"], 512), tensor_scale(d["x"], 512)
    assert to_np(Sdy)[0] == S_dy and to_np(Sx)[0] == S_x
    rng = np.random.default_rng(103)
    o0 = int(rng.integers(0, F // 64)) * 64
    h0 = int(rng.integers(0, H // 64)) * 64
    qo, so = orc.nvfp4_1x16_pass2(np.ascontiguousarray(d["dy"][:, o0:o0 + 64]), o0, F, S_dy, True, True, rs, True, ss)
    qh, sh = orc.nvfp4_1x16_pass2(np.ascontiguousarray(d["x"][:, h0:h0 + 64]), h0, H, S_x, True, True, rs, False, 0)
    assert np.array_equal(to_np(qdy[o0:o0 + 64]), qo), first_mismatch(to_np(qdy[o0:o0 + 64]), qo)
    assert np.array_equal(laid_rows(orc, to_np(sdy), F, T // 16, np.arange(o0, o0 + 64)), so)
    assert np.array_equal(to_np(qx[h0:h0 + 64]), qh)
    assert np.array_equal(laid_rows(orc, to_np(sx), H, T // 16, np.arange(h0, h0 + 64)), sh)
    A = orc.decode_nvfp4_f64(qo, so) * np.float64(S_dy)
    B = orc.decode_nvfp4_f64(qh, sh) * np.float64(S_x)
    got = dw.float().cpu().numpy()[o0:o0 + 64, h0:h0 + 64]
    check_block(orc, got, A @ B.T, np.abs(A) @ np.abs(B).T)


# ------------------------------------------------------------------------------------------------
# weight_sync: Q -> DQ -> re-Q byte identity on sampled layers, and codes vs the oracle
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("layer", [0, 47])
@pytest.mark.parametrize("fused", [False, True])
def test_weight_sync_layer(mx, orc, layer, fused):
    d = synthetic.weight_sync_layer(layer)
    cnt = torch.zeros(1, dtype=torch.int64, device=DEV)
    for name in ("down", "gate", "up"):
        w = d[name]
        G, O, H = w.shape
        wd = bf16_dev(w)
        m8 = mx.alloc_mxfp8(G * O, H, DEV)
        amax_w = torch.empty(G, dtype=torch.int32, device=DEV)
        if fused:
            mx.mx_quantize_mxfp8_amax(wd.view(G * O, H), O, amax_w, **m8)
        else:
            mx.mx_quantize_mxfp8(wd.view(G * O, H), **m8)
        y = torch.empty((G * O, H), dtype=torch.bfloat16, device=DEV)
        mx.mx_dequantize_bf16(mx.MX_FMT_MXFP8, m8["q_row"], m8["s_row"], None, 0, G * O, H, y)
        m8b = mx.alloc_mxfp8(G * O, H, DEV, colwise=False)
        mx.mx_quantize_mxfp8(y, **m8b)
        mx.mx_count_mismatch(m8["q_row"], m8b["q_row"], cnt)
        mx.mx_count_mismatch(m8["s_row"], m8b["s_row"], cnt)
        n4 = mx.alloc_nvfp4_weight_2d(G, O, H, DEV)
        y2 = torch.empty((G * O, H), dtype=torch.bfloat16, device=DEV)
        n4b = mx.alloc_nvfp4_weight_2d(G, O, H, DEV)
        if fused:
            # the maxima carried from the MXFP8 quantize and the NVFP4 dequantize (the weight-sync bench's chain)
            amax_y = torch.empty(G, dtype=torch.int32, device=DEV)
            mx.mx_nvfp4_quantize_weight_2d_given_amax(wd, n4["q_row"], n4["s_row"], n4["q_col"], n4["s_col"], n4["s_w"],
                                                      amax_w)
            mx.mx_dequantize_nvfp4_amax(n4["q_row"], n4["s_row"], n4["s_w"], O, G * O, H, y2, amax_y)
            mx.mx_nvfp4_quantize_weight_2d_given_amax(y2.view(G, O, H), n4b["q_row"], n4b["s_row"], n4b["q_col"],
                                                      n4b["s_col"], n4b["s_w"], amax_y)
        else:
            mx.mx_nvfp4_quantize_weight_2d(wd, n4["q_row"], n4["s_row"], n4["q_col"], n4["s_col"], n4["s_w"], n4["ws"])
            mx.mx_dequantize_bf16(mx.MX_FMT_NVFP4, n4["q_row"], n4["s_row"], n4["s_w"], mx.MX_SCOPE_GROUP, G * O, H, y2,
                                  group_rows=O)
            mx.mx_nvfp4_quantize_weight_2d(y2.view(G, O, H), n4b["q_row"], n4b["s_row"], n4b["q_col"], n4b["s_col"],
                                           n4b["s_w"], n4b["ws"])
        for k in ("q_row", "s_row", "q_col", "s_col"):
            mx.mx_count_mismatch(n4[k], n4b[k], cnt)
        torch.cuda.synchronize()
        y2_np = to_np_u16(y2)
        # sampled experts against the oracle
        for g in (0, G - 1):
            we = np.ascontiguousarray(w[g])
            qr, sr = orc.mxfp8_quantize_rowwise(we)
            assert np.array_equal(to_np(m8["q_row"][g * O:(g + 1) * O]), qr), (name, g)
            q2r, q2c, st, sw = orc.nvfp4_quantize_weight_2d(we)
            assert np.array_equal(to_np(n4["q_row"][g]), q2r), (name, g)
            assert to_np(n4["s_w"])[g] == sw
            assert np.array_equal(y2_np[g * O:(g + 1) * O],
                                  orc.dequant_nvfp4(q2r, orc.weight_2d_operand_scales(st, "row"), sw, per_row=False))
    assert int(cnt.item()) == 0, f"{int(cnt.item())} bytes changed on re-quantization"
