"""Parity past 2^31 elements: a 65600 x 32768 BF16 tensor (2 149 580 800 elements), so that element, code
and scale offsets of the sampled outputs lie beyond the 32-bit range: MXFP8 row and column quantize, the
MXFP8 GEMM with that tensor as A, the MXFP8 dequantize, the NVFP4 column-wise quantizer with RHT and SR,
the per-token NVFP4 quantizer and the 16x16 weight quantizer (the tensor as 41 stacked matrices).

The tensor is built on the device from a host-drawn 64-row block: row r is block row r % 64 times
2^(((r // 64) % 7) - 3), an exact scaling of BF16 values.  Every oracle input is rebuilt on the host from the
same block (sampled rows, full-height column slabs, and one 448-row period, which holds every 16-row group of
the tensor and so its per-tensor maximum); nothing the device computes feeds the oracle.
"""
import numpy as np
import pytest
import torch

import synthetic
from gpu_util import DEV, bf16_dev, first_mismatch, to_np, to_np_u16

pytestmark = pytest.mark.gpu

T, N = 65600, 32768
RHT_SEED, SR_SEED = 81, 82
BLOCK = synthetic.random_bf16(5150, (64, N), "normal", 1.0)


def exponents(rows):
    return ((np.asarray(rows, dtype=np.int64) // 64) % 7) - 3


def host_rows(rows, c0=0, c1=N):
    """Rows of the tensor (columns [c0, c1)) as BF16 bit patterns, built on the host."""
    rows = np.asarray(rows, dtype=np.int64)
    f = (BLOCK[rows % 64, c0:c1].astype(np.uint32) << 16).view(np.float32)
    f = f * np.float32(2.0) ** exponents(rows).astype(np.float32)[:, None]
    return (f.view(np.uint32) >> 16).astype(np.uint16)


@pytest.fixture(scope="module")
def big():
    import microscaled_precision_numerics_gb300 as mx
    mx.lib()
    blk = bf16_dev(BLOCK)
    scale = torch.from_numpy((2.0 ** exponents(np.arange(T))).astype(np.float32)).to(DEV).to(torch.bfloat16)
    x = blk.view(1, 64, N).expand(T // 64 + 1, 64, N).reshape(-1, N)[:T] * scale[:, None]
    del blk
    torch.cuda.synchronize()
    assert x.numel() > 2 ** 31
    # the device construction equals the host one (rows across the 2^31-element boundary)
    for r in (0, 65535, 65536, T - 1):
        assert np.array_equal(to_np_u16(x[r]), host_rows([r])[0])
    yield mx, x
    del x
    torch.cuda.empty_cache()


SAMPLE_ROWS = [0, 1, 4097, 65535, 65536, 65537, T - 1]


def test_mxfp8_row_and_column_past_2g(big, orc):
    mx, x = big
    out = mx.alloc_mxfp8(T, N, DEV)
    mx.mx_quantize_mxfp8(x, **out)
    torch.cuda.synchronize()
    mx.check_device_status()
    rows = np.array(SAMPLE_ROWS)
    qr, sr = orc.mxfp8_quantize_rowwise(host_rows(rows))
    got_q = to_np(out["q_row"][torch.from_numpy(rows).to(DEV)])
    assert np.array_equal(got_q, qr), first_mismatch(got_q, qr)
    assert np.array_equal(orc.scales_from_gemm_layout(to_np(out["s_row"]), T, N // 32)[rows], sr)
    for c0 in (0, N - 64):
        qc, sc = orc.mxfp8_quantize_colwise(host_rows(np.arange(T), c0, c0 + 64))
        got = to_np(out["q_col"][c0:c0 + 64])
        assert np.array_equal(got, qc), first_mismatch(got, qc)
        assert np.array_equal(orc.scales_from_gemm_layout(to_np(out["s_col"]), N, T // 32)[c0:c0 + 64], sc)
    # FPROP-shaped GEMM with this tensor as A (2^31+ codes) and a 256-row B: sampled output rows against the
    # FP64 product of the oracle's quantization of the same rows
    b = synthetic.random_bf16(5151, (256, N), "normal", 0.02)
    ob = mx.alloc_mxfp8(256, N, DEV, colwise=False)
    mx.mx_quantize_mxfp8(bf16_dev(b), **ob)
    d = torch.empty((T, 256), dtype=torch.bfloat16, device=DEV)
    mx.mx_scaled_gemm(mx.MX_FMT_MXFP8, out["q_row"], out["s_row"], None, 0, ob["q_row"], ob["s_row"], None, 0,
                      T, 256, N, d)
    torch.cuda.synchronize()
    mx.check_device_status()
    A = orc.decode_mxfp8_f64(qr, sr)
    B = orc.decode_mxfp8_f64(*orc.mxfp8_quantize_rowwise(b))
    got_d = d[torch.from_numpy(rows).to(DEV)].float().cpu().numpy().astype(np.float64)
    ref = A @ B.T
    assert orc.rel_fro_error(got_d, ref) <= 1e-2
    assert not (np.abs(got_d - ref) > 2.0 ** -7 * np.abs(ref) + 2.0 ** -15 * (np.abs(A) @ np.abs(B).T) + 1e-30).any()
    del d
    # the dequantize of the whole row-wise copy, sampled rows against the oracle's decode
    y = torch.empty((T, N), dtype=torch.bfloat16, device=DEV)
    mx.mx_dequantize_bf16(mx.MX_FMT_MXFP8, out["q_row"], out["s_row"], None, 0, T, N, y)
    torch.cuda.synchronize()
    got_y = to_np_u16(y[torch.from_numpy(rows).to(DEV)])
    want_y = orc.dequant_mxfp8(qr, sr)
    assert np.array_equal(got_y, want_y), first_mismatch(got_y, want_y)
    del out, y


def test_nvfp4_colwise_rht_sr_past_2g(big, orc):
    mx, x = big
    q = torch.empty((N, T // 2), dtype=torch.uint8, device=DEV)
    s = torch.empty(mx.scale_bytes(N, T, 16), dtype=torch.uint8, device=DEV)
    S = torch.empty(1, dtype=torch.float32, device=DEV)
    ws = torch.empty(16, dtype=torch.uint8, device=DEV)
    mx.mx_nvfp4_quantize_1x16(x, True, True, RHT_SEED, True, SR_SEED, q, s, S, ws)
    torch.cuda.synchronize()
    mx.check_device_status()
    # per-tensor scale from one 448-row period (every 16-row group of the tensor occurs in it), slab by slab
    period = host_rows(np.arange(448))
    amax = max(orc.nvfp4_1x16_amax(np.ascontiguousarray(period[:, c:c + 4096]), rht=True, rht_seed=RHT_SEED)
               for c in range(0, N, 4096))
    S_ref = orc.nvfp4_second_scale(amax)
    assert to_np(S).view(np.uint32)[0] == np.float32(S_ref).view(np.uint32)
    laid = orc.scales_from_gemm_layout(to_np(s), N, T // 16)
    for c0 in (0, N - 64):
        qo, so = orc.nvfp4_1x16_pass2(host_rows(np.arange(T), c0, c0 + 64), c0, N, S_ref, True, True, RHT_SEED,
                                      True, SR_SEED)
        got = to_np(q[c0:c0 + 64])
        assert np.array_equal(got, qo), first_mismatch(got, qo)
        assert np.array_equal(laid[c0:c0 + 64], so)
    del q, s


def test_nvfp4_per_token_past_2g(big, orc):
    """Rows of 2048 blocks (the kernel's streaming path, rows re-read between the passes)."""
    mx, x = big
    out = mx.alloc_nvfp4_rows(T, N, DEV)
    mx.mx_nvfp4_quantize_per_token(x, out["q"], out["s"], out["s2"])
    torch.cuda.synchronize()
    mx.check_device_status()
    rows = np.array(SAMPLE_ROWS)
    q, s, st = orc.nvfp4_quantize_per_token(host_rows(rows))
    sel = torch.from_numpy(rows).to(DEV)
    got = to_np(out["q"][sel])
    assert np.array_equal(got, q), first_mismatch(got, q)
    assert np.array_equal(orc.scales_from_gemm_layout(to_np(out["s"]), T, N // 16)[rows], s)
    assert np.array_equal(to_np(out["s2"][sel]).view(np.uint32), st.view(np.uint32))
    del out


def test_nvfp4_weight_2d_past_2g(big, orc):
    """The tensor as 41 stacked 1600 x 32768 matrices; the last one lies past element 2^31."""
    mx, x = big
    G, O = 41, T // 41
    w = x.view(G, O, N)
    out = mx.alloc_nvfp4_weight_2d(G, O, N, DEV)
    mx.mx_nvfp4_quantize_weight_2d(w, out["q_row"], out["s_row"], out["q_col"], out["s_col"], out["s_w"], out["ws"])
    torch.cuda.synchronize()
    mx.check_device_status()
    g = G - 1
    qr, qc, st, sw = orc.nvfp4_quantize_weight_2d(host_rows(np.arange(g * O, (g + 1) * O)))
    assert out["s_w"][g].item() == float(sw)
    got = to_np(out["q_row"][g])
    assert np.array_equal(got, qr), first_mismatch(got, qr)
    got = to_np(out["q_col"][g])
    assert np.array_equal(got, qc), first_mismatch(got, qc)
    srb, scb = orc.scale_layout_bytes(O, N // 16), orc.scale_layout_bytes(N, O // 16)
    assert np.array_equal(to_np(out["s_row"][g * srb:(g + 1) * srb]),
                          orc.scales_to_gemm_layout(orc.weight_2d_operand_scales(st, "row")))
    assert np.array_equal(to_np(out["s_col"][g * scb:(g + 1) * scb]),
                          orc.scales_to_gemm_layout(orc.weight_2d_operand_scales(st, "col")))
    del out
