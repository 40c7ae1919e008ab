"""GPU parity of the whole weight-sync sweep: all 48 layers of the Qwen3-30B-A3B expert weights, run
through the chain `bench.py --workload weight_sync` times (MXFP8 quantize with the matrix maxima,
dequantize, re-quantize, byte compare; NVFP4 16x16 quantize from the carried maxima, dequantize with
maxima, re-quantize, byte compare), with the same per-layer device draws (seed 1000 + layer).

Per layer: the re-quantized bytes of every matrix of the layer equal the first quantization's (the
E2E page's abstract: synchronized weights are byte-identical with the learner's; its Table 11: the
byte comparison), and for one seeded expert of each of the three matrices (down, gate, up) every
output is compared with the oracle: the MXFP8 row-wise and column-wise codes and scales, the NVFP4
row-wise and column-wise codes and tile scales and the matrix scale, and both dequantized tensors."""
import numpy as np
import pytest
import torch

import bench
from gpu_util import DEV, first_mismatch, to_np, to_np_u16

pytestmark = pytest.mark.gpu
LAYERS = 48


@pytest.fixture(scope="module")
def mx():
    import microscaled_precision_numerics_gb300 as m
    m.lib()
    return m


@pytest.fixture(scope="module")
def sweep(mx):
    return bench.WeightSync(mx, torch, torch.device(DEV), layers=LAYERS)


def expert_of(layer):
    """One seeded expert per matrix (down, gate, up) of this layer."""
    return [int(g) for g in np.random.default_rng(5000 + layer).integers(0, 128, size=3)]


@pytest.mark.parametrize("layer", range(LAYERS))
def test_weight_sync_sweep_layer(mx, orc, sweep, layer):
    ops = sweep.ops()
    per_shape = len(ops) // len(sweep.shapes)
    sweep.draw(layer)
    sweep.count.zero_()
    picks = expert_of(layer)
    snap = []
    for si, ((G, O, H), b) in enumerate(zip(sweep.shapes, sweep.bufs)):
        g = picks[si]
        base = si * per_shape
        ops[base][4]()                       # MXFP8 quantize (+ matrix maxima)
        ops[base + 1][4]()                   # MXFP8 dequantize into b["y"]
        snap.append({"w": to_np_u16(b["w"][g]), "dq8": to_np_u16(b["y"][g * O:(g + 1) * O])})
        for i in range(2, per_shape):
            ops[base + i][4]()
    torch.cuda.synchronize()
    assert mx.mx_check_device_status() == mx.MX_OK
    changed = int(sweep.count.item())
    assert changed == 0, f"layer {layer}: {changed} bytes changed on re-quantization"

    for si, ((G, O, H), b) in enumerate(zip(sweep.shapes, sweep.bufs)):
        g, s = picks[si], snap[si]
        tag = (layer, si, g)
        w = s["w"]
        m8, n4 = b["m8"], b["n4"]
        # MXFP8: row-wise (blocks along H) and column-wise (blocks along the stacked rows, stored transposed)
        qr, sr = orc.mxfp8_quantize_rowwise(w)
        qc, sc = orc.mxfp8_quantize_colwise(w)
        got = to_np(m8["q_row"][g * O:(g + 1) * O])
        assert np.array_equal(got, qr), (tag, first_mismatch(got, qr))
        s_row = orc.scales_from_gemm_layout(to_np(m8["s_row"]), G * O, H // 32)[g * O:(g + 1) * O]
        assert np.array_equal(s_row, sr), tag
        got = to_np(m8["q_col"][:, g * O:(g + 1) * O])
        assert np.array_equal(got, qc), (tag, first_mismatch(got, qc))
        s_col = orc.scales_from_gemm_layout(to_np(m8["s_col"]), H, G * O // 32)[:, g * O // 32:(g + 1) * O // 32]
        assert np.array_equal(s_col, sc), tag
        dq8 = orc.dequant_mxfp8(qr, sr)
        assert np.array_equal(s["dq8"], dq8), (tag, first_mismatch(s["dq8"], dq8))
        # NVFP4 16x16: codes in both orientations, tile scales in both GEMM layouts, the matrix scale
        q2r, q2c, st, sw = orc.nvfp4_quantize_weight_2d(w)
        got = to_np(n4["q_row"][g])
        assert np.array_equal(got, q2r), (tag, first_mismatch(got, q2r))
        got = to_np(n4["q_col"][g])
        assert np.array_equal(got, q2c), (tag, first_mismatch(got, q2c))
        srb = orc.scale_layout_bytes(O, H // 16)
        scb = orc.scale_layout_bytes(H, O // 16)
        assert np.array_equal(to_np(n4["s_row"][g * srb:(g + 1) * srb]),
                              orc.scales_to_gemm_layout(orc.weight_2d_operand_scales(st, "row"))), tag
        assert np.array_equal(to_np(n4["s_col"][g * scb:(g + 1) * scb]),
                              orc.scales_to_gemm_layout(orc.weight_2d_operand_scales(st, "col"))), tag
        assert to_np(n4["s_w"])[g] == sw, tag
        dq4 = orc.dequant_nvfp4(q2r, orc.weight_2d_operand_scales(st, "row"), sw, per_row=False)
        got = to_np_u16(b["y"][g * O:(g + 1) * O])
        assert np.array_equal(got, dq4), (tag, first_mismatch(got, dq4))
