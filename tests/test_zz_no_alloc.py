"""The allocation-free 2D weight quantizer gives the same bytes as the regular entry point.

mx_nvfp4_quantize_weight_2d_noalloc serves callers that cannot allocate device memory (a plugin in
a host framework that owns all device memory, or a loop that must not call cudaMalloc because it
synchronizes the device): its per-matrix scratch is a fixed array inside the library rather than a
caller workspace.  Through the C ABI, two calls in a row -- the second with a smaller weight
magnitude and fewer matrices, so stale scratch from the first call would change its scales -- must
match mx_nvfp4_quantize_weight_2d byte for byte (the quantizer tolerance is bit-exactness), and the CPU
oracle's codes, tile scales and matrix scales for every matrix.
This file is collected last so that a run stopping at the first failure has run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import synthetic
from gpu_util import DEV, bf16_dev

pytestmark = pytest.mark.gpu


def _outputs(mx, G, O, H):
    return mx.alloc_nvfp4_weight_2d(G, O, H, DEV)


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(orc):
    import microscaled_precision_numerics_gb300 as mx
    L = mx.lib()
    f = L.mx_nvfp4_quantize_weight_2d_noalloc
    P, I64 = ctypes.c_void_p, ctypes.c_int64
    f.restype = ctypes.c_int
    f.argtypes = [P, I64, I64, I64, P, P, P, P, P, P]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())

    for call, (G, O, H, std, seed) in enumerate([(5, 64, 96, 1.0, 401), (3, 48, 80, 0.02, 402)]):
        w = bf16_dev(synthetic.random_bf16(seed, (G, O, H), "student_t", std))
        ref = _outputs(mx, G, O, H)
        mx.mx_nvfp4_quantize_weight_2d(w, ref["q_row"], ref["s_row"], ref["q_col"], ref["s_col"], ref["s_w"],
                                       ref["ws"])
        got = _outputs(mx, G, O, H)
        for k in ("q_row", "s_row", "q_col", "s_col"):
            got[k].fill_(0xA5)
        got["s_w"].fill_(-1.0)
        status = f(ptr(w), G, O, H, ptr(got["q_row"]), ptr(got["s_row"]), ptr(got["q_col"]), ptr(got["s_col"]),
                   ptr(got["s_w"]), stream)
        assert status == 0, f"call {call}: status {status}"
        torch.cuda.synchronize()
        for k in ("q_row", "s_row", "q_col", "s_col", "s_w"):
            a, b = got[k].cpu().numpy(), ref[k].cpu().numpy()
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), f"call {call}: {k} differs"
        # and the oracle, matrix by matrix
        w_np = w.view(torch.int16).cpu().numpy().view(np.uint16)
        srb, scb = orc.scale_layout_bytes(O, H // 16), orc.scale_layout_bytes(H, O // 16)
        for g in range(G):
            qr, qc, st, sw = orc.nvfp4_quantize_weight_2d(np.ascontiguousarray(w_np[g]))
            assert np.array_equal(got["q_row"][g].cpu().numpy(), qr), f"call {call}: q_row of matrix {g}"
            assert np.array_equal(got["q_col"][g].cpu().numpy(), qc), f"call {call}: q_col of matrix {g}"
            assert np.array_equal(got["s_row"][g * srb:(g + 1) * srb].cpu().numpy(),
                                  orc.scales_to_gemm_layout(orc.weight_2d_operand_scales(st, "row")))
            assert np.array_equal(got["s_col"][g * scb:(g + 1) * scb].cpu().numpy(),
                                  orc.scales_to_gemm_layout(orc.weight_2d_operand_scales(st, "col")))
            assert got["s_w"][g].item() == float(sw), f"call {call}: s_w of matrix {g}"


def test_noalloc_rejects_more_matrices_than_its_scratch():
    import microscaled_precision_numerics_gb300 as mx
    f = mx.lib().mx_nvfp4_quantize_weight_2d_noalloc
    P, I64 = ctypes.c_void_p, ctypes.c_int64
    f.restype = ctypes.c_int
    f.argtypes = [P, I64, I64, I64, P, P, P, P, P, P]
    a = ctypes.c_void_p(0x10000)   # never dereferenced: the size check comes first
    assert f(a, mx.MX_NOALLOC_MAX_MATRICES + 1, 16, 16, a, a, a, a, a, None) == 3
