"""The C ABI loads and exports every symbol include/mxnum.h declares, and host-side validation
returns the documented status codes before anything touches a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mxnum.h")


@pytest.fixture(scope="module")
def lib():
    from microscaled_precision_numerics_gb300 import _build
    import microscaled_precision_numerics_gb300 as mx
    _build.build()
    return mx.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mx_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["mx_quantize_mxfp8", "mx_quantize_mxfp8_batched", "mx_quantize_mxfp8_amax",
                     "mx_nvfp4_quantize_weight_2d_given_amax", "mx_dequantize_nvfp4_amax", "mx_nvfp4_quantize_per_token", "mx_nvfp4_quantize_weight_2d", "mx_rht16",
                     "mx_nvfp4_quantize_1x16", "mx_dequantize_bf16", "mx_scaled_gemm", "mx_grouped_scaled_gemm",
                     "mx_fp8_blockwise_quantize_1x128", "mx_fp8_blockwise_quantize_128x128", "mx_gemm_bf16_dq_nvfp4",
                     "mx_wgrad_bf16_dq_nvfp4", "mx_fp8_blockwise_gemm"]:
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, text in [(0, b"MX_OK"), (1, b"MX_ERR_INVALID_ARG"), (2, b"MX_ERR_ALIGNMENT"), (3, b"MX_ERR_UNSUPPORTED"),
                       (4, b"MX_ERR_CUDA"), (5, b"MX_ERR_TIMEOUT")]:
        assert lib.mx_status_string(code) == text


def test_scale_and_workspace_sizes(lib):
    assert lib.mx_scale_bytes(256, 1024, 32) == 2 * 8 * 512
    assert lib.mx_scale_bytes(130, 48, 16) == 2 * 1 * 512
    assert lib.mx_scale_bytes(1, 16, 16) == 512
    assert lib.mx_scale_bytes(0, 16, 16) == 0
    assert lib.mx_scale_bytes(16, 16, 8) == 0
    assert lib.mx_workspace_bytes(0, 128, 0) == 512
    assert lib.mx_workspace_bytes(1, 0, 0) == 16


# Fake, never-dereferenced device addresses: validation must reject before any launch.
A16 = ctypes.c_void_p(0x10000)
A8 = ctypes.c_void_p(0x10008)
NUL = None


def test_mxfp8_validation(lib):
    f = lib.mx_quantize_mxfp8
    assert f(NUL, 32, 32, 32, A16, A16, NUL, NUL, NUL) == 1            # null input
    assert f(A16, 32, 32, 32, NUL, NUL, NUL, NUL, NUL) == 1            # no output
    assert f(A16, 32, 32, 32, A16, NUL, NUL, NUL, NUL) == 1            # codes without scales
    assert f(A8, 32, 32, 32, A16, A16, NUL, NUL, NUL) == 2             # misaligned input
    assert f(A16, 32, 48, 48, A16, A16, NUL, NUL, NUL) == 3            # cols % 32
    assert f(A16, 48, 32, 32, NUL, NUL, A16, A16, NUL) == 3            # rows % 32 for column-wise
    assert f(A16, 32, 36, 36, A16, A16, NUL, NUL, NUL) == 2            # cols % 8 (16-byte rows)
    assert f(A16, -1, 32, 32, A16, A16, NUL, NUL, NUL) == 1


def test_mxfp8_batched_validation(lib):
    from microscaled_precision_numerics_gb300 import _Mxfp8Tensor
    f = lib.mx_quantize_mxfp8_batched
    both = _Mxfp8Tensor(0x10000, 32, 32, 32, 0x10000, 0x10000, 0x10000, 0x10000)
    row = _Mxfp8Tensor(0x10000, 32, 32, 32, 0x10000, 0x10000, None, None)
    bad = _Mxfp8Tensor(0x10008, 32, 32, 32, 0x10000, 0x10000, 0x10000, 0x10000)

    def call(items, count=None):
        arr = (_Mxfp8Tensor * max(len(items), 1))(*items)
        return f(ctypes.cast(arr, ctypes.c_void_p), len(items) if count is None else count, None)

    assert f(None, 1, None) == 1                                        # no descriptors
    assert call([both], 0) == 1                                         # empty batch
    assert call([both] * 5) == 1                                        # above MX_MXFP8_MAX_BATCH
    assert call([both, row]) == 1                                       # mixed orientations
    assert call([both, bad]) == 2                                       # one descriptor misaligned
    assert call([both, _Mxfp8Tensor(0x10000, 32, 48, 48, 0x10000, 0x10000, 0x10000, 0x10000)]) == 3


def test_fused_maxima_validation(lib):
    f = lib.mx_quantize_mxfp8_amax
    assert f(A16, 256, 64, 64, A16, A16, NUL, NUL, 128, NUL, NUL) == 1          # no maxima buffer
    assert f(A16, 256, 64, 64, NUL, NUL, A16, A16, 128, A16, NUL) == 1          # row-wise output required
    assert f(A16, 256, 64, 64, A16, A16, NUL, NUL, 96, A16, NUL) == 3           # matrix_rows % 128
    assert f(A16, 384, 64, 64, A16, A16, NUL, NUL, 256, A16, NUL) == 3          # rows % matrix_rows
    assert f(A16, 256, 64, 64, A16, A16, NUL, NUL, 128, A8, NUL) == 2           # misaligned maxima
    g = lib.mx_nvfp4_quantize_weight_2d_given_amax
    assert g(A16, 2, 32, 32, A16, A16, A16, A16, A16, NUL, NUL) == 1
    assert g(A16, 2, 24, 32, A16, A16, A16, A16, A16, A16, NUL) == 3            # O % 16
    d = lib.mx_dequantize_nvfp4_amax
    assert d(A16, A16, A16, 128, 256, 64, A16, NUL, NUL) == 1
    assert d(A16, A16, A16, 64, 256, 64, A16, A16, NUL) == 3                    # group_rows % 128


def test_nvfp4_validation(lib):
    assert lib.mx_nvfp4_quantize_per_token(A16, 4, 24, 24, A16, A16, A16, NUL) == 3
    assert lib.mx_nvfp4_quantize_per_token(A16, 4, 32, 32, A16, A16, NUL, NUL) == 1
    assert lib.mx_nvfp4_quantize_weight_2d(A16, 1, 24, 32, A16, A16, A16, A16, A16, A16, 16, NUL) == 3
    assert lib.mx_nvfp4_quantize_weight_2d(A16, 4, 32, 32, A16, A16, A16, A16, A16, A16, 8, NUL) == 1
    assert lib.mx_rht16(A16, 24, 8, 0, ctypes.c_void_p(0x20000), NUL) == 3
    assert lib.mx_rht16(A16, 32, 8, 0, A16, NUL) == 1                   # in place not allowed
    assert lib.mx_nvfp4_quantize_1x16(A16, 32, 32, 0, 1, 0, 0, 0, A16, A16, A16, A16, 16, NUL) == 3   # row-wise RHT
    assert lib.mx_nvfp4_quantize_1x16(A16, 40, 32, 1, 0, 0, 0, 0, A16, A16, A16, A16, 16, NUL) == 3   # T % 16
    assert lib.mx_nvfp4_quantize_1x16(A16, 32, 32, 1, 0, 0, 7, 0, A16, A16, A16, A16, 16, NUL) == 1   # bad rounding
    assert lib.mx_nvfp4_quantize_1x16(A16, 32, 32, 1, 0, 0, 0, 0, A16, A16, A16, A16, 4, NUL) == 1    # workspace


def test_fp8_blockwise_validation(lib):
    f = lib.mx_fp8_blockwise_quantize_1x128
    assert f(A16, 128, 256, 256, 0, NUL, NUL, NUL, NUL, NUL, NUL, NUL) == 1           # no output
    assert f(A16, 128, 256, 256, 2, A16, A16, NUL, NUL, NUL, NUL, NUL) == 1           # pow2 not 0/1
    assert f(A16, 128, 256, 256, 0, A16, A16, A16, NUL, NUL, NUL, NUL) == 1           # E8M0 layout needs pow2
    assert f(A16, 128, 192, 192, 1, A16, A16, NUL, NUL, NUL, NUL, NUL) == 3           # cols % 128 (row-wise)
    assert f(A16, 96, 256, 256, 1, NUL, NUL, NUL, A16, A16, NUL, NUL) == 3            # rows % 128 (column-wise)
    assert f(A16, 128, 200, 200, 1, NUL, NUL, NUL, A16, A16, NUL, NUL) == 3           # cols % 16
    assert f(A8, 128, 256, 256, 1, A16, A16, NUL, NUL, NUL, NUL, NUL) == 2            # misaligned input
    assert f(A16, 128, 256, 252, 1, A16, A16, NUL, NUL, NUL, NUL, NUL) == 1           # ldx < cols
    w = lib.mx_fp8_blockwise_quantize_128x128
    assert w(A16, 1, 200, 256, 0, A16, A16, NUL, NUL, NUL, NUL) == 1                  # no scale output
    assert w(A16, 1, 200, 256, 1, A16, A16, A16, A16, NUL, NUL) == 3                  # E8M0 layout needs O % 128
    assert w(A16, 1, 200, 250, 1, A16, A16, A16, NUL, NUL, NUL) == 3                  # H % 16
    assert w(A16, 0, 256, 256, 1, A16, A16, A16, NUL, NUL, NUL) == 1                  # G = 0
    assert w(A16, 1, 256, 256, 0, A16, A16, A16, NUL, A16, NUL) == 1                  # E8M0 layout needs pow2


def test_gemm_validation(lib):
    g = lib.mx_scaled_gemm
    assert g(0, A16, A16, NUL, 0, A16, A16, NUL, 0, 128, 128, 96, A16, 128, NUL) == 3   # K % 128 (MXFP8)
    assert g(1, A16, A16, NUL, 0, A16, A16, NUL, 0, 128, 128, 128, A16, 128, NUL) == 3  # K % 256 (NVFP4)
    assert g(2, A16, A16, NUL, 0, A16, A16, NUL, 0, 128, 128, 128, A16, 128, NUL) == 1  # bad format
    assert g(0, A16, A16, NUL, 2, A16, A16, NUL, 0, 128, 128, 128, A16, 128, NUL) == 1  # scope without pointer
    assert g(0, A8, A16, NUL, 0, A16, A16, NUL, 0, 128, 128, 128, A16, 128, NUL) == 2
    assert g(0, A16, A16, NUL, 0, A16, A16, NUL, 0, 128, 128, 128, A16, 100, NUL) == 1  # ldd < N
    assert g(0, A16, A16, NUL, 0, A16, A16, NUL, 0, 128, 100, 128, A16, 100, NUL) == 2  # N % 8
    gg = lib.mx_grouped_scaled_gemm
    assert gg(1, 0, A16, 16, A16, A16, NUL, A16, A16, NUL, 256, 256, A16, NUL) == 1      # G = 0
    assert gg(1, 5000, A16, 16, A16, A16, NUL, A16, A16, NUL, 256, 256, A16, NUL) == 1   # too many groups
    assert gg(1, 4, A16, 16, A16, A16, NUL, A16, A16, NUL, 256, 200, A16, NUL) == 3      # K % 256


def test_dq_gemm_validation(lib):
    g = lib.mx_gemm_bf16_dq_nvfp4
    assert g(A16, NUL, 0, A16, A16, A16, 1, 128, 128, 96, A16, 128, NUL) == 3      # K % 64
    assert g(A16, NUL, 0, A16, A16, A16, 0, 128, 128, 128, A16, 128, NUL) == 1     # second-level scope
    assert g(A16, NUL, 2, A16, A16, A16, 1, 128, 128, 128, A16, 128, NUL) == 1     # alpha scope without pointer
    assert g(A16, NUL, 0, A16, A16, A16, 1, 128, 100, 128, A16, 100, NUL) == 2     # N % 8
    assert g(A8, NUL, 0, A16, A16, A16, 1, 128, 128, 128, A16, 128, NUL) == 2
    w = lib.mx_wgrad_bf16_dq_nvfp4
    assert w(A16, A16, A16, A16, 2, 96, 128, 128, A16, 128, NUL) == 3              # T % 64
    assert w(A16, A16, A16, A16, 2, 128, 128, 80, A16, 80, NUL) == 3               # H % 32
    assert w(A16, A16, A16, A16, 2, 128, 100, 128, A16, 128, NUL) == 2             # O % 8 (dY row pitch)
    assert w(A16, A16, A16, A16, 3, 128, 128, 128, A16, 128, NUL) == 1             # scope
    assert w(A16, A16, A16, NUL, 2, 128, 128, 128, A16, 128, NUL) == 1             # no scales


def test_fp8_blockwise_gemm_validation(lib):
    f = lib.mx_fp8_blockwise_gemm
    assert f(A16, A16, A16, A16, 128, 128, 96, A16, 128, NUL) == 3      # K % 128
    assert f(A16, A16, A16, NUL, 128, 128, 128, A16, 128, NUL) == 1     # no B scales
    assert f(A16, A16, A16, A16, 128, 100, 128, A16, 100, NUL) == 2     # N % 8
    assert f(A8, A16, A16, A16, 128, 128, 128, A16, 128, NUL) == 2      # misaligned codes
    assert f(A16, A16, A16, A16, 128, 128, 128, A16, 120, NUL) == 1     # ldd < N


def test_mismatch_validation(lib):
    assert lib.mx_count_mismatch(A16, A16, -1, A16, NUL) == 1
    assert lib.mx_count_mismatch(A8, A16, 16, A16, NUL) == 2
    assert lib.mx_count_mismatch(A16, A16, 0, A16, NUL) == 0


def test_binding_refuses_cpu_tensors():
    import torch
    import microscaled_precision_numerics_gb300 as mx
    x = torch.zeros((32, 32), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        mx.mx_quantize_mxfp8(x, q_row=torch.zeros((32, 32), dtype=torch.uint8), s_row=torch.zeros(512, dtype=torch.uint8))


def test_binding_checks_buffer_sizes_before_any_device_call():
    """The C ABI takes bare pointers, so the binding refuses undersized or non-contiguous buffers and
    badly strided inputs itself (checked here on host tensors: the checks run before any pointer is taken)."""
    import torch
    import microscaled_precision_numerics_gb300 as mx
    x = torch.zeros((256, 64), dtype=torch.bfloat16)
    sb = mx.scale_bytes(256, 64, 32)
    with pytest.raises(ValueError, match="q_row holds 16383 bytes, 16384 needed"):
        mx.mx_quantize_mxfp8(x, q_row=torch.zeros(256 * 64 - 1, dtype=torch.uint8), s_row=torch.zeros(sb, dtype=torch.uint8))
    with pytest.raises(ValueError, match="s_col holds"):
        mx.mx_quantize_mxfp8(x, q_col=torch.zeros(256 * 64, dtype=torch.uint8),
                             s_col=torch.zeros(mx.scale_bytes(64, 256, 32) - 16, dtype=torch.uint8))
    with pytest.raises(ValueError, match="unit column stride"):
        mx.mx_quantize_mxfp8(torch.zeros((64, 256), dtype=torch.bfloat16).t())
    with pytest.raises(ValueError, match="contiguous"):
        mx.mx_nvfp4_quantize_weight_2d(torch.zeros((2, 32, 64), dtype=torch.bfloat16).transpose(1, 2), None, None,
                                       None, None, None, torch.zeros(16, dtype=torch.uint8))
    with pytest.raises(ValueError, match="s_tok holds"):
        mx.mx_nvfp4_quantize_per_token(x, torch.zeros(256 * 32, dtype=torch.uint8),
                                       torch.zeros(mx.scale_bytes(256, 64, 16), dtype=torch.uint8),
                                       torch.zeros(255, dtype=torch.float32))
    with pytest.raises(ValueError, match="y holds"):
        mx.mx_dequantize_bf16(mx.MX_FMT_MXFP8, torch.zeros(256 * 64, dtype=torch.uint8),
                              torch.zeros(sb, dtype=torch.uint8), None, 0, 256, 64, torch.zeros((255, 64), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="d must be a 2-D view"):
        mx.mx_scaled_gemm(mx.MX_FMT_MXFP8, torch.zeros(128 * 128, dtype=torch.uint8),
                          torch.zeros(mx.scale_bytes(128, 128, 32), dtype=torch.uint8), None, 0,
                          torch.zeros(64 * 128, dtype=torch.uint8), torch.zeros(mx.scale_bytes(64, 128, 32), dtype=torch.uint8),
                          None, 0, 128, 64, 128, torch.zeros((128, 32), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="count holds"):
        mx.mx_count_mismatch(torch.zeros(64, dtype=torch.uint8), torch.zeros(64, dtype=torch.uint8),
                             torch.zeros(1, dtype=torch.int32))


def test_grid_limits_refused_before_launch(lib):
    """Shapes beyond the launch grids' y / z limits are refused on the host (MX_ERR_UNSUPPORTED)."""
    w2 = lib.mx_nvfp4_quantize_weight_2d
    assert w2(A16, 65536, 32, 32, A16, A16, A16, A16, A16, A16, 1 << 20, NUL) == 3     # G > 65535
    assert w2(A16, 1, 65535 * 64 + 16, 32, A16, A16, A16, A16, A16, A16, 16, NUL) == 3  # O / 64 > 65535
    assert lib.mx_nvfp4_quantize_weight_2d_46(A16, 65536, 32, 32, A16, A16, A16, A16, A16, A16, 1 << 20, NUL) == 3
    assert lib.mx_nvfp4_quantize_weight_2d_given_amax(A16, 65536, 32, 32, A16, A16, A16, A16, A16, A16, NUL) == 3
    f = lib.mx_nvfp4_quantize_weight_2d_noalloc
    f.restype, f.argtypes = ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64] + \
        [ctypes.c_void_p] * 6
    assert f(A16, 1, 65535 * 64 + 16, 32, A16, A16, A16, A16, A16, NUL) == 3
    # column-wise 1x16: one grid row per 128 tokens
    assert lib.mx_nvfp4_quantize_1x16(A16, 65535 * 128 + 16, 32, 1, 0, 0, 0, 0, A16, A16, A16, A16, 16, NUL) == 3


def test_binding_alloc_helpers_satisfy_its_size_checks():
    """Buffers from the alloc_* helpers pass the binding's size checks for ragged shapes: on host tensors the
    call then stops only at the device check."""
    import torch
    import microscaled_precision_numerics_gb300 as mx
    cpu = "cpu"
    only_cuda = "CUDA tensors only"
    for R, K in [(130, 96), (256, 1024), (1, 32)]:
        x = torch.zeros((R, K), dtype=torch.bfloat16)
        with pytest.raises(ValueError, match=only_cuda):
            mx.mx_quantize_mxfp8(x, **mx.alloc_mxfp8(R, K, cpu, colwise=R % 32 == 0))
        if K % 16 == 0:
            o = mx.alloc_nvfp4_rows(R, K, cpu)
            with pytest.raises(ValueError, match=only_cuda):
                mx.mx_nvfp4_quantize_per_token(x, o["q"], o["s"], o["s2"])
    for G, O, H in [(3, 48, 96), (1, 256, 2048)]:
        w = torch.zeros((G, O, H), dtype=torch.bfloat16)
        with pytest.raises(ValueError, match=only_cuda):
            mx.mx_nvfp4_quantize_weight_2d(w, **{k: v for k, v in mx.alloc_nvfp4_weight_2d(G, O, H, cpu).items()
                                                 if k != "ws"}, workspace=mx.alloc_nvfp4_weight_2d(G, O, H, cpu)["ws"])
    offs = torch.tensor([0, 100, 100, 300], dtype=torch.int64)
    x = torch.zeros((300, 64), dtype=torch.bfloat16)
    o = mx.alloc_nvfp4_rows_grouped(300, 3, 64, cpu)
    with pytest.raises(ValueError, match=only_cuda):
        mx.mx_nvfp4_quantize_per_token_grouped(x, offs, o["q"], o["s"], o["s2"])


def test_watchdog_selftest_validation(lib):
    f = lib.mx_watchdog_selftest
    assert f(0, 999, NUL) == 1                 # limit below 1 us
    assert f(0, 1_000_000_001, NUL) == 1       # limit above 1 s
    assert f(2, 1_000_000, NUL) == 1           # unknown unit
    assert f(-1, 1_000_000, NUL) == 1


def test_fp8_blockwise_wgrad_validation(lib):
    f = lib.mx_fp8_blockwise_gemm_wgrad
    assert f(NUL, A16, A16, A16, 128, 128, 128, A16, 128, NUL) == 1     # null A
    assert f(A16, A16, A16, A16, 128, 128, 128, A16, 64, NUL) == 1      # ldd < N
    assert f(A8, A16, A16, A16, 128, 128, 128, A16, 128, NUL) == 2      # misaligned A
    assert f(A16, A16, A16, A16, 128, 132, 128, A16, 136, NUL) == 2     # N % 8
    assert f(A16, A16, A16, A16, 128, 128, 192, A16, 128, NUL) == 3     # K % 128


# Every entry point with a size argument, as (function, a call that would pass its size checks, the
# positions of its size arguments).  Each size set to 0, then to -1, must come back MX_ERR_INVALID_ARG from
# the host-side checks (the addresses are never dereferenced: nothing is launched).
def _sized_calls(lib):
    A20 = ctypes.c_void_p(0x20000)
    return [
        ("mx_quantize_mxfp8", (A16, 32, 32, 32, A16, A16, A16, A16, NUL), [1, 2]),
        ("mx_quantize_mxfp8_grouped", (A16, 32, 32, 32, 2, A16, A16, A16, NUL), [1, 2, 4]),
        ("mx_quantize_mxfp8_amax", (A16, 256, 64, 64, A16, A16, NUL, NUL, 128, A16, NUL), [1, 2, 8]),
        ("mx_nvfp4_quantize_per_token", (A16, 32, 32, 32, A16, A16, A16, NUL), [1, 2]),
        ("mx_nvfp4_quantize_per_token_46", (A16, 32, 32, 32, A16, A16, A16, NUL), [1, 2]),
        ("mx_nvfp4_quantize_per_token_grouped", (A16, 32, 32, 32, 2, A16, A16, A16, A16, NUL), [1, 2, 4]),
        ("mx_nvfp4_quantize_weight_2d", (A16, 2, 32, 32, A16, A16, A16, A16, A16, A16, 4096, NUL), [1, 2, 3]),
        ("mx_nvfp4_quantize_weight_2d_46", (A16, 2, 32, 32, A16, A16, A16, A16, A16, A16, 4096, NUL), [1, 2, 3]),
        ("mx_nvfp4_quantize_weight_2d_noalloc", (A16, 2, 32, 32, A16, A16, A16, A16, A16, NUL), [1, 2, 3]),
        ("mx_nvfp4_quantize_weight_2d_given_amax", (A16, 2, 32, 32, A16, A16, A16, A16, A16, A16, NUL), [1, 2, 3]),
        ("mx_fp8_blockwise_quantize_1x128", (A16, 128, 128, 128, 0, A16, A16, NUL, A16, A16, NUL, NUL), [1, 2]),
        ("mx_fp8_blockwise_quantize_128x128", (A16, 1, 128, 128, 0, A16, A16, A16, NUL, NUL, NUL), [1, 2, 3]),
        ("mx_rht16", (A16, 32, 16, 0, A20, NUL), [1, 2]),
        ("mx_nvfp4_quantize_1x16", (A16, 32, 32, 1, 0, 0, 0, 0, A16, A16, A16, A16, 16, NUL), [1, 2]),
        ("mx_dequantize_bf16", (0, A16, A16, NUL, 0, 0, 32, 32, A16, NUL), [6, 7]),
        ("mx_dequantize_nvfp4_amax", (A16, A16, A16, 128, 256, 64, A16, A16, NUL), [3, 4, 5]),
        ("mx_scaled_gemm", (0, A16, A16, NUL, 0, A16, A16, NUL, 0, 128, 128, 128, A16, 128, NUL), [9, 10, 11]),
        ("mx_grouped_scaled_gemm", (0, 2, A16, 256, A16, A16, NUL, A16, A16, NUL, 128, 128, A16, NUL), [1, 3, 10, 11]),
        ("mx_gemm_bf16_dq_nvfp4", (A16, NUL, 0, A16, A16, A16, 1, 128, 128, 256, A16, 128, NUL), [7, 8, 9]),
        ("mx_wgrad_bf16_dq_nvfp4", (A16, A16, A16, A16, 1, 128, 128, 128, A16, 128, NUL), [5, 6, 7]),
        ("mx_fp8_blockwise_gemm", (A16, A16, A16, A16, 128, 128, 128, A16, 128, NUL), [4, 5, 6]),
        ("mx_fp8_blockwise_gemm_wgrad", (A16, A16, A16, A16, 128, 128, 128, A16, 128, NUL), [4, 5, 6]),
    ]


def test_zero_and_negative_sizes_are_rejected_before_any_launch(lib):
    covered = set()
    for name, args, sizes in _sized_calls(lib):
        f = getattr(lib, name)
        f.restype = ctypes.c_int
        covered.add(name)
        for i in sizes:
            for bad in (0, -1):
                call = list(args)
                call[i] = bad
                assert f(*[ctypes.c_int64(a) if isinstance(a, int) and j in sizes else a
                           for j, a in enumerate(call)]) == 1, f"{name}: argument {i} = {bad}"
    # every declared entry point that takes a size is in the table
    sized = {n for n in declared_functions() if n not in (
        "mx_status_string", "mx_scale_bytes", "mx_grouped_scale_bytes", "mx_workspace_bytes", "mx_check_device_status",
        "mx_check_stream_status", "mx_watchdog_selftest", "mx_quantize_mxfp8_batched", "mx_count_mismatch")}
    assert sized <= covered, sorted(sized - covered)


def test_empty_comparison_is_a_no_op(lib):
    """Comparing zero bytes counts nothing and launches nothing (the one zero-size call that succeeds)."""
    f = lib.mx_count_mismatch
    assert f(A16, A16, 0, A16, NUL) == 0
    assert f(A16, A16, -1, A16, NUL) == 1
