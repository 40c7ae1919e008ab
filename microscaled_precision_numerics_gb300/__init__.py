"""Python binding of libmxnum.so (block-scaled microscaling numerics on GB300, sm_103a).

Argument marshalling only: every function passes ``tensor.data_ptr()`` values, sizes, seeds and the
current CUDA stream to the C ABI declared in ``include/mxnum.h`` and raises ``MXError`` on a non-OK
status.  No arithmetic happens here and there is no CPU fallback: if the CUDA library is missing or
a tensor is not on a CUDA device, the call raises.  ``alloc_*`` helpers only create output tensors
of the right sizes (``torch.empty`` on the input's device).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmxnum.so")

MX_OK, MX_ERR_INVALID_ARG, MX_ERR_ALIGNMENT, MX_ERR_UNSUPPORTED, MX_ERR_CUDA, MX_ERR_TIMEOUT = range(6)
MX_FMT_MXFP8, MX_FMT_NVFP4 = 0, 1
MX_ROUND_RNE, MX_ROUND_SR = 0, 1
MX_SCOPE_NONE, MX_SCOPE_TENSOR, MX_SCOPE_ROW, MX_SCOPE_GROUP = 0, 1, 2, 3
MX_WS_WEIGHT_2D, MX_WS_1X16 = 0, 1
MX_NOALLOC_MAX_MATRICES = 4096

_lock = threading.Lock()
_lib = None


class MXError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn} failed: {text} ({status})")
        self.status = status


def lib() -> ctypes.CDLL:
    """Load libmxnum.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
            L = ctypes.CDLL(LIB_PATH)
            P, I64, U64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int, ctypes.c_size_t
            sigs = {
                "mx_status_string": (ctypes.c_char_p, [I32]),
                "mx_scale_bytes": (I64, [I64, I64, I32]),
                "mx_workspace_bytes": (SZ, [I32, I64, I64]),
                "mx_quantize_mxfp8": (I32, [P, I64, I64, I64, P, P, P, P, P]),
                "mx_quantize_mxfp8_batched": (I32, [P, I32, P]),
                "mx_quantize_mxfp8_amax": (I32, [P, I64, I64, I64, P, P, P, P, I64, P, P]),
                "mx_nvfp4_quantize_weight_2d_given_amax": (I32, [P, I64, I64, I64, P, P, P, P, P, P, P]),
                "mx_dequantize_nvfp4_amax": (I32, [P, P, P, I64, I64, I64, P, P, P]),
                "mx_nvfp4_quantize_per_token": (I32, [P, I64, I64, I64, P, P, P, P]),
                "mx_nvfp4_quantize_per_token_46": (I32, [P, I64, I64, I64, P, P, P, P]),
                "mx_nvfp4_quantize_per_token_grouped": (I32, [P, I64, I64, I64, I64, P, P, P, P, P]),
                "mx_quantize_mxfp8_grouped": (I32, [P, I64, I64, I64, I64, P, P, P, P]),
                "mx_grouped_scale_bytes": (I64, [I64, I64, I64, I32]),
                "mx_nvfp4_quantize_weight_2d": (I32, [P, I64, I64, I64, P, P, P, P, P, P, SZ, P]),
                "mx_nvfp4_quantize_weight_2d_46": (I32, [P, I64, I64, I64, P, P, P, P, P, P, SZ, P]),
                "mx_nvfp4_quantize_weight_2d_noalloc": (I32, [P, I64, I64, I64, P, P, P, P, P, P]),
                "mx_rht16": (I32, [P, I64, I64, U64, P, P]),
                "mx_fp8_blockwise_quantize_1x128": (I32, [P, I64, I64, I64, I32, P, P, P, P, P, P, P]),
                "mx_fp8_blockwise_quantize_128x128": (I32, [P, I64, I64, I64, I32, P, P, P, P, P, P]),
                "mx_nvfp4_quantize_1x16": (I32, [P, I64, I64, I32, I32, U64, I32, U64, P, P, P, P, SZ, P]),
                "mx_dequantize_bf16": (I32, [I32, P, P, P, I32, I64, I64, I64, P, P]),
                "mx_scaled_gemm": (I32, [I32, P, P, P, I32, P, P, P, I32, I64, I64, I64, P, I64, P]),
                "mx_grouped_scaled_gemm": (I32, [I32, I64, P, I64, P, P, P, P, P, P, I64, I64, P, P]),
                "mx_count_mismatch": (I32, [P, P, I64, P, P]),
                "mx_gemm_bf16_dq_nvfp4": (I32, [P, P, I32, P, P, P, I32, I64, I64, I64, P, I64, P]),
                "mx_wgrad_bf16_dq_nvfp4": (I32, [P, P, P, P, I32, I64, I64, I64, P, I64, P]),
                "mx_fp8_blockwise_gemm": (I32, [P, P, P, P, I64, I64, I64, P, I64, P]),
                "mx_fp8_blockwise_gemm_wgrad": (I32, [P, P, P, P, I64, I64, I64, P, I64, P]),
                "mx_check_device_status": (I32, []),
                "mx_check_stream_status": (I32, [P]),
                "mx_watchdog_selftest": (I32, [I32, U64, P]),
            }
            for name, (res, args) in sigs.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise MXError(fn, status, lib().mx_status_string(status).decode())


def _p(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError("mxnum operates on CUDA tensors only (no CPU path)")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"tensor on {t.device} but the current device is cuda:{torch.cuda.current_device()}")
    return ctypes.c_void_p(t.data_ptr())


def _need(fn: str, name: str, t, nbytes) -> None:
    """Raise unless t (when given) is contiguous and holds at least nbytes bytes: the C ABI takes bare
    pointers, so the sizes of the buffers it reads and writes are checked here."""
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{fn}: {name} must be a torch.Tensor")
    if not t.is_contiguous():
        raise ValueError(f"{fn}: {name} must be contiguous")
    have = t.numel() * t.element_size()
    if have < nbytes:
        raise ValueError(f"{fn}: {name} holds {have} bytes, {int(nbytes)} needed")


def _need_out2d(fn: str, name: str, d, rows: int, cols: int) -> None:
    """A row-major [rows, cols] output that may be a view with a row stride (unit column stride)."""
    if d.dim() != 2 or d.shape[0] < rows or d.shape[1] < cols or d.stride(1) != 1:
        raise ValueError(f"{fn}: {name} must be a 2-D view of at least [{rows}, {cols}] with unit column stride")


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _bf16_bits(t: torch.Tensor, dims: int = 2) -> torch.Tensor:
    """A BF16 input: [rows, cols] with unit column stride (any row stride), or a contiguous [G, rows, cols]."""
    if t.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError("BF16 input expected (bfloat16 or its 16-bit bit pattern)")
    if t.dim() != dims:
        raise ValueError(f"a {dims}-D BF16 tensor expected, got shape {tuple(t.shape)}")
    if dims == 2 and t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError("BF16 input must have unit column stride")
    if dims != 2 and not t.is_contiguous():
        raise ValueError("stacked BF16 input must be contiguous")
    return t


def scale_bytes(rows: int, k: int, block: int) -> int:
    return int(lib().mx_scale_bytes(rows, k, block))


def _mxfp8_outputs(fn, rows, cols, q_row, s_row, q_col, s_col):
    _need(fn, "q_row", q_row, rows * cols)
    _need(fn, "s_row", s_row, scale_bytes(rows, cols, 32))
    _need(fn, "q_col", q_col, rows * cols)
    _need(fn, "s_col", s_col, scale_bytes(cols, rows, 32))


def workspace_bytes(op: int, groups: int = 0) -> int:
    return int(lib().mx_workspace_bytes(op, groups, 0))


def check_device_status() -> None:
    _check("mx_check_device_status", lib().mx_check_device_status())


def mx_check_device_status() -> int:
    """The raw status (MX_OK, MX_ERR_TIMEOUT, MX_ERR_CUDA): synchronizes the device, clears the watchdog words."""
    return int(lib().mx_check_device_status())


def mx_check_stream_status(stream=None) -> int:
    """The raw status after waiting for `stream` (default: the current stream) only."""
    return int(lib().mx_check_stream_status(_stream(stream)))


MX_WATCHDOG_GEMM, MX_WATCHDOG_MXFP8 = 0, 1


def mx_watchdog_selftest(unit: int, limit_ns: int, stream=None) -> None:
    """Test hook: one kernel whose bounded waits expire after limit_ns (see include/mxnum.h)."""
    _check("mx_watchdog_selftest", lib().mx_watchdog_selftest(int(unit), int(limit_ns), _stream(stream)))


# ------------------------------------------------------------------------------------------------
# quantizers
# ------------------------------------------------------------------------------------------------

def mx_quantize_mxfp8(x, q_row=None, s_row=None, q_col=None, s_col=None, stream=None):
    x = _bf16_bits(x)
    rows, cols = x.shape
    _mxfp8_outputs("mx_quantize_mxfp8", rows, cols, q_row, s_row, q_col, s_col)
    _check("mx_quantize_mxfp8", lib().mx_quantize_mxfp8(
        _p(x), rows, cols, x.stride(0), _p(q_row), _p(s_row), _p(q_col), _p(s_col), _stream(stream)))


MX_MXFP8_MAX_BATCH = 4


class _Mxfp8Tensor(ctypes.Structure):
    """mx_mxfp8_tensor: one tensor of mx_quantize_mxfp8_batched."""
    _fields_ = [("x", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("ldx", ctypes.c_int64),
                ("q_row", ctypes.c_void_p), ("s_row", ctypes.c_void_p), ("q_col", ctypes.c_void_p),
                ("s_col", ctypes.c_void_p)]


def mx_quantize_mxfp8_batched(jobs, stream=None):
    """mx_quantize_mxfp8 over several tensors in one launch.  `jobs`: a list of (x, outputs) pairs, outputs a
    dict with the keyword arguments of mx_quantize_mxfp8 (q_row, s_row, q_col, s_col)."""
    arr = (_Mxfp8Tensor * max(len(jobs), 1))()
    keep = []
    for i, (x, out) in enumerate(jobs):
        x = _bf16_bits(x)
        keep.append(x)
        rows, cols = x.shape
        _mxfp8_outputs("mx_quantize_mxfp8_batched", rows, cols, out.get("q_row"), out.get("s_row"), out.get("q_col"),
                       out.get("s_col"))
        arr[i] = _Mxfp8Tensor(_p(x), rows, cols, x.stride(0), _p(out.get("q_row")), _p(out.get("s_row")),
                              _p(out.get("q_col")), _p(out.get("s_col")))
    _check("mx_quantize_mxfp8_batched", lib().mx_quantize_mxfp8_batched(ctypes.cast(arr, ctypes.c_void_p),
                                                                        len(jobs), _stream(stream)))


def mx_quantize_mxfp8_amax(x, matrix_rows: int, amax, q_row=None, s_row=None, q_col=None, s_col=None, stream=None):
    """mx_quantize_mxfp8 of stacked matrices plus each matrix's max |x| (int32 words, BF16 bits << 16)."""
    x = _bf16_bits(x)
    rows, cols = x.shape
    _mxfp8_outputs("mx_quantize_mxfp8_amax", rows, cols, q_row, s_row, q_col, s_col)
    _need("mx_quantize_mxfp8_amax", "amax", amax, 4 * (rows // max(int(matrix_rows), 1)))
    _check("mx_quantize_mxfp8_amax", lib().mx_quantize_mxfp8_amax(
        _p(x), rows, cols, x.stride(0), _p(q_row), _p(s_row), _p(q_col), _p(s_col), matrix_rows, _p(amax),
        _stream(stream)))


def _weight_2d_outputs(fn, G, O, H, q_row, s_row, q_col, s_col, s_w):
    _need(fn, "q_row", q_row, G * O * H // 2)
    _need(fn, "s_row", s_row, G * scale_bytes(O, H, 16))
    _need(fn, "q_col", q_col, G * O * H // 2)
    _need(fn, "s_col", s_col, G * scale_bytes(H, O, 16))
    _need(fn, "s_w", s_w, 4 * G)


def mx_nvfp4_quantize_weight_2d_given_amax(w, q_row, s_row, q_col, s_col, s_w, amax, stream=None):
    w = _bf16_bits(w, 3)
    G, O, H = w.shape
    _weight_2d_outputs("mx_nvfp4_quantize_weight_2d_given_amax", G, O, H, q_row, s_row, q_col, s_col, s_w)
    _need("mx_nvfp4_quantize_weight_2d_given_amax", "amax", amax, 4 * G)
    _check("mx_nvfp4_quantize_weight_2d_given_amax", lib().mx_nvfp4_quantize_weight_2d_given_amax(
        _p(w), G, O, H, _p(q_row), _p(s_row), _p(q_col), _p(s_col), _p(s_w), _p(amax), _stream(stream)))


def mx_dequantize_nvfp4_amax(q, s, s2, group_rows: int, rows: int, cols: int, y, amax, stream=None):
    fn, ng = "mx_dequantize_nvfp4_amax", rows // max(int(group_rows), 1)
    _need(fn, "q", q, rows * cols // 2)
    _need(fn, "s", s, scale_bytes(rows, cols, 16))
    _need(fn, "s2", s2, 4 * ng)
    _need(fn, "y", y, 2 * rows * cols)
    _need(fn, "amax", amax, 4 * ng)
    _check("mx_dequantize_nvfp4_amax", lib().mx_dequantize_nvfp4_amax(
        _p(q), _p(s), _p(s2), group_rows, rows, cols, _p(y), _p(amax), _stream(stream)))


def _per_token_outputs(fn, T, H, q, s_bytes, s, s_tok):
    _need(fn, "q", q, T * H // 2)
    _need(fn, "s", s, s_bytes)
    _need(fn, "s_tok", s_tok, 4 * T)


def mx_nvfp4_quantize_per_token(x, q, s, s_tok, stream=None):
    x = _bf16_bits(x)
    T, H = x.shape
    _per_token_outputs("mx_nvfp4_quantize_per_token", T, H, q, scale_bytes(T, H, 16), s, s_tok)
    _check("mx_nvfp4_quantize_per_token", lib().mx_nvfp4_quantize_per_token(
        _p(x), T, H, x.stride(0), _p(q), _p(s), _p(s_tok), _stream(stream)))


def mx_nvfp4_quantize_per_token_46(x, q, s, s_tok, stream=None):
    x = _bf16_bits(x)
    T, H = x.shape
    _per_token_outputs("mx_nvfp4_quantize_per_token_46", T, H, q, scale_bytes(T, H, 16), s, s_tok)
    _check("mx_nvfp4_quantize_per_token_46", lib().mx_nvfp4_quantize_per_token_46(
        _p(x), T, H, x.stride(0), _p(q), _p(s), _p(s_tok), _stream(stream)))


def mx_nvfp4_quantize_per_token_grouped(x, group_offsets, q, s, s_tok, stream=None):
    x = _bf16_bits(x)
    T, H = x.shape
    G = group_offsets.numel() - 1
    _need("mx_nvfp4_quantize_per_token_grouped", "group_offsets", group_offsets, 8 * (G + 1))
    _per_token_outputs("mx_nvfp4_quantize_per_token_grouped", T, H, q, grouped_scale_bytes(T, G, H, 16), s, s_tok)
    _check("mx_nvfp4_quantize_per_token_grouped", lib().mx_nvfp4_quantize_per_token_grouped(
        _p(x), T, H, x.stride(0), group_offsets.numel() - 1, _p(group_offsets), _p(q), _p(s), _p(s_tok),
        _stream(stream)))


def mx_quantize_mxfp8_grouped(x, group_offsets, q_row, s_row, stream=None):
    x = _bf16_bits(x)
    rows, cols = x.shape
    G = group_offsets.numel() - 1
    _need("mx_quantize_mxfp8_grouped", "group_offsets", group_offsets, 8 * (G + 1))
    _need("mx_quantize_mxfp8_grouped", "q_row", q_row, rows * cols)
    _need("mx_quantize_mxfp8_grouped", "s_row", s_row, grouped_scale_bytes(rows, G, cols, 32))
    _check("mx_quantize_mxfp8_grouped", lib().mx_quantize_mxfp8_grouped(
        _p(x), rows, cols, x.stride(0), group_offsets.numel() - 1, _p(group_offsets), _p(q_row), _p(s_row),
        _stream(stream)))


def grouped_scale_bytes(rows: int, G: int, k: int, block: int) -> int:
    return int(lib().mx_grouped_scale_bytes(rows, G, k, block))


def mx_nvfp4_quantize_weight_2d(w, q_row, s_row, q_col, s_col, s_w, workspace, stream=None):
    w = _bf16_bits(w, 3)
    G, O, H = w.shape
    _weight_2d_outputs("mx_nvfp4_quantize_weight_2d", G, O, H, q_row, s_row, q_col, s_col, s_w)
    _check("mx_nvfp4_quantize_weight_2d", lib().mx_nvfp4_quantize_weight_2d(
        _p(w), G, O, H, _p(q_row), _p(s_row), _p(q_col), _p(s_col), _p(s_w), _p(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def mx_nvfp4_quantize_weight_2d_46(w, q_row, s_row, q_col, s_col, s_w, workspace, stream=None):
    w = _bf16_bits(w, 3)
    G, O, H = w.shape
    _weight_2d_outputs("mx_nvfp4_quantize_weight_2d_46", G, O, H, q_row, s_row, q_col, s_col, s_w)
    _check("mx_nvfp4_quantize_weight_2d_46", lib().mx_nvfp4_quantize_weight_2d_46(
        _p(w), G, O, H, _p(q_row), _p(s_row), _p(q_col), _p(s_col), _p(s_w), _p(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def mx_nvfp4_quantize_weight_2d_noalloc(w, q_row, s_row, q_col, s_col, s_w, stream=None):
    """Same as mx_nvfp4_quantize_weight_2d without a workspace, for callers that cannot allocate
    device memory: the library keeps the per-matrix scratch in a fixed internal array (at most
    MX_NOALLOC_MAX_MATRICES matrices per call).  Calls that may overlap on the GPU share that array
    and must be serialized by the caller."""
    w = _bf16_bits(w, 3)
    G, O, H = w.shape
    _weight_2d_outputs("mx_nvfp4_quantize_weight_2d_noalloc", G, O, H, q_row, s_row, q_col, s_col, s_w)
    f = lib().mx_nvfp4_quantize_weight_2d_noalloc
    if G > MX_NOALLOC_MAX_MATRICES:
        raise ValueError(f"{G} matrices exceed the allocation-free limit of {MX_NOALLOC_MAX_MATRICES}")
    _check("mx_nvfp4_quantize_weight_2d_noalloc", f(
        _p(w), G, O, H, _p(q_row), _p(s_row), _p(q_col), _p(s_col), _p(s_w), _stream(stream)))


def mx_fp8_blockwise_quantize_1x128(x, pow2: bool, q_row=None, s_row=None, sf_row=None, q_col=None, s_col=None,
                                    sf_col=None, stream=None):
    """Blockwise FP8 of activations / gradients in [1, 128] tiles: row-wise (q_row [R, C], s_row
    [R, C/128]) and/or column-wise stored transposed (q_col [C, R], s_col [C, R/128]); with pow2 the
    E8M0 scales may also be written in the MXFP8 GEMM layout (sf_row / sf_col)."""
    x = _bf16_bits(x)
    rows, cols = x.shape
    fn = "mx_fp8_blockwise_quantize_1x128"
    _need(fn, "q_row", q_row, rows * cols)
    _need(fn, "s_row", s_row, 4 * rows * (cols // 128))
    _need(fn, "sf_row", sf_row, scale_bytes(rows, cols, 32))
    _need(fn, "q_col", q_col, rows * cols)
    _need(fn, "s_col", s_col, 4 * cols * (rows // 128))
    _need(fn, "sf_col", sf_col, scale_bytes(cols, rows, 32))
    _check("mx_fp8_blockwise_quantize_1x128", lib().mx_fp8_blockwise_quantize_1x128(
        _p(x), rows, cols, x.stride(0), int(bool(pow2)), _p(q_row), _p(s_row), _p(sf_row), _p(q_col), _p(s_col),
        _p(sf_col), _stream(stream)))


def mx_fp8_blockwise_quantize_128x128(w, pow2: bool, q_row, q_col, s, sf_row=None, sf_col=None, stream=None):
    """Blockwise FP8 of G stacked weights [G, O, H] in [128, 128] blocks: q_row [G, O, H], q_col
    [G, H, O], s [G, ceil(O/128), ceil(H/128)]; with pow2 optionally the MXFP8-layout E8M0 scales."""
    w = _bf16_bits(w, 3)
    G, O, H = w.shape
    fn = "mx_fp8_blockwise_quantize_128x128"
    _need(fn, "q_row", q_row, G * O * H)
    _need(fn, "q_col", q_col, G * O * H)
    _need(fn, "s", s, 4 * G * ((O + 127) // 128) * ((H + 127) // 128))
    _need(fn, "sf_row", sf_row, G * scale_bytes(O, H, 32))
    _need(fn, "sf_col", sf_col, G * scale_bytes(H, O, 32))
    _check("mx_fp8_blockwise_quantize_128x128", lib().mx_fp8_blockwise_quantize_128x128(
        _p(w), G, O, H, int(bool(pow2)), _p(q_row), _p(q_col), _p(s), _p(sf_row), _p(sf_col), _stream(stream)))


def mx_rht16(x, seed: int, y, stream=None):
    x = _bf16_bits(x)
    T, N = x.shape
    _need("mx_rht16", "x", x, 2 * T * N)
    _need("mx_rht16", "y", y, 2 * T * N)
    _check("mx_rht16", lib().mx_rht16(_p(x), T, N, seed, _p(y), _stream(stream)))


def mx_nvfp4_quantize_1x16(x, colwise: bool, rht: bool, rht_seed: int, sr: bool, sr_seed: int, q, s, s_tensor,
                           workspace, stream=None):
    x = _bf16_bits(x)
    T, N = x.shape
    fn = "mx_nvfp4_quantize_1x16"
    _need(fn, "x", x, 2 * T * N)
    _need(fn, "q", q, T * N // 2)
    _need(fn, "s", s, scale_bytes(N, T, 16) if colwise else scale_bytes(T, N, 16))
    _need(fn, "s_tensor", s_tensor, 4)
    _check("mx_nvfp4_quantize_1x16", lib().mx_nvfp4_quantize_1x16(
        _p(x), T, N, int(colwise), int(rht), rht_seed, MX_ROUND_SR if sr else MX_ROUND_RNE, sr_seed,
        _p(q), _p(s), _p(s_tensor), _p(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def mx_dequantize_bf16(fmt: int, q, s, s2, s2_scope: int, rows: int, cols: int, y, stream=None, group_rows: int = 0):
    fn, fp4 = "mx_dequantize_bf16", fmt == MX_FMT_NVFP4
    _need(fn, "q", q, rows * cols // 2 if fp4 else rows * cols)
    _need(fn, "s", s, scale_bytes(rows, cols, 16 if fp4 else 32))
    if fp4:
        n2 = {MX_SCOPE_ROW: rows, MX_SCOPE_GROUP: rows // max(int(group_rows), 1)}.get(s2_scope, 1)
        _need(fn, "s2", s2, 4 * n2)
    _need(fn, "y", y, 2 * rows * cols)
    _check("mx_dequantize_bf16", lib().mx_dequantize_bf16(
        fmt, _p(q), _p(s), _p(s2), s2_scope, group_rows, rows, cols, _p(y), _stream(stream)))


def _alpha_count(scope: int, n: int) -> int:
    return n if scope == MX_SCOPE_ROW else (1 if scope == MX_SCOPE_TENSOR else 0)


def mx_scaled_gemm(fmt: int, a, sa, alpha_a, alpha_a_scope: int, b, sb, alpha_b, alpha_b_scope: int,
                   M: int, N: int, K: int, d, stream=None):
    fn, fp4 = "mx_scaled_gemm", fmt == MX_FMT_NVFP4
    _need(fn, "a", a, M * K // 2 if fp4 else M * K)
    _need(fn, "b", b, N * K // 2 if fp4 else N * K)
    _need(fn, "sa", sa, scale_bytes(M, K, 16 if fp4 else 32))
    _need(fn, "sb", sb, scale_bytes(N, K, 16 if fp4 else 32))
    _need(fn, "alpha_a", alpha_a, 4 * _alpha_count(alpha_a_scope, M))
    _need(fn, "alpha_b", alpha_b, 4 * _alpha_count(alpha_b_scope, N))
    _need_out2d(fn, "d", d, M, N)
    _check("mx_scaled_gemm", lib().mx_scaled_gemm(
        fmt, _p(a), _p(sa), _p(alpha_a), alpha_a_scope, _p(b), _p(sb), _p(alpha_b), alpha_b_scope,
        M, N, K, _p(d), d.stride(0), _stream(stream)))


def mx_gemm_bf16_dq_nvfp4(a, qb, sb, sb2, sb2_scope, M: int, N: int, K: int, d, alpha_a=None, alpha_a_scope=0,
                          stream=None):
    """D = BF16(alpha_a * A @ DQ(B)^T) with A BF16 [M, K] and B NVFP4 codes [N, K/2] + GEMM-layout scales + FP32
    second-level scale(s) sb2 (MX_SCOPE_TENSOR or MX_SCOPE_ROW), B expanded to BF16 inside the GEMM."""
    a = _bf16_bits(a)
    if a.stride(0) != K or a.stride(1) != 1:
        raise ValueError("A must be a contiguous [M, K] BF16 tensor")
    fn = "mx_gemm_bf16_dq_nvfp4"
    _need(fn, "a", a, 2 * M * K)
    _need(fn, "alpha_a", alpha_a, 4 * _alpha_count(alpha_a_scope, M))
    _need(fn, "qb", qb, N * K // 2)
    _need(fn, "sb", sb, scale_bytes(N, K, 16))
    _need(fn, "sb2", sb2, 4 * _alpha_count(sb2_scope, N))
    _need_out2d(fn, "d", d, M, N)
    _check("mx_gemm_bf16_dq_nvfp4", lib().mx_gemm_bf16_dq_nvfp4(
        _p(a), _p(alpha_a), int(alpha_a_scope), _p(qb), _p(sb), _p(sb2), int(sb2_scope), M, N, K, _p(d), d.stride(0),
        _stream(stream)))


def mx_wgrad_bf16_dq_nvfp4(dy, qx, sx, sx2, sx2_scope, dw, stream=None):
    """dW = BF16(dY^T @ DQ(X)) with dY BF16 [T, O] and X as NVFP4 codes [T, H/2] + GEMM-layout scales + FP32
    second-level scale(s) (MX_SCOPE_ROW: per token, MX_SCOPE_TENSOR), X expanded to BF16 inside the GEMM."""
    dy = _bf16_bits(dy)
    T, O = dy.shape
    H = qx.shape[1] * 2
    if dy.stride(0) != O or dy.stride(1) != 1:
        raise ValueError("dY must be a contiguous [T, O] BF16 tensor")
    fn = "mx_wgrad_bf16_dq_nvfp4"
    _need(fn, "qx", qx, T * H // 2)
    _need(fn, "sx", sx, scale_bytes(T, H, 16))
    _need(fn, "sx2", sx2, 4 * _alpha_count(sx2_scope, T))
    _need_out2d(fn, "dw", dw, O, H)
    _check("mx_wgrad_bf16_dq_nvfp4", lib().mx_wgrad_bf16_dq_nvfp4(
        _p(dy), _p(qx), _p(sx), _p(sx2), int(sx2_scope), T, O, H, _p(dw), dw.stride(0), _stream(stream)))


def mx_fp8_blockwise_gemm(a, sa, b, sb, M: int, N: int, K: int, d, stream=None):
    """D = BF16(sum over 128-deep K blocks of sa[m, kb] * sb[n / 128, kb] * A_kb B_kb^T): E4M3 a [M, K] with
    FP32 [1, 128]-tile scales sa [M, K/128], E4M3 b [N, K] with FP32 [128, 128]-block scales sb."""
    fn = "mx_fp8_blockwise_gemm"
    _need(fn, "a", a, M * K)
    _need(fn, "sa", sa, 4 * M * (K // 128))
    _need(fn, "b", b, N * K)
    _need(fn, "sb", sb, 4 * ((N + 127) // 128) * (K // 128))
    _need_out2d(fn, "d", d, M, N)
    _check("mx_fp8_blockwise_gemm", lib().mx_fp8_blockwise_gemm(
        _p(a), _p(sa), _p(b), _p(sb), M, N, K, _p(d), d.stride(0), _stream(stream)))


def mx_fp8_blockwise_gemm_wgrad(a, sa, b, sb, M: int, N: int, K: int, d, stream=None):
    """D = BF16(sum over 128-deep K blocks of sa[m, kb] * sb[n, kb] * A_kb B_kb^T): both operands column-wise
    [1, 128]-tile copies (K = tokens) with FP32 scales sa [M, K/128], sb [N, K/128]."""
    fn = "mx_fp8_blockwise_gemm_wgrad"
    _need(fn, "a", a, M * K)
    _need(fn, "sa", sa, 4 * M * (K // 128))
    _need(fn, "b", b, N * K)
    _need(fn, "sb", sb, 4 * N * (K // 128))
    _need_out2d(fn, "d", d, M, N)
    _check(fn, lib().mx_fp8_blockwise_gemm_wgrad(
        _p(a), _p(sa), _p(b), _p(sb), M, N, K, _p(d), d.stride(0), _stream(stream)))


def mx_grouped_scaled_gemm(fmt: int, group_offsets, a, sa, alpha_a_rows, b, sb, alpha_b_groups, N: int, K: int, d,
                           stream=None):
    G = group_offsets.numel() - 1
    fn, fp4, rows = "mx_grouped_scaled_gemm", fmt == MX_FMT_NVFP4, a.shape[0]
    _need(fn, "group_offsets", group_offsets, 8 * (G + 1))
    _need(fn, "a", a, rows * K // 2 if fp4 else rows * K)
    _need(fn, "b", b, G * N * K // 2 if fp4 else G * N * K)
    _need(fn, "alpha_a_rows", alpha_a_rows, 4 * rows if alpha_a_rows is not None else 0)
    _need(fn, "alpha_b_groups", alpha_b_groups, 4 * G if alpha_b_groups is not None else 0)
    _need(fn, "d", d, 2 * rows * N)
    _check("mx_grouped_scaled_gemm", lib().mx_grouped_scaled_gemm(
        fmt, G, _p(group_offsets), a.shape[0], _p(a), _p(sa), _p(alpha_a_rows), _p(b), _p(sb), _p(alpha_b_groups),
        N, K, _p(d), _stream(stream)))


def mx_count_mismatch(x, y, count, stream=None):
    n = x.numel() * x.element_size()
    if y.numel() * y.element_size() != n:
        raise ValueError("byte sizes differ")
    _need("mx_count_mismatch", "x", x, n)
    _need("mx_count_mismatch", "y", y, n)
    _need("mx_count_mismatch", "count", count, 8)
    _check("mx_count_mismatch", lib().mx_count_mismatch(_p(x), _p(y), n, _p(count), _stream(stream)))


# ------------------------------------------------------------------------------------------------
# output allocation helpers (torch.empty only)
# ------------------------------------------------------------------------------------------------

def _u8(n: int, device) -> torch.Tensor:
    return torch.empty(n, dtype=torch.uint8, device=device)


def alloc_mxfp8(rows: int, cols: int, device, rowwise: bool = True, colwise: bool = True):
    out = {}
    if rowwise:
        out["q_row"] = torch.empty((rows, cols), dtype=torch.uint8, device=device)
        out["s_row"] = _u8(scale_bytes(rows, cols, 32), device)
    if colwise:
        out["q_col"] = torch.empty((cols, rows), dtype=torch.uint8, device=device)
        out["s_col"] = _u8(scale_bytes(cols, rows, 32), device)
    return out


def alloc_nvfp4_rows(rows: int, k: int, device):
    """Codes [rows, k/2], GEMM-layout scales and one FP32 second-level scale per row."""
    return {"q": torch.empty((rows, k // 2), dtype=torch.uint8, device=device),
            "s": _u8(scale_bytes(rows, k, 16), device),
            "s2": torch.empty(rows, dtype=torch.float32, device=device)}


def alloc_nvfp4_rows_grouped(rows: int, G: int, k: int, device):
    """Like alloc_nvfp4_rows with the scales sized for the grouped scale layout."""
    return {"q": torch.empty((rows, k // 2), dtype=torch.uint8, device=device),
            "s": _u8(grouped_scale_bytes(rows, G, k, 16), device),
            "s2": torch.empty(rows, dtype=torch.float32, device=device)}


def alloc_nvfp4_weight_2d(G: int, O: int, H: int, device):
    return {"q_row": torch.empty((G, O, H // 2), dtype=torch.uint8, device=device),
            "s_row": _u8(G * scale_bytes(O, H, 16), device),
            "q_col": torch.empty((G, H, O // 2), dtype=torch.uint8, device=device),
            "s_col": _u8(G * scale_bytes(H, O, 16), device),
            "s_w": torch.empty(G, dtype=torch.float32, device=device),
            "ws": _u8(max(16, workspace_bytes(MX_WS_WEIGHT_2D, G)), device)}
