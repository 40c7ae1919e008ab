"""CPU oracle for block-scaled microscaling numerics.

TEST INFRASTRUCTURE ONLY.  This package is the independent reference the CUDA
library is checked against; only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import it.  It shares no code with
the CUDA library: the per-element arithmetic lives in ``mxoracle.c`` (plain
C, FP32 round-to-nearest, no FMA contraction, no fast-math) and the FP64
GEMM reference below uses numpy's matmul as a library step.

Sources are the pages named in ``mxoracle.c``'s header.  Every function here
states the passage it follows.  Arrays are numpy; BF16 tensors are carried as
``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxoracle.c")
_LIB_PATH = os.path.join(_HERE, "libmxoracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-fexcess-precision=standard", "-fopenmp"]


def build(force: bool = False) -> str:
    """Compile ``mxoracle.c`` into ``libmxoracle.so`` with gcc (no GPU needed).

    ``MXORACLE_LIB`` names a prebuilt library to load instead; the oracle's
    mutation test uses it to run the pins against a deliberately broken copy."""
    override = os.environ.get("MXORACLE_LIB")
    if override:
        return override
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            U64 = ctypes.c_uint64
            sig = {
                "orc_e4m3_value": (ctypes.c_double, [ctypes.c_uint8]),
                "orc_e2m1_value": (ctypes.c_double, [ctypes.c_uint8]),
                "orc_e8m0_value": (ctypes.c_double, [ctypes.c_uint8]),
                "orc_e4m3_encode": (ctypes.c_uint8, [ctypes.c_double]),
                "orc_e2m1_encode": (ctypes.c_uint8, [ctypes.c_double]),
                "orc_e2m1_encode_sr": (ctypes.c_uint8, [ctypes.c_float, ctypes.c_uint32]),
                "orc_float_to_bf16": (ctypes.c_uint16, [ctypes.c_float]),
                "orc_philox4x32_10": (None, [P, P, P]),
                "orc_sr_bits16": (ctypes.c_uint32, [U64, U64]),
                "orc_rht16_signs": (None, [U64, P]),
                "orc_rht16_vec_f32": (None, [P, U64, P]),
                "orc_scale_layout_bytes": (I64, [I64, I64]),
                "orc_scale_layout_offset": (I64, [I64, I64, I64]),
                "orc_scales_to_gemm_layout": (None, [P, I64, I64, P]),
                "orc_scales_from_gemm_layout": (None, [P, I64, I64, P]),
                "orc_grouped_padded_rows": (I64, [I64, P]),
                "orc_scales_to_grouped_layout": (None, [P, I64, I64, I64, P, P, I64]),
                "orc_mxfp8_quantize_rowwise": (None, [P, I64, I64, I64, P, P]),
                "orc_mxfp8_quantize_colwise": (None, [P, I64, I64, I64, P, P]),
                "orc_nvfp4_second_scale": (ctypes.c_float, [ctypes.c_float]),
                "orc_nvfp4_block_scale": (ctypes.c_uint8, [ctypes.c_float, ctypes.c_float]),
                "orc_nvfp4_block_recip": (ctypes.c_float, [ctypes.c_uint8, ctypes.c_float]),
                "orc_nvfp4_quantize_per_token": (None, [P, I64, I64, I64, P, P, P]),
                "orc_nvfp4_quantize_weight_2d": (None, [P, I64, I64, P, P, P, P]),
                "orc_nvfp4_quantize_weight_2d_46": (None, [P, I64, I64, P, P, P, P]),
                "orc_nvfp4_quantize_per_token_46": (None, [P, I64, I64, I64, P, P, P]),
                "orc_fp8_blockwise_1x128": (None, [P, I64, I64, I64, ctypes.c_int, P, P, P]),
                "orc_fp8_blockwise_128x128": (None, [P, I64, I64, ctypes.c_int, P, P, P, P]),
                "orc_rht16": (None, [P, I64, I64, U64, P]),
                "orc_nvfp4_quantize_1x16": (None, [P, I64, I64, ctypes.c_int, ctypes.c_int, U64,
                                                   ctypes.c_int, U64, P, P, P]),
                "orc_nvfp4_1x16_amax": (ctypes.c_float, [P, I64, I64, ctypes.c_int, U64]),
                "orc_nvfp4_1x16_pass2": (None, [P, I64, I64, I64, I64, ctypes.c_int, ctypes.c_int, U64, ctypes.c_int, U64,
                                                ctypes.c_float, P, P]),
                "orc_dequant_mxfp8": (None, [P, P, I64, I64, P]),
                "orc_dequant_nvfp4": (None, [P, P, P, ctypes.c_int, I64, I64, P]),
                "orc_decode_mxfp8_f64": (None, [P, P, I64, I64, P]),
                "orc_decode_nvfp4_f64": (None, [P, P, I64, I64, P]),
                "orc_set_threads": (None, [ctypes.c_int]),
                "orc_get_threads": (ctypes.c_int, []),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _bf16(x) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint16:
        raise TypeError("BF16 inputs are passed as uint16 bit patterns")
    return x


def set_threads(n: int) -> None:
    _load().orc_set_threads(int(n))


def get_threads() -> int:
    return int(_load().orc_get_threads())


# ---------------------------------------------------------------------------
# Formats (public OCP MX / NVFP4 field definitions; the pages name E4M3, E2M1
# and E8M0: Miles "cada bloco de 32 valores E4M3 compartilha uma escala
# E8M0", "NVFP4 armazena valores E2M1 ... com uma escala E4M3").
# ---------------------------------------------------------------------------

def e4m3_value(code: int) -> float:
    return _load().orc_e4m3_value(code)


def e2m1_value(code: int) -> float:
    return _load().orc_e2m1_value(code)


def e8m0_value(code: int) -> float:
    return _load().orc_e8m0_value(code)


def e4m3_encode(v: float) -> int:
    return int(_load().orc_e4m3_encode(float(v)))


def e2m1_encode(v: float) -> int:
    return int(_load().orc_e2m1_encode(float(v)))


def e2m1_encode_sr(v: float, k16: int) -> int:
    return int(_load().orc_e2m1_encode_sr(float(np.float32(v)), int(k16)))


def float_to_bf16(f: float) -> int:
    return int(_load().orc_float_to_bf16(float(np.float32(f))))


def e4m3_table() -> np.ndarray:
    return np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def e2m1_table() -> np.ndarray:
    return np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)


def bf16_to_f32(x: np.ndarray) -> np.ndarray:
    """BF16 bit patterns -> float32 (exact widening)."""
    return (np.asarray(x, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# Counter-based RNG (Philox4x32-10, Salmon et al., SC'11) used for the SR
# uniforms and the RHT signs (MaxText: "random Hadamard transform",
# "stochastic rounding").
# ---------------------------------------------------------------------------

def philox4x32_10(ctr, key) -> tuple:
    c = np.asarray(ctr, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    out = np.zeros(4, dtype=np.uint32)
    _load().orc_philox4x32_10(_p(c), _p(k), _p(out))
    return tuple(int(v) for v in out)


def sr_bits16(seed: int, i: int) -> int:
    return int(_load().orc_sr_bits16(seed, i))


def rht16_signs(seed: int) -> np.ndarray:
    out = np.zeros(16, dtype=np.int32)
    _load().orc_rht16_signs(seed, _p(out))
    return out


def rht16_vec_f32(v: np.ndarray, seed: int) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.zeros(16, dtype=np.float32)
    _load().orc_rht16_vec_f32(_p(v), seed, _p(out))
    return out


# ---------------------------------------------------------------------------
# Scale-factor layout of the block-scaled GEMM (E2E, Table 6 "scale
# rearrangement" and F3 "stale swizzled scales": the GEMM consumes scales in
# an interleaved layout; the quantizer writes it directly).
# ---------------------------------------------------------------------------

def scale_layout_bytes(rows: int, scols: int) -> int:
    return int(_load().orc_scale_layout_bytes(rows, scols))


def scales_to_gemm_layout(compact: np.ndarray) -> np.ndarray:
    compact = np.ascontiguousarray(compact, dtype=np.uint8)
    rows, scols = compact.shape
    out = np.zeros(scale_layout_bytes(rows, scols), dtype=np.uint8)
    _load().orc_scales_to_gemm_layout(_p(compact), rows, scols, _p(out))
    return out


def scales_from_gemm_layout(laid: np.ndarray, rows: int, scols: int) -> np.ndarray:
    laid = np.ascontiguousarray(laid, dtype=np.uint8)
    out = np.zeros((rows, scols), dtype=np.uint8)
    _load().orc_scales_from_gemm_layout(_p(laid), rows, scols, _p(out))
    return out


def grouped_padded_rows(group_offsets) -> int:
    off = np.ascontiguousarray(group_offsets, dtype=np.int64)
    return int(_load().orc_grouped_padded_rows(off.size - 1, _p(off)))


def scales_to_grouped_layout(compact: np.ndarray, group_offsets, out_bytes: int = None) -> np.ndarray:
    """Compact scales [rows, scols] of expert-sorted rows -> the grouped GEMM layout (each group's
    rows start on a 128-row tile)."""
    compact = np.ascontiguousarray(compact, dtype=np.uint8)
    off = np.ascontiguousarray(group_offsets, dtype=np.int64)
    rows, scols = compact.shape
    if out_bytes is None:
        out_bytes = scale_layout_bytes(max(1, grouped_padded_rows(off)), scols)
    out = np.zeros(out_bytes, dtype=np.uint8)
    _load().orc_scales_to_grouped_layout(_p(compact), rows, scols, off.size - 1, _p(off), _p(out), out_bytes)
    return out


# ---------------------------------------------------------------------------
# Quantizers
# ---------------------------------------------------------------------------

def mxfp8_quantize_rowwise(x: np.ndarray):
    """MXFP8 1x32 blocks along the last dim (Miles: 32 E4M3 + one E8M0).
    Returns (codes uint8 [R, K], scales compact uint8 [R, K/32])."""
    x = _bf16(x)
    R, K = x.shape
    q = np.zeros((R, K), dtype=np.uint8)
    s = np.zeros((R, K // 32), dtype=np.uint8)
    _load().orc_mxfp8_quantize_rowwise(_p(x), R, K, K, _p(q), _p(s))
    return q, s


def mxfp8_quantize_colwise(x: np.ndarray):
    """MXFP8 32x1 blocks along rows, stored transposed (Miles: row-wise and
    column-wise copies both made from the high-precision input).
    Returns (codes [K, R], scales compact [K, R/32])."""
    x = _bf16(x)
    R, K = x.shape
    q = np.zeros((K, R), dtype=np.uint8)
    s = np.zeros((K, R // 32), dtype=np.uint8)
    _load().orc_mxfp8_quantize_colwise(_p(x), R, K, K, _p(q), _p(s))
    return q, s


def nvfp4_quantize_per_token(x: np.ndarray):
    """NVFP4 1x16 with a per-token FP32 scale (Miles, 4bitter).
    Returns (codes [T, H/2], scales compact [T, H/16], s_tok f32 [T])."""
    x = _bf16(x)
    T, H = x.shape
    q = np.zeros((T, H // 2), dtype=np.uint8)
    s = np.zeros((T, H // 16), dtype=np.uint8)
    st = np.zeros(T, dtype=np.float32)
    _load().orc_nvfp4_quantize_per_token(_p(x), T, H, H, _p(q), _p(s), _p(st))
    return q, s, st


def nvfp4_quantize_weight_2d(w: np.ndarray):
    """NVFP4 16x16 2D weight blocks under a per-matrix FP32 scale (MaxText).
    Returns (q_row [O, H/2], q_col [H, O/2], tile scales [O/16, H/16], s_w)."""
    w = _bf16(w)
    O, H = w.shape
    q_row = np.zeros((O, H // 2), dtype=np.uint8)
    q_col = np.zeros((H, O // 2), dtype=np.uint8)
    st = np.zeros((O // 16, H // 16), dtype=np.uint8)
    sw = np.zeros(1, dtype=np.float32)
    _load().orc_nvfp4_quantize_weight_2d(_p(w), O, H, _p(q_row), _p(q_col), _p(st), _p(sw))
    return q_row, q_col, st, np.float32(sw[0])


def nvfp4_quantize_per_token_46(x: np.ndarray):
    """Per-token NVFP4 with Four-over-Six block scales (NVIDIA RL blog, "Four-Over-Six"): each block
    keeps the scale mapping its maximum to 4 or to 6, whichever gives the smaller largest
    dequantization error (ties keep 6).  Returns as nvfp4_quantize_per_token."""
    x = _bf16(x)
    T, H = x.shape
    q = np.zeros((T, H // 2), dtype=np.uint8)
    s = np.zeros((T, H // 16), dtype=np.uint8)
    st = np.zeros(T, dtype=np.float32)
    _load().orc_nvfp4_quantize_per_token_46(_p(x), T, H, H, _p(q), _p(s), _p(st))
    return q, s, st


def nvfp4_quantize_weight_2d_46(w: np.ndarray):
    """16x16 2D weight NVFP4 with Four-over-Six tile scales.  Returns as nvfp4_quantize_weight_2d."""
    w = _bf16(w)
    O, H = w.shape
    q_row = np.zeros((O, H // 2), dtype=np.uint8)
    q_col = np.zeros((H, O // 2), dtype=np.uint8)
    st = np.zeros((O // 16, H // 16), dtype=np.uint8)
    sw = np.zeros(1, dtype=np.float32)
    _load().orc_nvfp4_quantize_weight_2d_46(_p(w), O, H, _p(q_row), _p(q_col), _p(st), _p(sw))
    return q_row, q_col, st, np.float32(sw[0])


def fp8_blockwise_1x128(x: np.ndarray, pow2: bool):
    """Blockwise FP8 of activations / gradients (PT page, "FP8 nas camadas lineares": E4M3 in [1, 128]
    tiles with one FP32 scale each; optionally power-of-two scales).
    Returns (codes uint8 [R, K], scales FP32 [R, K/128], E8M0 codes [R, K/128] (power of two only))."""
    x = _bf16(x)
    R, K = x.shape
    q = np.zeros((R, K), dtype=np.uint8)
    s = np.zeros((R, K // 128), dtype=np.float32)
    e8 = np.zeros((R, K // 128), dtype=np.uint8)
    _load().orc_fp8_blockwise_1x128(_p(x), R, K, K, int(pow2), _p(q), _p(s), _p(e8))
    return q, s, e8


def fp8_blockwise_128x128(w: np.ndarray, pow2: bool):
    """Blockwise FP8 of weights in [128, 128] blocks, both orientations.
    Returns (q_row [O, H], q_col [H, O], scales FP32 [ceil(O/128), ceil(H/128)], E8M0 codes of that shape)."""
    w = _bf16(w)
    O, H = w.shape
    q_row = np.zeros((O, H), dtype=np.uint8)
    q_col = np.zeros((H, O), dtype=np.uint8)
    bo, bh = (O + 127) // 128, (H + 127) // 128
    s = np.zeros((bo, bh), dtype=np.float32)
    e8 = np.zeros((bo, bh), dtype=np.uint8)
    _load().orc_fp8_blockwise_128x128(_p(w), O, H, int(pow2), _p(q_row), _p(q_col), _p(s), _p(e8))
    return q_row, q_col, s, e8


def fp8_blockwise_e8m0_rowwise(e8: np.ndarray, block: int = 128) -> np.ndarray:
    """E8M0 codes of power-of-two [1, 128] tiles repeated over their four 32-element sub-blocks: the MXFP8
    row-wise scale array [R, K/32] that decodes the same codes to the same values."""
    return np.repeat(np.asarray(e8, dtype=np.uint8), block // 32, axis=1)


def fp8_blockwise_e8m0_weight(e8: np.ndarray, O: int, H: int, orientation: str) -> np.ndarray:
    """E8M0 codes of power-of-two [128, 128] weight blocks as MXFP8 scales of one operand orientation:
    "row" gives [O, H/32] for the codes q_row [O, H]; "col" gives [H, O/32] for q_col [H, O]."""
    e8 = np.asarray(e8, dtype=np.uint8)
    if orientation == "row":
        return e8[np.arange(O)[:, None] // 128, (np.arange(H // 32) * 32)[None, :] // 128]
    if orientation == "col":
        return e8[(np.arange(O // 32) * 32)[None, :] // 128, np.arange(H)[:, None] // 128]
    raise ValueError(orientation)


def weight_2d_operand_scales(s_tile: np.ndarray, orientation: str) -> np.ndarray:
    """Expand 16x16 tile scales to the per-row 1x16 scale matrix a GEMM
    operand carries: 'row' -> [O, H/16], 'col' -> [H, O/16]."""
    if orientation == "row":
        return np.repeat(s_tile, 16, axis=0)
    return np.repeat(s_tile.T, 16, axis=0)


def rht16(x: np.ndarray, seed: int) -> np.ndarray:
    x = _bf16(x)
    T, N = x.shape
    y = np.zeros_like(x)
    _load().orc_rht16(_p(x), T, N, seed, _p(y))
    return y


def nvfp4_quantize_1x16(x: np.ndarray, colwise: bool, rht: bool = False, rht_seed: int = 0,
                        sr: bool = False, sr_seed: int = 0):
    """NVFP4 1x16 with a per-tensor FP32 scale (MaxText), optional RHT along
    tokens and SR.  Returns (codes, scales compact, S)."""
    x = _bf16(x)
    T, N = x.shape
    if colwise:
        q = np.zeros((N, T // 2), dtype=np.uint8)
        s = np.zeros((N, T // 16), dtype=np.uint8)
    else:
        q = np.zeros((T, N // 2), dtype=np.uint8)
        s = np.zeros((T, N // 16), dtype=np.uint8)
    st = np.zeros(1, dtype=np.float32)
    _load().orc_nvfp4_quantize_1x16(_p(x), T, N, int(colwise), int(rht), rht_seed, int(sr), sr_seed,
                                    _p(q), _p(s), _p(st))
    return q, s, np.float32(st[0])


def nvfp4_1x16_amax(x: np.ndarray, rht: bool = False, rht_seed: int = 0) -> np.float32:
    """Pass 1 of the per-tensor 1x16 quantizer on a [T, N] tensor or column slab (MaxText recipe:
    per-tensor FP32 scale; RHT on WGRAD inputs)."""
    x = _bf16(x)
    T, N = x.shape
    return np.float32(_load().orc_nvfp4_1x16_amax(_p(x), T, N, int(rht), rht_seed))


def nvfp4_1x16_pass2(x_slab: np.ndarray, n_offset: int, N_total: int, S, colwise: bool, rht: bool = False,
                     rht_seed: int = 0, sr: bool = False, sr_seed: int = 0):
    """Pass 2 on columns [n_offset, n_offset + N) of a [T, N_total] tensor with a given per-tensor
    scale S; SR indices use the global element index t * N_total + n."""
    x = _bf16(x_slab)
    T, N = x.shape
    if colwise:
        q = np.zeros((N, T // 2), dtype=np.uint8)
        s = np.zeros((N, T // 16), dtype=np.uint8)
    else:
        q = np.zeros((T, N // 2), dtype=np.uint8)
        s = np.zeros((T, N // 16), dtype=np.uint8)
    _load().orc_nvfp4_1x16_pass2(_p(x), T, N, n_offset, N_total, int(colwise), int(rht), rht_seed, int(sr), sr_seed,
                                 float(np.float32(S)), _p(q), _p(s))
    return q, s


def nvfp4_second_scale(amax) -> np.float32:
    return np.float32(_load().orc_nvfp4_second_scale(float(np.float32(amax))))


# ---------------------------------------------------------------------------
# Dequantize (4bitter: y = x * DQ(Q(w_bf16))) and exact decode
# ---------------------------------------------------------------------------

def dequant_mxfp8(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.uint8)
    R, K = q.shape
    y = np.zeros((R, K), dtype=np.uint16)
    _load().orc_dequant_mxfp8(_p(q), _p(s), R, K, _p(y))
    return y


def dequant_nvfp4(q: np.ndarray, s: np.ndarray, s2, per_row: bool) -> np.ndarray:
    """s2 is the FP32 second-level scale: one per row (per token) when
    ``per_row``, else a single per-tensor value."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.uint8)
    s2 = np.ascontiguousarray(np.atleast_1d(np.asarray(s2, dtype=np.float32)))
    R, K2 = q.shape
    K = K2 * 2
    if per_row and s2.size != R:
        raise ValueError("per-row second-level scale needs one value per row")
    y = np.zeros((R, K), dtype=np.uint16)
    _load().orc_dequant_nvfp4(_p(q), _p(s), _p(s2), int(bool(per_row)), R, K, _p(y))
    return y


def decode_mxfp8_f64(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.uint8)
    R, K = q.shape
    out = np.zeros((R, K), dtype=np.float64)
    _load().orc_decode_mxfp8_f64(_p(q), _p(s), R, K, _p(out))
    return out


def decode_nvfp4_f64(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.uint8)
    R, K2 = q.shape
    out = np.zeros((R, K2 * 2), dtype=np.float64)
    _load().orc_decode_nvfp4_f64(_p(q), _p(s), R, K2 * 2, _p(out))
    return out


# ---------------------------------------------------------------------------
# FP64 GEMM reference (MaxText: the three GEMMs take quantized inputs and emit
# BF16; Miles: MXFP8 forward, weight-gradient and data-gradient GEMMs).
#   ref[m, n] = alpha_a[m] * alpha_b[n] * sum_k DQ(A)[m, k] * DQ(B)[n, k]
# with DQ the exact decoded values; numpy's float64 matmul is the library step.
# ---------------------------------------------------------------------------

def gemm_ref_mxfp8(qa, sa, qb, sb) -> np.ndarray:
    return decode_mxfp8_f64(qa, sa) @ decode_mxfp8_f64(qb, sb).T


def gemm_ref_nvfp4(qa, sa, alpha_a, qb, sb, alpha_b) -> np.ndarray:
    A = decode_nvfp4_f64(qa, sa)
    B = decode_nvfp4_f64(qb, sb)
    ref = A @ B.T
    aa = np.asarray(alpha_a, dtype=np.float64).reshape(-1, 1) if np.ndim(alpha_a) else np.float64(alpha_a)
    ab = np.asarray(alpha_b, dtype=np.float64).reshape(1, -1) if np.ndim(alpha_b) else np.float64(alpha_b)
    return ref * aa * ab


def gemm_ref_bf16_dq_nvfp4(a: np.ndarray, qb, sb, sb2, per_row: bool, alpha_a=None) -> np.ndarray:
    """The dequantized-backward GEMM (4-bitter page, "dequantized backward": BF16 operands rebuilt from the
    forward's NVFP4 values): ref = alpha_a * A @ DQ(B)^T with A BF16 [M, K] and DQ(B) the BF16 values of
    dequant_nvfp4 (sb the compact [N, K/16] scales); numpy's float64 matmul is the library step."""
    A = bf16_to_f32(_bf16(a)).astype(np.float64)
    B = bf16_to_f32(dequant_nvfp4(qb, sb, sb2, per_row)).astype(np.float64)
    ref = A @ B.T
    if alpha_a is not None:
        aa = np.asarray(alpha_a, dtype=np.float64)
        ref = ref * (aa.reshape(-1, 1) if aa.ndim else aa)
    return ref


def fp8_blockwise_decode_f64(q: np.ndarray, s: np.ndarray, block_rows: int, block_cols: int) -> np.ndarray:
    """Exact values of blockwise FP8 codes: E4M3 value of each code times its block's FP32 scale, with one
    scale per block_rows x block_cols block (1 x 128 for activations and gradients, 128 x 128 for weights;
    s holds ceil(R / block_rows) x ceil(C / block_cols) scales)."""
    q = np.asarray(q, dtype=np.uint8)
    R, C = q.shape
    mag = e4m3_table()[q & 0x7F].astype(np.float64) * np.where(q & 0x80, -1.0, 1.0)
    sx = np.repeat(np.repeat(np.asarray(s, dtype=np.float64), block_rows, 0), block_cols, 1)[:R, :C]
    return mag * sx


def gemm_ref_fp8_blockwise(qa, sa, qb, sb) -> np.ndarray:
    """The blockwise FP8 GEMM (NeMo RL FP8 page, DeepSeek-V3 recipe: [1, 128] activation tiles, [128, 128]
    weight blocks, FP32 scales): ref = DQ(A) @ DQ(B)^T in FP64, DQ the exact decoded values."""
    return fp8_blockwise_decode_f64(qa, sa, 1, 128) @ fp8_blockwise_decode_f64(qb, sb, 128, 128).T


def gemm_ref_fp8_blockwise_wgrad(qa, sa, qb, sb) -> np.ndarray:
    """The blockwise FP8 weight-gradient GEMM (NeMo RL FP8 page, "FP8 nas camadas lineares": activations and
    output gradients in [1, 128] tiles with FP32 scales; the weight gradient contracts both over tokens, so
    both operands are [1, 128]-tiled along K): ref = DQ(A) @ DQ(B)^T in FP64, DQ the exact decoded values,
    sa [M, K/128] and sb [N, K/128]."""
    return fp8_blockwise_decode_f64(qa, sa, 1, 128) @ fp8_blockwise_decode_f64(qb, sb, 1, 128).T


def rel_fro_error(d: np.ndarray, ref: np.ndarray) -> float:
    """||D - ref||_F / ||ref||_F."""
    d = np.asarray(d, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(d - ref) / den) if den > 0 else float(np.linalg.norm(d))
