"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws random tensors and routes tokens; it holds none of the
quantization, transform or GEMM arithmetic, so both the CUDA path's tests and
the CPU oracle can take their inputs from it.

BF16 tensors are returned as numpy ``uint16`` bit patterns (the FP32 draws are
rounded to BF16 by round-to-nearest-even through ``torch``'s conversion).

Workloads (stand-ins for the pages' models; no dataset or weight is needed
because the bytes moved depend only on shapes and value distributions):

* ``tiny``        -- activation 256x1024 ~ N(0,1) with 0.5% outliers x50, one
                     all-zero 32-block (row 0, cols 0..31) and one
                     subnormal-only block (row 1, cols 0..31); weight
                     512x1024 ~ N(0, 0.02); seed 0.
* ``dense_mlp``   -- Qwen3-8B-shaped MLP linear: X 8192x4096 Student-t(3),
                     W 12288x4096 N(0, 0.02), dY 8192x12288 N(0, 1e-3);
                     seeds 1, 2, 3.
* ``moe``         -- Qwen3-30B-A3B expert layer: X 8192x2048 Student-t(3) and
                     a uniform top-8-of-128 router (seed 4), giving 65536
                     expert-sorted rows; a 65536x768 down-projection input;
                     128 experts x (gate 768x2048, up 768x2048, down 2048x768)
                     N(0, 0.02) (seed 5).
* ``wgrad``       -- Llama-3-8B-shaped WGRAD inputs: X 32768x4096
                     Student-t(3) (seed 6), dY 32768x14336 N(0, 1e-3) (seed 7);
                     RHT seed 8, SR seed 9.
* ``weight_sync`` -- per layer l (48 layers): 128 experts x {2048x768,
                     768x2048, 768x2048} N(0, 0.02), seed 1000 + l.
"""
from __future__ import annotations

import os

import numpy as np
import torch


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """FP32 array -> BF16 bit patterns (round to nearest even)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# Tensors of at least this many elements are drawn in fixed chunks of independent streams (seeded from
# one draw of the caller's generator), filled by a thread pool: the values depend on the seed only, not
# on the number of threads.  Smaller tensors come straight from the caller's generator.
_BIG = 1 << 22
_CHUNK = 1 << 22


def _chunked_f32(rng: np.random.Generator, shape, fill) -> np.ndarray:
    """A float32 array of `shape` whose chunk i is fill(Generator_i, out_chunk_i)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    seeds = np.random.SeedSequence(int(rng.integers(0, 2 ** 63))).spawn((n + _CHUNK - 1) // _CHUNK)

    def work(i):
        fill(np.random.default_rng(seeds[i]), out[i * _CHUNK:(i + 1) * _CHUNK])

    import concurrent.futures as cf
    with cf.ThreadPoolExecutor(max_workers=min(len(seeds), os.cpu_count() or 1)) as ex:
        list(ex.map(work, range(len(seeds))))
    return out.reshape(shape)


def normal(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    if int(np.prod(shape)) >= _BIG:
        def fill(g, o):
            g.standard_normal(out=o, dtype=np.float32)
            o *= np.float32(std)
        return to_bf16_bits(_chunked_f32(rng, shape, fill))
    return to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(std))


def student_t(rng: np.random.Generator, shape, nu: float = 3.0, scale: float = 1.0) -> np.ndarray:
    if int(np.prod(shape)) >= _BIG and nu == 3.0:
        # Student-t with 3 degrees of freedom as z / sqrt(chi2_3 / 3), chi2_3 a sum of three squared
        # standard normals (the textbook construction; the same distribution as Generator.standard_t(3))
        def fill(g, o):
            z = g.standard_normal(o.shape[0], dtype=np.float32)
            c = np.zeros(o.shape[0], dtype=np.float32)
            for _ in range(3):
                u = g.standard_normal(o.shape[0], dtype=np.float32)
                c += u * u
            o[:] = z / np.sqrt(c / np.float32(3.0)) * np.float32(scale)
        return to_bf16_bits(_chunked_f32(rng, shape, fill))
    return to_bf16_bits((rng.standard_t(nu, size=shape) * scale).astype(np.float32))


# ---------------------------------------------------------------------------
# tiny
# ---------------------------------------------------------------------------

def tiny(seed: int = 0, rows: int = 256, cols: int = 1024, out_features: int = 512):
    """Returns dict(x, w) of BF16 bits."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, cols), dtype=np.float32)
    n_out = int(round(0.005 * rows * cols))
    idx = rng.choice(rows * cols, size=n_out, replace=False)
    x.reshape(-1)[idx] *= np.float32(50.0)
    xb = to_bf16_bits(x)
    # one all-zero 32-block: row 0, cols 0..31
    xb[0, 0:32] = 0
    # one subnormal-only block: row 1, cols 0..31, values +-k * 2^-133, k in 1..127
    if rows > 1:
        k = rng.integers(1, 128, size=32).astype(np.uint16)      # BF16 subnormal mantissa
        sign = (rng.integers(0, 2, size=32).astype(np.uint16) << 15)
        xb[1, 0:32] = sign | k
    w = normal(rng, (out_features, cols), 0.02)
    return {"x": xb, "w": w}


# ---------------------------------------------------------------------------
# dense_mlp
# ---------------------------------------------------------------------------

def dense_mlp(tokens: int = 8192, hidden: int = 4096, ffn: int = 12288):
    x = student_t(np.random.default_rng(1), (tokens, hidden))
    w = normal(np.random.default_rng(2), (ffn, hidden), 0.02)
    dy = normal(np.random.default_rng(3), (tokens, ffn), 1e-3)
    return {"x": x, "w": w, "dy": dy}


# ---------------------------------------------------------------------------
# moe
# ---------------------------------------------------------------------------

def route_uniform_topk(rng: np.random.Generator, tokens: int, experts: int, topk: int):
    """Uniform router: each token's experts are the first ``topk`` entries of
    a seeded Fisher-Yates permutation of 0..experts-1.  Rows are then sorted
    stably by (expert, token).  Returns (row_token [tokens*topk] int64,
    group_offsets [experts+1] int64)."""
    # one Fisher-Yates shuffle per token, back to front, all tokens at once (token t's uniforms are row t)
    u = rng.random((tokens, experts - 1))
    perm = np.tile(np.arange(experts, dtype=np.int64), (tokens, 1))
    rows = np.arange(tokens)
    for i in range(experts - 1, 0, -1):
        j = (u[:, experts - 1 - i] * (i + 1)).astype(np.int64)
        pi = perm[:, i].copy()
        perm[:, i] = perm[rows, j]
        perm[rows, j] = pi
    choice = perm[:, :topk]
    expert_of_row = choice.reshape(-1)
    token_of_row = np.repeat(np.arange(tokens, dtype=np.int64), topk)
    order = np.lexsort((token_of_row, expert_of_row))   # primary: expert, then token
    counts = np.bincount(expert_of_row, minlength=experts)
    offsets = np.zeros(experts + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    return token_of_row[order], offsets


def moe(tokens: int = 8192, hidden: int = 2048, ffn: int = 768, experts: int = 128, topk: int = 8,
        with_weights: bool = True):
    rng = np.random.default_rng(4)
    x = student_t(rng, (tokens, hidden))
    row_token, offsets = route_uniform_topk(rng, tokens, experts, topk)
    down_in = student_t(rng, (tokens * topk, ffn))
    out = {"x": x, "row_token": row_token, "group_offsets": offsets, "down_in": down_in}
    if with_weights:
        wr = np.random.default_rng(5)
        out["w_gate_up"] = normal(wr, (experts, 2 * ffn, hidden), 0.02)   # gate rows then up rows
        out["w_down"] = normal(wr, (experts, hidden, ffn), 0.02)
    return out


# ---------------------------------------------------------------------------
# wgrad
# ---------------------------------------------------------------------------

def wgrad(tokens: int = 32768, hidden: int = 4096, ffn: int = 14336):
    x = student_t(np.random.default_rng(6), (tokens, hidden))
    dy = normal(np.random.default_rng(7), (tokens, ffn), 1e-3)
    return {"x": x, "dy": dy, "rht_seed": 8, "sr_seed": 9}


def dense_nvfp4(tokens: int = 32768, hidden: int = 4096, ffn: int = 14336):
    """The NVFP4 pretraining linear layer at the MaxText benchmark's Llama-3-8B MLP shapes: the WGRAD
    inputs of ``wgrad`` plus the weight [ffn, hidden] N(0, 0.02) (seed 10)."""
    d = wgrad(tokens, hidden, ffn)
    d["w"] = normal(np.random.default_rng(10), (ffn, hidden), 0.02)
    return d


# ---------------------------------------------------------------------------
# weight_sync
# ---------------------------------------------------------------------------

def weight_sync_layer(layer: int, experts: int = 128, hidden: int = 2048, ffn: int = 768):
    rng = np.random.default_rng(1000 + layer)
    return {
        "down": normal(rng, (experts, hidden, ffn), 0.02),
        "gate": normal(rng, (experts, ffn, hidden), 0.02),
        "up": normal(rng, (experts, ffn, hidden), 0.02),
    }


def random_bf16(seed: int, shape, kind: str = "normal", scale: float = 1.0) -> np.ndarray:
    """Small helper for parity cases of arbitrary shape."""
    rng = np.random.default_rng(seed)
    if kind == "normal":
        return normal(rng, shape, scale)
    if kind == "student_t":
        return student_t(rng, shape, 3.0, scale)
    raise ValueError(kind)
