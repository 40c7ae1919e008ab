"""GPU parity: quantizers, RHT, dequantize and the byte comparator against the CPU oracle.

Bit-exact for every code, scale byte (including the zero padding of the GEMM layout) and FP32
second-level scale, SR included.  Shapes span several CTA tiles and ragged tails; inputs include
zero blocks, subnormals, the largest finite BF16 values and negative zeros (the pages' quantizer
contract: random values, boundary cases, zero tensors and max-representable values).
"""
import numpy as np
import pytest
import torch

import synthetic
from gpu_util import DEV, bf16_dev, first_mismatch, to_np, to_np_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    import microscaled_precision_numerics_gb300 as m
    m.lib()
    return m


def edge_tensor(seed, shape):
    """Random values with planted boundary cases."""
    rng = np.random.default_rng(seed)
    x = synthetic.random_bf16(seed, shape, "student_t")
    flat = x.reshape(-1)
    n = flat.size
    idx = rng.choice(n, size=min(n, 64), replace=False)
    specials = np.array([0x7F7F, 0xFF7F, 0x0001, 0x8001, 0x007F, 0x8000, 0x0000, 0x0080, 0x3F80, 0x4380,
                         0x43E0, 0x43E1, 0xC3E0], dtype=np.uint16)   # max, -max, subnormals, -0, 0, 1, 256, 448
    flat[idx] = specials[np.arange(idx.size) % specials.size]
    return x


# ------------------------------------------------------------------------------------------------
# MXFP8
# ------------------------------------------------------------------------------------------------
MXFP8_SHAPES = [(256, 1024), (512, 1024), (96, 160), (32, 32), (160, 64), (384, 416), (992, 96)]


@pytest.mark.parametrize("shape", MXFP8_SHAPES)
def test_mxfp8_row_and_col(mx, orc, shape):
    R, K = shape
    x = synthetic.tiny(rows=R, cols=K, out_features=32)["x"] if shape == (256, 1024) else edge_tensor(R * 7 + K, shape)
    if R % 32:
        pytest.skip("column-wise needs rows % 32 == 0")
    out = mx.alloc_mxfp8(R, K, DEV)
    for v in out.values():
        v.fill_(0xAB)          # the quantizer must overwrite every byte, padding included
    mx.mx_quantize_mxfp8(bf16_dev(x), **out)
    torch.cuda.synchronize()
    qr, sr = orc.mxfp8_quantize_rowwise(x)
    qc, sc = orc.mxfp8_quantize_colwise(x)
    assert np.array_equal(to_np(out["q_row"]), qr), first_mismatch(to_np(out["q_row"]), qr)
    assert np.array_equal(to_np(out["s_row"]), orc.scales_to_gemm_layout(sr))
    assert np.array_equal(to_np(out["q_col"]), qc), first_mismatch(to_np(out["q_col"]), qc)
    assert np.array_equal(to_np(out["s_col"]), orc.scales_to_gemm_layout(sc))


def test_mxfp8_row_codes_16_byte_aligned_output(mx, orc):
    """Row-wise codes into a buffer that is 16-byte but not 32-byte aligned: the row pass then writes
    each thread's 32 code bytes as two 16-byte stores instead of one 32-byte store."""
    R, K = 384, 416
    x = edge_tensor(R * 5 + K, (R, K))
    out = mx.alloc_mxfp8(R, K, DEV)
    q_row = torch.full((R * K + 32,), 0xAB, dtype=torch.uint8, device=DEV)[16:16 + R * K].view(R, K)
    assert q_row.data_ptr() % 32 == 16
    mx.mx_quantize_mxfp8(bf16_dev(x), q_row=q_row, s_row=out["s_row"], q_col=out["q_col"], s_col=out["s_col"])
    torch.cuda.synchronize()
    qr, sr = orc.mxfp8_quantize_rowwise(x)
    qc, _ = orc.mxfp8_quantize_colwise(x)
    assert np.array_equal(to_np(q_row), qr), first_mismatch(to_np(q_row), qr)
    assert np.array_equal(to_np(out["s_row"]), orc.scales_to_gemm_layout(sr))
    assert np.array_equal(to_np(out["q_col"]), qc)


@pytest.mark.parametrize("which", ["both", "row", "col"])
def test_mxfp8_batched(mx, orc, which):
    """One launch over tensors of different shapes (ragged tiles, one strided) gives each tensor exactly the
    codes and scales of the oracle's per-tensor quantizer."""
    shapes = [(256, 1024), (96, 160), (384, 416), (64, 128)]
    xs = [edge_tensor(31 * i + R + K, (R, K)) for i, (R, K) in enumerate(shapes)]
    jobs, outs = [], []
    for i, ((R, K), x) in enumerate(zip(shapes, xs)):
        out = mx.alloc_mxfp8(R, K, DEV, rowwise=which != "col", colwise=which != "row")
        for v in out.values():
            v.fill_(0xAB)
        xd = bf16_dev(x)
        if i == 3:                                # a row pitch of 192 elements
            wide = torch.zeros((R, 192), dtype=torch.bfloat16, device=DEV)
            wide[:, :K] = xd
            xd = wide[:, :K]
        jobs.append((xd, out))
        outs.append(out)
    mx.mx_quantize_mxfp8_batched(jobs)
    torch.cuda.synchronize()
    mx.check_device_status()
    for x, out in zip(xs, outs):
        if which != "col":
            qr, sr = orc.mxfp8_quantize_rowwise(x)
            assert np.array_equal(to_np(out["q_row"]), qr), first_mismatch(to_np(out["q_row"]), qr)
            assert np.array_equal(to_np(out["s_row"]), orc.scales_to_gemm_layout(sr))
        if which != "row":
            qc, sc = orc.mxfp8_quantize_colwise(x)
            assert np.array_equal(to_np(out["q_col"]), qc), first_mismatch(to_np(out["q_col"]), qc)
            assert np.array_equal(to_np(out["s_col"]), orc.scales_to_gemm_layout(sc))


def test_mxfp8_rowwise_only_ragged_rows(mx, orc):
    x = edge_tensor(5, (37, 96))
    out = mx.alloc_mxfp8(37, 96, DEV, colwise=False)
    out["s_row"].fill_(0xCD)
    mx.mx_quantize_mxfp8(bf16_dev(x), **out)
    qr, sr = orc.mxfp8_quantize_rowwise(x)
    assert np.array_equal(to_np(out["q_row"]), qr)
    assert np.array_equal(to_np(out["s_row"]), orc.scales_to_gemm_layout(sr))


def test_mxfp8_strided_input(mx, orc):
    base = edge_tensor(6, (64, 192))
    xt = bf16_dev(base)[:, :128]          # ldx = 192
    out = mx.alloc_mxfp8(64, 128, DEV)
    mx.mx_quantize_mxfp8(xt, **out)
    sub = np.ascontiguousarray(base[:, :128])
    qr, sr = orc.mxfp8_quantize_rowwise(sub)
    qc, sc = orc.mxfp8_quantize_colwise(sub)
    assert np.array_equal(to_np(out["q_row"]), qr)
    assert np.array_equal(to_np(out["q_col"]), qc)


def test_mxfp8_zero_tensor(mx, orc):
    x = np.zeros((64, 64), dtype=np.uint16)
    out = mx.alloc_mxfp8(64, 64, DEV)
    mx.mx_quantize_mxfp8(bf16_dev(x), **out)
    assert int(out["q_row"].sum()) == 0 and int(out["s_row"].sum()) == 0 and int(out["q_col"].sum()) == 0


def test_mxfp8_negative_zero_and_tiny_negatives(mx, orc):
    row = np.full(32, 0x8000, dtype=np.uint16)      # -0
    row[0] = 0x4300                                   # 128 (sets the block scale)
    row[1:8] = 0x8001                                 # tiny negative subnormals -> round to -0
    x = np.tile(row, (32, 1))
    out = mx.alloc_mxfp8(32, 32, DEV)
    mx.mx_quantize_mxfp8(bf16_dev(x), **out)
    qr, _ = orc.mxfp8_quantize_rowwise(x)
    assert np.array_equal(to_np(out["q_row"]), qr), first_mismatch(to_np(out["q_row"]), qr)


# ------------------------------------------------------------------------------------------------
# NVFP4 per-token
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("shape", [(256, 1024), (100, 48), (65, 768), (8, 2048), (300, 4160)])
def test_nvfp4_per_token(mx, orc, shape):
    T, H = shape
    x = edge_tensor(T + 3 * H, shape)
    x[min(2, T - 1)] = 0                              # a zero token
    out = mx.alloc_nvfp4_rows(T, H, DEV)
    out["s"].fill_(0xEE)
    mx.mx_nvfp4_quantize_per_token(bf16_dev(x), out["q"], out["s"], out["s2"])
    q, s, st = orc.nvfp4_quantize_per_token(x)
    assert np.array_equal(to_np(out["q"]), q), first_mismatch(to_np(out["q"]), q)
    assert np.array_equal(to_np(out["s"]), orc.scales_to_gemm_layout(s))
    assert np.array_equal(to_np(out["s2"]).view(np.uint32), st.view(np.uint32))


def e4m3_tie_tensor(seed, T, H, per_tensor):
    """Blocks whose scale quotient amax_b / 6 / S lands exactly on an E4M3 rounding midpoint (and one BF16
    step either side of it): S is a power of two (token or tensor amax 2688 * 2^k), so the quotient is
    exact, and the device's fast block-scale path must hand these blocks to the IEEE divisions."""
    rng = np.random.default_rng(seed)
    e4 = np.array([(1 + i / 8) * 2.0 ** e for e in range(-6, 9) for i in range(8)] + [i * 2.0 ** -9 for i in range(1, 8)])
    e4 = np.unique(e4[e4 <= 448])
    mids = (e4[:-1] + e4[1:]) / 2                                   # all exactly representable
    x = np.zeros((T, H), dtype=np.float32)
    k_all = rng.integers(-20, 20)
    for t in range(T):
        k = k_all if per_tensor else rng.integers(-20, 20)
        for b in range(H // 16):
            blk = x[t, 16 * b:16 * b + 16]
            if b == 0:
                amax = 2688.0 * 2.0 ** k                            # the token (tensor) maximum: S = 2^k
            else:
                m = mids[rng.integers(0, mids.size)] * 6.0 * 2.0 ** k
                step = rng.integers(-1, 2)                          # on the midpoint or one BF16 step off
                amax = float(np.float32(m)) * (1 + step * 2.0 ** -7)
            blk[:] = rng.uniform(-1, 1, 16).astype(np.float32) * amax * 0.9
            blk[rng.integers(0, 16)] = amax * rng.choice([-1.0, 1.0])
    u = x.view(np.uint32)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def test_nvfp4_subnormal_tokens_and_blocks(mx, orc):
    """Tokens made only of BF16 subnormals (so S, the block scales and every maximum come from subnormal
    values) and subnormal-only blocks inside ordinary tokens, per token and per tensor."""
    T, H = 64, 128
    rng = np.random.default_rng(21)
    x = synthetic.random_bf16(22, (T, H), "normal")
    sub = (rng.integers(1, 128, size=(T, H)) | (rng.integers(0, 2, size=(T, H)) << 15)).astype(np.uint16)
    x[::3] = sub[::3]                                   # whole tokens of subnormals
    x[1::3, 16:32] = sub[1::3, 16:32]                   # one subnormal-only block in other tokens
    out = mx.alloc_nvfp4_rows(T, H, DEV)
    mx.mx_nvfp4_quantize_per_token(bf16_dev(x), out["q"], out["s"], out["s2"])
    q, s, st = orc.nvfp4_quantize_per_token(x)
    assert np.array_equal(to_np(out["q"]), q), first_mismatch(to_np(out["q"]), q)
    assert np.array_equal(to_np(out["s"]), orc.scales_to_gemm_layout(s))
    assert np.array_equal(to_np(out["s2"]).view(np.uint32), st.view(np.uint32))
    xs = np.ascontiguousarray(sub)                      # a whole tensor of subnormals, row- and column-wise
    for colwise in (False, True):
        qd = torch.empty((H, T // 2) if colwise else (T, H // 2), dtype=torch.uint8, device=DEV)
        sd = torch.empty(mx.scale_bytes(H, T, 16) if colwise else mx.scale_bytes(T, H, 16), dtype=torch.uint8, device=DEV)
        S = torch.empty(1, dtype=torch.float32, device=DEV)
        ws = torch.empty(16, dtype=torch.uint8, device=DEV)
        mx.mx_nvfp4_quantize_1x16(bf16_dev(xs), colwise, False, 0, False, 0, qd, sd, S, ws)
        qo, so, So = orc.nvfp4_quantize_1x16(xs, colwise=colwise)
        assert to_np(S).view(np.uint32)[0] == np.float32(So).view(np.uint32)
        assert np.array_equal(to_np(qd), qo), first_mismatch(to_np(qd), qo)
        assert np.array_equal(to_np(sd), orc.scales_to_gemm_layout(so))


def test_weight_sync_fused_maxima(mx, orc):
    """The weight-sync chain with the matrix maxima carried between calls: MXFP8 quantize that also
    returns each matrix's max |w|, the 2D NVFP4 quantizer fed that maximum, and the NVFP4 dequantize that
    returns each matrix's max |y| -- every output identical to the plain calls and to the oracle, the
    maxima equal to the exact ones."""
    G, O, H = 3, 256, 384
    w = synthetic.random_bf16(31, (G, O, H), "normal", 0.02)
    w[1, 5, 7] = 0x4100                                      # a spike in one matrix (8.0)
    wd = bf16_dev(w)
    exact = (w.astype(np.uint32) & 0x7FFF).reshape(G, -1).max(axis=1) << 16
    # MXFP8 with the maxima
    m8 = mx.alloc_mxfp8(G * O, H, DEV)
    amax = torch.full((G,), -1, dtype=torch.int32, device=DEV)
    mx.mx_quantize_mxfp8_amax(wd.view(G * O, H), O, amax, **m8)
    ref8 = mx.alloc_mxfp8(G * O, H, DEV)
    mx.mx_quantize_mxfp8(wd.view(G * O, H), **ref8)
    for k in ("q_row", "s_row", "q_col", "s_col"):
        assert torch.equal(m8[k], ref8[k]), k
    assert np.array_equal(to_np(amax).view(np.uint32), exact.astype(np.uint32))
    # the 2D quantizer given those maxima
    n4 = mx.alloc_nvfp4_weight_2d(G, O, H, DEV)
    mx.mx_nvfp4_quantize_weight_2d_given_amax(wd, n4["q_row"], n4["s_row"], n4["q_col"], n4["s_col"], n4["s_w"], amax)
    ref4 = mx.alloc_nvfp4_weight_2d(G, O, H, DEV)
    mx.mx_nvfp4_quantize_weight_2d(wd, ref4["q_row"], ref4["s_row"], ref4["q_col"], ref4["s_col"], ref4["s_w"], ref4["ws"])
    for k in ("q_row", "s_row", "q_col", "s_col", "s_w"):
        assert torch.equal(n4[k], ref4[k]), k
    for g in range(G):
        qr, qc, st, sw = orc.nvfp4_quantize_weight_2d(np.ascontiguousarray(w[g]))
        assert np.array_equal(to_np(n4["q_row"][g]), qr)
        assert np.float32(to_np(n4["s_w"])[g]) == np.float32(sw)
    # the NVFP4 dequantize with the maxima of its output
    y = torch.empty((G * O, H), dtype=torch.bfloat16, device=DEV)
    amy = torch.full((G,), -1, dtype=torch.int32, device=DEV)
    mx.mx_dequantize_nvfp4_amax(n4["q_row"], n4["s_row"], n4["s_w"], O, G * O, H, y, amy)
    yref = torch.empty_like(y)
    mx.mx_dequantize_bf16(mx.MX_FMT_NVFP4, n4["q_row"], n4["s_row"], n4["s_w"], mx.MX_SCOPE_GROUP, G * O, H, yref,
                          group_rows=O)
    torch.cuda.synchronize()
    mx.check_device_status()
    assert torch.equal(y.view(torch.int16), yref.view(torch.int16))
    yb = to_np_u16(y).astype(np.uint32)
    assert np.array_equal(to_np(amy).view(np.uint32), ((yb & 0x7FFF).reshape(G, -1).max(axis=1) << 16).astype(np.uint32))


@pytest.mark.parametrize("H", [16, 48, 2064])
def test_dequant_nvfp4_amax_row_widths(mx, H):
    """The dequantize that also returns each matrix's max |y| walks its blocks with a running
    (row, block column) pair: rows of 1, 3 and 129 blocks (fewer, and not a multiple of, the 32 blocks a
    warp steps by) give the same bytes as the plain dequantize, which the oracle pins, and exact maxima."""
    G, O = 3, 128
    w = synthetic.random_bf16(40 + H, (G, O, H), "normal", 0.02)
    w[2, 100, H - 1] = 0xC0C0                                # a spike in the last matrix (-6.0)
    n4 = mx.alloc_nvfp4_weight_2d(G, O, H, DEV)
    mx.mx_nvfp4_quantize_weight_2d(bf16_dev(w), n4["q_row"], n4["s_row"], n4["q_col"], n4["s_col"], n4["s_w"], n4["ws"])
    y = torch.empty((G * O, H), dtype=torch.bfloat16, device=DEV)
    amy = torch.full((G,), -1, dtype=torch.int32, device=DEV)
    mx.mx_dequantize_nvfp4_amax(n4["q_row"], n4["s_row"], n4["s_w"], O, G * O, H, y, amy)
    yref = torch.empty_like(y)
    mx.mx_dequantize_bf16(mx.MX_FMT_NVFP4, n4["q_row"], n4["s_row"], n4["s_w"], mx.MX_SCOPE_GROUP, G * O, H, yref,
                          group_rows=O)
    torch.cuda.synchronize()
    mx.check_device_status()
    assert torch.equal(y.view(torch.int16), yref.view(torch.int16))
    yb = to_np_u16(y).astype(np.uint32)
    assert np.array_equal(to_np(amy).view(np.uint32), ((yb & 0x7FFF).reshape(G, -1).max(axis=1) << 16).astype(np.uint32))


def test_nvfp4_block_scale_ties(mx, orc):
    """Block scales at E4M3 rounding midpoints take the exact path on the device, per token and per tensor."""
    T, H = 96, 256
    x = e4m3_tie_tensor(11, T, H, per_tensor=False)
    out = mx.alloc_nvfp4_rows(T, H, DEV)
    mx.mx_nvfp4_quantize_per_token(bf16_dev(x), out["q"], out["s"], out["s2"])
    q, s, st = orc.nvfp4_quantize_per_token(x)
    assert np.array_equal(to_np(out["q"]), q), first_mismatch(to_np(out["q"]), q)
    assert np.array_equal(to_np(out["s"]), orc.scales_to_gemm_layout(s))
    xt = e4m3_tie_tensor(12, T, H, per_tensor=True)
    qd = torch.empty((T, H // 2), dtype=torch.uint8, device=DEV)
    sd = torch.empty(mx.scale_bytes(T, H, 16), dtype=torch.uint8, device=DEV)
    S = torch.empty(1, dtype=torch.float32, device=DEV)
    ws = torch.empty(16, dtype=torch.uint8, device=DEV)
    mx.mx_nvfp4_quantize_1x16(bf16_dev(xt), False, False, 0, False, 0, qd, sd, S, ws)
    qo, so, So = orc.nvfp4_quantize_1x16(xt, colwise=False)
    assert to_np(S)[0] == So
    assert np.array_equal(to_np(qd), qo), first_mismatch(to_np(qd), qo)
    assert np.array_equal(to_np(sd), orc.scales_to_gemm_layout(so))


def test_nvfp4_per_token_moe_gather_commutes(mx, orc):
    """quantize(gather(X)) == gather(quantize(X)) on the device (per-token scaling)."""
    d = synthetic.moe(tokens=256, hidden=512, ffn=128, experts=16, topk=4, with_weights=False)
    x = d["x"]
    xg = np.ascontiguousarray(x[d["row_token"]])
    out = mx.alloc_nvfp4_rows(xg.shape[0], 512, DEV)
    mx.mx_nvfp4_quantize_per_token(bf16_dev(xg), out["q"], out["s"], out["s2"])
    q, s, st = orc.nvfp4_quantize_per_token(x)
    assert np.array_equal(to_np(out["q"]), q[d["row_token"]])
    assert np.array_equal(to_np(out["s2"]), st[d["row_token"]])


# ------------------------------------------------------------------------------------------------
# NVFP4 per-tensor 1x16 (column-wise with RHT / SR, row-wise)
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("shape", [(256, 512), (48, 40), (1040, 264), (4096, 64)])
@pytest.mark.parametrize("rht,sr", [(False, False), (True, False), (False, True), (True, True)])
def test_nvfp4_colwise(mx, orc, shape, rht, sr):
    T, N = shape
    x = edge_tensor(T * 13 + N + rht * 2 + sr, shape) if not rht else synthetic.random_bf16(T + N, shape, "student_t")
    q = torch.empty((N, T // 2), dtype=torch.uint8, device=DEV)
    s = torch.full((mx.scale_bytes(N, T, 16),), 0x5A, dtype=torch.uint8, device=DEV)
    S = torch.empty(1, dtype=torch.float32, device=DEV)
    ws = torch.empty(16, dtype=torch.uint8, device=DEV)
    mx.mx_nvfp4_quantize_1x16(bf16_dev(x), True, rht, 8, sr, 9, q, s, S, ws)
    qo, so, So = orc.nvfp4_quantize_1x16(x, colwise=True, rht=rht, rht_seed=8, sr=sr, sr_seed=9)
    assert to_np(S).view(np.uint32)[0] == np.float32(So).view(np.uint32)
    assert np.array_equal(to_np(q), qo), first_mismatch(to_np(q), qo)
    assert np.array_equal(to_np(s), orc.scales_to_gemm_layout(so))


@pytest.mark.parametrize("sr", [False, True])
def test_nvfp4_rowwise_per_tensor(mx, orc, sr):
    x = edge_tensor(77, (130, 96))
    q = torch.empty((130, 48), dtype=torch.uint8, device=DEV)
    s = torch.empty(mx.scale_bytes(130, 96, 16), dtype=torch.uint8, device=DEV)
    S = torch.empty(1, dtype=torch.float32, device=DEV)
    ws = torch.empty(16, dtype=torch.uint8, device=DEV)
    mx.mx_nvfp4_quantize_1x16(bf16_dev(x), False, False, 0, sr, 1234, q, s, S, ws)
    qo, so, So = orc.nvfp4_quantize_1x16(x, colwise=False, sr=sr, sr_seed=1234)
    assert to_np(S)[0] == So
    assert np.array_equal(to_np(q), qo), first_mismatch(to_np(q), qo)
    assert np.array_equal(to_np(s), orc.scales_to_gemm_layout(so))


def sr_grid_tensor(T, N, seed):
    """Blocks whose maximum is 6 units and whose other values sweep the E2M1 range densely: exact grid
    points, values just above / below each grid point and each binade edge (0.5, 1, 2, 4), tiny values
    and zeros, random signs -- every branch of the stochastic-rounding decision, under many random bits."""
    rng = np.random.default_rng(seed)
    unit = np.float32(2.0) ** rng.integers(-20, 20, size=(T, N // 16, 1)).astype(np.float32)
    frac = rng.random((T, N // 16, 16)).astype(np.float32) * 6.0
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6], dtype=np.float32)
    pick = rng.integers(0, 8, size=frac.shape)
    near = grid[pick] * (1 + rng.choice([-1, 0, 1], size=frac.shape) * np.float32(2.0 ** -7))
    vals = np.where(rng.random(frac.shape) < 0.4, near, frac)
    vals[..., 1] = rng.random((T, N // 16)) * 1e-3              # tiny values
    vals[..., 2] = 0.0
    vals[..., 0] = 6.0                                          # the block maximum
    vals = vals * unit * rng.choice([-1.0, 1.0], size=frac.shape).astype(np.float32)
    f = vals.reshape(T, N).astype(np.float32)
    return ((f.view(np.uint32) + 0x7FFF + ((f.view(np.uint32) >> 16) & 1)) >> 16).astype(np.uint16)


@pytest.mark.parametrize("colwise", [False, True])
def test_nvfp4_sr_dense_grid(mx, orc, colwise):
    """Stochastic rounding bit-exact against the oracle on values covering every E2M1 interval."""
    T, N = (512, 1024)
    x = sr_grid_tensor(T, N, 5 + colwise)
    if colwise:
        x = np.ascontiguousarray(x.T)                           # blocks of 16 along the rows for column-wise
        T, N = N, T
    q = torch.empty((N, T // 2) if colwise else (T, N // 2), dtype=torch.uint8, device=DEV)
    s = torch.empty(mx.scale_bytes(N, T, 16) if colwise else mx.scale_bytes(T, N, 16), dtype=torch.uint8, device=DEV)
    S = torch.empty(1, dtype=torch.float32, device=DEV)
    ws = torch.empty(16, dtype=torch.uint8, device=DEV)
    mx.mx_nvfp4_quantize_1x16(bf16_dev(x), colwise, False, 0, True, 4321, q, s, S, ws)
    qo, so, So = orc.nvfp4_quantize_1x16(x, colwise=colwise, sr=True, sr_seed=4321)
    assert np.array_equal(to_np(q), qo), first_mismatch(to_np(q), qo)
    assert np.array_equal(to_np(s), orc.scales_to_gemm_layout(so))


@pytest.mark.parametrize("shape", [(64, 48), (256, 1024), (32, 8)])
def test_rht16(mx, orc, shape):
    x = synthetic.random_bf16(sum(shape), shape, "student_t")
    y = torch.empty(shape, dtype=torch.bfloat16, device=DEV)
    mx.mx_rht16(bf16_dev(x), 8, y)
    assert np.array_equal(to_np_u16(y), orc.rht16(x, 8))


# ------------------------------------------------------------------------------------------------
# NVFP4 2D weights
# ------------------------------------------------------------------------------------------------
# (208, 384): full 64 x 128 tiles whose 32-byte transposed-code runs start 8 bytes off a 16-byte boundary
# (O / 2 = 104), plus a 16-row remainder tile; (48, 80) and (16, 16): partial tiles only
@pytest.mark.parametrize("G,O,H", [(3, 48, 80), (2, 256, 512), (1, 1536, 2048), (2, 2048, 768), (1, 16, 16),
                                   (2, 208, 384)])
def test_nvfp4_weight_2d(mx, orc, G, O, H):
    w = synthetic.random_bf16(G * O + H, (G, O, H), "normal", 0.02)
    w[0, 0, :16] = 0x7F7F if O * H < 10000 else w[0, 0, :16]
    out = mx.alloc_nvfp4_weight_2d(G, O, H, DEV)
    out["s_row"].fill_(0x33)
    out["s_col"].fill_(0x44)
    mx.mx_nvfp4_quantize_weight_2d(bf16_dev(w), out["q_row"], out["s_row"], out["q_col"], out["s_col"], out["s_w"],
                                   out["ws"])
    srb = orc.scale_layout_bytes(O, (H // 16))
    scb = orc.scale_layout_bytes(H, (O // 16))
    for g in range(G):
        qr, qc, st, sw = orc.nvfp4_quantize_weight_2d(np.ascontiguousarray(w[g]))
        assert np.array_equal(to_np(out["q_row"][g]), qr), first_mismatch(to_np(out["q_row"][g]), qr)
        assert np.array_equal(to_np(out["q_col"][g]), qc), first_mismatch(to_np(out["q_col"][g]), qc)
        assert np.array_equal(to_np(out["s_row"][g * srb:(g + 1) * srb]),
                              orc.scales_to_gemm_layout(orc.weight_2d_operand_scales(st, "row")))
        assert np.array_equal(to_np(out["s_col"][g * scb:(g + 1) * scb]),
                              orc.scales_to_gemm_layout(orc.weight_2d_operand_scales(st, "col")))
        assert to_np(out["s_w"])[g] == sw


# ------------------------------------------------------------------------------------------------
# Dequantize (fed the oracle's codes, so it is checked independently of the GPU quantizers)
# ------------------------------------------------------------------------------------------------
def output_at(shape, offset_elems):
    """A BF16 output whose first element sits offset_elems past a fresh (256-byte aligned) allocation."""
    n = shape[0] * shape[1]
    return torch.empty(n + 16, dtype=torch.bfloat16, device=DEV)[offset_elems:offset_elems + n].view(shape)


# offset 8 elements: a 16-byte but not 32-byte aligned output, written with two 16-byte stores per
# block instead of one 32-byte store
@pytest.mark.parametrize("offset", [0, 8])
@pytest.mark.parametrize("shape", [(256, 1024), (130, 96)])
def test_dequant_mxfp8(mx, orc, shape, offset):
    R, K = shape
    x = edge_tensor(R + K, shape)
    q, s = orc.mxfp8_quantize_rowwise(x)
    y = output_at(shape, offset)
    mx.mx_dequantize_bf16(mx.MX_FMT_MXFP8, torch.from_numpy(q).to(DEV),
                          torch.from_numpy(orc.scales_to_gemm_layout(s)).to(DEV), None, 0, R, K, y)
    ref = orc.dequant_mxfp8(q, s)
    assert np.array_equal(to_np_u16(y), ref), first_mismatch(to_np_u16(y), ref)


@pytest.mark.parametrize("offset", [0, 8])
@pytest.mark.parametrize("per_row", [True, False])
def test_dequant_nvfp4(mx, orc, per_row, offset):
    x = edge_tensor(99, (200, 320))
    if per_row:
        q, s, s2 = orc.nvfp4_quantize_per_token(x)
    else:
        q, s, s2 = orc.nvfp4_quantize_1x16(x, colwise=False)
        s2 = np.array([s2], dtype=np.float32)
    y = output_at((200, 320), offset)
    mx.mx_dequantize_bf16(mx.MX_FMT_NVFP4, torch.from_numpy(q).to(DEV),
                          torch.from_numpy(orc.scales_to_gemm_layout(s)).to(DEV), torch.from_numpy(s2).to(DEV),
                          mx.MX_SCOPE_ROW if per_row else mx.MX_SCOPE_TENSOR, 200, 320, y)
    ref = orc.dequant_nvfp4(q, s, s2, per_row=per_row)
    assert np.array_equal(to_np_u16(y), ref), first_mismatch(to_np_u16(y), ref)


def test_weight_sync_round_trip_on_device(mx, orc):
    """Q -> DQ -> Q on the device reproduces the bytes (the weight-sync invariant) and the byte
    comparator counts exactly the planted differences."""
    w = synthetic.random_bf16(123, (512, 768), "normal", 0.02)
    wd = bf16_dev(w)
    a = mx.alloc_mxfp8(512, 768, DEV, colwise=False)
    mx.mx_quantize_mxfp8(wd, **a)
    y = torch.empty((512, 768), dtype=torch.bfloat16, device=DEV)
    mx.mx_dequantize_bf16(mx.MX_FMT_MXFP8, a["q_row"], a["s_row"], None, 0, 512, 768, y)
    b = mx.alloc_mxfp8(512, 768, DEV, colwise=False)
    mx.mx_quantize_mxfp8(y, **b)
    cnt = torch.zeros(1, dtype=torch.int64, device=DEV)
    mx.mx_count_mismatch(a["q_row"], b["q_row"], cnt)
    mx.mx_count_mismatch(a["s_row"], b["s_row"], cnt)
    assert int(cnt.item()) == 0
    c = b["q_row"].clone()
    c.view(-1)[torch.tensor([0, 5, 777, 512 * 768 - 1], device=DEV)] ^= 1
    cnt.zero_()
    mx.mx_count_mismatch(a["q_row"], c, cnt)
    assert int(cnt.item()) == 4
    # odd byte counts use the scalar tail
    cnt.zero_()
    mx.mx_count_mismatch(a["q_row"].view(-1)[:1001], c.view(-1)[:1001], cnt)
    assert int(cnt.item()) == 3


def test_count_mismatch_many_vectors_per_thread(mx):
    """The byte comparator over a buffer of several 16-byte vectors per thread and a ragged tail counts
    exactly the planted differences (one to four per touched 16-byte vector)."""
    n = 152 * 6 * 256 * 16 * 9 + 12345
    g = torch.Generator(device="cpu").manual_seed(7)
    a = torch.randint(0, 256, (n,), dtype=torch.uint8, generator=g)
    pos = torch.randperm(n, generator=g)[:5000]
    b = a.clone()
    b[pos] ^= torch.randint(1, 256, (5000,), dtype=torch.uint8, generator=g)
    cnt = torch.zeros(1, dtype=torch.int64, device=DEV)
    mx.mx_count_mismatch(a.to(DEV), b.to(DEV), cnt)
    assert int(cnt.item()) == 5000
    cnt.zero_()
    mx.mx_count_mismatch(a.to(DEV), a.to(DEV), cnt)
    assert int(cnt.item()) == 0


def test_device_status_clean(mx):
    torch.cuda.synchronize()
    mx.check_device_status()


def test_dequant_nvfp4_stacked_2d_weights_group_scope(mx, orc):
    """Per-expert 2D weights stacked as one [G*O, H] operand dequantize in one launch with one FP32
    scale per expert (the dequantized backward's DQ(Q(w)) for all experts)."""
    G, O, H = 3, 256, 96
    w = synthetic.random_bf16(31, (G, O, H), "normal", 0.02)
    out = mx.alloc_nvfp4_weight_2d(G, O, H, DEV)
    mx.mx_nvfp4_quantize_weight_2d(bf16_dev(w), out["q_row"], out["s_row"], out["q_col"], out["s_col"], out["s_w"],
                                   out["ws"])
    y = torch.empty((G * O, H), dtype=torch.bfloat16, device=DEV)
    mx.mx_dequantize_bf16(mx.MX_FMT_NVFP4, out["q_row"], out["s_row"], out["s_w"], mx.MX_SCOPE_GROUP, G * O, H, y,
                          group_rows=O)
    got = to_np_u16(y).reshape(G, O, H)
    for g in range(G):
        qr, qc, st, sw = orc.nvfp4_quantize_weight_2d(np.ascontiguousarray(w[g]))
        ref = orc.dequant_nvfp4(qr, orc.weight_2d_operand_scales(st, "row"), sw, per_row=False)
        assert np.array_equal(got[g], ref), first_mismatch(got[g], ref)


@pytest.mark.parametrize("K", [256, 96])
@pytest.mark.parametrize("sizes", [[0, 130, 7, 300, 128, 1], [512] * 3, [1] * 40])
def test_grouped_quantizers_write_grouped_layout(mx, orc, sizes, K):
    """The *_grouped quantizers give the plain codes and the scales in the grouped layout, padding rows
    between groups and the unused tail zero (K = 256: whole scale words, zeroed by the kernels; K = 96:
    partial words, the layout cleared before the kernel)."""
    G = len(sizes)
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    R = int(offs[-1])
    x = edge_tensor(R + G, (R, K))
    offs_d = torch.from_numpy(offs).to(DEV)
    q = torch.empty((R, K // 2), dtype=torch.uint8, device=DEV)
    s = torch.full((mx.grouped_scale_bytes(R, G, K, 16),), 0x77, dtype=torch.uint8, device=DEV)
    st = torch.empty(R, dtype=torch.float32, device=DEV)
    mx.mx_nvfp4_quantize_per_token_grouped(bf16_dev(x), offs_d, q, s, st)
    qo, so, sto = orc.nvfp4_quantize_per_token(x)
    assert np.array_equal(to_np(q), qo)
    assert np.array_equal(to_np(st), sto)
    assert np.array_equal(to_np(s), orc.scales_to_grouped_layout(so, offs, s.numel()))
    q8 = torch.empty((R, K), dtype=torch.uint8, device=DEV)
    s8 = torch.full((mx.grouped_scale_bytes(R, G, K, 32),), 0x77, dtype=torch.uint8, device=DEV)
    mx.mx_quantize_mxfp8_grouped(bf16_dev(x), offs_d, q8, s8)
    q8o, s8o = orc.mxfp8_quantize_rowwise(x)
    assert np.array_equal(to_np(q8), q8o)
    assert np.array_equal(to_np(s8), orc.scales_to_grouped_layout(s8o, offs, s8.numel()))


# ------------------------------------------------------------------------------------------------
# Four-over-Six NVFP4 (per token, 2D weights)
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("shape", [(256, 512), (37, 48), (130, 2048), (64, 2560)])
def test_nvfp4_per_token_four_over_six(mx, orc, shape):
    T, H = shape
    x = synthetic.random_bf16(T * 7 + H, shape, "student_t")
    x[min(2, T - 1)] = 0                              # a zero token
    out = mx.alloc_nvfp4_rows(T, H, DEV)
    out["s"].fill_(0xEE)
    mx.mx_nvfp4_quantize_per_token_46(bf16_dev(x), out["q"], out["s"], out["s2"])
    q, s, st = orc.nvfp4_quantize_per_token_46(x)
    assert np.array_equal(to_np(out["q"]), q), first_mismatch(to_np(out["q"]), q)
    assert np.array_equal(to_np(out["s"]), orc.scales_to_gemm_layout(s))
    assert np.array_equal(to_np(out["s2"]).view(np.uint32), st.view(np.uint32))
    _, s6, _ = orc.nvfp4_quantize_per_token(x)
    assert (s != s6).any()                            # some blocks took the scale-to-4


@pytest.mark.parametrize("G,O,H", [(3, 96, 160), (2, 256, 512)])
def test_nvfp4_weight_2d_four_over_six(mx, orc, G, O, H):
    w = synthetic.random_bf16(G * O + H + 1, (G, O, H), "normal", 0.02)
    out = mx.alloc_nvfp4_weight_2d(G, O, H, DEV)
    out["s_row"].fill_(0x33)
    out["s_col"].fill_(0x44)
    mx.mx_nvfp4_quantize_weight_2d_46(bf16_dev(w), out["q_row"], out["s_row"], out["q_col"], out["s_col"], out["s_w"],
                                      out["ws"])
    srb = orc.scale_layout_bytes(O, (H // 16))
    scb = orc.scale_layout_bytes(H, (O // 16))
    for g in range(G):
        qr, qc, st, sw = orc.nvfp4_quantize_weight_2d_46(np.ascontiguousarray(w[g]))
        assert np.array_equal(to_np(out["q_row"][g]), qr), first_mismatch(to_np(out["q_row"][g]), qr)
        assert np.array_equal(to_np(out["q_col"][g]), qc), first_mismatch(to_np(out["q_col"][g]), qc)
        assert np.array_equal(to_np(out["s_row"][g * srb:(g + 1) * srb]),
                              orc.scales_to_gemm_layout(orc.weight_2d_operand_scales(st, "row")))
        assert np.array_equal(to_np(out["s_col"][g * scb:(g + 1) * scb]),
                              orc.scales_to_gemm_layout(orc.weight_2d_operand_scales(st, "col")))
        assert to_np(out["s_w"])[g] == sw


# ------------------------------------------------------------------------------------------------
# Non-finite inputs.  The pages quantize finite training values; a block that holds an infinity or a NaN
# gets unspecified codes and scale.  Every other block must be exact as before: the damage stays in the
# blocks (MXFP8), tokens (per-token NVFP4) or matrices (2D NVFP4) that hold the value.
# ------------------------------------------------------------------------------------------------
NONFINITE = (0x7FC0, 0x7F80, 0xFF80)          # BF16 NaN, +Inf, -Inf


def test_mxfp8_non_finite_values_stay_in_their_blocks(mx, orc):
    R, K = 256, 512
    x = synthetic.random_bf16(4040, (R, K), "normal", 1.0)
    spots = [(3, 40), (100, 300), (200, 7)]
    for (r, c), v in zip(spots, NONFINITE):
        x[r, c] = v
    out = mx.alloc_mxfp8(R, K, DEV)
    mx.mx_quantize_mxfp8(bf16_dev(x), **out)
    torch.cuda.synchronize()
    mx.check_device_status()
    qr, sr = orc.mxfp8_quantize_rowwise(x)
    qc, sc = orc.mxfp8_quantize_colwise(x)
    row_ok = np.ones((R, K // 32), dtype=bool)
    col_ok = np.ones((K, R // 32), dtype=bool)
    for r, c in spots:
        row_ok[r, c // 32] = False
        col_ok[c, r // 32] = False
    got_sr = orc.scales_from_gemm_layout(to_np(out["s_row"]), R, K // 32)
    got_sc = orc.scales_from_gemm_layout(to_np(out["s_col"]), K, R // 32)
    assert np.array_equal(got_sr[row_ok], sr[row_ok])
    assert np.array_equal(to_np(out["q_row"]).reshape(R, K // 32, 32)[row_ok], qr.reshape(R, K // 32, 32)[row_ok])
    assert np.array_equal(got_sc[col_ok], sc[col_ok])
    assert np.array_equal(to_np(out["q_col"]).reshape(K, R // 32, 32)[col_ok], qc.reshape(K, R // 32, 32)[col_ok])


def test_nvfp4_per_token_non_finite_values_stay_in_their_tokens(mx, orc):
    T, H = 64, 512
    x = synthetic.random_bf16(4041, (T, H), "student_t")
    rows = [5, 20, 41]
    for r, v in zip(rows, NONFINITE):
        x[r, 100 + r] = v
    out = mx.alloc_nvfp4_rows(T, H, DEV)
    mx.mx_nvfp4_quantize_per_token(bf16_dev(x), out["q"], out["s"], out["s2"])
    torch.cuda.synchronize()
    mx.check_device_status()
    q, s, st = orc.nvfp4_quantize_per_token(x)
    ok = np.setdiff1d(np.arange(T), rows)
    assert np.array_equal(to_np(out["q"])[ok], q[ok])
    assert np.array_equal(orc.scales_from_gemm_layout(to_np(out["s"]), T, H // 16)[ok], s[ok])
    assert np.array_equal(to_np(out["s2"]).view(np.uint32)[ok], st.view(np.uint32)[ok])


def test_nvfp4_weight_2d_non_finite_values_stay_in_their_matrix(mx, orc):
    G, O, H = 3, 64, 128
    w = synthetic.random_bf16(4042, (G, O, H), "normal", 0.02)
    w[1, 10, 20], w[1, 63, 127] = NONFINITE[0], NONFINITE[1]
    out = mx.alloc_nvfp4_weight_2d(G, O, H, DEV)
    mx.mx_nvfp4_quantize_weight_2d(bf16_dev(w), out["q_row"], out["s_row"], out["q_col"], out["s_col"], out["s_w"],
                                   out["ws"])
    torch.cuda.synchronize()
    mx.check_device_status()
    srb, scb = orc.scale_layout_bytes(O, H // 16), orc.scale_layout_bytes(H, O // 16)
    for g in (0, 2):
        qr, qc, st, sw = orc.nvfp4_quantize_weight_2d(np.ascontiguousarray(w[g]))
        assert np.array_equal(to_np(out["q_row"][g]), qr)
        assert np.array_equal(to_np(out["q_col"][g]), qc)
        assert np.array_equal(to_np(out["s_row"][g * srb:(g + 1) * srb]),
                              orc.scales_to_gemm_layout(orc.weight_2d_operand_scales(st, "row")))
        assert np.array_equal(to_np(out["s_col"][g * scb:(g + 1) * scb]),
                              orc.scales_to_gemm_layout(orc.weight_2d_operand_scales(st, "col")))
        assert out["s_w"][g].item() == float(sw)


@pytest.mark.parametrize("v", NONFINITE)
def test_nvfp4_per_tensor_non_finite(mx, orc, v):
    """One scale for the whole tensor (RHT + SR column-wise here).  The tensor maximum skips a NaN, as the
    oracle's does, so only the NaN's own block (its 16 tokens of one column, across which the transform
    spreads it) is unspecified and every other block is exact; an infinity makes the scale infinite on both
    sides.  Either way both passes run to the end with no device error."""
    T, N = 64, 256
    x = synthetic.random_bf16(4043, (T, N), "normal", 1.0)
    x[17, 33] = v
    q = torch.empty((N, T // 2), dtype=torch.uint8, device=DEV)
    s = torch.empty(mx.scale_bytes(N, T, 16), dtype=torch.uint8, device=DEV)
    S = torch.empty(1, dtype=torch.float32, device=DEV)
    ws = torch.empty(16, dtype=torch.uint8, device=DEV)
    mx.mx_nvfp4_quantize_1x16(bf16_dev(x), True, True, 7, True, 8, q, s, S, ws)
    torch.cuda.synchronize()
    mx.check_device_status()
    S_ref = orc.nvfp4_second_scale(orc.nvfp4_1x16_amax(x, rht=True, rht_seed=7))
    assert to_np(S).view(np.uint32)[0] == np.float32(S_ref).view(np.uint32)
    if v == NONFINITE[0]:
        qo, so = orc.nvfp4_1x16_pass2(x, 0, N, S_ref, True, True, 7, True, 8)
        ok = np.ones((N, T // 16), dtype=bool)
        ok[33, 17 // 16] = False
        assert np.array_equal(to_np(q).reshape(N, T // 16, 8)[ok], qo.reshape(N, T // 16, 8)[ok])
        assert np.array_equal(orc.scales_from_gemm_layout(to_np(s), N, T // 16)[ok], so[ok])
    else:
        assert np.isinf(to_np(S)[0])


def test_nvfp4_all_zero_tensors(mx, orc):
    """All-zero inputs put the second-level scale at 0 (S = 0, block scales 0, reciprocals 0): every NVFP4
    quantizer gives the oracle's bytes (all-zero codes and scales, S = 0), and the GEMM and the dequantize
    of those codes give zeros."""
    T, H = 64, 256
    x = np.zeros((T, H), dtype=np.uint16)
    xd = bf16_dev(x)
    out = mx.alloc_nvfp4_rows(T, H, DEV)
    for fn, ref in ((mx.mx_nvfp4_quantize_per_token, orc.nvfp4_quantize_per_token),
                    (mx.mx_nvfp4_quantize_per_token_46, orc.nvfp4_quantize_per_token_46)):
        out["q"].fill_(0xA5)
        out["s"].fill_(0xA5)
        fn(xd, out["q"], out["s"], out["s2"])
        q, s, st = ref(x)
        assert np.array_equal(to_np(out["q"]), q)
        assert np.array_equal(orc.scales_from_gemm_layout(to_np(out["s"]), T, H // 16), s)
        assert np.array_equal(to_np(out["s2"]).view(np.uint32), st.view(np.uint32))
    for colwise in (False, True):
        for rht, sr in ((False, False), (True, False), (False, True), (True, True)):
            if rht and not colwise:
                continue                                  # the transform runs along tokens (column-wise) only
            qd = torch.full((H, T // 2) if colwise else (T, H // 2), 0xA5, dtype=torch.uint8, device=DEV)
            sd = torch.full((mx.scale_bytes(H, T, 16) if colwise else mx.scale_bytes(T, H, 16),), 0xA5,
                            dtype=torch.uint8, device=DEV)
            S = torch.full((1,), -1.0, dtype=torch.float32, device=DEV)
            mx.mx_nvfp4_quantize_1x16(xd, colwise, rht, 5, sr, 6, qd, sd, S,
                                      torch.empty(16, dtype=torch.uint8, device=DEV))
            qo, so, So = orc.nvfp4_quantize_1x16(x, colwise=colwise, rht=rht, rht_seed=5, sr=sr, sr_seed=6)
            assert to_np(S)[0] == np.float32(So) == 0.0
            assert np.array_equal(to_np(qd), qo), (colwise, rht, sr)
            rows, k = (H, T) if colwise else (T, H)
            assert np.array_equal(orc.scales_from_gemm_layout(to_np(sd), rows, k // 16), so), (colwise, rht, sr)
    G, O = 2, 64
    w = np.zeros((G, O, H), dtype=np.uint16)
    wo = mx.alloc_nvfp4_weight_2d(G, O, H, DEV)
    for fn in (mx.mx_nvfp4_quantize_weight_2d, mx.mx_nvfp4_quantize_weight_2d_46):
        for k in ("q_row", "s_row", "q_col", "s_col"):
            wo[k].fill_(0xA5)
        fn(bf16_dev(w), wo["q_row"], wo["s_row"], wo["q_col"], wo["s_col"], wo["s_w"], wo["ws"])
        qr, qc, st, sw = orc.nvfp4_quantize_weight_2d(np.ascontiguousarray(w[0]))
        for g in range(G):
            assert np.array_equal(to_np(wo["q_row"][g]), qr) and np.array_equal(to_np(wo["q_col"][g]), qc)
            assert wo["s_w"][g].item() == float(sw) == 0.0
        assert int(wo["s_row"].sum()) == 0 and int(wo["s_col"].sum()) == 0
    # the codes of zeros through the GEMM (per-token S = 0 on A) and the dequantize
    mx.mx_nvfp4_quantize_per_token(xd, out["q"], out["s"], out["s2"])
    d = torch.full((T, O), float("nan"), dtype=torch.bfloat16, device=DEV)
    mx.mx_scaled_gemm(mx.MX_FMT_NVFP4, out["q"], out["s"], out["s2"], mx.MX_SCOPE_ROW, wo["q_row"][0],
                      wo["s_row"][:mx.scale_bytes(O, H, 16)], wo["s_w"][0:1], mx.MX_SCOPE_TENSOR, T, O, H, d)
    y = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    mx.mx_dequantize_bf16(mx.MX_FMT_NVFP4, out["q"], out["s"], out["s2"], mx.MX_SCOPE_ROW, T, H, y)
    torch.cuda.synchronize()
    mx.check_device_status()
    assert int(torch.count_nonzero(d.float())) == 0 and not torch.isnan(d.float()).any()
    assert int(torch.count_nonzero(y.float())) == 0 and not torch.isnan(y.float()).any()
