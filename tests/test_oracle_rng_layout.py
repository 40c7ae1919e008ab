"""Pins for the oracle's counter-based RNG, RHT signs and GEMM scale layout."""
import numpy as np

from conftest import read_golden


def test_philox_known_answers(orc):
    for row in read_golden("philox4x32_10_kat.txt"):
        vals = [int(v, 16) for v in row]
        ctr, key, out = vals[0:4], vals[4:6], vals[6:10]
        assert orc.philox4x32_10(ctr, key) == tuple(out)


def test_sr_bits_layout(orc):
    """Element i uses word (i>>1)&3 of the block i>>3, low half for even i."""
    seed = 0x1234_5678_9ABC_DEF0
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for blk in [0, 1, 12345, (1 << 33) + 7]:
        words = orc.philox4x32_10([blk & 0xFFFFFFFF, blk >> 32, 0, 0], key)
        for j in range(8):
            i = blk * 8 + j
            w = words[(i >> 1) & 3]
            assert orc.sr_bits16(seed, i) == ((w >> 16) if (i & 1) else (w & 0xFFFF))


def test_sr_bits_roughly_uniform(orc):
    bits = np.array([orc.sr_bits16(9, i) for i in range(20000)])
    assert 0 <= bits.min() and bits.max() < 65536
    hist = np.bincount(bits >> 12, minlength=16)
    expected = len(bits) / 16
    chi2 = float(((hist - expected) ** 2 / expected).sum())
    assert chi2 < 50.0            # 15 dof; p ~ 1e-5 threshold
    assert len(set(bits.tolist())) > 0.7 * len(bits)


def test_rht_signs_are_from_seeded_stream(orc):
    s8 = orc.rht16_signs(8)
    w = orc.philox4x32_10([0, 0, 1, 0], [8, 0])[0]
    assert [(-1 if (w >> j) & 1 else 1) for j in range(16)] == s8.tolist()
    assert set(s8.tolist()) <= {-1, 1}
    assert not np.array_equal(orc.rht16_signs(8), orc.rht16_signs(9))


def test_scale_layout_offsets_golden(orc):
    lib = orc._load()
    for r, c, scols, off in read_golden("scale_layout_offsets.txt"):
        assert lib.orc_scale_layout_offset(int(r), int(c), int(scols)) == int(off)


def test_scale_layout_round_trip_and_padding(orc):
    rng = np.random.default_rng(1)
    for rows, scols in [(1, 1), (128, 4), (130, 9), (300, 64), (256, 2)]:
        comp = rng.integers(1, 255, size=(rows, scols), dtype=np.uint8)
        laid = orc.scales_to_gemm_layout(comp)
        assert laid.size == ((rows + 127) // 128) * ((scols + 3) // 4) * 512
        np.testing.assert_array_equal(orc.scales_from_gemm_layout(laid, rows, scols), comp)
        # every real scale lands on a distinct byte; the rest is zero padding
        assert int((laid != 0).sum()) == rows * scols


def test_grouped_layout_places_each_group_on_a_tile(orc):
    """Groups of 3, 0, 130 and 1 rows: padded starts 0, 128, 128, 384 (the empty group takes no
    tile); within a group the plain layout applies from the group's first tile."""
    sizes = [3, 0, 130, 1]
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    rows, scols = int(off[-1]), 8
    comp = (np.arange(rows * scols, dtype=np.int64) % 251 + 1).astype(np.uint8).reshape(rows, scols)
    assert orc.grouped_padded_rows(off) == 128 + 256 + 128
    laid = orc.scales_to_grouped_layout(comp, off)
    plain = orc.scales_from_gemm_layout(laid, 512, scols)
    np.testing.assert_array_equal(plain[0:3], comp[0:3])
    assert not plain[3:128].any()
    np.testing.assert_array_equal(plain[128:258], comp[3:133])
    assert not plain[258:384].any()
    np.testing.assert_array_equal(plain[384], comp[133])
    assert int((laid != 0).sum()) == rows * scols
