"""Pins for the oracle's FP4 / E4M3 codec (no GPU).

The codec is checked against hand-worked encodings of the OCP formats, an
exhaustive round trip over every code and every finite positive scale, the
saturation and zero rules, and the byte counts the pages print.
"""

import numpy as np
import pytest

from conftest import read_golden
from oracle import fp4


def test_e2m1_and_e4m3_tables_match_hand_values():
    g = read_golden("fp_formats.txt")
    for code, val in g["e2m1"]:
        v = fp4.e2m1_value(int(code, 16))
        assert v == float(val) and np.signbit(v) == val.startswith("-")
    for byte, val in g["e4m3"]:
        assert fp4.e4m3_value(int(byte, 16)) == float(val)
    assert np.isnan(fp4.e4m3_value(0x7F)) and np.isnan(fp4.e4m3_value(0xFF))


def test_rounding_hand_cases():
    g = read_golden("fp_formats.txt")
    for x, byte in g["e4m3_rne"]:
        assert int(fp4.e4m3_rne(np.float64(np.float32(x)))) == int(byte, 16), x
    for x, code in g["e2m1_rne"]:
        assert int(fp4.e2m1_rne(np.float64(np.float32(x)))) == int(code), x


def test_e4m3_grid_is_the_format():
    # 126 distinct finite positive values, strictly increasing with the code,
    # consecutive ratio at most 1 + 1/8 in the normal range, max 448.
    grid = fp4._E4M3_GRID
    assert grid[0] == 0 and grid[-1] == 448.0 and len(grid) == 127
    assert np.all(np.diff(grid) > 0)
    normal = grid[8:]
    assert np.all(normal[1:] / normal[:-1] <= 1.125 + 1e-15)


def test_exhaustive_round_trip_every_code_every_scale():
    # Block = [6s, code_0*s, ..., code_15*s, 0...]: amax/6 == s exactly, so every
    # representable (code, scale) pair must come back unchanged.
    codes16 = np.arange(16, dtype=np.uint8)
    vals16 = fp4.e2m1_value(codes16)
    n_checked = 0
    for sb in range(1, 0x7F):
        s = float(fp4.e4m3_value(sb))
        block = np.zeros(32, dtype=np.float32)
        block[0] = np.float32(6 * s)
        block[1:17] = (vals16 * s).astype(np.float32)
        packed, scales = fp4.quantize_rows(block[None, :])
        assert int(scales[0, 0]) == sb
        got = fp4.unpack_codes(packed)[0]
        assert got[0] == 7
        np.testing.assert_array_equal(got[1:17], codes16)
        np.testing.assert_array_equal(fp4.dequantize_rows(packed, scales)[0],
                                      block.astype(np.float64))
        n_checked += 1
    assert n_checked == 126


def test_zero_tiny_and_saturating_blocks():
    z = np.zeros((1, 32), np.float32)
    p, s = fp4.quantize_rows(z)
    assert not p.any() and not s.any()
    tiny = np.full((1, 32), 6 * 2.0 ** -10, np.float32)     # amax/6 = 2^-10 -> ties to 0
    p, s = fp4.quantize_rows(tiny)
    assert not p.any() and not s.any()
    big = np.zeros((1, 32), np.float32)
    big[0, 0], big[0, 1] = 1e6, -3000.0
    p, s = fp4.quantize_rows(big)
    assert s[0, 0] == 0x7E
    c = fp4.unpack_codes(p)[0]
    assert c[0] == 0x7 and c[1] == 0xF       # both saturate to +-6
    neg0 = np.zeros((1, 32), np.float32)
    neg0[0, 0], neg0[0, 1] = 3.0, -0.0       # -0 in a live block keeps its sign
    c = fp4.unpack_codes(fp4.quantize_rows(neg0)[0])[0]
    assert c[1] == 0x8 and c[2] == 0x0


def test_nibble_packing_and_midpoints_in_a_block():
    # scale 0.5 (amax 3): u = v / 0.5 hits every E2M1 decision midpoint
    v = np.zeros((1, 32), np.float32)
    v[0, :10] = [3.0, 0.125, 0.375, 0.625, 0.875, 1.25, 1.75, 2.5, -0.125, -1.0]
    p, s = fp4.quantize_rows(v)
    assert fp4.e4m3_value(s[0, 0]) == 0.5
    c = fp4.unpack_codes(p)[0][:10]
    np.testing.assert_array_equal(c, [0x7, 0x0, 0x2, 0x2, 0x4, 0x4, 0x6, 0x6, 0x8, 0xC])
    assert p[0, 0] == (0x7 | (0x0 << 4))


def test_entry_sizes_printed_on_pages():
    # [P3] §六: indexer-K entry 68 B (128 codes + one scale per 32), main entry 288 B
    # (512 codes + one scale per 16 dims); 288 + 68 = 356.
    g = read_golden("layer_pattern.txt")
    p, s = fp4.quantize_rows(np.ones((1, 128), np.float32))
    assert p.nbytes + s.nbytes == int(g["index_entry_bytes"][0][0])
    assert 512 // 2 + 512 // 16 == int(g["main_entry_bytes"][0][0])
    assert int(g["main_entry_bytes"][0][0]) + int(g["index_entry_bytes"][0][0]) == \
        int(g["entry_bytes"][0][0])


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_dequantised_error_bound(seed):
    # |v - v_hat| <= half an E2M1 step times the scale (1 * s above 4, 0.25 * s below 0.5),
    # for unsaturated blocks: a property of nearest rounding on this grid.
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((64, 128)).astype(np.float32)
    p, s = fp4.quantize_rows(v)
    vh = fp4.dequantize_rows(p, s)
    sc = np.repeat(fp4.e4m3_value(s), 32, axis=-1)
    u = np.abs(v / sc)
    half_step = np.where(u > 4, 1.0, np.where(u > 2, 0.5, np.where(u > 0.5, 0.25, 0.25)))
    sat = u > 6
    assert np.all((np.abs(v - vh) <= half_step * sc + 1e-12) | sat)


# ---------------------------------------------------------------- FP4 main KV (16-channel groups)
def test_main_kv_entry_takes_the_pages_288_bytes():
    # [P3] section 六: one main-KV entry is about 288 bytes (512 channels)
    from oracle import csa2_ref as R
    codes, scales = R.main_kv_fp4(np.linspace(-3, 3, 2 * 512).reshape(2, 512))
    assert codes.shape == (2, 256) and scales.shape == (2, 32)
    assert codes.shape[-1] + scales.shape[-1] == 288


def test_main_kv_groups_are_16_channels_and_independent():
    from oracle import csa2_ref as R
    rng = np.random.default_rng(5)
    v = rng.standard_normal(512).astype(np.float32)
    c0, s0 = R.main_kv_fp4(v)
    w = v.copy()
    w[16:32] *= np.float32(8.0)              # only channel group 1 changes
    c1, s1 = R.main_kv_fp4(w)
    assert s1[1] != s0[1]
    np.testing.assert_array_equal(np.delete(s1, 1), np.delete(s0, 1))
    np.testing.assert_array_equal(c1[:8], c0[:8])
    np.testing.assert_array_equal(c1[16:], c0[16:])
    # codes are unchanged by the exact power-of-two rescaling (scale moves by 2^3)
    np.testing.assert_array_equal(c1[8:16], c0[8:16])


def test_main_kv_representable_groups_round_trip_exactly():
    # a group whose values are E2M1 grid points times 2^e, with max magnitude 6 * 2^e,
    # has scale 2^e exactly and decodes to itself
    from oracle import csa2_ref as R
    from oracle import fp4
    rng = np.random.default_rng(6)
    rows = []
    for g in range(32):
        e = int(rng.integers(-6, 7))
        mag = fp4.E2M1_MAG[rng.integers(0, 8, 16)]
        mag[int(rng.integers(0, 16))] = 6.0
        sign = np.where(rng.integers(0, 2, 16) == 1, -1.0, 1.0)
        rows.append(mag * sign * 2.0 ** e)
    v = np.concatenate(rows)
    codes, scales = R.main_kv_fp4(v)
    np.testing.assert_array_equal(R.main_kv_dequant(codes, scales), v)


def test_main_kv_error_within_half_the_grid_gap_times_the_scale():
    from oracle import csa2_ref as R
    from oracle import fp4
    rng = np.random.default_rng(7)
    v = (rng.standard_normal((50, 512)) * np.exp(rng.standard_normal((50, 512)))).astype(np.float32)
    codes, scales = R.main_kv_fp4(v)
    d = R.main_kv_dequant(codes, scales).reshape(50, 32, 16)
    s = fp4.e4m3_value(scales)[..., None]
    amax = np.abs(v.reshape(50, 32, 16)).max(-1, keepdims=True)
    # E2M1 gaps are at most 2 (between 4 and 6); the scale's own rounding adds at most
    # 1/16 relative, and values above 6 s saturate by at most amax - 6 s
    bound = 1.0 * s + np.maximum(amax - 6 * s, 0.0) + 1e-12
    assert np.all(np.abs(d - v.reshape(50, 32, 16)) <= bound)
