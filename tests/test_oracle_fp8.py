"""Pins for the oracle's FP8 window-KV codec (no GPU): E4M3 elements with one power-of-two
scale per 64 channels.

The scale rule is checked against a brute-force search, the element codes against
hand-worked encodings of the OCP E4M3 format, the round trip against values built on the
grid, and the rounding error against the format's half-ulp bound.
"""

import numpy as np

import synth
from oracle import csa2_ref as R
from oracle import fp4, fp8


def _brute_k(amax):
    for k in range(-126, 300):
        if amax <= 448.0 * 2.0 ** k:
            return k
    raise AssertionError


def test_scale_exponent_is_the_smallest_power_that_fits():
    rng = np.random.default_rng(5)
    vals = list(np.float64(np.float32(rng.lognormal(0, 12, 4000))))
    for k in (-126, -20, -9, -8, 0, 3, 40):
        t = 448.0 * 2.0 ** k
        vals += [t, np.nextafter(t, 0), np.nextafter(t, np.inf), 0.875 * 2.0 ** k, 2.0 ** k]
    vals += [0.0, 2.0 ** -149, 2.0 ** -130, 1e-38]
    got = fp8.scale_exponent(np.array(vals))
    for a, k in zip(vals, got):
        assert k == _brute_k(a), a


def test_hand_encoded_group():
    # one 64-channel group with amax 1: k = -8 (448 / 256 = 1.75 >= 1 > 0.875), byte 119;
    # u = 256 v: 1 -> 2^8 = E4M3 0x78 (exponent field 15); -0.5 -> 2^7 -> 0xF0; 0.3 -> 76.8,
    # between 72 and 80 on the step-8 grid of 64..128, nearer 80 (exponent field 13, mantissa
    # 2: 0x6A); 2^-20 -> 2^-12, below half the smallest subnormal 2^-9: code 0; -0.0 -> 0x80.
    v = np.zeros(64)
    v[:5] = [1.0, -0.5, 0.3, 2.0 ** -20, -0.0]
    codes, scales = fp8.quantize_rows(v)
    assert scales.tolist() == [119]
    assert codes[:5].tolist() == [0x78, 0xF0, 0x6A, 0x00, 0x80]
    assert np.all(codes[5:] == 0)
    d = fp8.dequantize_rows(codes, scales)
    assert d[:3].tolist() == [1.0, -0.5, 80.0 / 256.0]


def test_round_trip_exact_on_the_grid():
    rng = np.random.default_rng(7)
    grid = fp4._E4M3_GRID
    for _ in range(50):
        k = int(rng.integers(-126, 100))
        c = rng.integers(0, 127, 64)
        c[rng.integers(0, 64)] = rng.integers(0x70, 0x7F)    # a value in (224, 448]: scale is 2^k
        sgn = np.where(rng.random(64) < 0.5, -1.0, 1.0)
        v = sgn * grid[c] * 2.0 ** k
        codes, scales = fp8.quantize_rows(v)
        assert int(scales[0]) == k + 127
        np.testing.assert_array_equal(fp8.dequantize_rows(codes, scales), v)


def test_error_bound_and_no_saturation():
    v = synth.normal_f32(3, 1, 0, 64 * 512).astype(np.float64).reshape(64, 512)
    v = v * np.exp2(np.repeat(np.arange(-6, 2), 64))          # groups over a range of sizes
    v = R.bf16_to_f64(R.f64_to_bf16_bits(v))
    codes, scales = R.swa_kv_fp8(v)
    assert codes.shape == (64, 512) and scales.shape == (64, 8)
    assert codes.shape[-1] + scales.shape[-1] == 520            # bytes per row
    d = R.swa_kv_dequant(codes, scales)
    s = np.repeat(np.exp2(scales.astype(np.float64) - 127), 64, axis=-1)
    err = np.abs(d - v)
    assert np.all(err <= np.maximum(np.abs(v) * 2.0 ** -4, 2.0 ** -10 * s))
    u = np.abs(v) / s
    gmax = u.reshape(64, 8, 64).max(axis=-1)
    assert np.all((gmax > 224) & (gmax <= 448))


def test_groups_are_independent():
    v = synth.normal_f32(4, 1, 0, 512).astype(np.float64)
    c0, s0 = fp8.quantize_rows(v)
    w = v.copy()
    w[3 * 64 + 5] = 1000.0
    c1, s1 = fp8.quantize_rows(w)
    changed = np.nonzero((c0 != c1).reshape(8, 64).any(axis=1) | (s0 != s1))[0].tolist()
    assert changed == [3]
