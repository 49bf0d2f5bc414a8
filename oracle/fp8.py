"""FP8 (E4M3) sliding-window KV rows with one power-of-two scale per 64 channels -- oracle side.

Test infrastructure: imported only by the tests, the smoke check and the CPU baseline.

[P3] section 七 "FP4 Main KV": the window (SWA) KV reacts more to quantisation than the main KV
and is kept in FP8.  The pages give no more; READINGS, each the plainest one:
  * elements are OCP E4M3 ("FN": bias 7, largest finite 448), nearest-even;
  * one scale per group of 64 channels (8 per 512-channel row; the last group is exactly the
    64 RoPE dims), a power of two 2^k stored as the byte k + 127;
  * k is the smallest integer >= -126 with amax <= 448 * 2^k, so no element saturates and a
    dequantised value (E4M3 value times 2^k, 4 significant bits) is exact in bf16 wherever
    bf16 is normal;
  * u = v / 2^k (exact); code = signbit(u) << 7 | E4M3_RNE(|u|) (so -0 gives 0x80).
A row is 512 code bytes plus 8 scale bytes (520 B against 1024 B in bf16).
"""

import numpy as np

from . import fp4

GROUP = 64
K_MIN = -126


def scale_exponent(amax):
    """Smallest integer k >= -126 with amax <= 448 * 2^k (amax >= 0, float64 exact)."""
    amax = np.asarray(amax, dtype=np.float64)
    f, e = np.frexp(amax)            # amax = f * 2^e, f in [0.5, 1) (0 for amax = 0)
    # 448 = 0.875 * 2^9: f * 2^e <= 0.875 * 2^(k + 9)  <=>  k >= e - 9 + [f > 0.875]
    k = e.astype(np.int64) - 9 + (f > 0.875).astype(np.int64)
    k = np.where(amax == 0, K_MIN, k)
    return np.maximum(k, K_MIN)


def quantize_rows(v):
    """bf16-valued rows v[..., D] (D a multiple of 64) -> (codes uint8 [..., D],
    scales uint8 [..., D/64])."""
    v = np.asarray(v, dtype=np.float64)
    d = v.shape[-1]
    assert d % GROUP == 0
    g = v.reshape(v.shape[:-1] + (d // GROUP, GROUP))
    k = scale_exponent(np.max(np.abs(g), axis=-1))
    u = g * np.power(2.0, -k.astype(np.float64))[..., None]       # exact: a power of two
    mag = fp4.e4m3_rne(np.abs(u))
    sign = np.signbit(u).astype(np.uint8) << 7
    codes = (mag | sign).astype(np.uint8).reshape(v.shape)
    return codes, (k + 127).astype(np.uint8)


def dequantize_rows(codes, scales):
    """codes/scales -> float64 values (E4M3 value times the group's 2^k, exact)."""
    vals = fp4.e4m3_value(np.asarray(codes, dtype=np.uint8))
    d = vals.shape[-1]
    s = np.power(2.0, np.asarray(scales, dtype=np.int64) - 127)
    g = vals.reshape(vals.shape[:-1] + (d // GROUP, GROUP)) * s[..., None]
    return g.reshape(vals.shape)
