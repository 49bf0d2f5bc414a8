"""FP4 (E2M1) codes with one E4M3 scale per block of values -- oracle side.

Storage format of the indexer keys: [P1] section "indexer K 改由 main KV 投影"
(FP4, one scale per 32 dims) and [P3] section 六 "890 B/Token 是怎样算出来的"
(68 bytes per indexer-K entry: 128 four-bit codes = 64 B plus 4 one-byte scales).
The main KV entries use the same element formats with 16-value blocks: [P3] section 六
(288 bytes per main-KV entry) and section 七 "FP4 Main KV" (E2M1 data, channel groups
sharing an E4M3 scale).  READING: 288 = 256 B of codes + 32 one-byte scales, i.e. groups
of 16 of the 512 channels.

Element formats follow the OCP 8-bit floating point spec (E4M3, "FN" variant:
bias 7, no infinities, S.1111.111 is NaN, largest finite 448) and the OCP
Microscaling spec (E2M1: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6).

Rounding readings (the pages state none):
  * scale  s = E4M3_RNE(float32(amax) / 6)  (IEEE float32 divide, then nearest-
    even over the E4M3 grid, saturating at 448; subnormals kept);
  * a block whose scale rounds to 0 stores code 0 for every element;
  * element u = float32(v) / s (IEEE float32 divide) -> nearest-even E2M1,
    saturating at +-6; the sign bit is the sign bit of u (so -0 gives 0x8);
  * element 2i of a row sits in the low nibble of byte i.

Rounding is written as "nearest value of the finite grid, ties to the even
code" over an explicit table of representable values, independently of any
bit-twiddling conversion.
"""

import numpy as np

E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
BLOCK = 32
E4M3_MAX = 448.0


def e4m3_value(b):
    """Decode E4M3 byte(s) to float64 (NaN for the NaN codes)."""
    b = np.asarray(b, dtype=np.int64)
    s = np.where((b >> 7) & 1, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 7
    sub = m * 2.0 ** -9
    nrm = (1.0 + m / 8.0) * np.power(2.0, e - 7)
    v = np.where(e == 0, sub, nrm) * s
    return np.where((e == 15) & (m == 7), np.nan, v)


# positive finite grid: codes 0x00..0x7E, ascending in both code and value
_E4M3_CODES = np.arange(0x7F, dtype=np.int64)
_E4M3_GRID = e4m3_value(_E4M3_CODES)


def _nearest_even(x, grid, codes):
    """Nearest grid point to x >= 0 (grid ascending); ties -> even code.

    Values above the last grid point saturate to it.
    """
    x = np.asarray(x, dtype=np.float64)
    hi = np.clip(np.searchsorted(grid, x, side="left"), 0, len(grid) - 1)
    lo = np.clip(hi - 1, 0, len(grid) - 1)
    dlo = np.abs(x - grid[lo])
    dhi = np.abs(grid[hi] - x)
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (codes[hi] % 2 == 0))
    out = np.where(pick_hi, codes[hi], codes[lo])
    return np.where(x >= grid[-1], codes[-1], out)


def e4m3_rne(x):
    """float32 magnitude(s) >= 0 -> E4M3 code byte, nearest-even, satfinite."""
    return _nearest_even(x, _E4M3_GRID, _E4M3_CODES).astype(np.uint8)


def e2m1_rne(x):
    """magnitude(s) >= 0 -> 3-bit E2M1 magnitude code, nearest-even, satfinite 6."""
    return _nearest_even(x, E2M1_MAG, np.arange(8, dtype=np.int64)).astype(np.uint8)


def e2m1_value(code):
    code = np.asarray(code, dtype=np.int64)
    return np.where(code & 8, -1.0, 1.0) * E2M1_MAG[code & 7]


def quantize_rows(v, block=BLOCK):
    """Quantise float32 rows v[..., D] (D a multiple of `block`).

    Returns (codes uint8 [..., D/2], scales uint8 [..., D/block]).
    """
    v = np.asarray(v, dtype=np.float32)
    d = v.shape[-1]
    assert d % block == 0
    blocks = v.reshape(v.shape[:-1] + (d // block, block))
    amax = np.max(np.abs(blocks), axis=-1)                       # float32, exact
    s_f32 = amax / np.float32(6.0)                               # IEEE float32 divide
    sb = e4m3_rne(s_f32.astype(np.float64))
    s = e4m3_value(sb).astype(np.float32)                        # exact in float32
    safe = np.where(s == 0, np.float32(1.0), s).astype(np.float32)
    u = blocks / safe[..., None]                                 # IEEE float32 divide
    mag = e2m1_rne(np.abs(u).astype(np.float64))
    sign = np.signbit(u).astype(np.uint8) << 3
    code = (mag | sign).astype(np.uint8)
    code = np.where((s == 0)[..., None], np.uint8(0), code)
    code = code.reshape(v.shape[:-1] + (d,))
    packed = (code[..., 0::2] | (code[..., 1::2] << 4)).astype(np.uint8)
    return packed, sb.astype(np.uint8)


def unpack_codes(packed):
    packed = np.asarray(packed, dtype=np.uint8)
    lo = packed & 0xF
    hi = packed >> 4
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def dequantize_rows(packed, scales):
    """codes/scales -> float64 values (code value times block scale, exact); the block
    size is the row length over the number of scales."""
    codes = unpack_codes(packed)
    vals = e2m1_value(codes)
    d = vals.shape[-1]
    s = e4m3_value(scales)
    block = d // s.shape[-1]
    return (vals.reshape(vals.shape[:-1] + (d // block, block)) * s[..., None]).reshape(vals.shape)
