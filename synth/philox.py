"""NumPy implementation of the seeded input generator (see package docstring)."""

import numpy as np

_M0 = np.uint64(0xD2511F53)
_M1 = np.uint64(0xCD9E8D57)
_W0 = 0x9E3779B9
_W1 = 0xBB67AE85
_MASK = np.uint64(0xFFFFFFFF)
_SHIFT = np.uint64(32)

# sqrt(3) / 2^23 rounded once to float32: scales the centred Irwin-Hall integer
# (variance 2^46 / 3) to unit variance.
IH_SCALE = np.float32(np.sqrt(3.0) / float(1 << 23))


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Philox4x32 with 10 rounds.

    c0..c3: uint32-valued integer arrays (any integer dtype), k0, k1: ints.
    Each round multiplies words 0 and 2 by the two Philox constants, swaps the
    high/low halves into new positions and mixes in the key; the key is bumped
    by the two Weyl constants between rounds.  Returns four uint32 arrays.
    """
    c0 = np.asarray(c0, dtype=np.uint64) & _MASK
    c1 = np.asarray(c1, dtype=np.uint64) & _MASK
    c2 = np.asarray(c2, dtype=np.uint64) & _MASK
    c3 = np.asarray(c3, dtype=np.uint64) & _MASK
    k0 = int(k0) & 0xFFFFFFFF
    k1 = int(k1) & 0xFFFFFFFF
    for _ in range(10):
        p0 = _M0 * c0
        p1 = _M1 * c2
        hi0, lo0 = p0 >> _SHIFT, p0 & _MASK
        hi1, lo1 = p1 >> _SHIFT, p1 & _MASK
        c0, c1, c2, c3 = (hi1 ^ c1 ^ np.uint64(k0), lo1,
                          hi0 ^ c3 ^ np.uint64(k1), lo0)
        k0 = (k0 + _W0) & 0xFFFFFFFF
        k1 = (k1 + _W1) & 0xFFFFFFFF
    return (c0.astype(np.uint32), c1.astype(np.uint32),
            c2.astype(np.uint32), c3.astype(np.uint32))


def _words(seed, stream, start, n):
    idx = np.arange(int(start), int(start) + int(n), dtype=np.uint64)
    lo = idx & _MASK
    hi = idx >> _SHIFT
    z = np.zeros_like(lo)
    return philox4x32_10(lo, hi, z, z, seed, stream)


def uniform_u32(seed, stream, start, n):
    """First Philox word of each element: n uint32 values."""
    return _words(seed, stream, start, n)[0]


def normal_f32(seed, stream, start, n, sigma=1.0):
    """n float32 values, approximately N(0, sigma^2) (Irwin-Hall of 4)."""
    r = _words(seed, stream, start, n)
    acc = np.zeros(int(n), dtype=np.int64)
    for w in r:
        acc += 2 * (w.astype(np.int64) >> 10) + 1
    acc -= 1 << 24
    z = acc.astype(np.float32) * IH_SCALE
    return (z * np.float32(sigma)).astype(np.float32)


def f32_to_bf16_bits(x):
    """Round float32 to bfloat16 bits, nearest-even (finite inputs)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return b.astype(np.uint16)


def bf16_bits_to_f32(b):
    """Exact widening of bfloat16 bits to float32."""
    b = np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def normal_bf16_bits(seed, stream, start, n, sigma=1.0):
    """n bfloat16 values (as uint16 bits): normal_f32 rounded nearest-even."""
    return f32_to_bf16_bits(normal_f32(seed, stream, start, n, sigma))
