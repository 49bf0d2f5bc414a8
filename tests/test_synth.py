"""The seeded input generator (host side): known-answer vectors and value mapping."""

import numpy as np

from conftest import read_golden
import synth


def test_philox_known_answers():
    for row in read_golden("philox_kat.txt")["kat"]:
        c = [int(v, 16) for v in row[:4]]
        k = [int(v, 16) for v in row[4:6]]
        exp = [int(v, 16) for v in row[7:11]]
        out = synth.philox4x32_10(*[np.array([v]) for v in c], *k)
        assert [int(o[0]) for o in out] == exp


def test_normal_mapping_moments_and_chunking():
    z = synth.normal_f32(7, 3, 0, 200_000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    assert np.abs(z).max() < 3.4642            # Irwin-Hall(4) support: |z| < sqrt(12)
    # element i does not depend on where a chunk starts
    np.testing.assert_array_equal(synth.normal_f32(7, 3, 1000, 50), z[1000:1050])
    b = synth.normal_bf16_bits(7, 3, 0, 1000, sigma=0.02)
    f = synth.bf16_bits_to_f32(b)
    ref = synth.normal_f32(7, 3, 0, 1000, sigma=0.02)
    assert np.all(np.abs(f - ref) <= np.abs(ref) * 2.0 ** -8)
    assert not np.array_equal(synth.uniform_u32(7, 3, 0, 8), synth.uniform_u32(7, 4, 0, 8))
