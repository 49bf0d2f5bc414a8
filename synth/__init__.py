"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds no arithmetic of the attention method: only a counter-based
random number generator and the mapping of its words to the input values.  It
has two implementations that produce identical bits:

* ``synth.philox``  -- NumPy, used on the host (oracle side, small inputs);
* ``synth.gpu``     -- a CUDA kernel in ``libcsa2_synth.so`` for inputs too large
                      to make on the host (caches of 1M-token contexts).

Generator: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers:
as easy as 1, 2, 3", SC 2011).  Element ``i`` of stream ``stream`` under ``seed``
uses counter (i mod 2^32, i div 2^32, 0, 0) and key (seed, stream).

Normal values use the Irwin-Hall sum of the four 32-bit words (each reduced to
a 22-bit uniform with a half-step offset), centred and scaled to unit variance.
The sum is an integer below 2^24 in magnitude, so its conversion to float32 is
exact and the only rounding is one float32 multiply by sqrt(3)/2^23, one by
sigma, and (for bf16 tensors) one round-to-nearest-even to bfloat16: the same
IEEE operations on host and device, hence bit-identical results.
"""

from .philox import (  # noqa: F401
    philox4x32_10,
    normal_f32,
    normal_bf16_bits,
    uniform_u32,
    bf16_bits_to_f32,
    f32_to_bf16_bits,
)
