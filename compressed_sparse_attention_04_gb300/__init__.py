"""CSA2 global-attention hot path (DeepSeek-V4.1-Flash) for one GB300 (sm_103a).

The compute lives in ``libcsa2.so`` (hand-written CUDA kernels behind the C ABI of
``include/csa2.h``); ``ops`` marshals torch tensors into those calls.  There is no
CPU fallback: importing ``ops`` works without a GPU, calling it needs the library
and a CUDA device.
"""

from . import _lib  # noqa: F401
from . import ops  # noqa: F401

__all__ = ["ops"]
