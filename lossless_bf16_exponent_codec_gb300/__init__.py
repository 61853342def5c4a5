"""libexpzip: lossless BF16 exponent codecs (ZipCCL 3-bit exponent code and
CIERA cross-iteration exponent reuse) as hand-written CUDA kernels for sm_103a
behind a C ABI (include/expzip.h).

``binding`` is the ctypes marshalling of that ABI, ``codec.Codec`` allocates
the caller-owned buffers of one plan with torch, ``build`` compiles the
library in-tree, ``breakeven`` is the host-side break-even model and ``bsc``
the benefit-driven choice of the shards to send with exponent reuse.
"""
from . import binding, breakeven, bsc  # noqa: F401

__all__ = ["binding", "breakeven", "bsc", "codec", "build"]
