"""libexpzip: lossless BF16 exponent codecs (ZipCCL 3-bit exponent code and
CIERA cross-iteration exponent reuse) as hand-written CUDA kernels for sm_103a
behind a C ABI (include/expzip.h).

``binding`` is the ctypes marshalling of that ABI, ``codec.Codec`` allocates
the caller-owned buffers of one plan with torch, ``build`` compiles the
library in-tree, ``breakeven`` is the host-side break-even model.
"""
from . import binding, breakeven  # noqa: F401

__all__ = ["binding", "breakeven", "codec", "build"]
