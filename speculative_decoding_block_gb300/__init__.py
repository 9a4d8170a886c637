"""GB300 (sm_103a) greedy block-verify step of block speculative decoding.

The work runs in libvsd.so (C ABI in include/vsd.h); `binding` mirrors its
entry points for torch tensors and `target` builds the model object from
BF16 master weights.  Importing the package does not need a GPU; calling
into the library needs the built shared library and a CUDA device.
"""
from . import binding  # noqa: F401
from .binding import VsdError, lib  # noqa: F401
