"""GB300-native RESOLVE step of a two-level (host pool / GPU hot cache) KV cache.

The compute path is the CUDA library ``libhs.so`` built from ``csrc/`` for
sm_103a and exposed through the C ABI in ``include/hs.h``; :mod:`.hs` is its
thin Python binding.  There is no CPU implementation of the path: importing
the binding works anywhere, but any call fails loudly when the library cannot
be built or no GPU is present.
"""
from . import hs  # noqa: F401
from .hs import HsError, Pool  # noqa: F401
