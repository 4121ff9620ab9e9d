"""Layerwise weight-streaming DiT forward for one GB300 (sm_103a).

Python binding of the C ABI declared in ``include/dlo.h``: the same function
names, argument marshalling only.  Every step of the forward runs in the CUDA
library ``_lib/libdlo.so``; there is no Python or CPU fallback - if the
library has not been built, every call raises ``DloLibraryMissing``.

Pointers may be given as ints, torch tensors (``data_ptr()``) or numpy arrays;
streams as ints, ``torch.cuda.Stream`` objects or None (legacy default stream).
"""
from __future__ import annotations

from ._binding import *  # noqa: F401,F403
from ._binding import __all__  # noqa: F401
