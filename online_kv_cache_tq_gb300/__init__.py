"""GB300-native TurboQuant KV-cache engine.

The compute path is the C-ABI library ``_lib/libtq.so`` (hand-written CUDA for
sm_103a, sources in ``csrc/``, ABI in ``include/tq.h``).  ``binding`` wraps its
entry points under the same names; ``cache`` allocates the paged cache fields
and the decode workspace as torch device tensors (memory only).  Importing the
package does not load the library; the first binding call does, and raises if
the library has not been built.
"""
from . import binding  # noqa: F401
