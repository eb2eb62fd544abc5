"""Plain fp64 CPU oracle for FAVOR+: projections, forward passes and their gradients (test infrastructure only).

This package is the oracle the CUDA library is tested against.  It is imported
only by the tests, by ``__graft_entry__.smoke()`` and by ``bench.py``'s CPU
baseline / reference arm.  The product path (``linear_softmax_attention_gb300``)
never imports it, and it never imports the product path.
"""

from .favor import *  # noqa: F401,F403
