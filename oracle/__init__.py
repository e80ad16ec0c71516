"""CPU oracle for Hadamard-rotated, block-quantized KV-cache attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and
its Python binding) may import, call or link this package.  Only the tests,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` use it.  It shares no code, tables or helpers with the
CUDA path.

Parity status of each function is listed in the module ``kvq_oracle``.
"""

from .kvq_oracle import *  # noqa: F401,F403
