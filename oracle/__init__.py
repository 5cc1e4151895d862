"""fp64 CPU oracle for the causal-convolution stack (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use this package. The CUDA path never imports it.
"""

from .reference import *  # noqa: F401,F403
from .reference import __all__  # noqa: F401
