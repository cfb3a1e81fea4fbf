"""CPU float64 oracle for fused attention: test infrastructure only.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. It shares no code with the CUDA library.
"""
from . import kvcache  # noqa: F401
from .attention import (  # noqa: F401
    backward,
    backward_dq_rows,
    forward,
    forward_rows,
    probabilities,
    valid_length,
)
