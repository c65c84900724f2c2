"""Float64 CPU oracle for exact softmax attention (forward and backward).

TEST INFRASTRUCTURE ONLY: imported by the test suite, by the smoke check in
``__graft_entry__`` and by the CPU-baseline leg of ``bench.py``, never by the
library.  It shares no code with the CUDA path and imports nothing from it.

Every function is pinned by tests/test_oracle.py (no function here is
"parity unpinned").
"""

from . import fp8  # noqa: F401
from .attention import (  # noqa: F401
    attention_backward,
    attention_backward_head,
    attention_backward_head_sampled,
    attention_forward,
    attention_forward_head,
    default_scale,
)
