"""Exact softmax attention (forward and backward) for NVIDIA GB300 (sm_103a).

The computation lives in ``libattn.so`` (C ABI: include/attn.h), built
in-tree from ``csrc/`` by ``__graft_entry__.build()``.  ``attn`` is its
ctypes binding; ``inputs`` draws the seeded synthetic workloads; ``flops``
counts the algorithmic work used for throughput reports.
"""

from . import flops, inputs  # noqa: F401

__version__ = "0.1.0"

