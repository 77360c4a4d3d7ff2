"""CPU oracle for the routed-MoE layer hot path (fp64, numpy).

TEST INFRASTRUCTURE ONLY. This package is the independent reference the CUDA
path is checked against. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import it. It shares no code with the CUDA
path: the two meet only through the seeded inputs of the ``inputs`` module.
"""
from . import formats, moe, backward  # noqa: F401
