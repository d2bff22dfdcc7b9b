"""Float64 CPU oracle for exact attention (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  The CUDA library neither imports nor links it.
"""
from .oracle import Oracle, bwd, bwd_rows, default, default_threads, fwd, fwd_rows  # noqa: F401
