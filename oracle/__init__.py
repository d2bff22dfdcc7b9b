"""Float64 CPU oracle for exact attention (test infrastructure only).

``oracle.fp8`` states the e4m3 block quantiser of the low-precision forward in
numpy; the attention on quantised inputs is the same oracle applied to their
dequantised values.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  The CUDA library neither imports nor links it.
"""
from .oracle import Oracle, bwd, bwd_rows, default, default_threads, fwd, fwd_rows  # noqa: F401
