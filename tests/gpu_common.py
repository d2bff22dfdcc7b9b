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


# Unit roundoff of bf16 (8 significant bits) and of fp32 (24).
U_BF16 = 2.0 ** -8
U_FP32 = 2.0 ** -24


def grad_bounds(q, k, v, do, causal, scale, sigmas=6.0):
    """Per-element bounds on the kernel's dQ, dK, dV errors against the exact
    gradients, float64 (q, k, v, do float64 [BH, N, d]), from where the kernel rounds.
    Each round-to-nearest to bf16 multiplies a value by (1 + e), e within +-u
    (u = 2^-8), taken as independent errors of variance u^2 / 3:

      O    the forward rounds P to bf16 for its P V product, then O to bf16:
           var dO_ic = u^2/3 (O_ic^2 + sum_j P_ij^2 V_jc^2)   (P normalised)
      D_i  = sum_c dO_ic O_ic from that O: var dD_i = sum_c dO_ic^2 var dO_ic
      dS   = P o (dP - D) in fp32 from fp32 P, rounded to bf16 for dK and dQ:
           d dS_ij = -P_ij dD_i + e_ij dS_ij
      dQ   = scale dS K:   var = scale^2 ((P K)_ic^2 var dD_i + u^2/3 sum_j dS_ij^2 K_jc^2)
      dK   = scale dS^T Q: var = scale^2 sum_i (P_ij^2 Q_ic^2 var dD_i + u^2/3 dS_ij^2 Q_ic^2)
      dV   = P^T dO, P rounded to bf16: var = u^2/3 sum_i P_ij^2 dO_ic^2

    The bound is `sigmas` standard deviations plus the fp32 accumulation error
    (n u32 times the sum of magnitudes, n the reduction length).  dD_i enters a dQ row
    coherently (one error times the whole row of P K), which is why it is not summed
    in quadrature there."""
    BH, N, d = q.shape
    s = scale * np.einsum("bid,bjd->bij", q, k)
    if causal:
        s = np.where(np.tril(np.ones((N, N), dtype=bool))[None], s, -np.inf)
    s -= s.max(axis=2, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=2, keepdims=True)
    p2 = p * p
    o = np.einsum("bij,bjd->bid", p, v)
    dp = np.einsum("bid,bjd->bij", do, v)
    ds = p * (dp - (do * o).sum(axis=2, keepdims=True))
    ds2 = ds * ds
    w = U_BF16 * U_BF16 / 3.0
    var_o = w * (o * o + np.einsum("bij,bjd->bid", p2, v * v))
    var_dd = (do * do * var_o).sum(axis=2, keepdims=True)                  # [BH, N, 1]
    pk = np.einsum("bij,bjd->bid", p, k)
    var_dq = scale * scale * (pk * pk * var_dd + w * np.einsum("bij,bjd->bid", ds2, k * k))
    var_dk = scale * scale * (np.einsum("bij,bid->bjd", p2 * var_dd, q * q) +
                              w * np.einsum("bij,bid->bjd", ds2, q * q))
    var_dv = w * np.einsum("bij,bid->bjd", p2, do * do)
    ads = np.abs(ds)
    acc = N * U_FP32
    b_dq = sigmas * np.sqrt(var_dq) + acc * scale * np.einsum("bij,bjd->bid", ads, np.abs(k))
    b_dk = sigmas * np.sqrt(var_dk) + acc * scale * np.einsum("bij,bid->bjd", ads, np.abs(q))
    b_dv = sigmas * np.sqrt(var_dv) + acc * np.einsum("bij,bid->bjd", p, np.abs(do))
    return b_dq + 1e-6, b_dk + 1e-6, b_dv + 1e-6
