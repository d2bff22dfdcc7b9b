"""The derived gradient bound (gpu_common.grad_bounds) against an emulation of the
backward kernel's roundings, on the CPU.

The emulation repeats, in numpy, the places where the kernel rounds: the forward's P
to bf16 for its P V product and O to bf16; the backward's P = exp(S scale - L) in
fp32, D_i from the bf16 O, dS = P (dP - D) in fp32 then rounded to bf16 for the dK and
dQ products, P rounded to bf16 for dV.  Every element of its error against the exact
gradients must sit inside the bound, at the extreme scales the GPU test uses and at
1/sqrt(d); and the bound must not be slack (its largest ratio of error to bound is
above 0.2 at every scale, so a bound inflated tenfold would fail)."""
import numpy as np
import pytest
import torch

from exact_attention_26_gb300.inputs import normal_qkv, to_f64
from gpu_common import grad_bounds


def _bf16(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).double().numpy()


def _f32(x):
    return np.asarray(x, dtype=np.float32).astype(np.float64)


@pytest.mark.parametrize("scale", [1.5, 0.02, 1.0 / np.sqrt(128)])
@pytest.mark.parametrize("causal", [False, True])
def test_bound_covers_the_kernels_roundings(scale, causal):
    q, k, v, do = normal_qkv(1, 2, 400, 128, seed=11, with_do=True)
    q, k, v, do = (to_f64(t).reshape(2, 400, 128) for t in (q, k, v, do))
    N = q.shape[1]
    s = scale * np.einsum("bid,bjd->bij", q, k)
    if causal:
        s = np.where(np.tril(np.ones((N, N), dtype=bool))[None], s, -np.inf)
    m = s.max(axis=2, keepdims=True)
    e = np.exp(s - m)
    l_ = e.sum(axis=2, keepdims=True)
    p, lse = e / l_, m + np.log(l_)
    # exact gradients
    o = p @ v
    dp = do @ v.transpose(0, 2, 1)
    ds = p * (dp - (do * o).sum(axis=2, keepdims=True))
    exact = (scale * ds @ k, scale * ds.transpose(0, 2, 1) @ q, p.transpose(0, 2, 1) @ do)
    # the kernel's roundings
    o_k = _bf16((_bf16(e) @ v) / l_)
    p_k = _f32(np.exp(_f32(s) - _f32(lse)))
    d_k = _f32((do * o_k).sum(axis=2, keepdims=True))
    ds_k = _bf16(_f32(p_k * (_f32(dp) - d_k)))
    kernel = (scale * ds_k @ k, scale * ds_k.transpose(0, 2, 1) @ q,
              _bf16(p_k).transpose(0, 2, 1) @ do)
    for name, g, r, b in zip(("dQ", "dK", "dV"), kernel, exact,
                             grad_bounds(q, k, v, do, causal, scale)):
        ratio = np.abs(g - r) / b
        assert ratio.max() <= 1.0, (name, float(ratio.max()))
        assert ratio.max() > 0.2, (name, float(ratio.max()))
