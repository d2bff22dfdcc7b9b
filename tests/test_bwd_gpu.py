"""Backward parity on the GPU: fa_bwd (through the C ABI) against the float64 oracle."""
import numpy as np
import pytest
import torch

from exact_attention_26_gb300.inputs import normal_qkv, to_f64
from gpu_common import grad_bounds, GRAD_ABS, assert_abs_close, load_fa
from oracle import Oracle

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def fa():
    return load_fa()


@pytest.fixture(scope="module")
def orc():
    return Oracle()


def _grads(fa, q, k, v, do, causal, scale=None, workspace=None):
    q, k, v, do = (t.to(DEV) for t in (q, k, v, do))
    o, lse = fa.forward(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=causal, scale=scale, workspace=workspace)
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == 0
    return [t.cpu().numpy() for t in (dq, dk, dv)]


def _check(got, ref, what):
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        assert_abs_close(g, r, GRAD_ABS, f"{what} {name}")


SMALL = [
    (1, 1, 1, 64), (1, 1, 2, 128), (1, 2, 100, 64), (1, 1, 128, 128), (2, 1, 129, 128),
    (1, 2, 300, 64), (1, 1, 513, 128), (2, 2, 640, 128), (1, 1, 1000, 64), (1, 1, 1, 96),
    (1, 2, 130, 96), (2, 1, 513, 96),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s)))
def test_bwd_small(fa, orc, shape, causal):
    B, H, N, d = shape
    q, k, v, do = normal_qkv(B, H, N, d, seed=3 * N + d, with_do=True)
    got = _grads(fa, q, k, v, do, causal)
    ref = orc.bwd(to_f64(q), to_f64(k), to_f64(v), to_f64(do), causal=causal)
    _check(got, ref, f"{shape} causal={causal}")


def test_bwd_b2_h16_n4096_d128_causal(fa, orc):
    """The full fwd+bwd workload in the benchmark's launch configuration; the
    oracle recomputes three whole heads (heads are independent)."""
    B, H, N, d = 2, 16, 4096, 128
    q, k, v, do = normal_qkv(B, H, N, d, seed=0, with_do=True)
    got = _grads(fa, q, k, v, do, True)
    for (b, h) in [(0, 0), (1, 7), (1, 15)]:
        sl = (slice(b, b + 1), slice(h, h + 1))
        ref = orc.bwd(to_f64(q[sl]), to_f64(k[sl]), to_f64(v[sl]), to_f64(do[sl]), causal=True)
        _check([g[sl] for g in got], ref, f"head ({b},{h})")
    # properties that hold for every head at any size: sum_j dK_j = 0, sum_j dV_j = sum_i dO_i
    dk_sum = got[1].sum(axis=2)
    dv_sum = got[2].sum(axis=2)
    do_sum = do.double().sum(dim=2).numpy()
    assert np.max(np.abs(dk_sum)) < 0.5, np.max(np.abs(dk_sum))
    assert np.max(np.abs(dv_sum - do_sum)) < 0.5, np.max(np.abs(dv_sum - do_sum))


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_b2_h4_n2048_d64(fa, orc, causal):
    q, k, v, do = normal_qkv(2, 4, 2048, 64, seed=4, with_do=True)
    got = _grads(fa, q, k, v, do, causal)
    sl = (slice(1, 2), slice(2, 4))
    ref = orc.bwd(to_f64(q[sl]), to_f64(k[sl]), to_f64(v[sl]), to_f64(do[sl]), causal=causal)
    _check([g[sl] for g in got], ref, "2048x64")


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_b2_h8_n2048_d96(fa, orc, causal):
    """Head dimension 96 at a size that fills the GPU: two whole heads against the
    oracle, the gradient sums on every head."""
    q, k, v, do = normal_qkv(2, 8, 2048, 96, seed=5, with_do=True)
    got = _grads(fa, q, k, v, do, causal)
    sl = (slice(1, 2), slice(3, 5))
    ref = orc.bwd(to_f64(q[sl]), to_f64(k[sl]), to_f64(v[sl]), to_f64(do[sl]), causal=causal)
    _check([g[sl] for g in got], ref, "2048x96")
    assert np.max(np.abs(got[1].sum(axis=2))) < 0.5
    assert np.max(np.abs(got[2].sum(axis=2) - do.double().sum(dim=2).numpy())) < 0.5


@pytest.mark.parametrize("scale", [1.5, 0.02])
def test_bwd_extreme_scales(fa, orc, scale):
    """Far from 1/sqrt(d) the gradients grow with `scale` and the kernel's bf16
    roundings (of P and dS for the products, of O inside D_i) are relative, so a fixed
    absolute bound does not apply.  Each element is held to the bound derived from
    those roundings (gpu_common.grad_bounds: six standard deviations of independent
    round-to-nearest errors, plus fp32 accumulation).  At the usual 1/sqrt(d) the
    derived bound is tighter than the stated 2e-2: everywhere without a mask, and for
    at least 99.5% of elements with one (the first causal rows, whose P sits on few
    keys, get a wider bound)."""
    q, k, v, do = normal_qkv(1, 2, 400, 128, seed=11, with_do=True)
    qf, kf, vf, dof = (to_f64(t).reshape(2, 400, 128) for t in (q, k, v, do))
    for causal in (False, True):
        got = _grads(fa, q, k, v, do, causal, scale=scale)
        ref = orc.bwd(to_f64(q), to_f64(k), to_f64(v), to_f64(do), causal=causal, scale=scale)
        bounds = grad_bounds(qf, kf, vf, dof, causal, scale)
        for name, g, r, b in zip(("dQ", "dK", "dV"), got, ref, bounds):
            g, r = g.reshape(b.shape), r.reshape(b.shape)
            err = np.abs(g - r)
            worst = np.unravel_index(np.argmax(err / b), err.shape)
            print(f"scale={scale} causal={causal} {name}: max|ref| {np.abs(r).max():.3g} "
                  f"max-abs err {err.max():.3g}, worst err/bound {err[worst] / b[worst]:.3f}")
            assert np.all(np.isfinite(g))
            assert np.all(err <= b), (name, worst, float(err[worst]), float(b[worst]))
    # at the usual scale the derived bound is tighter than the stated tolerance
    for causal in (False, True):
        for b in grad_bounds(qf, kf, vf, dof, causal, 1.0 / np.sqrt(128)):
            tight = float(np.percentile(b, 99.5)) if causal else float(b.max())
            assert tight < GRAD_ABS


def test_bwd_workspace_contents_do_not_matter(fa):
    q, k, v, do = normal_qkv(1, 2, 333, 128, seed=12, with_do=True)
    need = fa.fa_bwd_workspace_bytes(1, 2, 333, 128)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device=DEV)  # NaN bit patterns
    a = _grads(fa, q, k, v, do, True, workspace=ws)
    b = _grads(fa, q, k, v, do, True)
    for x, y in zip(a, b):
        assert np.allclose(x, y, atol=1e-6, rtol=0)


def test_bwd_dk_dv_deterministic(fa):
    """dK and dV are owned by one CTA each, so they are bit-reproducible."""
    q, k, v, do = normal_qkv(2, 2, 777, 128, seed=13, with_do=True)
    a = _grads(fa, q, k, v, do, True)
    b = _grads(fa, q, k, v, do, True)
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    assert np.allclose(a[0], b[0], atol=1e-5, rtol=0)


def test_bwd_long_sequence_65536(fa, orc):
    """N = 65536 (the longest sequence of the pages' table), B1 H2 d128 causal.  With a
    causal mask the last 128 keys receive gradient only from the last 128 queries, so
    the oracle restricted to those rows (plus 16 sampled rows for dQ) gives their dK,
    dV exactly; dQ is checked on every row the oracle ran."""
    from exact_attention_26_gb300.inputs import sample_rows
    B, H, N, d = 1, 2, 65536, 128
    q, k, v, do = normal_qkv(B, H, N, d, seed=21, with_do=True)
    got = _grads(fa, q, k, v, do, True)
    tail = np.arange(N - 128, N)
    rows = np.unique(np.concatenate([sample_rows(N, 16, seed=3).numpy(), tail]))
    rq, rk, rv = orc.bwd_rows(to_f64(q), to_f64(k), to_f64(v), to_f64(do), rows, causal=True)
    assert_abs_close(got[0][:, :, rows], rq, GRAD_ABS, "65536 dQ rows")
    assert_abs_close(got[1][:, :, tail], rk[:, :, tail], GRAD_ABS, "65536 dK last keys")
    assert_abs_close(got[2][:, :, tail], rv[:, :, tail], GRAD_ABS, "65536 dV last keys")
    dv_sum = got[2].astype(np.float64).sum(axis=2)
    assert np.max(np.abs(dv_sum - do.double().sum(dim=2).numpy())) < 2.0
