"""Low-precision forward on the GPU: the e4m3 quantiser (fa_quantize_fp8) against
the oracle's quantiser, and attention on e4m3 inputs (fa_fwd_fp8) against the
float64 oracle applied to the dequantised inputs.

Codes are integers, so the quantiser must agree bit for bit (both sides take each
rounding decision in IEEE fp32); with incoherent processing the GPU's Hadamard
butterflies round differently from the oracle's exact transform, so there each
code must be a correct rounding of the exact transformed value.

The attention inputs are quantised by the oracle on the CPU and uploaded, so
nothing the oracle sees comes from the CUDA path.  The kernel differs from the
definition applied to the dequantised inputs only by the rounding of P to e4m3
before the PV product; with P_ij = exp(s_ij - max_j s_ij) the rounding error of
each P (relative to the kernel's running reference, which only scales P up by at
most 2^8) is at most max(2^-4 P, 2^-10), so per element

    |O_ic - O_ref,ic| <= sum_j max(2^-4 P_ij, 2^-10) |V_jc| / sum_j P_ij
                         + 2^-8 |O_ref,ic| (bf16 output) + 1e-4 (fp32 sums),

which the tests evaluate in float64.  L is computed from P before rounding and
keeps the 1e-3 tolerance.
"""
import numpy as np
import pytest
import torch

from exact_attention_26_gb300.inputs import hadamard_signs, outlier_qkv, sample_rows, to_f64
from gpu_common import L_ABS, assert_abs_close, load_fa
from oracle import Oracle
from oracle import fp8 as ofp8

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def fa():
    return load_fa()


@pytest.fixture(scope="module")
def orc():
    return Oracle()


# ---------------------------------------------------------------- quantiser

QUANT = [  # (BH, N, d, block_rows, transpose)
    (3, 300, 128, 128, False), (2, 1, 64, 0, False), (1, 1000, 256, 256, False),
    (4, 129, 128, 0, True), (2, 300, 64, 128, True), (1, 640, 128, 384, False), (2, 17, 256, 0, True),
]


def _quant_input(BH, N, d, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((BH, N, d), generator=g) * 3.0
    x[0, :min(N, 130)] *= 1e-4  # tiny values: subnormal codes
    if BH > 1:
        x[1] = 0.0  # an all-zero head
    x[-1, N // 2, d // 3] = 700.0  # an outlier
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("case", QUANT, ids=lambda c: "x".join(map(str, c)))
def test_quantize_matches_oracle_bit_for_bit(fa, case):
    BH, N, d, br, tr = case
    x = _quant_input(BH, N, d, seed=N + d)
    codes, descale = fa.quantize_fp8(x.to(DEV), block_rows=br, transpose=tr)
    torch.cuda.synchronize()
    ref_codes, ref_descale = ofp8.quantize(x.float().numpy(), block_rows=br, transpose=tr)
    assert np.array_equal(descale.cpu().numpy(), ref_descale), "descale"
    got = codes.cpu().numpy()
    bad = np.argwhere(got != ref_codes)
    assert bad.size == 0, f"{len(bad)} codes differ, first at {bad[:3].tolist()}"


@pytest.mark.parametrize("d", [64, 128, 256])
def test_quantize_incoherent_rounds_the_exact_transform(fa, d):
    BH, N = 2, 260
    x = _quant_input(BH, N, d, seed=d)
    s = hadamard_signs(d, seed=d)
    codes, descale = fa.quantize_fp8(x.to(DEV), block_rows=128, signs=s.to(DEV))
    torch.cuda.synchronize()
    codes, descale = codes.cpu().numpy(), descale.cpu().numpy().astype(np.float64)
    y = (x.double().numpy() * s.double().numpy()) @ ofp8.hadamard(d) / np.sqrt(d)  # exact
    for bi, r0 in enumerate(range(0, N, 128)):
        yb = y[:, r0:r0 + 128]
        amax = np.abs(yb).max(axis=(1, 2))
        ds = descale[:, bi]
        ref_ds = np.where(amax > 0, amax / 448.0, 1.0)
        assert np.all(np.abs(ds - ref_ds) <= 1e-5 * ref_ds), "descale"
        t = yb / ds[:, None, None]
        val = ofp8.e4m3_value(codes[:, r0:r0 + 128])
        half_q = np.maximum(np.abs(t) * 2.0 ** -4, 2.0 ** -10)
        assert np.all(np.abs(val - t) <= half_q * (1 + 1e-3) + 1e-4 * np.abs(t)), "not a rounding of y"


# ---------------------------------------------------------------- attention

def _quantised(q, k, v, signs=None):
    """The oracle's quantisation of one attention problem: numpy codes and scales
    shaped the way fa_fwd_fp8 takes them."""
    qc, qd = ofp8.quantize(q.float().numpy(), 128, signs)
    kc, kd = ofp8.quantize(k.float().numpy(), 128, signs)
    vc, vd = ofp8.quantize(v.float().numpy(), 0, None, transpose=True)
    return qc, qd, kc, kd, vc, vd


def _dequantised(qc, qd, kc, kd, vc, vd, N):
    return (ofp8.dequantize(qc, qd, 128), ofp8.dequantize(kc, kd, 128),
            ofp8.dequantize(vc, vd, 0, transposed=True, N=N))


def _run_fp8(fa, qc, qd, kc, kd, vc, vd, causal, scale=None):
    t = [torch.from_numpy(np.ascontiguousarray(a)).to(DEV) for a in (qc, kc, vc, qd, kd, vd)]
    o, lse = fa.forward_fp8(t[0], t[1], t[2], t[3], t[4], t[5], causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == 0
    return o.float().cpu().numpy(), lse.cpu().numpy()


def _o_bound(q, k, v, causal, scale, rows=None):
    """The per-element bound of the module docstring, float64 (q [.., n, d] rows)."""
    N = k.shape[-2]
    idx = np.arange(q.shape[-2]) if rows is None else np.asarray(rows)
    s = scale * np.einsum("bhid,bhjd->bhij", q, k)
    if causal:
        s = np.where(np.arange(N)[None, :] <= idx[:, None], s, -np.inf)
    p = np.exp(s - s.max(axis=-1, keepdims=True))
    l = p.sum(axis=-1, keepdims=True)
    w = np.where(np.isfinite(s), np.maximum(p * 2.0 ** -4, 2.0 ** -10), 0.0)
    o = np.einsum("bhij,bhjd->bhid", p, v) / l
    return np.einsum("bhij,bhjd->bhid", w, np.abs(v)) / l + 2.0 ** -8 * np.abs(o) + 1e-4


def _check_fp8(orc, o, lse, qf, kf, vf, causal, scale, what, rows=None):
    H, Hkv = qf.shape[1], kf.shape[1]
    ke, ve = (np.repeat(t, H // Hkv, axis=1) for t in (kf, vf))
    if rows is None:
        ro, rl = orc.fwd(qf, ke, ve, causal=causal, scale=scale)
        bound = _o_bound(qf, ke, ve, causal, scale)
    else:
        ro, rl = orc.fwd_rows(qf, ke, ve, rows, causal=causal, scale=scale)
        bound = _o_bound(qf[:, :, rows], ke, ve, causal, scale, rows)
        o, lse = o[:, :, rows], lse[:, :, rows]
    err = np.abs(o - ro)
    worst = np.unravel_index(np.argmax(err / bound), err.shape)
    assert np.all(err <= bound), f"{what}: O error {err[worst]:.3g} > bound {bound[worst]:.3g} at {worst}"
    assert_abs_close(lse, rl, L_ABS, f"{what} L")
    return float(err.max()), float(np.sqrt((err ** 2).mean()))


FWD = [  # (B, H, Hkv, N)
    (1, 1, 1, 1), (1, 2, 2, 200), (2, 4, 2, 513), (1, 3, 1, 130), (1, 2, 2, 1024), (1, 1, 1, 383),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", FWD, ids=lambda s: "x".join(map(str, s)))
def test_fwd_fp8_small(fa, orc, shape, causal):
    B, H, Hkv, N = shape
    d = 128
    q, k, v = outlier_qkv(B, H, Hkv, N, d, seed=N + H)
    qz = _quantised(q, k, v)
    o, lse = _run_fp8(fa, *qz, causal)
    qf, kf, vf = _dequantised(*qz, N)
    _check_fp8(orc, o, lse, qf, kf, vf, causal, d ** -0.5, f"{shape} causal={causal}")


@pytest.mark.parametrize("scale", [0.02, 0.5])
def test_fwd_fp8_scales(fa, orc, scale):
    q, k, v = outlier_qkv(1, 2, 2, 700, 128, seed=3)
    qz = _quantised(q, k, v)
    o, lse = _run_fp8(fa, *qz, True, scale=scale)
    qf, kf, vf = _dequantised(*qz, 700)
    _check_fp8(orc, o, lse, qf, kf, vf, True, scale, f"scale={scale}")


def test_fwd_fp8_incoherent_inputs(fa, orc):
    """Inputs quantised after the random-sign Hadamard transform (Q and K with the
    same signs) and outlier channels: the kernel is the same, the oracle gets the
    dequantised transformed inputs."""
    q, k, v = outlier_qkv(1, 4, 2, 600, 128, seed=9, n_outliers=4)
    qz = _quantised(q, k, v, signs=hadamard_signs(128, seed=1).numpy())
    o, lse = _run_fp8(fa, *qz, False)
    qf, kf, vf = _dequantised(*qz, 600)
    _check_fp8(orc, o, lse, qf, kf, vf, False, 128 ** -0.5, "incoherent")


def test_fwd_fp8_long_context_workload(fa, orc):
    """B=1, H=16, N=16384, d=128, causal, in the launch configuration the benchmark
    times; 48 rows per head checked against the oracle."""
    B, H, N, d = 1, 16, 16384, 128
    q, k, v = outlier_qkv(B, H, H, N, d, seed=0)
    qz = _quantised(q, k, v)
    o, lse = _run_fp8(fa, *qz, True)
    qf, kf, vf = _dequantised(*qz, N)
    rows = sample_rows(N, 48, seed=2).numpy()
    mx, rms = _check_fp8(orc, o, lse, qf, kf, vf, True, d ** -0.5, "16384 sampled", rows=rows)
    print(f"long context: max |O err| {mx:.4g}, rms {rms:.4g}")


def test_incoherent_processing_lowers_the_error(fa, orc):
    """End to end on outlier channels: bf16 inputs -> GPU quantiser -> fp8 forward,
    against the exact attention of the bf16 inputs.  With the random-sign Hadamard
    transform on Q and K the error is lower than without (the pages: incoherent
    processing contains outlier-driven quantisation error)."""
    B, H, N, d = 1, 4, 1024, 128
    q, k, v = outlier_qkv(B, H, H, N, d, seed=5, n_outliers=4, outlier_mult=30.0)
    ro, _ = orc.fwd(to_f64(q), to_f64(k), to_f64(v), causal=False)
    errs = {}
    for name, signs in (("plain", None), ("incoherent", hadamard_signs(d, seed=2).to(DEV))):
        qc, qd = fa.quantize_fp8(q.to(DEV), 128, signs=signs)
        kc, kd = fa.quantize_fp8(k.to(DEV), 128, signs=signs)
        vc, vd = fa.quantize_fp8(v.to(DEV), 0, transpose=True)
        o, _ = fa.forward_fp8(qc, kc, vc, qd, kd, vd)
        torch.cuda.synchronize()
        errs[name] = float(np.sqrt(((o.float().cpu().numpy() - ro) ** 2).mean()))
    print(f"rms error vs exact attention: {errs}")
    assert errs["incoherent"] < errs["plain"], errs
