"""Forward parity on the GPU: fa_fwd (through the C ABI) against the float64 oracle.

Small shapes span several 128-row tiles and ragged tails; the full-size
workloads run in the launch configuration the benchmark times and are checked on
sampled rows the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

from exact_attention_26_gb300.inputs import boosted_qkv, normal_qkv, sample_rows, to_f64
from gpu_common import L_ABS, assert_abs_close, assert_o_close, load_fa
from oracle import Oracle

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def fa():
    return load_fa()


@pytest.fixture(scope="module")
def orc():
    return Oracle()


def _run(fa, q, k, v, causal, scale=None):
    o, lse = fa.forward(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == 0
    return o.float().cpu().numpy(), lse.cpu().numpy()


SMALL = [
    (1, 1, 1, 64), (1, 2, 2, 128), (1, 1, 100, 64), (1, 1, 128, 64), (2, 1, 129, 128),
    (1, 2, 256, 128), (1, 1, 300, 256), (1, 2, 383, 64), (1, 1, 513, 128), (1, 1, 200, 256),
    (2, 3, 640, 64), (1, 1, 1000, 256), (1, 1, 1, 96), (1, 2, 200, 96), (2, 1, 513, 96),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s)))
def test_fwd_small(fa, orc, shape, causal):
    B, H, N, d = shape
    q, k, v = normal_qkv(B, H, N, d, seed=N + d)
    o, lse = _run(fa, q, k, v, causal)
    ro, rl = orc.fwd(to_f64(q), to_f64(k), to_f64(v), causal=causal)
    assert_o_close(o, ro, f"{shape} causal={causal}")
    assert_abs_close(lse, rl, L_ABS, f"{shape} causal={causal} L")


@pytest.mark.parametrize("causal", [False, True])
def test_fwd_smallest_workload(fa, orc, causal):
    """B=1, H=1, N=128, d=64, N(0,1) from seed 0, scale 1/sqrt(d): every row."""
    q, k, v = normal_qkv(1, 1, 128, 64, seed=0)
    o, lse = _run(fa, q, k, v, causal)
    ro, rl = orc.fwd(to_f64(q), to_f64(k), to_f64(v), causal=causal)
    assert_o_close(o, ro, "128x64")
    assert_abs_close(lse, rl, L_ABS, "128x64 L")


def _sampled(fa, orc, q, k, v, causal, nrows, seed=2):
    B, H, N, d = q.shape
    rows = sample_rows(N, nrows, seed=seed).numpy()
    o, lse = _run(fa, q, k, v, causal)
    ro, rl = orc.fwd_rows(to_f64(q), to_f64(k), to_f64(v), rows, causal=causal)
    assert_o_close(o[:, :, rows], ro, f"{tuple(q.shape)} causal={causal} sampled")
    assert_abs_close(lse[:, :, rows], rl, L_ABS, f"{tuple(q.shape)} L sampled")
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
def test_fwd_b4_h16_n4096_d96(fa, orc, causal):
    q, k, v = normal_qkv(4, 16, 4096, 96, seed=0)
    _sampled(fa, orc, q, k, v, causal, 48)


@pytest.mark.parametrize("causal", [False, True])
def test_fwd_b8_h16_n2048_d64(fa, orc, causal):
    q, k, v = normal_qkv(8, 16, 2048, 64, seed=0)
    _sampled(fa, orc, q, k, v, causal, 64)


def test_fwd_b1_h16_n16384_d128_causal(fa, orc):
    """Long-context batch-1 workload; 256 seeded rows per head."""
    q, k, v = normal_qkv(1, 16, 16384, 128, seed=0)
    _sampled(fa, orc, q, k, v, True, 256)


def test_fwd_b4_h8_n8192_d256_boosted(fa, orc):
    """Half-scale inputs with one +4 key per 128-key block: the row max keeps moving."""
    q, k, v = boosted_qkv(4, 8, 8192, 256, seed=0)
    _sampled(fa, orc, q, k, v, False, 96)


def test_fwd_b2_h16_n4096_d128_causal(fa, orc):
    q, k, v = normal_qkv(2, 16, 4096, 128, seed=0)
    _sampled(fa, orc, q, k, v, True, 128)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_fwd_causal_row_zero_is_v0(fa, d):
    """Causal row 0 sees only key 0: P = 1 exactly, so O_0 = V_0 bit for bit."""
    q, k, v = normal_qkv(2, 2, 300, d, seed=5)
    o, lse = _run(fa, q, k, v, True)
    assert np.array_equal(o[:, :, 0], v[:, :, 0].float().numpy())
    s = (q[:, :, 0].double() * k[:, :, 0].double()).sum(-1).numpy() / np.sqrt(d)
    assert_abs_close(lse[:, :, 0], s, L_ABS, "L_0")


@pytest.mark.parametrize("d", [64, 128, 256])
def test_fwd_identical_keys_give_mean(fa, orc, d):
    q, k, v = normal_qkv(1, 2, 333, d, seed=6)
    k = k[:, :, :1].expand(-1, -1, 333, -1).contiguous()
    for causal in (False, True):
        o, lse = _run(fa, q, k, v, causal)
        ro, rl = orc.fwd(to_f64(q), to_f64(k), to_f64(v), causal=causal)
        assert_o_close(o, ro, f"identical keys d={d}")
        assert_abs_close(lse, rl, L_ABS, "identical keys L")


@pytest.mark.parametrize("scale", [2.0, 0.01])
def test_fwd_extreme_scales(fa, orc, scale):
    """A large scale makes rows nearly one-hot (many max moves); a tiny one makes them flat."""
    q, k, v = normal_qkv(1, 2, 700, 128, seed=7)
    for causal in (False, True):
        o, lse = _run(fa, q, k, v, causal, scale=scale)
        ro, rl = orc.fwd(to_f64(q), to_f64(k), to_f64(v), causal=causal, scale=scale)
        assert_o_close(o, ro, f"scale={scale}")
        assert_abs_close(lse, rl, L_ABS, f"scale={scale} L")


def test_fwd_deterministic(fa):
    q, k, v = normal_qkv(2, 4, 1111, 128, seed=8)
    a = _run(fa, q, k, v, True)
    b = _run(fa, q, k, v, True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_fwd_writes_nothing_outside_outputs(fa):
    """Guard bands around O and L keep their sentinel values."""
    B, H, N, d = 1, 2, 257, 64
    q, k, v = (t.to(DEV) for t in normal_qkv(B, H, N, d, seed=9))
    pad = 4096
    o_buf = torch.full((B * H * N * d + 2 * pad,), 7.0, dtype=torch.bfloat16, device=DEV)
    l_buf = torch.full((B * H * N + 2 * pad,), 7.0, dtype=torch.float32, device=DEV)
    o = o_buf[pad:pad + B * H * N * d].view(B, H, N, d)
    lse = l_buf[pad:pad + B * H * N].view(B, H, N)
    fa.forward(q, k, v, causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    for buf in (o_buf, l_buf):
        assert torch.all(buf[:pad] == 7.0) and torch.all(buf[-pad:] == 7.0)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


@pytest.mark.parametrize("d", [64, 96, 128, 256])
def test_fwd_output_on_a_16_byte_boundary(fa, d):
    """An O base that is 16- but not 32-byte aligned takes the epilogue's 16-byte
    stores instead of its 32-byte ones: the same values, and nothing written outside
    the output."""
    B, H, N = 1, 2, 300
    q, k, v = (t.to(DEV) for t in normal_qkv(B, H, N, d, seed=d))
    ref, ref_l = fa.forward(q, k, v, causal=True)
    n = B * H * N * d
    buf = torch.full((n + 64,), 7.0, dtype=torch.bfloat16, device=DEV)
    off = next(i for i in range(0, 32, 8) if (buf.data_ptr() + 2 * i) % 32 == 16)
    o = buf[off:off + n].view(B, H, N, d)
    assert o.data_ptr() % 32 == 16
    _, lse = fa.forward(q, k, v, causal=True, out=o)
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == 0
    assert torch.equal(o, ref) and torch.equal(lse, ref_l)
    assert torch.all(buf[:off] == 7.0) and torch.all(buf[off + n:] == 7.0)


@pytest.mark.parametrize("shape", [(1, 2, 65536, 128), (1, 1, 131072, 64)], ids=["65536x128", "131072x64"])
def test_fwd_long_sequences(fa, orc, shape):
    """The longest sequences of the pages' table and beyond, causal, sampled rows
    (row indices times d pass 2^23 here)."""
    B, H, N, d = shape
    q, k, v = normal_qkv(B, H, N, d, seed=N + d)
    _sampled(fa, orc, q, k, v, True, 24)
