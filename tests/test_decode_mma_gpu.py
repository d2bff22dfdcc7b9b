"""Tensor-core decode (several query rows per key/value head) against the float64
oracle, through the C ABI.

R = (H / Hkv) * Nq >= 2 rows per key/value head and d <= 128 run on the tcgen05
kernel: the CTA's rows as M = 128 against 64-key tiles of the cache (128 at
d = 64), two S slots,
the forward's online softmax per row.  Cases: Nq in {2, 4, 8, 16}, grouped
queries, more than 128 rows (several row blocks), ragged key counts and ranges,
every head dimension it serves, and the B=8 H=32 Nq=4 Nk=32768 d=128 workload.
"""
import numpy as np
import pytest
import torch

from exact_attention_26_gb300.inputs import decode_qkv, to_f64
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


def _expand(x, g):
    return np.repeat(x, g, axis=1)


def _check(fa, orc, B, H, Hkv, Nq, Nk, d, splits, seed, what):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, H, Nq, d), generator=g).to(torch.bfloat16)
    _, k, v = decode_qkv(B, Hkv, 1, Nk, d, seed=seed + 1)
    o, lse = fa.decode(q.to(DEV), k.to(DEV), v.to(DEV), num_splits=splits)
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == 0
    grp = H // Hkv
    ro, rl = orc.decode(to_f64(q), _expand(to_f64(k), grp), _expand(to_f64(v), grp))
    assert_o_close(o.float().cpu().numpy(), ro, what)
    assert_abs_close(lse.cpu().numpy(), rl, L_ABS, f"{what} L")


@pytest.mark.parametrize("Nq", [2, 4, 8, 16])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_decode_rows(fa, orc, Nq, splits):
    """Nq rows per head (multi-head: R = Nq)."""
    B, H, Nk, d = 2, 4, 3001, 128
    assert fa.fa_decode_uses_tensor_cores(H, H, Nq, d, 0) == 1
    _check(fa, orc, B, H, H, Nq, Nk, d, splits, Nq * 10 + splits, f"Nq={Nq} splits={splits}")


# (B, H, Hkv, Nq, Nk, d, splits)
SHAPES = [
    (1, 8, 2, 1, 1000, 128, 0),     # grouped queries, one new token: R = 4
    (2, 4, 2, 1, 999, 64, 3),       # R = 2, d = 64 (128-key tiles)
    (1, 2, 2, 3, 129, 64, 0),       # d = 64, a ragged second tile
    (2, 32, 4, 2, 777, 64, 0),      # R = 16, d = 64
    (1, 16, 1, 16, 700, 64, 2),     # R = 256: two row blocks of 128
    (1, 8, 1, 16, 513, 128, 0),     # R = 128 exactly
    (1, 43, 1, 3, 300, 128, 1),     # R = 129: a second block with one row
    (1, 4, 4, 4, 65, 96, 2),        # d = 96; ranges of 64 keys and 1 key
    (3, 2, 2, 5, 1, 128, 0),        # a single cached key
    (1, 2, 2, 4, 64 * 7, 128, 7),   # one 64-key tile per range
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_decode_shapes(fa, orc, shape):
    B, H, Hkv, Nq, Nk, d, splits = shape
    assert fa.fa_decode_uses_tensor_cores(H, Hkv, Nq, d, 0) == 1
    _check(fa, orc, B, H, Hkv, Nq, Nk, d, splits, Nk + d + Nq, f"{shape}")


def test_decode_rows_boosted_keys(fa, orc):
    """One key per 128-key block carries +4: the reference max moves, O is rescaled."""
    q, k, v = decode_qkv(1, 4, 8, 3000, 128, seed=5, mult=0.5, boost=4.0)
    o, lse = fa.decode(q.to(DEV), k.to(DEV), v.to(DEV), num_splits=2)
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == 0
    ro, rl = orc.decode(to_f64(q), to_f64(k), to_f64(v))
    assert_o_close(o.float().cpu().numpy(), ro, "boosted")
    assert_abs_close(lse.cpu().numpy(), rl, L_ABS, "boosted L")


def test_decode_rows_deterministic(fa):
    q, k, v = (t.to(DEV) for t in decode_qkv(2, 2, 8, 5000, 128, seed=3))
    a = fa.decode(q, k, v)
    b = fa.decode(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_decode_rows_paged_stays_on_cuda_cores(fa):
    assert fa.fa_decode_uses_tensor_cores(8, 2, 4, 128, 1) == 0
    assert fa.fa_decode_uses_tensor_cores(8, 2, 4, 256, 0) == 0
    assert fa.fa_decode_uses_tensor_cores(8, 8, 1, 128, 0) == 0


def test_decode_four_rows_workload(fa, orc):
    """B=8 x 32 heads, Nq = 4 new tokens, Nk = 32768, d = 128, automatic key ranges:
    the benchmark's multi-row decode configuration; eight heads against the oracle."""
    B, H, Nq, Nk, d = 8, 32, 4, 32768, 128
    q, k, v = decode_qkv(B, H, Nq, Nk, d, seed=0, device=DEV)
    assert fa.fa_decode_uses_tensor_cores(H, H, Nq, d, 0) == 1
    o, lse = fa.decode(q, k, v)
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == 0
    heads = [(b, h) for b in range(B) for h in range(H)][:: (B * H) // 8][:8]
    for b, h in heads:
        ro, rl = orc.decode(to_f64(q[b:b + 1, h:h + 1].cpu()), to_f64(k[b:b + 1, h:h + 1].cpu()),
                            to_f64(v[b:b + 1, h:h + 1].cpu()))
        assert_o_close(o[b:b + 1, h:h + 1].float().cpu().numpy(), ro, f"head ({b},{h})")
        assert_abs_close(lse[b:b + 1, h:h + 1].cpu().numpy(), rl, L_ABS, f"head ({b},{h}) L")
