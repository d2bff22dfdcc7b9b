"""Decode parity on the GPU: fa_decode (split key ranges + LSE merge, through the C
ABI) against the float64 oracle's decode rows.

Small shapes cover one and several key ranges, ragged last ranges and stages,
query blocks with a ragged tail, every head dimension, and key counts below one
pipeline stage.  The long-context workload (B=8, H=32, Nk=32768, d=128, one query
row) runs in the launch configuration the benchmark times, with the cache drawn
on the GPU and a sample of heads checked against the oracle.
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


def _run(fa, q, k, v, scale=None, splits=0):
    o, lse = fa.decode(q.to(DEV), k.to(DEV), v.to(DEV), scale=scale, num_splits=splits)
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == 0
    return o.float().cpu().numpy(), lse.cpu().numpy()


# (B, H, Nq, Nk, d, requested key ranges; 0 = automatic)
SMALL = [
    (1, 1, 1, 1, 128, 0), (1, 2, 1, 100, 64, 0), (2, 3, 1, 1000, 128, 0), (1, 2, 1, 1000, 128, 1),
    (1, 2, 1, 1000, 128, 7), (1, 1, 3, 777, 64, 3), (2, 2, 8, 500, 128, 0), (1, 1, 9, 300, 128, 2),
    (1, 2, 5, 1234, 256, 0), (1, 1, 1, 4097, 256, 5), (1, 1, 20, 2000, 64, 4), (1, 1, 1, 100, 128, 50),
    (1, 1, 2, 10, 128, 3), (3, 1, 1, 64, 64, 1), (1, 3, 4, 129, 256, 2), (1, 1, 16, 65, 128, 2),
    (1, 2, 1, 1000, 96, 0), (2, 1, 3, 777, 96, 3), (1, 1, 9, 129, 96, 1),
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s)))
def test_decode_small(fa, orc, shape):
    B, H, Nq, Nk, d, splits = shape
    q, k, v = decode_qkv(B, H, Nq, Nk, d, seed=Nk + d + Nq)
    o, lse = _run(fa, q, k, v, splits=splits)
    ro, rl = orc.decode(to_f64(q), to_f64(k), to_f64(v))
    assert_o_close(o, ro, f"{shape}")
    assert_abs_close(lse, rl, L_ABS, f"{shape} L")


def test_decode_split_count_is_clamped(fa):
    """Requests beyond the number of pipeline stages shrink to one range per stage.
    The automatic count spreads a short cache that fits one wave over one stage per
    range (it is latency-bound), and splits a large batch only a few ways."""
    assert fa.fa_decode_num_splits(1, 1, 1, 1, 100, 128, 50) == 2
    assert fa.fa_decode_num_splits(1, 1, 1, 1, 10, 128, 3) == 1
    assert fa.fa_decode_num_splits(1, 1, 1, 1, 64 * 40, 128, 0) == 40
    assert 1 < fa.fa_decode_num_splits(8, 32, 32, 1, 32768, 128, 0) < 16
    assert fa.fa_decode_workspace_bytes(1, 1, 1, 1, 1000, 128, 1) == 0
    assert fa.fa_decode_workspace_bytes(1, 1, 1, 1, 1000, 128, 4) > 0


@pytest.mark.parametrize("splits", [1, 3, 0])
def test_decode_boosted_keys(fa, orc, splits):
    """One key per 128-key block carries +4: the key range holding the largest
    score dominates the merge, and the others must be scaled down exactly."""
    q, k, v = decode_qkv(1, 4, 2, 3000, 128, seed=5, mult=0.5, boost=4.0)
    o, lse = _run(fa, q, k, v, splits=splits)
    ro, rl = orc.decode(to_f64(q), to_f64(k), to_f64(v))
    assert_o_close(o, ro, f"boosted splits={splits}")
    assert_abs_close(lse, rl, L_ABS, f"boosted splits={splits} L")


@pytest.mark.parametrize("scale", [0.01, 1.5])
def test_decode_extreme_scales(fa, orc, scale):
    q, k, v = decode_qkv(1, 2, 3, 900, 64, seed=9)
    o, lse = _run(fa, q, k, v, scale=scale, splits=4)
    ro, rl = orc.decode(to_f64(q), to_f64(k), to_f64(v), scale=scale)
    assert_o_close(o, ro, f"scale={scale}")
    assert_abs_close(lse, rl, L_ABS, f"scale={scale} L")


def test_decode_is_deterministic(fa):
    q, k, v = decode_qkv(2, 2, 1, 5000, 128, seed=3)
    a = fa.decode(q.to(DEV), k.to(DEV), v.to(DEV))
    b = fa.decode(q.to(DEV), k.to(DEV), v.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_decode_rejects_small_workspace(fa):
    q, k, v = (t.to(DEV) for t in decode_qkv(1, 1, 1, 2000, 128, seed=1))
    o = torch.empty_like(q)
    lse = torch.empty((1, 1, 1), dtype=torch.float32, device=DEV)
    need = fa.fa_decode_workspace_bytes(1, 1, 1, 1, 2000, 128, 4)
    ws = torch.empty(need - 16, dtype=torch.uint8, device=DEV)
    rc = fa.fa_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 1, 1,
                      1, 2000, 128, 0.1, 4, ws.data_ptr(), ws.numel(), None)
    assert rc == fa.fa.FA_ERR_WORKSPACE
    rc = fa.fa_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 1, 1,
                      1, 2000, 128, 0.1, 4, None, 0, None)
    assert rc == fa.fa.FA_ERR_WORKSPACE


@pytest.mark.parametrize("B", [8, 1])
def test_decode_long_context_workload(fa, orc, B):
    """B x 32 heads, one query row, Nk = 32768, d = 128, automatic key ranges (the
    benchmark's configuration); eight heads are checked against the oracle."""
    H, Nk, d = 32, 32768, 128
    q, k, v = decode_qkv(B, H, 1, Nk, d, seed=0, device=DEV)
    o, lse = fa.decode(q, k, v)
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == 0
    assert fa.fa_decode_num_splits(B, H, H, 1, Nk, d, 0) > 1
    heads = [(b, h) for b in range(B) for h in range(H)][:: max(1, (B * H) // 8)][:8]
    for b, h in heads:
        ro, rl = orc.decode(to_f64(q[b:b + 1, h:h + 1].cpu()), to_f64(k[b:b + 1, h:h + 1].cpu()),
                            to_f64(v[b:b + 1, h:h + 1].cpu()))
        assert_o_close(o[b:b + 1, h:h + 1].float().cpu().numpy(), ro, f"B{B} head ({b},{h})")
        assert_abs_close(lse[b:b + 1, h:h + 1].cpu().numpy(), rl, L_ABS, f"B{B} head ({b},{h}) L")
