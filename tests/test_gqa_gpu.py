"""Grouped-query attention on the GPU (forward, backward, decode, paged decode).

Reading of the definition: query head h of a batch uses key/value head
h / (H / Hkv); a key/value head shared by a group of query heads gets as its
gradient the sum of the gradients it would receive as each head's private copy
(the chain rule for a shared input).  So the oracle runs on K and V repeated over
each group (plain indexing), and its dK, dV are summed over each group.
"""
import numpy as np
import pytest
import torch

from exact_attention_26_gb300.inputs import decode_qkv, gqa_qkv, paged_cache, to_f64
from gpu_common import GRAD_ABS, L_ABS, assert_abs_close, assert_o_close, load_fa
from oracle import Oracle

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def fa():
    return load_fa()


@pytest.fixture(scope="module")
def orc():
    return Oracle()


def _expand(x, group):
    """[B, Hkv, N, d] -> [B, Hkv * group, N, d], each head repeated over its group."""
    return np.repeat(x, group, axis=1)


def _fold(g, group):
    """Sum [B, Hkv * group, N, d] over each group -> [B, Hkv, N, d]."""
    B, H, N, d = g.shape
    return g.reshape(B, H // group, group, N, d).sum(axis=2)


FWD = [(1, 4, 1, 300, 64), (2, 8, 2, 256, 128), (1, 6, 3, 129, 256), (1, 4, 4, 200, 128),
       (1, 16, 2, 640, 64), (1, 4, 2, 333, 96)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", FWD, ids=lambda s: "x".join(map(str, s)))
def test_gqa_forward(fa, orc, shape, causal):
    B, H, Hkv, N, d = shape
    q, k, v = gqa_qkv(B, H, Hkv, N, d, seed=N + H)
    o, lse = fa.forward(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == 0
    g = H // Hkv
    ro, rl = orc.fwd(to_f64(q), _expand(to_f64(k), g), _expand(to_f64(v), g), causal=causal)
    assert_o_close(o.float().cpu().numpy(), ro, f"{shape} causal={causal}")
    assert_abs_close(lse.cpu().numpy(), rl, L_ABS, f"{shape} causal={causal} L")


def test_gqa_forward_equals_repeated_heads(fa):
    """The shared head gives exactly the result of a private copy per query head."""
    q, k, v = (t.to(DEV) for t in gqa_qkv(2, 8, 2, 777, 128, seed=3))
    o1, l1 = fa.forward(q, k, v, causal=True)
    o2, l2 = fa.forward(q, k.repeat_interleave(4, dim=1).contiguous(),
                        v.repeat_interleave(4, dim=1).contiguous(), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


BWD = [(1, 4, 2, 300, 128), (2, 4, 1, 256, 64), (1, 8, 2, 513, 128), (1, 3, 3, 129, 64),
       (1, 4, 2, 257, 96)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", BWD, ids=lambda s: "x".join(map(str, s)))
def test_gqa_backward(fa, orc, shape, causal):
    B, H, Hkv, N, d = shape
    q, k, v, do = gqa_qkv(B, H, Hkv, N, d, seed=N + d, with_do=True)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = fa.forward(qd, kd, vd, causal=causal)
    dq, dk, dv = fa.backward(qd, kd, vd, o, lse, dod, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == 0
    assert dk.shape == k.shape and dv.shape == v.shape
    g = H // Hkv
    rq, rk, rv = orc.bwd(to_f64(q), _expand(to_f64(k), g), _expand(to_f64(v), g), to_f64(do),
                         causal=causal)
    assert_abs_close(dq.cpu().numpy(), rq, GRAD_ABS, f"{shape} dQ")
    assert_abs_close(dk.cpu().numpy(), _fold(rk, g), GRAD_ABS, f"{shape} dK")
    assert_abs_close(dv.cpu().numpy(), _fold(rv, g), GRAD_ABS, f"{shape} dV")


DEC = [(2, 8, 2, 1, 1000, 128, 0), (1, 32, 8, 1, 4096, 128, 0), (1, 4, 1, 3, 500, 64, 2),
       (2, 6, 2, 2, 777, 256, 3), (1, 16, 1, 1, 2000, 128, 1)]


@pytest.mark.parametrize("shape", DEC, ids=lambda s: "x".join(map(str, s)))
def test_gqa_decode(fa, orc, shape):
    B, H, Hkv, Nq, Nk, d, splits = shape
    g = torch.Generator().manual_seed(Nk)
    q = torch.randn((B, H, Nq, d), generator=g).to(torch.bfloat16)
    _, k, v = decode_qkv(B, Hkv, 1, Nk, d, seed=Nk + 1)
    o, lse = fa.decode(q.to(DEV), k.to(DEV), v.to(DEV), num_splits=splits)
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == 0
    grp = H // Hkv
    ro, rl = orc.decode(to_f64(q), _expand(to_f64(k), grp), _expand(to_f64(v), grp))
    assert_o_close(o.float().cpu().numpy(), ro, f"{shape}")
    assert_abs_close(lse.cpu().numpy(), rl, L_ABS, f"{shape} L")


def test_gqa_paged_decode(fa, orc):
    B, H, Hkv, Nq, P, ps, d = 3, 8, 2, 1, 20, 16, 128
    g = torch.Generator().manual_seed(11)
    q = torch.randn((B, H, Nq, d), generator=g).to(torch.bfloat16)
    _, k, v = decode_qkv(B, Hkv, 1, P * ps, d, seed=12)
    kc, vc, bt = paged_cache(k, v, ps)
    lens = torch.tensor([P * ps, 100, 7], dtype=torch.int32)
    o, lse = fa.decode_paged(q.to(DEV), kc.to(DEV), vc.to(DEV), bt.to(DEV), lens.to(DEV), num_splits=3)
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == 0
    grp = H // Hkv
    for b in range(B):
        n = int(lens[b])
        ro, rl = orc.decode(to_f64(q[b:b + 1]), _expand(to_f64(k[b:b + 1, :, :n]), grp),
                            _expand(to_f64(v[b:b + 1, :, :n]), grp))
        assert_o_close(o[b:b + 1].float().cpu().numpy(), ro, f"paged GQA seq {b}")
        assert_abs_close(lse[b:b + 1].cpu().numpy(), rl, L_ABS, f"paged GQA seq {b} L")
