"""Packed variable-length forward on the GPU (fa_fwd_varlen) against the oracle run
on each sequence separately.

Sequences include lengths 1, exact tile multiples, ragged tails and an empty one;
grouped key/value heads; every head dimension; causal masks taken per sequence.
The tokens after a sequence belong to the next one, so a key read past a
sequence's end is real data that must be masked, not zero fill.
"""
import numpy as np
import pytest
import torch

from exact_attention_26_gb300.inputs import normal_qkv, to_f64, varlen_qkv
from gpu_common import L_ABS, assert_abs_close, assert_o_close, load_fa
from oracle import Oracle

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
FA_ERR_BAD_INDEX = 7


@pytest.fixture(scope="module")
def fa():
    return load_fa()


@pytest.fixture(scope="module")
def orc():
    return Oracle()


CASES = [
    ([200, 129, 1, 513], 4, 2, 128), ([300, 0, 77], 2, 2, 64), ([256, 256], 3, 1, 256),
    ([1, 2, 3], 4, 4, 128), ([1000, 17, 640], 8, 2, 64),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c[0])) + f"_h{c[1]}kv{c[2]}d{c[3]}")
def test_varlen_forward(fa, orc, case, causal):
    lens, H, Hkv, d = case
    q, k, v, cu = varlen_qkv(lens, H, Hkv, d, seed=sum(lens) + d)
    o, lse = fa.forward_varlen(q.to(DEV), k.to(DEV), v.to(DEV), cu.to(DEV), max(lens), causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == 0
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    g = H // Hkv
    for b, n in enumerate(lens):
        if n == 0:
            continue
        a = int(cu[b])
        qs = to_f64(q[a:a + n].permute(1, 0, 2).unsqueeze(0))
        ks = np.repeat(to_f64(k[a:a + n].permute(1, 0, 2).unsqueeze(0)), g, axis=1)
        vs = np.repeat(to_f64(v[a:a + n].permute(1, 0, 2).unsqueeze(0)), g, axis=1)
        ro, rl = orc.fwd(qs, ks, vs, causal=causal)
        assert_o_close(o[a:a + n].transpose(1, 0, 2)[None], ro, f"seq {b} (len {n})")
        assert_abs_close(lse[:, a:a + n][None], rl, L_ABS, f"seq {b} L")


def test_varlen_equals_fixed_layout(fa):
    """Equal lengths: the packed layout gives the fixed layout's results bit for bit."""
    B, H, N, d = 3, 4, 700, 128
    q, k, v = (t.to(DEV) for t in normal_qkv(B, H, N, d, seed=6))
    o1, l1 = fa.forward(q, k, v, causal=True)
    pack = lambda x: x.permute(0, 2, 1, 3).reshape(B * N, H, d).contiguous()
    cu = torch.arange(0, B * N + 1, N, dtype=torch.int32, device=DEV)
    o2, l2 = fa.forward_varlen(pack(q), pack(k), pack(v), cu, N, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(pack(o1), o2)
    assert torch.equal(l1.permute(1, 0, 2).reshape(H, B * N), l2)


def test_varlen_bad_offsets_are_reported(fa):
    """Decreasing offsets, and a sequence longer than max_seqlen, are caught on the
    device (no access outside the tensors): FA_ERR_BAD_INDEX, and the context works."""
    q, k, v, cu = varlen_qkv([100, 50], 2, 2, 64, seed=1)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    assert fa.fa_device_status(None) == 0
    bad = torch.tensor([0, 120, 100], dtype=torch.int32, device=DEV)
    fa.forward_varlen(qd, kd, vd, bad, 150)
    assert fa.fa_device_status(None) == FA_ERR_BAD_INDEX
    fa.forward_varlen(qd, kd, vd, cu.to(DEV), 64)  # first sequence is longer than 64
    assert fa.fa_device_status(None) == FA_ERR_BAD_INDEX
    fa.forward_varlen(qd, kd, vd, cu.to(DEV), 100)
    assert fa.fa_device_status(None) == 0
