"""Packed variable-length forward and backward on the GPU (fa_fwd_varlen,
fa_bwd_varlen) against the oracle run on each sequence separately.

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
    ([1, 2, 3], 4, 4, 128), ([1000, 17, 640], 8, 2, 64), ([70, 300, 129], 4, 2, 96),
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


BWD_CASES = [([200, 129, 1, 513], 4, 2, 128), ([300, 0, 77], 2, 2, 64), ([1, 2, 3], 4, 4, 128),
             ([640, 17], 8, 2, 64), ([384, 256], 2, 1, 128), ([200, 1, 65], 4, 2, 96)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", BWD_CASES, ids=lambda c: "-".join(map(str, c[0])) + f"_h{c[1]}kv{c[2]}d{c[3]}")
def test_varlen_backward(fa, orc, case, causal):
    from gpu_common import GRAD_ABS
    lens, H, Hkv, d = case
    q, k, v, cu = varlen_qkv(lens, H, Hkv, d, seed=sum(lens) + 3 * d)
    g = torch.Generator().manual_seed(sum(lens))
    do = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    qd, kd, vd, dod, cud = (t.to(DEV) for t in (q, k, v, do, cu))
    o, lse = fa.forward_varlen(qd, kd, vd, cud, max(lens), causal=causal)
    dq, dk, dv = fa.backward_varlen(qd, kd, vd, o, lse, dod, cud, max(lens), causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == 0
    dq, dk, dv = (x.cpu().numpy() for x in (dq, dk, dv))
    grp = H // Hkv
    for b, n in enumerate(lens):
        if n == 0:
            continue
        a = int(cu[b])
        head_major = lambda x: to_f64(x[a:a + n].permute(1, 0, 2).unsqueeze(0))
        qs, dos = head_major(q), head_major(do)
        ks, vs = (np.repeat(head_major(x), grp, axis=1) for x in (k, v))
        rq, rk, rv = orc.bwd(qs, ks, vs, dos, causal=causal)
        fold = lambda r: r.reshape(1, H // grp, grp, n, d).sum(axis=2)[0].transpose(1, 0, 2)
        assert_abs_close(dq[a:a + n], rq[0].transpose(1, 0, 2), GRAD_ABS, f"seq {b} dQ")
        assert_abs_close(dk[a:a + n], fold(rk), GRAD_ABS, f"seq {b} dK")
        assert_abs_close(dv[a:a + n], fold(rv), GRAD_ABS, f"seq {b} dV")


def test_varlen_backward_equals_fixed_layout(fa):
    """Equal lengths: packed-layout dK and dV equal the fixed layout's bit for bit; dQ
    is summed over key blocks by bulk adds whose order varies, so it agrees to fp32
    rounding.  The shape gives the fixed layout at least as many CTAs as SMs, so it
    does not split key blocks over two CTAs (whose partial dK, dV sums would round
    differently from the packed layout's single pass)."""
    B, H, N, d = 4, 8, 640, 128
    q, k, v, do = (t.to(DEV) for t in normal_qkv(B, H, N, d, seed=8, with_do=True))
    o1, l1 = fa.forward(q, k, v, causal=True)
    g1 = fa.backward(q, k, v, o1, l1, do, causal=True)
    pack = lambda x: x.permute(0, 2, 1, 3).reshape(B * N, H, d).contiguous()
    cu = torch.arange(0, B * N + 1, N, dtype=torch.int32, device=DEV)
    o2, l2 = fa.forward_varlen(pack(q), pack(k), pack(v), cu, N, causal=True)
    g2 = fa.backward_varlen(pack(q), pack(k), pack(v), o2, l2, pack(do), cu, N, causal=True)
    torch.cuda.synchronize()
    assert torch.allclose(pack(g1[0]), g2[0], rtol=1e-5, atol=1e-6)
    for x, y in zip(g1[1:], g2[1:]):
        assert torch.equal(pack(x), y)


def test_varlen_backward_leaves_other_rows_and_reports_bad_offsets(fa, orc):
    """Tokens after the last sequence keep what the gradient buffers held; bad offsets
    are caught on the device (FA_ERR_BAD_INDEX) and the context keeps working."""
    from gpu_common import GRAD_ABS
    lens, H, Hkv, d = [90, 40], 2, 1, 64
    q, k, v, cu = varlen_qkv(lens + [30], H, Hkv, d, seed=12)  # 30 trailing tokens
    cu = cu[:3].clone()
    T = q.shape[0]
    g = torch.Generator().manual_seed(12)
    do = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    qd, kd, vd, dod, cud = (t.to(DEV) for t in (q, k, v, do, cu))
    o, lse = fa.forward_varlen(qd, kd, vd, cud, 90, causal=True)
    grads = [torch.full(t.shape, 7.0, dtype=torch.float32, device=DEV) for t in (q, k, v)]
    fa.backward_varlen(qd, kd, vd, o, lse, dod, cud, 90, causal=True, dq=grads[0], dk=grads[1],
                       dv=grads[2])
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == 0
    for t in grads:
        assert bool((t[130:] == 7.0).all())
    a, n = 90, 40
    head_major = lambda x: to_f64(x[a:a + n].permute(1, 0, 2).unsqueeze(0))
    rq, rk, rv = orc.bwd(head_major(q), np.repeat(head_major(k), H, axis=1),
                         np.repeat(head_major(v), H, axis=1), head_major(do), causal=True)
    assert_abs_close(grads[0][a:a + n].cpu().numpy(), rq[0].transpose(1, 0, 2), GRAD_ABS, "dQ")
    assert_abs_close(grads[1][a:a + n].cpu().numpy(), rk.sum(axis=1)[:, None][0].transpose(1, 0, 2),
                     GRAD_ABS, "dK")
    bad = torch.tensor([0, 100, 90], dtype=torch.int32, device=DEV)
    fa.backward_varlen(qd, kd, vd, o, lse, dod, bad, 100)
    assert fa.fa_device_status(None) == FA_ERR_BAD_INDEX
    fa.backward_varlen(qd, kd, vd, o, lse, dod, cud, 64)  # first sequence is longer than 64
    assert fa.fa_device_status(None) == FA_ERR_BAD_INDEX
    fa.backward_varlen(qd, kd, vd, o, lse, dod, cud, 90)
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == 0
    assert T == 160
