"""Paged decode on the GPU: fa_decode_paged (block-table gather, per-sequence
lengths, split key ranges, LSE merge) against the float64 oracle's decode rows of
each sequence's own keys.

The cache is written contiguously first and then scattered into randomly
permuted pages (``inputs.paged_cache``), so the test's gather (plain slicing of
the contiguous copy) is independent of the kernel's (block-table lookups).
Device-side index checks are exercised with out-of-range table entries and
lengths, which the kernel rejects before reading anything.
"""
import numpy as np
import pytest
import torch

from exact_attention_26_gb300.inputs import decode_qkv, paged_cache, to_f64
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


def _lens(B, nk_max, seed):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    lens = torch.randint(1, nk_max + 1, (B,), generator=g)
    lens[0] = nk_max  # one full-length sequence
    return lens.to(torch.int32)


def _check(fa, orc, q, k, v, lens, page_size, splits, what):
    kc, vc, bt = paged_cache(k, v, page_size)
    o, lse = fa.decode_paged(q.to(DEV), kc.to(DEV), vc.to(DEV), bt.to(DEV), lens.to(DEV),
                             num_splits=splits)
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == 0
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    for b in range(q.shape[0]):
        n = int(lens[b])
        ro, rl = orc.decode(to_f64(q[b:b + 1]), to_f64(k[b:b + 1, :, :n]), to_f64(v[b:b + 1, :, :n]))
        assert_o_close(o[b:b + 1], ro, f"{what} seq {b} (len {n})")
        assert_abs_close(lse[b:b + 1], rl, L_ABS, f"{what} seq {b} L")


# (B, H, Nq, pages per sequence, page_size, d, requested key ranges)
SMALL = [
    (3, 2, 1, 8, 16, 128, 0), (2, 1, 1, 5, 64, 64, 3), (4, 2, 3, 6, 16, 256, 0),
    (2, 2, 1, 30, 7, 128, 4), (1, 3, 1, 2, 256, 128, 2), (5, 1, 2, 40, 16, 64, 0),
    (2, 2, 9, 12, 32, 128, 1), (3, 1, 1, 64, 1, 128, 0), (2, 2, 1, 10, 16, 96, 0),
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s)))
def test_decode_paged_small(fa, orc, shape):
    B, H, Nq, P, ps, d, splits = shape
    nk_max = P * ps
    q, k, v = decode_qkv(B, H, Nq, nk_max, d, seed=nk_max + d)
    _check(fa, orc, q, k, v, _lens(B, nk_max, seed=B + P), ps, splits, f"{shape}")


def test_decode_paged_matches_contiguous(fa):
    """Identity table and full lengths: the same keys in the same ranges, so the
    result equals fa_decode's bit for bit."""
    B, H, Nq, Nk, d, ps = 2, 4, 1, 4096, 128, 64
    q, k, v = (t.to(DEV) for t in decode_qkv(B, H, Nq, Nk, d, seed=4))
    P = Nk // ps
    kc = k.reshape(B, H, P, ps, d).permute(0, 2, 1, 3, 4).reshape(B * P, H, ps, d).contiguous()
    vc = v.reshape(B, H, P, ps, d).permute(0, 2, 1, 3, 4).reshape(B * P, H, ps, d).contiguous()
    bt = torch.arange(B * P, dtype=torch.int32, device=DEV).reshape(B, P)
    lens = torch.full((B,), Nk, dtype=torch.int32, device=DEV)
    for splits in (1, 5):
        o1, l1 = fa.decode(q, k, v, num_splits=splits)
        o2, l2 = fa.decode_paged(q, kc, vc, bt, lens, num_splits=splits)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2), f"splits={splits}"


def test_decode_paged_bad_indices_are_reported(fa, orc):
    """A table entry past the pool, and lengths of 0 and past the table, are caught
    on the device before any access: FA_ERR_BAD_INDEX, then the context still works."""
    B, H, Nq, P, ps, d = 2, 2, 1, 4, 16, 128
    q, k, v = decode_qkv(B, H, Nq, P * ps, d, seed=8)
    kc, vc, bt = (t.to(DEV) for t in paged_cache(k, v, ps))
    qd = q.to(DEV)
    lens = torch.full((B,), P * ps, dtype=torch.int32, device=DEV)
    bad_bt = bt.clone()
    bad_bt[1, 2] = kc.shape[0]  # one past the last physical page
    assert fa.fa_device_status(None) == 0
    fa.decode_paged(qd, kc, vc, bad_bt, lens, num_splits=1)
    assert fa.fa_device_status(None) == FA_ERR_BAD_INDEX
    assert fa.fa_device_status(None) == 0
    for bad_len in (0, P * ps + 1):
        bl = lens.clone()
        bl[0] = bad_len
        fa.decode_paged(qd, kc, vc, bt, bl, num_splits=2)
        assert fa.fa_device_status(None) == FA_ERR_BAD_INDEX
    # the context is intact and the same call with good indices is correct
    lens_h = lens.cpu()
    _check(fa, orc, q, k, v, lens_h, ps, 2, "after bad indices")


def test_decode_paged_long_context_workload(fa, orc):
    """B=8, H=32, one query row, 32768-token sequences in 16-token pages scattered
    at random over the pool, automatic key ranges; eight heads checked."""
    B, H, Nk, d, ps = 8, 32, 32768, 128, 16
    q, k, v = decode_qkv(B, H, 1, Nk, d, seed=0, device=DEV)
    kc, vc, bt = paged_cache(k, v, ps)
    lens = torch.full((B,), Nk, dtype=torch.int32, device=DEV)
    lens[3] = 20000
    o, lse = fa.decode_paged(q, kc, vc, bt, lens)
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == 0
    for b, h in [(0, 0), (1, 5), (3, 9), (3, 31), (5, 17), (7, 30)]:
        n = int(lens[b])
        ro, rl = orc.decode(to_f64(q[b:b + 1, h:h + 1].cpu()), to_f64(k[b:b + 1, h:h + 1, :n].cpu()),
                            to_f64(v[b:b + 1, h:h + 1, :n].cpu()))
        assert_o_close(o[b:b + 1, h:h + 1].float().cpu().numpy(), ro, f"head ({b},{h})")
        assert_abs_close(lse[b:b + 1, h:h + 1].cpu().numpy(), rl, L_ABS, f"head ({b},{h}) L")
