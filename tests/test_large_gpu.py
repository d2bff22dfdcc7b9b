"""Tensors past 2^31 elements: forward and backward on B1 H1040 N16384 d128 causal,
where q, k, v, o, dO hold 2.18e9 elements each (4.4 GB bf16; dQ, dK, dV 8.7 GB fp32),
so every element offset of the last heads exceeds the int32 range.

The inputs are drawn on the GPU by the seeded generator of the inputs module (q, k,
v from one draw, dO from a second with its own seed); only the heads the oracle
checks are copied to the host.  In the last head (element offsets from 2.18e9) the
oracle checks O and L on sampled rows, dQ on those rows, and dK and dV of the last
128 keys, which with the causal mask receive gradient only from the last 128
queries; the first head is checked the same way as a control."""
import numpy as np
import pytest
import torch

from exact_attention_26_gb300.inputs import decode_qkv, sample_rows
from gpu_common import GRAD_ABS, L_ABS, assert_abs_close, assert_o_close, load_fa
from oracle import Oracle

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def test_fwd_bwd_beyond_2_31_elements():
    fa = load_fa()
    orc = Oracle()
    B, H, N, d = 1, 1040, 16384, 128
    assert B * H * N * d > 2 ** 31
    q, k, v = decode_qkv(B, H, N, N, d, seed=31, device=DEV)
    do = decode_qkv(B, H, N, 1, d, seed=32, device=DEV)[0]
    o, lse = fa.forward(q, k, v, causal=True)
    dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == 0

    tail = np.arange(N - 128, N)
    rows = np.unique(np.concatenate([sample_rows(N, 24, seed=5).numpy(), tail]))
    ridx = torch.from_numpy(rows).to(DEV)

    def host(t, h, idx=None):  # head h of a device tensor (rows idx) as float64 numpy
        t = t[:, h:h + 1]
        if idx is not None:
            t = t.index_select(2, idx)
        return t.to(torch.float64).cpu().numpy()

    for h in (H - 1, 0):
        assert (h * N * d > 2 ** 31) == (h == H - 1)
        qh, kh, vh, doh = (host(t, h) for t in (q, k, v, do))
        ro, rl = orc.fwd_rows(qh, kh, vh, rows, causal=True)
        assert_o_close(host(o, h, ridx), ro, f"head {h} O")
        assert_abs_close(host(lse.unsqueeze(-1), h, ridx)[..., 0], rl, L_ABS, f"head {h} L")
        rq, rk, rv = orc.bwd_rows(qh, kh, vh, doh, rows, causal=True)
        assert_abs_close(host(dq, h, ridx), rq, GRAD_ABS, f"head {h} dQ rows")
        tidx = torch.from_numpy(tail).to(DEV)
        assert_abs_close(host(dk, h, tidx), rk[:, :, tail], GRAD_ABS, f"head {h} dK last keys")
        assert_abs_close(host(dv, h, tidx), rv[:, :, tail], GRAD_ABS, f"head {h} dV last keys")
    del q, k, v, do, o, lse, dq, dk, dv
    torch.cuda.empty_cache()
