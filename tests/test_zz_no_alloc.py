"""fa_bwd_noalloc: the backward entry point for callers that cannot allocate.

It must give the oracle's gradients within the tolerance, the same dK and dV bits
as fa_bwd with a caller workspace (dQ within the tolerance: its partial sums arrive
in a varying order), on two calls in a row that share the library's scratch array,
and refuse sizes that do not fit that array.  This file is collected last on
purpose.
"""
import ctypes

import numpy as np
import pytest

from gpu_common import GRAD_ABS

DEV = "cuda:0"
FA_ERR_WORKSPACE = 6


def _lib():
    from exact_attention_26_gb300 import build as fb
    if fb.needs_build():
        fb.build()
    lib = ctypes.CDLL(fb.LIB)
    vp, i = ctypes.c_void_p, ctypes.c_int
    lib.fa_bwd_noalloc.argtypes = [vp] * 9 + [i] * 5 + [ctypes.c_float, vp]
    lib.fa_bwd_noalloc.restype = i
    return lib


def _call(lib, q, k, v, o, lse, do, dq, dk, dv, causal, scale, stream):
    B, H, N, d = q.shape
    return lib.fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                              lse.data_ptr(), do.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                              dv.data_ptr(), B, H, N, d, int(causal), scale, stream)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = _lib()
    ptr = 0x10000  # never dereferenced: the size check comes first
    # B*H*roundup(N,128) = 8 * 16 * 16384 = 2,097,152 rows > 1,048,576
    rc = lib.fa_bwd_noalloc(*([ptr] * 9), 8, 16, 16384, 128, 1, 0.088, None)
    assert rc == FA_ERR_WORKSPACE
    # one 128-row block past the limit
    rc = lib.fa_bwd_noalloc(*([ptr] * 9), 1, 1, 1048576 + 128, 128, 1, 0.088, None)
    assert rc == FA_ERR_WORKSPACE


@pytest.mark.gpu
def test_noalloc_matches_fa_bwd_on_two_calls():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_26_gb300 as fa
    from exact_attention_26_gb300.inputs import normal_qkv

    from exact_attention_26_gb300.inputs import to_f64
    from oracle import Oracle

    lib = _lib()
    orc = Oracle()
    # the larger case first, so the second case runs on scratch that still holds the
    # first one's vectors in rows it does not own
    cases = [((2, 4, 1000, 128), True), ((1, 3, 777, 64), False)]
    for (B, H, N, d), causal in cases:
        qh, kh, vh, doh = normal_qkv(B, H, N, d, seed=N + d, with_do=True)
        q, k, v, do = (t.to(DEV) for t in (qh, kh, vh, doh))
        scale = 1.0 / np.sqrt(d)
        o, lse = fa.forward(q, k, v, causal=causal)
        ws_path = [t.cpu().numpy() for t in fa.backward(q, k, v, o, lse, do, causal=causal)]
        oracle = orc.bwd(to_f64(qh), to_f64(kh), to_f64(vh), to_f64(doh), causal=causal)
        stream = torch.cuda.current_stream().cuda_stream
        for _ in range(2):  # two calls in a row share the scratch array
            out = [torch.full(q.shape, float("nan"), dtype=torch.float32, device=DEV)
                   for _ in range(3)]
            rc = _call(lib, q, k, v, o, lse, do, *out, causal, scale, stream)
            assert rc == 0, rc
            torch.cuda.synchronize()
            assert fa.fa_device_status(None) == 0
            for name, g, w, r in zip(("dQ", "dK", "dV"), out, ws_path, oracle):
                g = g.cpu().numpy()
                assert np.all(np.isfinite(g)), name
                # against the float64 oracle, within the gradient tolerance
                err = float(np.max(np.abs(g - r)))
                assert err <= GRAD_ABS, (name, err)
                if name == "dQ":
                    # dQ's fp32 partial sums arrive in a varying order
                    assert float(np.max(np.abs(g - w))) <= GRAD_ABS, name
                else:
                    # dK and dV are summed on chip in a fixed order: the same bits as
                    # with a caller's workspace
                    assert np.array_equal(g, w), name
