"""Bounded waits: a wait that runs out reports FA_ERR_TIMEOUT and leaves the GPU usable.

The self-test kernel waits, with the same bounded wait the attention kernels use,
on a barrier nothing arrives on.  Nothing here faults, traps or hangs a GPU: the
wait gives up after its limit and the kernel returns.
"""
import time

import numpy as np
import pytest

FA_ERR_INVALID_ARG = 1
FA_ERR_TIMEOUT = 5


@pytest.fixture(scope="module")
def fa_lib():
    from exact_attention_26_gb300 import build as fb
    if fb.needs_build():
        fb.build()
    import exact_attention_26_gb300 as fa
    fa.load()
    return fa


def test_selftest_rejects_bad_limits(fa_lib):
    # checked on the host before anything touches CUDA
    assert fa_lib.fa.fa_selftest_wait_timeout(0, None) == FA_ERR_INVALID_ARG
    assert fa_lib.fa.fa_selftest_wait_timeout(10_000_000_000, None) == FA_ERR_INVALID_ARG


@pytest.mark.gpu
def test_wait_timeout_is_reported_and_context_survives(fa_lib):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_26_gb300.inputs import normal_qkv, to_f64
    from gpu_common import L_ABS, assert_abs_close, assert_o_close
    from oracle import Oracle

    fa = fa_lib
    assert fa.fa_device_status(None) == 0
    limit_ns = 20_000_000  # 20 ms
    t0 = time.perf_counter()
    assert fa.fa.fa_selftest_wait_timeout(limit_ns, None) == 0
    status = fa.fa_device_status(None)  # synchronises
    elapsed = time.perf_counter() - t0
    assert status == FA_ERR_TIMEOUT
    assert elapsed >= 0.9 * limit_ns * 1e-9
    assert fa.fa_device_status(None) == 0  # the record is cleared once read

    # the context still runs the real kernels correctly
    q, k, v = normal_qkv(1, 2, 300, 128, seed=31)
    o, lse = fa.forward(q.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    assert fa.fa_device_status(None) == 0
    ro, rl = Oracle().fwd(to_f64(q), to_f64(k), to_f64(v), causal=True)
    assert_o_close(o.float().cpu().numpy(), ro, "after timeout")
    assert_abs_close(lse.cpu().numpy(), rl, L_ABS, "after timeout L")
