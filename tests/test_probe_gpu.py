"""The unit-rate probes (fa_probe_unit_rates) on the GPU: one CTA per SM issuing
dense bf16 MMAs (M = 128, N = 256 and N = 64) or MUFU ex2, timed with clock64.

The checks are what the hardware fixes: an MMA of M x N x K = 128 x N x 16 is
2 * 128 * N * 16 FLOPs, so the per-SM rate is a positive multiple of nothing in
particular but cannot exceed the tensor core's datapath; the N = 64 shape cannot
beat the N = 256 one; and the measured rates times the SM count and clock must
bracket the measured cuBLAS GEMM peak from above (a GEMM cannot outrun its
tensor cores) without being absurdly far from it."""
import json
import os

import pytest
import torch

from gpu_common import load_fa

pytestmark = pytest.mark.gpu


def test_unit_rates_are_consistent():
    fa = load_fa()
    r = fa.probe_unit_rates(2048)
    assert fa.fa_device_status(None) == 0
    n256, n64, ex2 = (r["mma_bf16_n256_flop_per_clk"], r["mma_bf16_n64_flop_per_clk"],
                      r["ex2_per_clk"])
    print(f"per SM clock: MMA N=256 {n256:.0f} FLOP, N=64 {n64:.0f} FLOP, ex2 {ex2:.2f}")
    assert 1024 <= n256 <= 32768
    assert 0 < n64 <= n256 * 1.02
    assert 4 <= ex2 <= 256
    peaks = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                         "MEASURED_PEAKS.json")
    if os.path.exists(peaks):
        with open(peaks) as f:
            gemm = json.load(f).get("bf16_tflops")
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        # any SM clock the part runs at (1.0-2.2 GHz) must leave the GEMM below the
        # probe's rate at that clock's upper end
        if gemm:
            assert gemm <= n256 * sms * 2.2e9 / 1e12


def test_unit_rates_reject_bad_arguments():
    fa = load_fa()
    import ctypes
    rates = (ctypes.c_double * 3)()
    assert fa.fa_probe_unit_rates(rates, 8, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_probe_unit_rates(None, 2048, None) == fa.FA_ERR_INVALID_ARG


def test_read_bandwidth_probe():
    """The HBM read rate over a 2 GiB buffer (16x the L2): a plausible GB300 figure,
    and no slower than a device-to-device copy moves its read half."""
    fa = load_fa()
    x = torch.zeros(1 << 30, dtype=torch.bfloat16, device="cuda:0")
    gbs = fa.probe_read_bandwidth(x, iters=3)
    y = torch.empty_like(x)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    y.copy_(x)
    a.record()
    y.copy_(x)
    b.record()
    b.synchronize()
    copy_read_gbs = x.numel() * 2 / (a.elapsed_time(b) * 1e-3) / 1e9
    assert 1000.0 < gbs < 12000.0, gbs
    assert gbs > copy_read_gbs, (gbs, copy_read_gbs)
