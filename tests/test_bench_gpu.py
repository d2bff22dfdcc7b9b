"""The benchmark's output contract on the GPU: a short `bench.py` run prints one JSON
line with the keys and units the measurement plan fixes, consistent with each
other (value from ms_per_step and the FLOP convention, the roofline fraction from
achieved and peak, the launch count from the steps), and the single-forward mode
prints its own line."""
import json
import os
import subprocess
import sys

import pytest

from gpu_common import require_gpu

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    require_gpu()
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def test_bench_line_keeps_the_contract():
    steps = 6
    r = _run("--steps", str(steps), "--warmup", "3", "--no-extra", "--cpu-seconds", "1")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in r, key
    assert r["n_gpus"] == 1 and r["steps"] == steps and r["warmup"] == 3
    assert r["higher_is_better"] is True and r["scaling"] == "weak"
    assert r["unit"] == "TFLOPS" and r["dtype"] == "bf16" and r["vs_baseline"] is None
    assert "workload" in r["config"]
    B, H, N, d = (r["config"][k] for k in ("B", "H", "N", "d"))
    flops = (4.0 + 10.0) * B * H * N * N * d * (0.5 if r["config"]["causal"] else 1.0)
    assert r["value"] == pytest.approx(flops / (r["ms_per_step"] * 1e-3) / 1e12, rel=1e-3)
    rl = r["roofline"]
    assert rl["bound"] == "tensor" and rl["unit"] == "TFLOP/s"
    assert rl["frac"] == pytest.approx(rl["achieved"] / rl["peak"], abs=1e-3)
    assert 0.05 < rl["frac"] < 1.5
    assert rl["peak_clock_derived"] > rl["peak"] * 0.9
    e2e = r["e2e"]
    assert e2e["unit"] == "TFLOPS" and 0 < e2e["value"] < r["value"]
    assert e2e["h2d_bytes_per_step"] == 4 * B * H * N * d * 2
    assert e2e["d2h_bytes_per_step"] == B * H * N * (d * 2 + 4 + 3 * d * 4)
    assert r["gpu_launches"] == 3 * steps
    assert r["clocks"]["sm_mhz"] is None or r["clocks"]["sm_mhz"] > 0
    # the line ends with the target configurations, checked against the oracle
    assert list(r)[-1] == "targets"
    t = r["targets"]
    for name in ("C1_B1H1N128d64", "C2_B8H16N2048d64", "C3_B1H16N16384d128", "C4_B4H8N8192d256",
                 "C5_B2H16N4096d128_causal"):
        assert name in t, name
    assert t["parity"]["ok"] is True
    c5 = t["C5_B2H16N4096d128_causal"]
    assert len(c5["err"]) == 5 and max(c5["err"][2:]) <= 2e-2
    assert c5["bwd"]["tflops"] == pytest.approx(r["bwd_tflops"], rel=2e-3)
    assert t["fwd_N16384_d128"]["frac"] == t["C3_B1H16N16384d128"]["frac"]
    assert r["cpu_baseline"]["cores"] >= 1


def test_single_forward_mode():
    r = _run("--only-forward", "1", "2", "1000", "128", "1", "--steps", "3", "--warmup", "3")
    assert r["only_forward"]["N"] == 1000 and r["only_forward"]["causal"] is True
    assert r["ms"] > 0 and r["tflops"] > 0


def test_single_backward_mode():
    r = _run("--only-backward", "1", "2", "1000", "64", "1", "--steps", "3", "--warmup", "3")
    assert r["only_backward"]["N"] == 1000 and r["only_backward"]["d"] == 64
    assert r["ms"] > 0 and r["tflops"] > 0


def test_single_decode_mode():
    r = _run("--only-decode", "1", "8", "2", "1", "3000", "128", "--steps", "3", "--warmup", "3")
    assert r["only_decode"]["Hkv"] == 2 and r["kernel"] == "tcgen05"
    assert r["ms"] > 0 and r["GB/s"] > 0 and r["splits"] >= 1
