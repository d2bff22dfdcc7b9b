"""The benchmark's multi-rank bookkeeping on two gloo processes (CPU): the job's
time is the slowest rank's, its throughput counts every rank's copy of the step,
and the reference arm prints from rank 0 only."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [0.8, 1.25][rank]
        step_ms = bench.max_over_ranks(local_ms, world, "cpu")
        # only rank 1 saw a thermal slowdown: both ranks must time the region again
        clocks = [{"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []},
                  {"sm_mhz": 1900.0, "sm_max_mhz": 2070.0, "reasons": ["hw_thermal_slowdown"]}]
        again = bench.max_over_ranks(1.0 if bench.clocks_rejected(clocks[rank]) else 0.0, world,
                                     "cpu") > 0
        out[rank] = (step_ms, bench.job_tflops(1e12, world, step_ms), again)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        step_ms, tf, again = res[rank]
        assert step_ms == 1.25
        assert tf == pytest.approx(2 * 1e12 / 1.25e-3 / 1e12)
        assert again


def test_clock_records_that_disqualify_a_timed_region():
    sys.path.insert(0, ROOT)
    import bench
    ok = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    assert not bench.clocks_rejected(ok)
    assert not bench.clocks_rejected(dict(ok, sm_mhz=1800.0, reasons=["sw_power_cap"]))
    for why in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert bench.clocks_rejected(dict(ok, reasons=[why]))
    assert bench.clocks_rejected(dict(ok, sm_mhz=1400.0))  # stuck low, no reason: a lock
    assert not bench.clocks_rejected({"sm_mhz": None, "sm_max_mhz": None,
                                      "reasons": ["nvidia-smi unavailable"]})


def test_single_rank_passes_values_through():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.7, 1, "cpu") == 0.7
    assert bench.job_tflops(2e12, 1, 1.0) == pytest.approx(2000.0)


def test_reference_arm_prints_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setattr(bench, "run_reference", lambda args: {"impl": "reference", "value": 1.0})
    for rank, expect in (("1", ""), ("0", "reference")):
        monkeypatch.setenv("RANK", rank)
        monkeypatch.setenv("WORLD_SIZE", "2")
        monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2"])
        buf = io.StringIO()
        with redirect_stdout(buf):
            bench.main()
        text = buf.getvalue().strip()
        if expect:
            assert json.loads(text)["impl"] == "reference"
        else:
            assert text == ""
