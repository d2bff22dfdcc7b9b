"""The e4m3 quantiser of the oracle against its pins, and planted mistakes in copies
of it, each of which must fail at least one pin.  CPU only."""
import importlib.util
import os

import pytest

import fp8_pins as pins
from oracle import fp8

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "fp8.py")


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(check):
    check(fp8)


MUTANTS = {
    "ties_away_from_zero": ("n = np.rint(a / quantum)", "n = np.floor(a / quantum + 0.5)"),
    "exponent_bias_8": ("np.exp2((ex - 7).astype", "np.exp2((ex - 8).astype"),
    "subnormal_floor_off_by_one": ("_MIN_EXP = -6", "_MIN_EXP = -7"),
    "no_saturation": ("v = np.minimum(n * quantum, E4M3_MAX)", "v = n * quantum"),
    "one_scale_per_head": ("amax = np.max(np.abs(blk), axis=(-2, -1))",
                           "amax = np.max(np.abs(x32), axis=(-2, -1))"),
    "descale_inverted": ("np.where(zero, np.float32(1), amax / f448)",
                         "np.where(zero, np.float32(1), f448 / amax)"),
    "hadamard_rows_swapped": ("np.block([[h, h], [h, -h]])", "np.block([[h, h], [-h, h]])"),
    "incoherent_not_normalised": ("@ hadamard(d) / np.sqrt(d)", "@ hadamard(d)"),
    "transpose_reshaped": ("out[..., :, :N] = np.swapaxes(codes, -1, -2)",
                           "out[..., :, :N] = codes.reshape(*lead, d, N)"),
    "sign_dropped": ("code = np.where(neg, code | 0x80, code)", "code = code"),
    "mantissa_truncated": ("n = np.rint(a / quantum)", "n = np.floor(a / quantum)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    with open(SRC) as fh:
        src = fh.read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"snippet for {name} no longer matches oracle/fp8.py exactly once"
    path = tmp_path / f"fp8_{name}.py"
    path.write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location(f"fp8_{name}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    failures = []
    for check in pins.ALL_CHECKS:
        try:
            check(mod)
        except (AssertionError, ValueError) as e:
            failures.append(f"{check.__name__}: {e}")
    assert failures, f"mutant {name} passed every pin"
