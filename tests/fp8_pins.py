"""Checks that pin the e4m3 quantiser of ``oracle/fp8.py`` to facts fixed outside it.

Each ``check_*`` takes the module (or a deliberately broken copy of it) and raises
AssertionError on a mismatch.  Sources:

* The OCP 8-bit floating point specification's e4m3 definition: the value of every
  code follows from sign, exponent (bias 7) and mantissa; 448 is the largest
  finite value; 2^-9 the smallest subnormal; S.1111.111 is NaN.
* Round to nearest, ties to even, by brute force over the whole code table.
* Library routines as independent references: torch's float8_e4m3fn conversion
  (in-range values) and ``scipy.linalg.hadamard``.
* Closed forms of the block quantiser: each block's largest magnitude maps to
  +-448; the dequantisation error is at most half a quantum; power-of-two data
  on the e4m3 grid comes back exactly.
* Orthogonality: the incoherent transform leaves Q K^T unchanged.
"""
from __future__ import annotations

import numpy as np
import scipy.linalg
import torch


def _rng(seed):
    return np.random.default_rng(seed)


FINITE = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


def check_value_table(f):
    codes = np.array([0x00, 0x01, 0x07, 0x08, 0x38, 0x40, 0x7E, 0x80, 0x81, 0xFE], dtype=np.uint8)
    want = [0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 2.0, 448.0, -0.0, -(2.0 ** -9), -448.0]
    got = f.e4m3_value(codes)
    assert np.array_equal(got, want), f"value table {got} != {want}"
    assert np.isnan(f.e4m3_value(np.array([0x7F, 0xFF], dtype=np.uint8))).all(), "NaN codes"
    pos = f.e4m3_value(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0), "codes 0x00..0x7e must increase strictly"


def check_round_trip_of_every_code(f):
    vals = f.e4m3_value(FINITE)
    back = f.e4m3_round(vals)
    assert np.array_equal(back, FINITE), "e4m3_round(value(c)) != c"


def check_round_is_nearest_ties_even(f):
    """Brute force: the chosen code's value is the nearest; on a tie, the one with
    the even mantissa (even code)."""
    table = f.e4m3_value(np.arange(0x7F, dtype=np.uint8))  # non-negative finite values
    r = _rng(1)
    mids = (table[1:] + table[:-1]) / 2
    x = np.concatenate([mids, table, r.uniform(0, 448, 4000), np.exp2(r.uniform(-12, 8.8, 4000))])
    x = x[x <= 448].astype(np.float32).astype(np.float64)
    for sgn in (1.0, -1.0):
        codes = f.e4m3_round(sgn * x)
        got = np.abs(f.e4m3_value(codes))
        dist = np.abs(table[None, :] - x[:, None])
        best = dist.min(axis=1)
        assert np.all(np.abs(got - x) == best), "not the nearest value"
        tie = (dist == best[:, None]).sum(axis=1) == 2
        assert np.all((codes[tie] & 1) == 0), "ties must go to the even code"
        assert np.all(((codes & 0x80) != 0) == (sgn < 0)), "sign bit"


def check_round_matches_torch(f):
    """torch's float8_e4m3fn conversion on in-range values (a library reference)."""
    r = _rng(2)
    table = f.e4m3_value(FINITE)
    mids = (np.sort(table)[1:] + np.sort(table)[:-1]) / 2
    bf = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).float().numpy()
    bf = bf[np.isfinite(bf) & (np.abs(bf) <= 448)]
    x = np.concatenate([table, mids, r.normal(0, 30, 20000), np.exp2(r.uniform(-14, 8.8, 20000)), bf])
    x = x[np.abs(x) <= 448].astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = f.e4m3_round(x.astype(np.float64))
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"{bad.size} mismatches vs torch, e.g. x={x[bad[:3]]} ours={got[bad[:3]]} torch={ref[bad[:3]]}"


def check_saturation(f):
    x = np.array([448.0, 449.0, 463.9, 464.0, 470.0, 1e6, -500.0, -448.0])
    got = f.e4m3_round(x)
    want = np.array([0x7E] * 6 + [0xFE, 0xFE], dtype=np.uint8)
    assert np.array_equal(got, want), f"saturation {got}"


def check_hadamard(f):
    for d in (1, 2, 4, 8, 64, 128, 256):
        h = f.hadamard(d)
        assert np.array_equal(h, scipy.linalg.hadamard(d)), f"Hadamard d={d} vs scipy"
        assert np.array_equal(h @ h.T, d * np.eye(d)), f"H H^T != d I (d={d})"


def check_incoherent_preserves_scores(f):
    r = _rng(3)
    for d in (64, 128):
        q = r.normal(size=(5, 40, d)).astype(np.float32)
        k = r.normal(size=(5, 40, d)).astype(np.float32)
        k[:, :, 7] *= 30.0  # an outlier column
        s = r.choice([-1.0, 1.0], size=d)
        qi = f.incoherent(q, s).astype(np.float64)
        ki = f.incoherent(k, s).astype(np.float64)
        ref = np.einsum("hnd,hmd->hnm", q.astype(np.float64), k.astype(np.float64))
        got = np.einsum("hnd,hmd->hnm", qi, ki)
        scale = np.abs(q).max() * np.abs(k).max() * d
        assert np.max(np.abs(got - ref)) <= 1e-6 * scale, "scores changed by the transform"
        # the outlier column is spread: the transformed K has a much smaller peak
        assert np.abs(ki).max() < 0.5 * np.abs(k).max(), "outlier not spread"


def _block_data(seed, shape=(2, 3, 300, 64)):
    r = _rng(seed)
    x = r.normal(size=shape).astype(np.float32)
    x[..., 5, 3] = 9.5  # the largest magnitude of the first block of every head
    if shape[-2] > 200:
        x[..., 200, 1] = -17.25  # ... and of the second block
    return x


def check_block_scale_maps_amax_to_448(f):
    x = _block_data(4)
    codes, descale = f.quantize(x, block_rows=128)
    assert codes.shape == x.shape and descale.shape == (2, 3, 3)
    assert np.all(codes[..., 5, 3] == 0x7E) and np.all(codes[..., 200, 1] == 0xFE), "amax -> 448"
    for bi, (r0, r1) in enumerate([(0, 128), (128, 256), (256, 300)]):
        amax = np.abs(x[..., r0:r1, :]).max(axis=(-2, -1)).astype(np.float32)
        assert np.array_equal(descale[..., bi], amax / np.float32(448)), "descale = amax / 448"


def check_dequantize_error_bound(f):
    x = _block_data(5)
    for br in (128, 0, 50):
        codes, descale = f.quantize(x, block_rows=br)
        deq = f.dequantize(codes, descale, block_rows=br)
        blocks = [(r0, min(r0 + (br or 300), 300)) for r0 in range(0, 300, br or 300)]
        for bi, (r0, r1) in enumerate(blocks):
            ds = descale[..., bi].astype(np.float64)[..., None, None]
            xb = x[..., r0:r1, :].astype(np.float64)
            t = np.abs(xb) / ds
            half_q = np.maximum(t * 2.0 ** -4, 2.0 ** -10)  # half a quantum, normal / subnormal
            bound = ds * half_q * (1 + 1e-6) + np.abs(xb) * 2.0 ** -22
            assert np.all(np.abs(deq[..., r0:r1, :] - xb) <= bound), f"error bound, block_rows={br}"


def check_blocks_are_independent(f):
    x = _block_data(6)
    y = x.copy()
    y[..., 130:, :] *= 100.0  # change every block but the first
    cx, dx = f.quantize(x, block_rows=128)
    cy, dy = f.quantize(y, block_rows=128)
    assert np.array_equal(cx[..., :128, :], cy[..., :128, :]), "first block's codes changed"
    assert np.array_equal(dx[..., 0], dy[..., 0]), "first block's scale changed"


def check_exact_on_grid(f):
    """Data that are e4m3 values times 2^-3, with 56 (= 448 / 8) in every block:
    the scale is exactly 1/8 and the codes come back exactly."""
    r = _rng(7)
    codes = r.choice(FINITE, size=(2, 256, 32)).astype(np.uint8)
    codes[:, 0, 0] = 0x7E
    codes[:, 128, 5] = 0xFE
    x = (f.e4m3_value(codes) / 8.0).astype(np.float32)
    got, descale = f.quantize(x, block_rows=128)
    assert np.all(descale == np.float32(1 / 8)), "scale must be exactly 1/8"
    want = np.where(f.e4m3_value(codes) == 0, 0, codes)  # -0 keeps its sign bit either way
    assert np.array_equal(np.where(f.e4m3_value(got) == 0, 0, got), want), "codes not recovered"
    assert np.array_equal(f.dequantize(got, descale, 128), x.astype(np.float64)), "values not exact"


def check_transposed_layout(f):
    x = _block_data(8, shape=(2, 100, 64))
    plain, d1 = f.quantize(x, block_rows=0)
    tr, d2 = f.quantize(x, block_rows=0, transpose=True)
    assert tr.shape == (2, 64, 112), f"transposed shape {tr.shape}"
    assert np.array_equal(tr[..., :100], np.swapaxes(plain, -1, -2)), "transposed codes"
    assert np.all(tr[..., 100:] == 0), "padding must be zero"
    assert np.array_equal(d1, d2)
    assert np.array_equal(f.dequantize(tr, d2, 0, transposed=True, N=100), f.dequantize(plain, d1, 0))


def check_zero_block(f):
    x = np.zeros((1, 130, 16), dtype=np.float32)
    x[0, 129, 0] = 3.0
    codes, descale = f.quantize(x, block_rows=128)
    assert np.all(codes[0, :128] == 0) and descale[0, 0] == 1.0, "all-zero block"
    assert codes[0, 129, 0] == 0x7E and descale[0, 1] == np.float32(3.0) / np.float32(448)


ALL_CHECKS = [
    check_value_table, check_round_trip_of_every_code, check_round_is_nearest_ties_even,
    check_round_matches_torch, check_saturation, check_hadamard, check_incoherent_preserves_scores,
    check_block_scale_maps_amax_to_448, check_dequantize_error_bound, check_blocks_are_independent,
    check_exact_on_grid, check_transposed_layout, check_zero_block,
]
