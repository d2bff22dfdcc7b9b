"""FP8 (e4m3) quantisation for the low-precision forward: the plain CPU statement.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU legs use this module; the CUDA library never does.  numpy, no GPU.

What the pages fix and what they leave open
-------------------------------------------
"FlashAttention: Move Less, Not Compute Less", section "FA1 to FA3: Optimization
Moves Closer to the Hardware", and the course page "10 FlashAttention", section
"FlashAttention-1 -> 2 -> 3", say only that the Hopper generation runs attention in
FP8, with block quantisation and "incoherent processing" to contain the error that
outliers cause.  Neither gives the format, the block shape or the transform, so
this module takes the plainest readings:

* FP8 is e4m3 as the OCP 8-bit floating point specification defines it (the "fn"
  variant: sign, 4 exponent bits with bias 7, 3 mantissa bits, no infinities, the
  all-ones pattern is NaN; largest finite value 448).  Conversion rounds to
  nearest, ties to even, and saturates finite values beyond +-448 to +-448.
* Block quantisation: each block of `block_rows` consecutive rows of one head
  (all d columns) gets its own scale, chosen so that the block's largest
  magnitude maps to 448.  The arithmetic is fp32 and fixed step by step, because
  the codes are integers that both sides must agree on: amax = max |x|,
  inv = 448 / amax, t = x * inv (each one IEEE fp32 operation, round to nearest),
  code = e4m3(t), descale = amax / 448.  A block of zeros takes inv = descale = 1.
  The dequantised value of a code is value(code) * descale.
* Incoherent processing: before quantisation each row of Q and of K is multiplied
  by M = diag(signs) H / sqrt(d), H the d x d Sylvester-Hadamard matrix and signs
  a vector of +-1 drawn by the caller.  M is orthogonal, so (Q M)(K M)^T = Q K^T:
  the scores are unchanged while an outlier column is spread over every column.
* The value tensor is stored transposed per head ([d][N rounded up to 16]), the
  layout the tensor-core product P V reads with keys contiguous.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
_MIN_EXP = -6  # exponent of the smallest normal number, 2^-6


def e4m3_value(codes) -> np.ndarray:
    """Value of each e4m3 code (uint8) as float64, from the format definition."""
    c = np.asarray(codes).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    ex = (c >> 3) & 0xF
    man = (c & 0x7).astype(np.float64)
    normal = (1.0 + man / 8.0) * np.exp2((ex - 7).astype(np.float64))
    sub = (man / 8.0) * 2.0 ** _MIN_EXP
    val = np.where(ex == 0, sub, normal)
    val = np.where((ex == 15) & (c & 0x7 == 7), np.nan, val)
    return sign * val


def e4m3_round(x) -> np.ndarray:
    """Round finite values to e4m3 codes: nearest, ties to even, saturating at 448."""
    x = np.asarray(x, dtype=np.float64)
    if not np.all(np.isfinite(x)):
        raise ValueError("e4m3_round takes finite values")
    neg = np.signbit(x)
    a = np.abs(x)
    # binade exponent e with 2^e <= a < 2^(e+1), floored at the subnormal range
    _, E = np.frexp(np.where(a > 0, a, 1.0))
    e = np.maximum(E - 1, _MIN_EXP)
    quantum = np.exp2((e - 3).astype(np.float64))  # 3 mantissa bits
    n = np.rint(a / quantum)                        # a / quantum is exact; rint ties to even
    v = np.minimum(n * quantum, E4M3_MAX)           # a carry may reach the next binade
    # encode v >= 0
    _, Ev = np.frexp(np.where(v > 0, v, 1.0))
    ev = Ev - 1
    is_sub = v < 2.0 ** _MIN_EXP
    exp_field = np.where(is_sub, 0, ev + 7)
    man_field = np.where(is_sub, np.rint(v / 2.0 ** (_MIN_EXP - 3)),
                         np.rint(v / np.exp2((ev - 3).astype(np.float64))) - 8)
    code = (exp_field.astype(np.int64) << 3) | man_field.astype(np.int64)
    code = np.where(neg, code | 0x80, code)
    return code.astype(np.uint8)


def hadamard(d: int) -> np.ndarray:
    """Sylvester construction: H_1 = [1], H_2n = [[H, H], [H, -H]]."""
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h


def incoherent(x, signs) -> np.ndarray:
    """Rows of x times diag(signs) H / sqrt(d), exact in float64, then rounded to fp32
    (the values the quantiser sees)."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    s = np.asarray(signs, dtype=np.float64).reshape(d)
    if not np.all(np.abs(s) == 1.0):
        raise ValueError("signs must be +-1")
    y = (x * s) @ hadamard(d) / np.sqrt(d)
    return y.astype(np.float32)


def _blocks(N: int, block_rows: int):
    R = N if block_rows <= 0 else block_rows
    return [(r0, min(r0 + R, N)) for r0 in range(0, N, R)]


def quantize(x, block_rows: int = 128, signs=None, transpose: bool = False):
    """Quantise [..., N, d] (fp32-representable values, e.g. bf16 upcast) to e4m3.

    Returns (codes, descale): codes uint8 [..., N, d], or [..., d, round_up(N, 16)]
    with zero padding when `transpose`; descale fp32 [..., n_blocks] with one entry
    per block of `block_rows` rows (block_rows <= 0: one block per head)."""
    x32 = incoherent(x, signs) if signs is not None else np.asarray(x, dtype=np.float32)
    *lead, N, d = x32.shape
    blocks = _blocks(N, block_rows)
    codes = np.zeros(x32.shape, dtype=np.uint8)
    descale = np.zeros((*lead, len(blocks)), dtype=np.float32)
    f448 = np.float32(E4M3_MAX)
    for bi, (r0, r1) in enumerate(blocks):
        blk = x32[..., r0:r1, :]
        amax = np.max(np.abs(blk), axis=(-2, -1)).astype(np.float32)
        zero = amax == 0
        inv = np.where(zero, np.float32(1), f448 / np.where(zero, np.float32(1), amax))
        descale[..., bi] = np.where(zero, np.float32(1), amax / f448)
        t = (blk * inv.astype(np.float32)[..., None, None]).astype(np.float32)
        codes[..., r0:r1, :] = e4m3_round(t.astype(np.float64))
    if transpose:
        Np = (N + 15) // 16 * 16
        out = np.zeros((*lead, d, Np), dtype=np.uint8)
        out[..., :, :N] = np.swapaxes(codes, -1, -2)
        codes = out
    return codes, descale


def dequantize(codes, descale, block_rows: int = 128, transposed: bool = False, N=None):
    """float64 [..., N, d] values of quantised data: value(code) * descale of its block."""
    codes = np.asarray(codes)
    if transposed:
        if N is None:
            raise ValueError("N is needed for a transposed tensor")
        codes = np.swapaxes(codes[..., :N], -1, -2)
    N = codes.shape[-2]
    out = e4m3_value(codes)
    descale = np.asarray(descale, dtype=np.float64)
    for bi, (r0, r1) in enumerate(_blocks(N, block_rows)):
        out[..., r0:r1, :] *= descale[..., bi][..., None, None]
    return out
