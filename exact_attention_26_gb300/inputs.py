"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module only draws random numbers and arranges them into tensors; it holds
none of the attention arithmetic, so neither side can inherit a mistake from the
other through it.

Recipes (one per workload of the measurement plan):

* ``normal_qkv``: Q, K, V (and optionally dO) are i.i.d. N(0, 1) drawn in fp32
  from one CPU ``torch.Generator`` seeded with ``seed`` in the order Q, K, V, dO,
  then rounded to bf16 (round-to-nearest-even, torch's ``.to(torch.bfloat16)``).
* ``boosted_qkv``: Q, K, V = bf16(0.5 * N(0, 1)) as above; then, from a second
  generator seeded with ``seed + 1``, for every (b, h) and every consecutive
  block of ``boost_block`` keys one key index is drawn uniformly and ``boost`` is
  added to every element of that K row (re-rounded to bf16).  The boosted keys
  raise the running row maximum at irregular points, so the online-softmax
  rescale path is exercised.
* ``sample_rows``: rows {0, N-1} plus distinct rows drawn by ``torch.randperm``
  from a generator seeded with ``seed``, sorted, ``count`` in total.

All tensors are contiguous ``[B, H, N, d]`` bf16 on the CPU; callers move them.
"""
from __future__ import annotations

import torch

__all__ = ["normal_qkv", "boosted_qkv", "sample_rows", "to_f64"]


def _draw(gen: torch.Generator, shape, mult: float = 1.0) -> torch.Tensor:
    x = torch.randn(shape, generator=gen, dtype=torch.float32)
    if mult != 1.0:
        x = x * mult
    return x.to(torch.bfloat16).contiguous()


def normal_qkv(B: int, H: int, N: int, d: int, seed: int = 0, with_do: bool = False,
               mult: float = 1.0):
    """Return (q, k, v) or (q, k, v, do): bf16 [B,H,N,d], N(0,1)*mult, one generator."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    shape = (B, H, N, d)
    q = _draw(gen, shape, mult)
    k = _draw(gen, shape, mult)
    v = _draw(gen, shape, mult)
    if with_do:
        do = _draw(gen, shape, mult)
        return q, k, v, do
    return q, k, v


def boosted_qkv(B: int, H: int, N: int, d: int, seed: int = 0, mult: float = 0.5,
                boost: float = 4.0, boost_block: int = 128):
    """Q/K/V = bf16(mult*N(0,1)); one key per block of ``boost_block`` keys gets +boost."""
    q, k, v = normal_qkv(B, H, N, d, seed=seed, mult=mult)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed + 1)
    nblk = (N + boost_block - 1) // boost_block
    kf = k.to(torch.float32)
    for b in range(B):
        for h in range(H):
            for blk in range(nblk):
                lo = blk * boost_block
                width = min(boost_block, N - lo)
                j = lo + int(torch.randint(0, width, (1,), generator=gen).item())
                kf[b, h, j, :] += boost
    return q, kf.to(torch.bfloat16).contiguous(), v


def sample_rows(N: int, count: int, seed: int = 2) -> torch.Tensor:
    """Sorted int64 row indices: {0, N-1} plus distinct seeded rows, ``count`` total."""
    count = min(count, N)
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    chosen = {0, N - 1}
    for r in torch.randperm(N, generator=gen).tolist():
        if len(chosen) >= count:
            break
        chosen.add(r)
    return torch.tensor(sorted(chosen), dtype=torch.int64)


def to_f64(t: torch.Tensor):
    """Exact upcast of a bf16 CPU tensor to a contiguous float64 numpy array."""
    return t.detach().to("cpu").to(torch.float64).contiguous().numpy()
