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
* ``decode_qkv``: decode shapes, q [B, H, Nq, d] and a key/value cache k, v
  [B, H, Nk, d], i.i.d. N(0, 1) * ``mult`` drawn in the order q, k, v from one
  generator seeded with ``seed`` on ``device`` (the cache of the long-context
  workload is drawn on the GPU; a test copies the heads it checks back to the
  host for the oracle), rounded to bf16.  With ``boost`` > 0, a second generator
  (``seed + 1``) picks one key per block of ``boost_block`` keys of every head and
  adds ``boost`` to that K row, so some key ranges dominate others.

* ``gqa_qkv``: grouped-query shapes, q (and dO) [B, H, N, d] and k, v [B, Hkv, N, d],
  i.i.d. N(0, 1) drawn in the order q, k, v, dO from one CPU generator seeded with
  ``seed``, rounded to bf16.
* ``varlen_qkv``: packed sequences of the given lengths, token-major q [T, H, d] and
  k, v [T, Hkv, d] (T = sum of the lengths), i.i.d. N(0, 1) drawn in the order q,
  k, v from one CPU generator seeded with ``seed``, rounded to bf16; plus
  cu_seqlens, the int32 prefix sums [0, l0, l0 + l1, ...].
* ``outlier_qkv``: q [B, H, N, d], k, v [B, Hkv, N, d], i.i.d. N(0, 1) drawn in the
  order q, k, v from one generator seeded with ``seed``; with ``n_outliers`` > 0,
  a second generator (``seed + 1``) draws that many columns by ``torch.randperm``
  and those columns of q and k are multiplied by ``outlier_mult`` before the bf16
  rounding (outlier channels, the case incoherent processing is for).
* ``hadamard_signs``: d values +-1 from ``torch.randint`` (seed ``seed``), fp32.
* ``paged_cache``: rearranges a contiguous cache k, v [B, H, Nk, d] (Nk a multiple
  of ``page_size``) into pages [num_pages, H, page_size, d]: logical page p of
  sequence b goes to physical page perm[b * Nk / page_size + p], where perm is
  ``torch.randperm`` of the B * Nk / page_size pages from a generator seeded with
  ``seed``; returns the paged k, v and the int32 block table [B, Nk / page_size].

All tensors are contiguous bf16, on the CPU unless a device is given; callers
move them.
"""
from __future__ import annotations

import torch

__all__ = ["normal_qkv", "boosted_qkv", "decode_qkv", "gqa_qkv", "varlen_qkv", "outlier_qkv",
           "hadamard_signs", "paged_cache", "sample_rows", "to_f64"]


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


def decode_qkv(B: int, H: int, Nq: int, Nk: int, d: int, seed: int = 0, mult: float = 1.0,
               boost: float = 0.0, boost_block: int = 128, device: str = "cpu"):
    """Return (q [B,H,Nq,d], k [B,H,Nk,d], v [B,H,Nk,d]) bf16 on ``device``."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)

    def draw(shape):
        x = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
        if mult != 1.0:
            x = x * mult
        return x.to(torch.bfloat16).contiguous()

    q = draw((B, H, Nq, d))
    k = draw((B, H, Nk, d))
    v = draw((B, H, Nk, d))
    if boost > 0:
        g2 = torch.Generator(device=device)
        g2.manual_seed(seed + 1)
        nblk = (Nk + boost_block - 1) // boost_block
        lo = torch.arange(nblk, device=device) * boost_block
        width = torch.clamp(Nk - lo, max=boost_block)
        r = torch.randint(0, boost_block, (B, H, nblk), generator=g2, device=device)
        idx = lo + r % width
        kf = k.to(torch.float32)
        kf.scatter_add_(2, idx[..., None].expand(B, H, nblk, d),
                        torch.full((B, H, nblk, d), float(boost), device=device))
        k = kf.to(torch.bfloat16).contiguous()
    return q, k, v


def gqa_qkv(B: int, H: int, Hkv: int, N: int, d: int, seed: int = 0, with_do: bool = False):
    """Return (q, k, v) or (q, k, v, do): q, do [B,H,N,d] and k, v [B,Hkv,N,d] bf16."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    q = _draw(gen, (B, H, N, d))
    k = _draw(gen, (B, Hkv, N, d))
    v = _draw(gen, (B, Hkv, N, d))
    if with_do:
        return q, k, v, _draw(gen, (B, H, N, d))
    return q, k, v


def outlier_qkv(B: int, H: int, Hkv: int, N: int, d: int, seed: int = 0, n_outliers: int = 0,
                outlier_mult: float = 20.0):
    """Return (q [B,H,N,d], k, v [B,Hkv,N,d]) bf16, N(0,1) drawn q, k, v from one
    generator; with n_outliers > 0 a second generator (seed + 1) picks that many
    head-dimension columns, and those columns of q and k are multiplied by
    outlier_mult (before rounding to bf16)."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    q = torch.randn((B, H, N, d), generator=gen, dtype=torch.float32)
    k = torch.randn((B, Hkv, N, d), generator=gen, dtype=torch.float32)
    v = torch.randn((B, Hkv, N, d), generator=gen, dtype=torch.float32)
    if n_outliers > 0:
        g2 = torch.Generator(device="cpu")
        g2.manual_seed(seed + 1)
        cols = torch.randperm(d, generator=g2)[:n_outliers]
        q[..., cols] *= outlier_mult
        k[..., cols] *= outlier_mult
    return tuple(t.to(torch.bfloat16).contiguous() for t in (q, k, v))


def hadamard_signs(d: int, seed: int = 0) -> torch.Tensor:
    """fp32 [d] of +-1 drawn uniformly (the random signs of incoherent processing)."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    return (torch.randint(0, 2, (d,), generator=gen) * 2 - 1).to(torch.float32)


def varlen_qkv(lens, H: int, Hkv: int, d: int, seed: int = 0):
    """Return (q [T,H,d], k [T,Hkv,d], v [T,Hkv,d], cu_seqlens int32 [len(lens)+1])."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    T = int(sum(lens))
    q = _draw(gen, (T, H, d))
    k = _draw(gen, (T, Hkv, d))
    v = _draw(gen, (T, Hkv, d))
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    return q, k, v, cu


def paged_cache(k: torch.Tensor, v: torch.Tensor, page_size: int, seed: int = 3):
    """Return (k_cache, v_cache [num_pages, H, page_size, d], block_table int32 [B, P])."""
    B, H, Nk, d = k.shape
    if Nk % page_size:
        raise ValueError("Nk must be a multiple of page_size")
    P = Nk // page_size
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    perm = torch.randperm(B * P, generator=gen).to(k.device)

    def pages(x):
        xp = x.reshape(B, H, P, page_size, d).permute(0, 2, 1, 3, 4).reshape(B * P, H, page_size, d)
        out = torch.empty_like(xp)
        out[perm] = xp
        return out.contiguous()

    return pages(k), pages(v), perm.reshape(B, P).to(torch.int32).contiguous()


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
