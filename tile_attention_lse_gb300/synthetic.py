"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

Holds no attention arithmetic: only random draws, rounding to the input dtype
and the packed-length recipe.  Both the CUDA path and the oracle consume what
these functions return.

Recipe:
* Q, K, V and the upstream gradient dO are N(0, 1) float32 draws from
  ``torch.Generator().manual_seed(seed + offset)`` on the CPU, in original
  token order, rounded to bfloat16 (round-to-nearest-even) for bf16 runs.
  Offsets: q 0, k 1, v 2, dO 3 (times 7919 so nearby seeds do not overlap).
* Packed sub-sequence lengths: numpy ``default_rng(seed)``; draw
  len = clip(round(exp(N(7.5, 1.0))), 128, 16384), round up to a multiple of
  2*cp, append while the total is below T; the last length is cut to the
  remainder, and a remainder below 128 is merged into the previous length.
"""

from __future__ import annotations

import numpy as np
import torch

_OFFSETS = {"q": 0, "k": 1, "v": 2, "do": 3}


def normal(shape, seed: int, which: str, dtype=torch.float32) -> torch.Tensor:
    """N(0,1) CPU tensor for input `which` ('q', 'k', 'v', 'do')."""
    g = torch.Generator().manual_seed(int(seed) + 7919 * _OFFSETS[which])
    x = torch.randn(tuple(shape), generator=g, dtype=torch.float32)
    return x.to(dtype)


def qkv(shape_q, shape_kv, seed: int, dtype=torch.bfloat16, with_do: bool = False):
    q = normal(shape_q, seed, "q", dtype)
    k = normal(shape_kv, seed, "k", dtype)
    v = normal(shape_kv, seed, "v", dtype)
    if with_do:
        return q, k, v, normal(shape_q, seed, "do", dtype)
    return q, k, v


def packed_lengths(total: int, cp: int, seed: int, mu: float = 7.5, sigma: float = 1.0,
                   lo: int = 128, hi: int = 16384) -> list[int]:
    """Sub-sequence lengths of a packed stream (all multiples of 2*cp, sum = total)."""
    align = 2 * cp
    assert total % align == 0
    rng = np.random.default_rng(seed)
    lens: list[int] = []
    acc = 0
    while acc < total:
        x = int(np.clip(np.round(np.exp(rng.normal(mu, sigma))), lo, hi))
        x = -(-x // align) * align
        x = min(x, total - acc)
        lens.append(x)
        acc += x
    if len(lens) > 1 and lens[-1] < lo:
        last = lens.pop()
        lens[-1] += last
    return lens


def cu_from_lengths(lengths) -> np.ndarray:
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return cu
