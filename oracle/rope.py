"""Rotary position embedding under the context-parallel split (float64).

Test infrastructure only: the test suite, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU legs may use it; the CUDA library shares no code with it.

"04 · Megatron-LM 实现" §5: a rotary embedding depends on the absolute
position, so the positions must be split by the same zigzag rule as the
tokens (under packed THD input the position is the offset inside the token's
own sub-sequence).  The pages name the embedding without printing its
formula; this module takes the rotate-half form: for i < d/2 the pair
(x_i, x_{i+d/2}) is rotated by the angle pos * base**(-2 i / d).
"""

from __future__ import annotations

import numpy as np


def inv_freq(head_dim: int, base: float = 10000.0) -> np.ndarray:
    """Angular frequency of pair i: base ** (-2 i / head_dim), i < head_dim / 2."""
    return float(base) ** (-2.0 * np.arange(head_dim // 2, dtype=np.float64) / head_dim)


def rotate(x, pos, base: float = 10000.0, inverse: bool = False) -> np.ndarray:
    """R(pos) x for x [..., T, H, d] and integer positions pos [T]; the
    transpose R(pos)^T x when `inverse` (the rotation by -angle)."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv_freq(d, base)[None, :]  # [T, d/2]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    if inverse:
        s = -s
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def permute_rope(x, idx, pos, base: float = 10000.0, inverse: bool = False) -> np.ndarray:
    """Token gather with the embedding applied at each token's own position.

    x [B, T, H, d]; idx [T] rank-local slot -> original token; pos [T] the
    position of every original token.
      inverse False: out[:, t] = R(pos[idx[t]]) x[:, idx[t]]
      inverse True:  out[:, idx[t]] = R(pos[idx[t]])^T x[:, t]
    """
    x = np.asarray(x, dtype=np.float64)
    idx = np.asarray(idx, dtype=np.int64).ravel()
    p = np.asarray(pos, dtype=np.int64)[idx]
    out = np.empty_like(x)
    if not inverse:
        out[:, :] = rotate(x[:, idx], p, base)
    else:
        out[:, idx] = rotate(x, p, base, inverse=True)
    return out
