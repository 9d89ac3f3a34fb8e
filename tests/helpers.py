"""Shared helpers of the GPU parity tests: seeded inputs, oracle evaluation on
row samples, and the tolerances of the parity bar."""

from __future__ import annotations

import numpy as np
import torch

from oracle import attention as A
from tile_attention_lse_gb300 import synthetic

# Parity bar (absolute): bf16 inputs with fp32 accumulation, float32 inputs,
# gradients relative to the largest gradient magnitude of the tensor.
TOL_O_BF16 = 2e-2
TOL_LSE_BF16 = 2e-3
TOL_F32 = 1e-5
TOL_GRAD_REL = 3e-2


def make_inputs(b, s, H, Hkv, d, seed, dtype, with_do=False, thd=False):
    shape_q = (s, H, d) if thd else (b, s, H, d)
    shape_kv = (s, Hkv, d) if thd else (b, s, Hkv, d)
    return synthetic.qkv(shape_q, shape_kv, seed, dtype, with_do)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def meta(cu):
    return A.token_meta_from_cu(cu)


def oracle_rows(q, k, v, rows, heads, cu, causal=True, scale=None, window=None):
    """Full-attention O and L of the listed rows and heads of one stream.

    q: [T, H, d], k/v: [T, Hkv, d] torch CPU tensors (any dtype).  Only the
    needed head slices are converted to float64.
    """
    seq, pos = meta(cu)
    rows = np.asarray(rows)
    vis = A.visibility(seq[rows], pos[rows], seq, pos, causal, window)
    H, Hkv = q.shape[1], k.shape[1]
    grp = H // Hkv
    out = {}
    for h in heads:
        g = h // grp
        qh = f64(q[rows, h:h + 1])
        kh = f64(k[:, g:g + 1])
        vh = f64(v[:, g:g + 1])
        o, l = A.masked_attention(qh, kh, vh, vis, scale)
        out[h] = (o[:, 0], l[:, 0])
    return out


def sample_rows(T, n, seed, chunk=None):
    """n rows of [0, T): both ends, every chunk boundary if given, the rest random."""
    rng = np.random.default_rng(seed)
    rows = {0, T - 1}
    if chunk:
        for c0 in range(0, T, chunk):
            rows.update({c0, min(T - 1, c0 + chunk - 1)})
    while len(rows) < n:
        rows.add(int(rng.integers(0, T)))
    return np.array(sorted(rows))


def max_abs(a, b):
    diff = np.abs(np.asarray(a, dtype=np.float64) - np.asarray(b, dtype=np.float64))
    return float(np.max(diff)) if diff.size else 0.0


# ---- inputs whose running row maximum rises across the key stream ---------
# The tensor-core forward keeps the running maximum m of a row lazily: O and
# l are rescaled by c = 2^(m - m') only when a key tile lifts the maximum by
# more than 8 in log2 units (5.55 in natural units).  With N(0, 1) inputs a
# row's first tile sets m for good, so these inputs scale key j by
# 1 + slope * pos_j / n: later keys score higher and the maximum keeps rising.
RESCALE_NATS = 8.0 * np.log(2.0)


def ramp_keys(k: torch.Tensor, slope: float, pos=None) -> torch.Tensor:
    """k [..., n, heads, d] (any float dtype) with key j scaled by
    1 + slope * pos_j / n (pos defaults to the row index), rounded back to
    k's dtype."""
    n = k.shape[-3]
    pos = torch.arange(n, dtype=torch.float64) if pos is None else torch.as_tensor(pos, dtype=torch.float64)
    g = (1.0 + slope * pos / n).to(torch.float32).view(n, 1, 1)
    return (k.float() * g).to(k.dtype)


def max_growth(q, k, vis, scale=None, span=128):
    """Per (row, head), a lower bound on how far the running maximum rises
    after the row's first streamed key tile: the max score over the visible
    keys minus the max over the row's first `span` visible keys (natural
    units).

    The zigzag kernels stream a row's keys in position order in tiles of at
    most 128 keys (one streaming part here), so the first tile holding a
    visible key holds only keys among the first 128 (span = 128); a striped
    segment holds every cp-th position, so there the first tile lies within
    the first 128 cp + cp visible keys.  Where the bound exceeds RESCALE_NATS
    the kernel must apply at least one correction with a finite running
    maximum.  q [n, H, d], k [m, Hkv, d] torch or numpy (any float type,
    converted one head at a time); vis [n, m] in key-position order."""
    H, Hkv = q.shape[1], k.shape[1]
    scale = 1.0 / np.sqrt(q.shape[-1]) if scale is None else scale
    first = vis & (np.cumsum(vis, axis=1) <= span)
    out = np.empty((q.shape[0], H))
    for h in range(H):
        qh = np.asarray(q[:, h], dtype=np.float64) if isinstance(q, np.ndarray) else f64(q[:, h])
        kg = k[:, h // (H // Hkv)]
        kh = np.asarray(kg, dtype=np.float64) if isinstance(kg, np.ndarray) else f64(kg)
        sc = scale * (qh @ kh.T)
        out[:, h] = np.where(vis, sc, -np.inf).max(1) - np.where(first, sc, -np.inf).max(1)
    return out
