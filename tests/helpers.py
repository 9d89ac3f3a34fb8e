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
