"""CPU check that the rising-maximum inputs of the GPU tests depend on the
online recurrence's correction ("上下文并行" 02 ONE ROW: c = e^(m - m'),
l' = c l + sum e^(S - m'), a' = c a + sum e^(S - m') V).

The tensor-core forward applies the correction lazily: it moves its running
maximum m only when a key tile lifts it by more than tau = 8 log2-units, and
otherwise exponentiates against a stale m (values up to e^tau, exact in the
final ratio).  Written out here in float64, that lazy recurrence equals the
oracle's plain softmax; leaving out the rescale of the accumulator or of the
denominator misses the oracle on the same inputs by far more than the parity
bar, so the GPU tests built on these inputs would catch such a mistake.
"""

import math

import numpy as np
import torch

from oracle import attention as A

from helpers import (RESCALE_NATS, TOL_LSE_BF16, TOL_O_BF16, f64, make_inputs, max_growth, ramp_keys)


def lazy_online(scores, v, tau, skip_o=False, skip_l=False):
    """One row through the lazy recurrence over 128-key tiles (natural units)."""
    m, ell, acc = -math.inf, 0.0, np.zeros(v.shape[1])
    for t0 in range(0, len(scores), 128):
        s, vb = scores[t0:t0 + 128], v[t0:t0 + 128]
        m_new = max(m, float(np.max(s)))
        if m_new > m + tau:                         # also when m is -inf
            c = math.exp(m - m_new) if m != -math.inf else 0.0
            if not skip_l:
                ell *= c
            if not skip_o:
                acc *= c
            m = m_new
        e = np.exp(s - m)
        ell += float(e.sum())
        acc += e @ vb
    return acc / ell, m + math.log(ell)


def _inputs():
    # the single-edge case of the GPU test: 256 queries, 1024 keys, no mask
    q, k, v = make_inputs(1, 1536, 2, 1, 128, seed=23, dtype=torch.bfloat16)
    k = ramp_keys(k, slope=10.0)
    return f64(q[0, :256]), f64(k[0, :1024]), f64(v[0, :1024])


def _run(q, k, v, **kw):
    o = np.empty((q.shape[0], q.shape[1], v.shape[-1]))
    lse = np.empty(q.shape[:2])
    for h in range(q.shape[1]):
        s = (q[:, h] @ k[:, 0].T) / math.sqrt(q.shape[-1])
        for i in range(q.shape[0]):
            o[i, h], lse[i, h] = lazy_online(s[i], v[:, 0], RESCALE_NATS, **kw)
    return o, lse


def test_inputs_lift_the_running_maximum():
    q, k, v = _inputs()
    vis = np.ones((q.shape[0], k.shape[0]), dtype=bool)
    assert np.mean(max_growth(q, k, vis) > RESCALE_NATS + 1.0) >= 0.5


def test_lazy_recurrence_equals_the_oracle():
    q, k, v = _inputs()
    vis = np.ones((q.shape[0], k.shape[0]), dtype=bool)
    ro, rl = A.masked_attention(q, k, v, vis)
    o, lse = _run(q, k, v)
    assert np.max(np.abs(o - ro)) < 1e-10 and np.max(np.abs(lse - rl)) < 1e-10


def test_skipped_corrections_miss_the_bar():
    q, k, v = _inputs()
    vis = np.ones((q.shape[0], k.shape[0]), dtype=bool)
    ro, rl = A.masked_attention(q, k, v, vis)
    o, _ = _run(q, k, v, skip_o=True)
    assert np.max(np.abs(o - ro)) > 10 * TOL_O_BF16
    _, lse = _run(q, k, v, skip_l=True)
    assert np.max(np.abs(lse - rl)) > 10 * TOL_LSE_BF16
