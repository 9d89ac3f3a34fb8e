"""Failure detection on the GPU without a fault: the tcgen05 kernels' bounded
waits.

cp_debug_set_wait_limit shortens the cycle budget of every main-loop wait of
the tensor-core forward and backward.  With a budget of one cycle every wait
that is not already complete runs out: the block raises its abort flag,
drains its own copies and MMAs (with the default budget), frees TMEM and
returns, and the host reads CP_ERR_TIMEOUT.  The context must stay usable: the
next call with the default budget is checked against the float64 oracle.
"""

import numpy as np
import pytest
import torch

from oracle import attention as A
from tile_attention_lse_gb300 import api

from helpers import TOL_GRAD_REL, TOL_LSE_BF16, TOL_O_BF16, f64, make_inputs, max_abs

pytestmark = pytest.mark.gpu
DEV = "cuda"
CP_ERR_TIMEOUT = -6


def _case():
    b, s, H, d, cp = 1, 2048, 2, 128, 4
    q, k, v, do = make_inputs(b, s, H, H, d, seed=17, dtype=torch.bfloat16, with_do=True)
    p = api.Problem(batch=b, heads_q=H, heads_kv=H, head_dim=d, cp=cp, seqlen=s)
    return p, q, k, v, do


def test_wait_limit_runs_out_then_recovers():
    p, q, k, v, do = _case()
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, do))
    assert api.device_error() == 0
    try:
        api.set_wait_limit(1)
        api.ring_attn_fwd(p, qd, kd, vd)                 # host status: launched
        assert api.device_error() == CP_ERR_TIMEOUT       # a forward wait ran out
        api.set_wait_limit(0)
        o_ok, l_ok = api.ring_attn_fwd(p, qd, kd, vd)    # backward input from a clean forward
        assert api.device_error() == 0
        api.set_wait_limit(1)
        api.ring_attn_bwd(p, qd, kd, vd, o_ok, l_ok, dod)
        assert api.device_error() == CP_ERR_TIMEOUT       # a backward wait ran out
    finally:
        api.set_wait_limit(0)
    # the word was read and cleared; the default budget gives correct results again
    assert api.device_error() == 0
    o, l = api.ring_attn_fwd(p, qd, kd, vd)
    dq, dk, dv = api.ring_attn_bwd(p, qd, kd, vd, o, l, dod)
    assert api.device_error() == 0
    ro, rl = A.attention_forward_bshd(f64(q), f64(k), f64(v))
    assert max_abs(f64(o[0]), ro[0]) <= TOL_O_BF16
    assert max_abs(f64(l[0]), rl[0]) <= TOL_LSE_BF16
    rq, rk, rv = A.attention_backward_bshd(f64(q), f64(k), f64(v), f64(do))
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        assert max_abs(f64(got[0]), ref[0]) <= TOL_GRAD_REL * float(np.max(np.abs(ref)))


def test_wait_limit_argument_checks():
    with pytest.raises(api.CpError) as e:
        api.set_wait_limit(10 ** 12)                     # above the default budget
    assert e.value.code == -1
    api.set_wait_limit(-5)                               # <= 0: the default
    api.set_wait_limit(0)
