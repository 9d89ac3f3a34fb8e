"""The allocation-free forward entry point, called through the C ABI.

cp_ring_attn_fwd_static_ws is for callers that cannot allocate device memory:
it runs the same ring forward as cp_ring_attn_fwd but on a static scratch
array inside the library.  On two calls in a row (the second reuses the
scratch the first left behind) its results must match the float64 oracle at
the parity bar and the workspace entry point's results at the same bar, for
the bf16 tensor-core path (BSHD and packed THD) and the float32 FFMA path; a
problem larger than the scratch must be refused with CP_ERR_WORKSPACE.  This
file is collected last on purpose.
"""

import ctypes

import numpy as np
import pytest
import torch

from oracle import attention as A
from tile_attention_lse_gb300 import api
from tile_attention_lse_gb300.synthetic import cu_from_lengths

from helpers import TOL_F32, TOL_LSE_BF16, TOL_O_BF16, f64, make_inputs, max_abs

pytestmark = pytest.mark.gpu
DEV = "cuda"
CP_ERR_WORKSPACE = next(code for code, name in api.STATUS.items() if name == "CP_ERR_WORKSPACE")


def _call_static(p, q, k, v, o, lse):
    return api.lib().cp_ring_attn_fwd_static_ws(
        p.desc, ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(o.data_ptr()),
        ctypes.c_void_p(lse.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


CASES = [
    # name, b, s, H, Hkv, d, cp, dtype, packed lengths (None: BSHD)
    ("bshd_gqa", 1, 1024, 4, 2, 128, 4, torch.bfloat16, None),
    ("bshd_b2", 2, 512, 2, 2, 128, 2, torch.bfloat16, None),
    ("thd", 1, None, 4, 2, 128, 4, torch.bfloat16, [8, 64, 200, 16, 1000, 8, 248]),
    ("f32_d64", 2, 512, 2, 1, 64, 4, torch.float32, None),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_static_ws_forward_matches_oracle_and_workspace_forward(case):
    _, b, s, H, Hkv, d, cp, dtype, lens = case
    cu = cu_from_lengths(lens) if lens is not None else None
    if cu is not None:
        s = int(cu[-1])
    q, k, v = make_inputs(b, s, H, Hkv, d, seed=21, dtype=dtype, thd=cu is not None)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    p = api.Problem(batch=b, heads_q=H, heads_kv=Hkv, head_dim=d, cp=cp, seqlen=s, dtype=dtype, cu_seqlens=cu)
    assert api.workspace_bytes(p, False) <= api.lib().cp_static_ws_capacity()
    tol_o = TOL_F32 if dtype == torch.float32 else TOL_O_BF16
    tol_l = TOL_F32 if dtype == torch.float32 else TOL_LSE_BF16
    # the float64 oracle on the same inputs
    if cu is None:
        ro, rl = A.attention_forward_bshd(f64(q), f64(k), f64(v))
    else:
        seq, pos = A.token_meta_from_cu(cu)
        ro, rl = A.attention_forward(f64(q), f64(k), f64(v), seq, pos)
    o_ref, l_ref = api.ring_attn_fwd(p, qd, kd, vd)       # the workspace entry point
    for _ in range(2):
        o = torch.full_like(qd, float("nan"))
        lse = torch.full(qd.shape[:-1], float("nan"), dtype=torch.float32, device=DEV)
        assert _call_static(p, qd, kd, vd, o, lse) == 0
        assert api.device_error() == 0
        torch.cuda.synchronize()
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        assert max_abs(f64(o), ro) <= tol_o
        assert max_abs(f64(lse), rl) <= tol_l
        assert (o.float() - o_ref.float()).abs().max().item() <= tol_o
        assert (lse - l_ref).abs().max().item() <= tol_l


def test_static_ws_rejects_oversized_problem():
    p = api.Problem(batch=1, heads_q=32, heads_kv=32, head_dim=128, cp=8, seqlen=32768)
    assert api.workspace_bytes(p, False) > api.lib().cp_static_ws_capacity()
    t = torch.empty(1, dtype=torch.bfloat16, device=DEV)
    assert _call_static(p, t, t, t, t, t.float()) == CP_ERR_WORKSPACE
