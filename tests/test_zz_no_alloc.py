"""The allocation-free forward entry point, called through the C ABI.

cp_ring_attn_fwd_static_ws is for callers that cannot allocate device memory:
it runs the same ring forward as cp_ring_attn_fwd but on a static scratch
array inside the library.  Its results must match the workspace entry point's
on two calls in a row (the second call reuses the scratch the first left
behind), and a problem larger than the scratch must be refused with
CP_ERR_WORKSPACE.  This file is collected last on purpose.
"""

import ctypes

import pytest
import torch

from tile_attention_lse_gb300 import api, synthetic

from helpers import TOL_LSE_BF16, TOL_O_BF16

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _call_static(p, q, k, v, o, lse):
    return api.lib().cp_ring_attn_fwd_static_ws(
        p.desc, ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(o.data_ptr()),
        ctypes.c_void_p(lse.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("b,s,H,Hkv,cp", [(1, 1024, 4, 2, 4), (2, 512, 2, 2, 2)])
def test_static_ws_forward_matches_workspace_forward(b, s, H, Hkv, cp):
    q, k, v = synthetic.qkv((b, s, H, 128), (b, s, Hkv, 128), seed=21, dtype=torch.bfloat16)
    q, k, v = q.to(DEV), k.to(DEV), v.to(DEV)
    p = api.Problem(batch=b, heads_q=H, heads_kv=Hkv, head_dim=128, cp=cp, seqlen=s)
    assert api.workspace_bytes(p, False) <= api.lib().cp_static_ws_capacity()
    o_ref, l_ref = api.ring_attn_fwd(p, q, k, v)
    for _ in range(2):
        o = torch.full_like(q, float("nan"))
        lse = torch.full((b, s, H), float("nan"), dtype=torch.float32, device=DEV)
        assert _call_static(p, q, k, v, o, lse) == 0
        assert api.device_error() == 0
        torch.cuda.synchronize()
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        assert (o.float() - o_ref.float()).abs().max().item() <= TOL_O_BF16
        assert (lse - l_ref).abs().max().item() <= TOL_LSE_BF16


def test_static_ws_rejects_oversized_problem():
    p = api.Problem(batch=1, heads_q=32, heads_kv=32, head_dim=128, cp=8, seqlen=32768)
    assert api.workspace_bytes(p, False) > api.lib().cp_static_ws_capacity()
    t = torch.empty(1, dtype=torch.bfloat16, device=DEV)
    assert _call_static(p, t, t, t, t, t.float()) == -4
