"""The five workloads at full size, through the C ABI, against the float64
oracle: every output where the oracle finishes in seconds, otherwise sampled
rows (both ends of every chunk plus random rows, every head) and invariants
that hold at any size."""

import numpy as np
import pytest
import torch

from oracle import attention as A
from tile_attention_lse_gb300 import api
from tile_attention_lse_gb300.synthetic import cu_from_lengths, packed_lengths

from helpers import (RESCALE_NATS, TOL_F32, TOL_GRAD_REL, TOL_LSE_BF16, TOL_O_BF16, f64, make_inputs,
                     max_abs, max_growth, oracle_rows, ramp_keys, sample_rows)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run_fwd(p, q, k, v):
    o, l = api.ring_attn_fwd(p, q.to(DEV), k.to(DEV), v.to(DEV))
    assert api.device_error() == 0
    return o.cpu(), l.cpu()


def _check_rows(o, l, q, k, v, rows, cu, tol_o, tol_l, heads=None, window=None):
    heads = range(q.shape[1]) if heads is None else heads
    ref = oracle_rows(q, k, v, rows, heads, cu, window=window)
    for h, (ro, rl) in ref.items():
        assert max_abs(f64(o[rows, h]), ro) <= tol_o, f"head {h}"
        assert max_abs(f64(l[rows, h]), rl) <= tol_l, f"head {h}"


def test_fp32_b1_h1_d64_s256_cp2_exact():
    """fp32, batch 1, 1 head, d 64, s 256, cp 2: every output at 1e-5."""
    s, d = 256, 64
    q, k, v = make_inputs(1, s, 1, 1, d, seed=0, dtype=torch.float32)
    p = api.Problem(batch=1, heads_q=1, heads_kv=1, head_dim=d, cp=2, seqlen=s, dtype=torch.float32)
    o, l = _run_fwd(p, q, k, v)
    ro, rl = A.attention_forward_bshd(f64(q), f64(k), f64(v))
    assert max_abs(f64(o), ro) <= TOL_F32
    assert max_abs(f64(l), rl) <= TOL_F32


def test_mha_h32_s16384_cp8():
    s, H, d = 16384, 32, 128
    q, k, v = make_inputs(1, s, H, H, d, seed=0, dtype=torch.bfloat16)
    p = api.Problem(batch=1, heads_q=H, heads_kv=H, head_dim=d, cp=8, seqlen=s)
    o, l = _run_fwd(p, q, k, v)
    rows = sample_rows(s, 64, seed=2, chunk=s // 16)
    _check_rows(o[0], l[0], q[0], k[0], v[0], rows, [0, s], TOL_O_BF16, TOL_LSE_BF16)


def test_mha_h32_s16384_cp8_rising_max():
    """The 16384-token, 32-head, cp = 8 ring with keys scaled up along the
    sequence (1 + 10 pos / s): most sampled rows' running maximum rises past
    the kernel's lazy threshold mid-stream, so the correction c = e^(m - m')
    of "上下文并行" 02 ONE ROW runs with a finite m; sampled rows on every
    head against the oracle."""
    s, H, d = 16384, 32, 128
    q, k, v = make_inputs(1, s, H, H, d, seed=6, dtype=torch.bfloat16)
    k = ramp_keys(k, slope=10.0)
    p = api.Problem(batch=1, heads_q=H, heads_kv=H, head_dim=d, cp=8, seqlen=s)
    o, l = _run_fwd(p, q, k, v)
    rows = sample_rows(s, 64, seed=7, chunk=s // 16)
    pos = np.arange(s)
    vis = A.visibility(np.zeros(len(rows)), rows, np.zeros(s), pos, True)
    assert np.mean(max_growth(q[0, rows], k[0], vis) > RESCALE_NATS + 1.0) >= 0.5
    _check_rows(o[0], l[0], q[0], k[0], v[0], rows, [0, s], TOL_O_BF16, TOL_LSE_BF16)


def test_thd_gqa_32_8_lognormal_t65536_cp4():
    T, H, Hkv, d, cp = 65536, 32, 8, 128, 4
    lens = packed_lengths(T, cp, seed=0)
    cu = cu_from_lengths(lens)
    q, k, v = make_inputs(1, T, H, Hkv, d, seed=0, dtype=torch.bfloat16, thd=True)
    p = api.Problem(batch=1, heads_q=H, heads_kv=Hkv, head_dim=d, cp=cp, seqlen=T, cu_seqlens=cu)
    o, l = _run_fwd(p, q, k, v)
    rng = np.random.default_rng(3)
    rows = set()
    for a, b in zip(cu[:-1], cu[1:]):                # both ends of every sub-sequence
        rows.update({int(a), int(b) - 1})
    rows.update(int(x) for x in rng.integers(0, T, 64))
    rows = np.array(sorted(rows))
    _check_rows(o, l, q, k, v, rows, cu, TOL_O_BF16, TOL_LSE_BF16)


def test_gqa_32_8_s131072_cp16():
    s, H, Hkv, d, cp = 131072, 32, 8, 128, 16
    q, k, v = make_inputs(1, s, H, Hkv, d, seed=0, dtype=torch.bfloat16)
    p = api.Problem(batch=1, heads_q=H, heads_kv=Hkv, head_dim=d, cp=cp, seqlen=s)
    o, l = _run_fwd(p, q, k, v)
    rows = sample_rows(s, 80, seed=4, chunk=s // 32)
    _check_rows(o[0], l[0], q[0], k[0], v[0], rows, [0, s], TOL_O_BF16, TOL_LSE_BF16)


def test_fwd_bwd_b2_h32_s32768_cp8():
    _fwd_bwd_b2_s32768_cp8(window=0)


def test_window4096_fwd_bwd_b2_s32768_cp8():
    """The same shape under a sliding window of 4096 (a sparser task graph)."""
    _fwd_bwd_b2_s32768_cp8(window=4096)


def _fwd_bwd_b2_s32768_cp8(window):
    b, s, H, d, cp = 2, 32768, 32, 128, 8
    w = window or None
    q, k, v, do = make_inputs(b, s, H, H, d, seed=0, dtype=torch.bfloat16, with_do=True)
    p = api.Problem(batch=b, heads_q=H, heads_kv=H, head_dim=d, cp=cp, seqlen=s,
                    order=api.CP_ORDER_RANK_LOCAL, window=window)
    # the bench's launch configuration: partition, gather, ring fwd, ring bwd
    idx, _ = api.partition_indices(p)
    ql, kl, vl, dol = (api.permute_tokens(p, idx, x.to(DEV)) for x in (q, k, v, do))
    o, l = api.ring_attn_fwd(p, ql, kl, vl)
    dq, dk, dv = api.ring_attn_bwd(p, ql, kl, vl, o, l, dol)
    assert api.device_error() == 0
    o, dq, dk, dv = (api.permute_tokens(p, idx, x, inverse=True).cpu() for x in (o, dq, dk, dv))
    lo = torch.empty_like(l)
    lo[:, idx.reshape(-1).long()] = l
    lo = lo.cpu()
    rows = sample_rows(s, 48, seed=5, chunk=s // 16)
    for bi in range(b):
        _check_rows(o[bi], lo[bi], q[bi], k[bi], v[bi], rows, [0, s], TOL_O_BF16, TOL_LSE_BF16,
                    heads=range(0, H, 3), window=w)
    # invariants at full size, every (batch, head): sum_j dK_j = 0 and
    # sum_j dV_j = sum_i dO_i (up to the rounding of s bf16 terms)
    dk64, dv64, do64 = (x.to(torch.float64) for x in (dk, dv, do))
    kmax = dk64.abs().amax(dim=(1, 3))
    assert torch.all(dk64.sum(1).abs().amax(-1) <= TOL_GRAD_REL * kmax * np.sqrt(s))
    dvs, dos = dv64.sum(1), do64.sum(1)
    assert torch.all((dvs - dos).abs().amax(-1) <= TOL_GRAD_REL * dv64.abs().amax(dim=(1, 3)) * np.sqrt(s))
    # exact gradients of two (batch, head) pairs, one in each batch entry,
    # against the oracle
    seq, pos = np.zeros(s, dtype=np.int64), np.arange(s)
    for bi, h in ((1, 5), (0, 22)):
        rq, rk, rv = A.attention_backward(f64(q[bi, :, h:h + 1]), f64(k[bi, :, h:h + 1]),
                                          f64(v[bi, :, h:h + 1]), f64(do[bi, :, h:h + 1]), seq, pos, window=w)
        for got, ref in ((dq[bi, :, h], rq[:, 0]), (dk[bi, :, h], rk[:, 0]), (dv[bi, :, h], rv[:, 0])):
            assert max_abs(f64(got), ref) <= TOL_GRAD_REL * float(np.max(np.abs(ref))), f"batch {bi} head {h}"


def test_gqa_32_8_s16384_cp8_fwd_bwd_sampled():
    """Grouped heads at length: 32 q-heads on 8 kv-heads, 16384 tokens, cp = 8,
    rank-local tensors.  dK/dV of a key tile sum the contributions of four
    q-heads and of every query tile that sees it (up to 128 of them) in TMEM;
    sampled key rows of dK/dV and sampled query rows of dQ of one kv-group
    are checked against the oracle's replay (exact row LSE and D)."""
    s, H, Hkv, d, cp = 16384, 32, 8, 128, 8
    q, k, v, do = make_inputs(1, s, H, Hkv, d, seed=8, dtype=torch.bfloat16, with_do=True)
    p = api.Problem(batch=1, heads_q=H, heads_kv=Hkv, head_dim=d, cp=cp, seqlen=s,
                    order=api.CP_ORDER_RANK_LOCAL)
    idx, _ = api.partition_indices(p)
    ql, kl, vl, dol = (api.permute_tokens(p, idx, x.to(DEV)) for x in (q, k, v, do))
    o, l = api.ring_attn_fwd(p, ql, kl, vl)
    dq, dk, dv = api.ring_attn_bwd(p, ql, kl, vl, o, l, dol)
    assert api.device_error() == 0
    o, dq, dk, dv = (api.permute_tokens(p, idx, x, inverse=True).cpu()[0] for x in (o, dq, dk, dv))
    g = 3
    hs = slice(g * (H // Hkv), (g + 1) * (H // Hkv))
    seq, pos = np.zeros(s, dtype=np.int64), np.arange(s)
    qg, kg, vg, dog = f64(q[0, :, hs]), f64(k[0, :, g:g + 1]), f64(v[0, :, g:g + 1]), f64(do[0, :, hs])
    ro, rl = A.attention_forward(qg, kg, vg, seq, pos)
    assert max_abs(f64(o[:, hs]), ro) <= TOL_O_BF16
    delta = np.einsum("nhd,nhd->nh", dog, ro)
    keys = sample_rows(s, 96, seed=9, chunk=s // 16)
    vis_k = A.visibility(seq, pos, seq[keys], pos[keys], True)
    _, rk, rv = A.block_backward(qg, kg[keys], vg[keys], dog, rl, delta, vis_k)
    for got, ref in ((dk[keys, g], rk[:, 0]), (dv[keys, g], rv[:, 0])):
        assert max_abs(f64(got), ref) <= TOL_GRAD_REL * float(np.max(np.abs(ref)))
    rows = sample_rows(s, 64, seed=10, chunk=s // 16)
    vis_q = A.visibility(seq[rows], pos[rows], seq, pos, True)
    rq, _, _ = A.block_backward(qg[rows], kg, vg, dog[rows], rl[rows], delta[rows], vis_q)
    assert max_abs(f64(dq[rows, hs]), rq) <= TOL_GRAD_REL * float(np.max(np.abs(rq)))
