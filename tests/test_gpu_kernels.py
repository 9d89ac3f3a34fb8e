"""GPU parity of each C-ABI entry point against the float64 oracle, at sizes
the oracle finishes in seconds (several tiles plus ragged tails)."""

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import hybrid as HY
from oracle import partition as P
from oracle import ring as R
from oracle import rope as RO
from tile_attention_lse_gb300 import api
from tile_attention_lse_gb300.synthetic import cu_from_lengths, packed_lengths

from helpers import (RESCALE_NATS, TOL_F32, TOL_GRAD_REL, TOL_LSE_BF16, TOL_O_BF16, f64, make_inputs, max_abs,
                     max_growth, ramp_keys)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _prob(**kw):
    return api.Problem(**kw)


# --------------------------------------------------------------- partition --
@pytest.mark.parametrize("s,cp", [(256, 2), (16384, 8), (131072, 16), (32768, 8), (8, 1), (24, 3)])
def test_partition_bshd_bitexact(s, cp):
    p = _prob(batch=1, heads_q=1, heads_kv=1, head_dim=64, cp=cp, seqlen=s)
    idx, _ = api.partition_indices(p)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), P.zigzag_indices(s, cp))


@pytest.mark.parametrize("seed,cp", [(0, 4), (1, 4), (2, 2), (3, 8)])
def test_partition_thd_bitexact(seed, cp):
    lens = packed_lengths(65536, cp, seed)
    cu = cu_from_lengths(lens)
    p = _prob(batch=1, heads_q=1, heads_kv=1, head_dim=64, cp=cp, seqlen=int(cu[-1]), cu_seqlens=cu)
    idx, local_cu = api.partition_indices(p)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), P.thd_partition_indices(cu, cp))
    assert np.array_equal(local_cu.cpu().numpy(), P.local_cu_seqlens(cu, cp))


def test_partition_thd_edge_cases():
    # sub-sequences of exactly 2cp tokens, and an empty one in the middle
    cu = np.array([0, 8, 8, 16, 48], dtype=np.int32)
    p = _prob(batch=1, heads_q=1, heads_kv=1, head_dim=64, cp=4, seqlen=48, cu_seqlens=cu)
    idx, _ = api.partition_indices(p)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), P.thd_partition_indices(cu, 4))


def test_partition_rejects_misaligned():
    p = _prob(batch=1, heads_q=1, heads_kv=1, head_dim=64, cp=4, seqlen=100)
    with pytest.raises(api.CpError) as e:
        api.partition_indices(p)
    assert e.value.code == -2


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_permute_and_inverse(dtype):
    b, s, H, d, cp = 2, 512, 3, 64, 4
    p = _prob(batch=b, heads_q=H, heads_kv=H, head_dim=d, cp=cp, seqlen=s, dtype=dtype)
    x = torch.randn(b, s, H, d, device=DEV).to(dtype)
    idx, _ = api.partition_indices(p)
    y = api.permute_tokens(p, idx, x)
    ref_idx = torch.from_numpy(P.zigzag_indices(s, cp).reshape(-1)).to(DEV)
    assert torch.equal(y, x[:, ref_idx])
    z = api.permute_tokens(p, idx, y, inverse=True)
    assert torch.equal(z, x)


# ------------------------------------------------------ striped partition --
STRIPED = dict(partition=api.CP_PARTITION_STRIPED, order=api.CP_ORDER_RANK_LOCAL)


@pytest.mark.parametrize("s,cp", [(256, 2), (32768, 8), (12, 4), (3000, 8), (8, 1)])
def test_partition_striped_bshd_bitexact(s, cp):
    p = _prob(batch=1, heads_q=1, heads_kv=1, head_dim=64, cp=cp, seqlen=s, **STRIPED)
    idx, _ = api.partition_indices(p)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), P.striped_indices(s, cp))


@pytest.mark.parametrize("cu,cp", [(None, 4), ([0, 12, 12, 36, 60, 64], 4), ([0, 3, 9, 9, 30], 3)])
def test_partition_striped_thd_bitexact(cu, cp):
    if cu is None:
        cu = cu_from_lengths(packed_lengths(65536, cp, 1))
    p = _prob(batch=1, heads_q=1, heads_kv=1, head_dim=64, cp=cp, seqlen=int(cu[-1]), cu_seqlens=cu,
              **STRIPED)
    idx, local_cu = api.partition_indices(p)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), P.thd_striped_indices(cu, cp))
    assert np.array_equal(local_cu.cpu().numpy(), P.local_cu_seqlens(cu, cp))


def test_permute_rope_striped_vs_oracle():
    # RoPE angles follow the original positions the striped gather brings in
    b, s, H, d, cp = 2, 1000, 2, 128, 8
    p = _prob(batch=b, heads_q=H, heads_kv=H, head_dim=d, cp=cp, seqlen=s, dtype=torch.bfloat16, **STRIPED)
    g = torch.Generator(device="cpu").manual_seed(4)
    x = torch.randn(b, s, H, d, generator=g).to(torch.bfloat16).to(DEV)
    idx, _ = api.partition_indices(p)
    y = api.permute_rope(p, idx, x)
    ref = RO.permute_rope(f64(x), P.striped_indices(s, cp).ravel(), np.arange(s))
    assert max_abs(f64(y), ref) <= TOL_O_BF16 * max(1.0, float(np.abs(ref).max()) / 4)


@pytest.mark.parametrize("case", ["bshd", "thd", "striped_thd", "hybrid"])
def test_token_seq_pos_bitexact(case):
    """Sub-sequence index and in-sequence position of every rank-local slot."""
    if case == "bshd":
        cu = cu_from_lengths([512])
        p = _prob(batch=1, heads_q=1, heads_kv=1, head_dim=64, cp=4, seqlen=512)
    else:
        cu = cu_from_lengths([8, 64, 0, 200, 16, 1000, 8, 248])
        kw = dict(batch=1, heads_q=1, heads_kv=1, head_dim=64, cp=4, seqlen=int(cu[-1]), cu_seqlens=cu,
                  order=api.CP_ORDER_RANK_LOCAL)
        if case == "striped_thd":
            kw["partition"] = api.CP_PARTITION_STRIPED
        if case == "hybrid":
            kw.update(seq_cp=[1, 2, 1, 4, 1, 4, 2, 2], seq_rank0=[3, 2, 0, 0, 1, 0, 0, 2])
        p = _prob(**kw)
    idx, _ = api.partition_indices(p)
    sp = api.token_seq_pos(p, idx)
    torch.cuda.synchronize()
    seq, pos = A.token_meta_from_cu(cu)
    t = idx.reshape(-1).cpu().numpy().astype(np.int64)
    got = sp.cpu().numpy()
    assert np.array_equal(got[:, 0], seq[t]) and np.array_equal(got[:, 1], pos[t])


# ----------------------------------------------- token gather with RoPE --
def _rope_case(dtype, d, cu=None, b=2, s=1024, H=3, cp=4, base=10000.0, seed=0):
    kw = dict(batch=b, heads_q=H, heads_kv=H, head_dim=d, cp=cp, seqlen=s, dtype=dtype)
    if cu is not None:
        kw.update(batch=1, seqlen=int(cu[-1]), cu_seqlens=cu)
    p = _prob(**kw)
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.randn(p.batch, p.seqlen, H, d, generator=g).to(dtype).to(DEV)
    idx, _ = api.partition_indices(p)
    if cu is None:
        pos = np.arange(p.seqlen)
    else:
        _, pos = A.token_meta_from_cu(cu)
    return p, x, idx, pos


def _rope_tol(dtype):
    # bf16 output of an exact rotation of bf16 inputs: one bf16 rounding
    # (2^-8 relative) of values up to ~|x|max; float32: sincos and products
    return (TOL_O_BF16, 0.0) if dtype == torch.bfloat16 else (TOL_F32, 0.0)


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.bfloat16, 64), (torch.float32, 64),
                                     (torch.float32, 128)])
def test_permute_rope_bshd_vs_oracle(dtype, d):
    p, x, idx, pos = _rope_case(dtype, d, base=500.0)
    y = api.permute_rope(p, idx, x, rope_base=500.0)
    ref = RO.permute_rope(f64(x), idx.cpu().numpy().ravel(), pos, base=500.0)
    tol, _ = _rope_tol(dtype)
    assert max_abs(f64(y), ref) <= tol * max(1.0, float(np.abs(ref).max()) / 4)
    # inverse gather of the result: back to the input (two roundings in bf16)
    z = api.permute_rope(p, idx, y, rope_base=500.0, inverse=True)
    ref_z = RO.permute_rope(f64(y), idx.cpu().numpy().ravel(), pos, base=500.0, inverse=True)
    assert max_abs(f64(z), ref_z) <= tol * max(1.0, float(np.abs(ref_z).max()) / 4)
    assert max_abs(f64(z), f64(x)) <= 2 * tol * max(1.0, float(np.abs(f64(x)).max()) / 4)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_permute_rope_thd_vs_oracle(dtype):
    lens = packed_lengths(8192, 4, seed=2, mu=6.0, sigma=1.0, lo=8, hi=2048)
    cu = cu_from_lengths(lens)
    p, x, idx, pos = _rope_case(dtype, 128, cu=cu, H=2)
    y = api.permute_rope(p, idx, x)
    ref = RO.permute_rope(f64(x), idx.cpu().numpy().ravel(), pos)
    tol, _ = _rope_tol(dtype)
    assert max_abs(f64(y), ref) <= tol * max(1.0, float(np.abs(ref).max()) / 4)


def test_permute_rope_long_positions_sampled():
    # positions up to 131071 (the 128K configuration): the angles are reduced
    # in float64 before the float32 sin/cos; sampled rows against the oracle
    p, x, idx, pos = _rope_case(torch.float32, 128, b=1, s=131072, H=2, cp=16)
    y = api.permute_rope(p, idx, x)
    ridx = idx.cpu().numpy().ravel()
    rows = np.random.default_rng(0).choice(p.seqlen, 512, replace=False)
    rows = np.concatenate([rows, [0, p.seqlen - 1, int(np.argmax(ridx))]])
    ref = RO.rotate(f64(x)[0, ridx[rows]], ridx[rows])
    assert max_abs(f64(y[0, torch.from_numpy(rows).to(DEV)]), ref) <= TOL_F32 * 4


def test_permute_rope_argument_errors():
    p, x, idx, _ = _rope_case(torch.bfloat16, 128)
    for bad in (dict(rope_base=0.0), dict(rope_base=-1.0)):
        with pytest.raises(api.CpError) as e:
            api.permute_rope(p, idx, x, **bad)
        assert e.value.code == -1
    with pytest.raises(api.CpError):
        api.permute_rope(p, idx, x, out=x)


@pytest.mark.parametrize("thd", [False, True])
def test_rope_then_ring_fwd_bwd(thd):
    """The rotary embedding at each token's own position, applied in the
    gather into rank-local order ("04 · Megatron-LM 实现" §5, §9: positions
    split by the same rule as the tokens), then the ring forward and backward,
    and the gradients of Q and K taken back through the transposed rotation.
    Oracle chain: rotate (float64, rounded to the bf16 of the gathered
    tensors) -> attention -> gradients -> transposed rotation."""
    cp, H, Hkv, d = 4, 4, 2, 128
    if thd:
        cu = cu_from_lengths([8, 64, 200, 16, 1000, 8, 248])
        b, s = 1, int(cu[-1])
        _, pos = A.token_meta_from_cu(cu)
    else:
        cu, b, s = None, 2, 1024
        pos = np.arange(s)
    q, k, v, do = make_inputs(b, s, H, Hkv, d, 37, torch.bfloat16, with_do=True, thd=thd)
    p = _prob(batch=b, heads_q=H, heads_kv=Hkv, head_dim=d, cp=cp, seqlen=s, cu_seqlens=cu,
              order=api.CP_ORDER_RANK_LOCAL)
    idx, _ = api.partition_indices(p)
    bat = (lambda x: x.unsqueeze(0)) if thd else (lambda x: x)     # the gathers take [b, s, h, d]
    unb = (lambda x: x[0]) if thd else (lambda x: x)
    qr, kr = (unb(api.permute_rope(p, idx, bat(x.to(DEV)))) for x in (q, k))
    vl, dol = (unb(api.permute_tokens(p, idx, bat(x.to(DEV)))) for x in (v, do))
    o, l = api.ring_attn_fwd(p, qr, kr, vl)
    dq, dk, dv = api.ring_attn_bwd(p, qr, kr, vl, o, l, dol)
    assert api.device_error() == 0
    dq, dk = (unb(api.permute_rope(p, idx, bat(x), inverse=True)) for x in (dq, dk))
    o, dv = (unb(api.permute_tokens(p, idx, bat(x), inverse=True)) for x in (o, dv))
    l = unb(_lse_to_original(p, bat(l), idx))
    torch.cuda.synchronize()
    to_bf16 = lambda x: torch.from_numpy(x).to(torch.bfloat16).double().numpy()  # noqa: E731
    qo, ko = (to_bf16(RO.rotate(f64(x), pos)) for x in (q, k))
    if thd:
        seq, _ = A.token_meta_from_cu(cu)
        ro, rl = A.attention_forward(qo, ko, f64(v), seq, pos)
        rq, rk, rv = A.attention_backward(qo, ko, f64(v), f64(do), seq, pos)
    else:
        ro, rl = A.attention_forward_bshd(qo, ko, f64(v))
        rq, rk, rv = A.attention_backward_bshd(qo, ko, f64(v), f64(do))
    rq, rk = (RO.rotate(x, pos, inverse=True) for x in (rq, rk))
    assert max_abs(f64(o), ro) <= TOL_O_BF16
    assert max_abs(f64(l), rl) <= TOL_LSE_BF16
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        assert max_abs(f64(got), ref) <= TOL_GRAD_REL * float(np.max(np.abs(ref)))


# ------------------------------------------------------------ tile forward --
EDGES = [
    # q_row0, q_pos0, q_len, kv_row0, kv_pos0, kv_len, causal
    (0, 0, 256, 0, 0, 256, True),        # diagonal edge, two full tiles
    (300, 300, 77, 0, 0, 200, True),     # full edge, ragged lengths
    (130, 130, 150, 100, 100, 181, True),  # diagonal crossing tiles, ragged
    (0, 0, 64, 200, 200, 64, True),      # every query before every key: empty rows
    (10, 10, 129, 400, 400, 111, False),  # non-causal
    # 256-row items of the bf16 kernel (two Q tiles per item):
    (0, 0, 300, 128, 128, 256, True),    # first Q tile sees no key, the second does; ragged tail item
    (40, 40, 256, 0, 0, 400, True),      # first Q tile sees a prefix of the second's key tiles
    (0, 0, 512, 0, 0, 512, True),        # two diagonal items
    (5, 5, 200, 0, 0, 512, False),       # non-causal, ragged second Q tile
]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("edge", EDGES)
def test_tile_attn_fwd_single_edge(dtype, edge):
    q_row0, q_pos0, q_len, kv_row0, kv_pos0, kv_len, causal = edge
    b, s, H, Hkv, d = 2, 512, 4, 2, (64 if dtype == torch.float32 else 128)
    q, k, v = make_inputs(b, s, H, Hkv, d, seed=11, dtype=dtype)
    p = _prob(batch=b, heads_q=H, heads_kv=Hkv, head_dim=d, cp=1, seqlen=s, dtype=dtype,
              causal=causal)
    o, l = api.tile_attn_fwd(p, q.to(DEV), k.to(DEV), v.to(DEV), q_row0, q_pos0, q_len,
                             kv_row0, kv_pos0, kv_len)
    torch.cuda.synchronize()
    qpos = np.arange(q_pos0, q_pos0 + q_len)
    kpos = np.arange(kv_pos0, kv_pos0 + kv_len)
    vis = A.visibility(np.zeros(q_len), qpos, np.zeros(kv_len), kpos, causal)
    tol_o = TOL_F32 if dtype == torch.float32 else TOL_O_BF16
    tol_l = TOL_F32 if dtype == torch.float32 else TOL_LSE_BF16
    for bi in range(b):
        ro, rl = A.masked_attention(f64(q[bi, q_row0:q_row0 + q_len]), f64(k[bi, kv_row0:kv_row0 + kv_len]),
                                    f64(v[bi, kv_row0:kv_row0 + kv_len]), vis)
        go, gl = f64(o[bi]), f64(l[bi])
        empty = ~vis.any(1)
        assert np.all(np.isneginf(gl[empty])) and np.all(go[empty] == 0)
        assert max_abs(go, ro) <= tol_o
        fin = ~empty
        assert max_abs(gl[fin], rl[fin]) <= tol_l


WINDOW_EDGES = [
    # q_row0, q_pos0, q_len, kv_row0, kv_pos0, kv_len, window
    (0, 0, 256, 0, 0, 256, 100),         # diagonal edge, band narrower than a tile
    (300, 300, 200, 0, 0, 400, 150),     # band cuts the key range on both sides
    (256, 256, 256, 0, 0, 256, 128),     # tile-aligned band: the second Q tile sees one key tile
    (40, 40, 300, 0, 0, 400, 1),         # every query sees its own key only
    (0, 400, 64, 0, 0, 64, 200),         # keys all older than the band: empty rows
]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("edge", WINDOW_EDGES)
def test_tile_attn_fwd_window(dtype, edge):
    q_row0, q_pos0, q_len, kv_row0, kv_pos0, kv_len, w = edge
    b, s, H, Hkv, d = 1, 512, 2, 1, (64 if dtype == torch.float32 else 128)
    q, k, v = make_inputs(b, s, H, Hkv, d, seed=12, dtype=dtype)
    p = _prob(batch=b, heads_q=H, heads_kv=Hkv, head_dim=d, cp=1, seqlen=s, dtype=dtype, window=w)
    o, l = api.tile_attn_fwd(p, q.to(DEV), k.to(DEV), v.to(DEV), q_row0, q_pos0, q_len,
                             kv_row0, kv_pos0, kv_len)
    torch.cuda.synchronize()
    qpos = np.arange(q_pos0, q_pos0 + q_len)
    kpos = np.arange(kv_pos0, kv_pos0 + kv_len)
    vis = A.visibility(np.zeros(q_len), qpos, np.zeros(kv_len), kpos, True, w)
    ro, rl = A.masked_attention(f64(q[0, q_row0:q_row0 + q_len]), f64(k[0, kv_row0:kv_row0 + kv_len]),
                                f64(v[0, kv_row0:kv_row0 + kv_len]), vis)
    go, gl = f64(o[0]), f64(l[0])
    empty = ~vis.any(1)
    assert np.all(np.isneginf(gl[empty])) and np.all(go[empty] == 0)
    assert max_abs(go, ro) <= (TOL_F32 if dtype == torch.float32 else TOL_O_BF16)
    assert max_abs(gl[~empty], rl[~empty]) <= (TOL_F32 if dtype == torch.float32 else TOL_LSE_BF16)


# ----------------------------------- forward: a rising running maximum --
RISING_EDGES = [
    # q_row0, q_pos0, q_len, kv_row0, kv_pos0, kv_len, causal
    (0, 0, 256, 0, 0, 1024, False),         # both Q tiles see all 8 key tiles
    (768, 768, 256, 0, 0, 1024, True),      # diagonal item: 7 and 8 key tiles
    (1024, 1024, 300, 0, 0, 1324, True),    # diagonal, ragged tail item and key tile
]


@pytest.mark.parametrize("edge", RISING_EDGES)
def test_tile_attn_fwd_rising_max(edge):
    """The correction of the online recurrence with a finite running maximum
    ("上下文并行" 02 ONE ROW: c = e^(m - m'), l' = c l + ..., a' = c a + ...):
    keys scaled up with position lift most rows' maximum mid-stream by more
    than the kernel's lazy threshold, so O and l must be rescaled in flight;
    a skipped or misapplied correction misses the oracle by far more than the
    parity bar."""
    q_row0, q_pos0, q_len, kv_row0, kv_pos0, kv_len, causal = edge
    b, s, H, Hkv, d = 1, 1536, 2, 1, 128
    q, k, v = make_inputs(b, s, H, Hkv, d, seed=23, dtype=torch.bfloat16)
    k = ramp_keys(k, slope=10.0)
    p = _prob(batch=b, heads_q=H, heads_kv=Hkv, head_dim=d, cp=1, seqlen=s, causal=causal)
    o, l = api.tile_attn_fwd(p, q.to(DEV), k.to(DEV), v.to(DEV), q_row0, q_pos0, q_len,
                             kv_row0, kv_pos0, kv_len)
    torch.cuda.synchronize()
    qpos = np.arange(q_pos0, q_pos0 + q_len)
    kpos = np.arange(kv_pos0, kv_pos0 + kv_len)
    vis = A.visibility(np.zeros(q_len), qpos, np.zeros(kv_len), kpos, causal)
    qs, ks, vs = q[0, q_row0:q_row0 + q_len], k[0, kv_row0:kv_row0 + kv_len], v[0, kv_row0:kv_row0 + kv_len]
    grow = max_growth(qs, ks, vis)
    assert np.mean(grow > RESCALE_NATS + 1.0) >= 0.5   # the inputs do drive the correction
    ro, rl = A.masked_attention(f64(qs), f64(ks), f64(vs), vis)
    assert max_abs(f64(o[0]), ro) <= TOL_O_BF16
    assert max_abs(f64(l[0]), rl) <= TOL_LSE_BF16


@pytest.mark.parametrize("part", [api.CP_PARTITION_ZIGZAG, api.CP_PARTITION_STRIPED])
def test_ring_fwd_bwd_window_rising_max(part):
    """The same correction on the sliding-window path (band masks on the
    boundary tiles), forward and backward against the oracle."""
    b, s, H, Hkv, d, cp, w = 1, 2048, 2, 2, 128, 4, 1000
    q, k, v, do = make_inputs(b, s, H, Hkv, d, 29, torch.bfloat16, with_do=True)
    k = ramp_keys(k, slope=20.0)
    p = _prob(batch=b, heads_q=H, heads_kv=Hkv, head_dim=d, cp=cp, seqlen=s, dtype=torch.bfloat16,
              order=api.CP_ORDER_RANK_LOCAL, partition=part, window=w)
    idx, _ = api.partition_indices(p)
    qd, kd, vd, dod = (api.permute_tokens(p, idx, x.to(DEV)) for x in (q, k, v, do))
    o, l = api.ring_attn_fwd(p, qd, kd, vd)
    dq, dk, dv = api.ring_attn_bwd(p, qd, kd, vd, o, l, dod)
    assert api.device_error() == 0
    o, dq, dk, dv = (api.permute_tokens(p, idx, x, inverse=True) for x in (o, dq, dk, dv))
    l = _lse_to_original(p, l, idx)
    torch.cuda.synchronize()
    pos = np.arange(s)
    vis = A.visibility(np.zeros(s), pos, np.zeros(s), pos, True, w)
    span = 128 if part == api.CP_PARTITION_ZIGZAG else 128 * cp + cp
    assert np.mean(max_growth(q[0], k[0], vis, span=span) > RESCALE_NATS + 1.0) >= 0.5
    ref_f = [x[0] for x in A.attention_forward_bshd(f64(q), f64(k), f64(v), window=w)]
    ref_b = [x[0] for x in A.attention_backward_bshd(f64(q), f64(k), f64(v), f64(do), window=w)]
    _ring_check(p, q, k, v, do, o[0], l[0], dq[0], dk[0], dv[0], torch.bfloat16, ref_f, ref_b)


# ------------------------------------------------------------------ merge --
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("n_parts,d", [(1, 128), (5, 64), (16, 128), (40, 128)])
def test_merge_partials(out_dtype, n_parts, d):
    rows, H = 333, 3
    g = torch.Generator().manual_seed(n_parts * 100 + d)
    o = torch.randn(n_parts, rows, H, d, generator=g)
    l = torch.randn(n_parts, rows, H, generator=g) * 4
    drop = torch.rand(n_parts, rows, H, generator=g) < 0.3
    l[drop] = float("-inf")
    l[:, 7, :] = float("-inf")        # a row whose partials are all empty
    o[drop] = 0.0
    go, gl = api.merge_partials(o.to(DEV), l.to(DEV), out_dtype)
    torch.cuda.synchronize()
    ro, rl = A.lse_merge(o.double().numpy(), l.double().numpy())
    tol = TOL_F32 if out_dtype == torch.float32 else TOL_O_BF16
    assert max_abs(f64(go), ro) <= tol
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(f64(gl)), fin)
    assert max_abs(f64(gl)[fin], rl[fin]) <= TOL_F32 * 10
    assert np.all(f64(go)[7] == 0)


# ------------------------------------------------------------- ring small --
def _ring_case(b, s, H, Hkv, d, cp, dtype, order, seed, cu=None):
    thd = cu is not None
    q, k, v, do = make_inputs(b, s, H, Hkv, d, seed, dtype, with_do=True, thd=thd)
    p = _prob(batch=b, heads_q=H, heads_kv=Hkv, head_dim=d, cp=cp, seqlen=s, dtype=dtype,
              cu_seqlens=cu, order=order)
    return p, q, k, v, do


def _to_order(p, x, idx):
    """Original -> the problem's token order (through the library's permute)."""
    if p.order == api.CP_ORDER_ORIGINAL:
        return x
    return api.permute_tokens(p, idx, x)


def _from_order(p, x, idx):
    if p.order == api.CP_ORDER_ORIGINAL:
        return x
    return api.permute_tokens(p, idx, x, inverse=True)


def _lse_to_original(p, l, idx):
    """Scatter a rank-local [.., s, H] LSE back to original order (test-side indexing)."""
    if p.order == api.CP_ORDER_ORIGINAL:
        return l
    out = torch.empty_like(l)
    out[..., idx.reshape(-1).long(), :] = l
    return out


RING = [
    # b, s, H, Hkv, d, cp, dtype, order
    (1, 256, 1, 1, 64, 2, torch.float32, api.CP_ORDER_ORIGINAL),
    (2, 512, 2, 1, 64, 4, torch.float32, api.CP_ORDER_RANK_LOCAL),
    (1, 1024, 4, 4, 128, 2, torch.bfloat16, api.CP_ORDER_ORIGINAL),
    (2, 2048, 4, 2, 128, 8, torch.bfloat16, api.CP_ORDER_RANK_LOCAL),
    (1, 768, 2, 2, 128, 3, torch.bfloat16, api.CP_ORDER_ORIGINAL),
    (1, 512, 2, 2, 128, 1, torch.bfloat16, api.CP_ORDER_ORIGINAL),
]


@pytest.mark.parametrize("case", RING)
def test_ring_fwd_bwd_bshd(case):
    b, s, H, Hkv, d, cp, dtype, order = case
    p, q, k, v, do = _ring_case(b, s, H, Hkv, d, cp, dtype, order, seed=5)
    idx, _ = api.partition_indices(p)
    qd, kd, vd, dod = (_to_order(p, x.to(DEV), idx) for x in (q, k, v, do))
    o, l = api.ring_attn_fwd(p, qd, kd, vd)
    dq, dk, dv = api.ring_attn_bwd(p, qd, kd, vd, o, l, dod)
    assert api.device_error() == 0
    o, dq, dk, dv = (_from_order(p, x, idx) for x in (o, dq, dk, dv))
    l = _lse_to_original(p, l, idx)
    torch.cuda.synchronize()
    tol_o = TOL_F32 if dtype == torch.float32 else TOL_O_BF16
    tol_l = TOL_F32 if dtype == torch.float32 else TOL_LSE_BF16
    for bi in range(b):
        ro, rl = A.attention_forward_bshd(f64(q[bi:bi + 1]), f64(k[bi:bi + 1]), f64(v[bi:bi + 1]))
        assert max_abs(f64(o[bi]), ro[0]) <= tol_o
        assert max_abs(f64(l[bi]), rl[0]) <= tol_l
        # the forward output the backward uses is the GPU's own (rounded) O, as in training;
        # gradients are compared against the oracle's exact gradients
        rq, rk, rv = A.attention_backward_bshd(f64(q[bi:bi + 1]), f64(k[bi:bi + 1]), f64(v[bi:bi + 1]),
                                               f64(do[bi:bi + 1]))
        for got, ref in ((dq[bi], rq[0]), (dk[bi], rk[0]), (dv[bi], rv[0])):
            scale = np.max(np.abs(ref))
            tol = TOL_F32 * max(1.0, scale) if dtype == torch.float32 else TOL_GRAD_REL * scale
            assert max_abs(f64(got), ref) <= tol


@pytest.mark.parametrize("order", [api.CP_ORDER_ORIGINAL, api.CP_ORDER_RANK_LOCAL])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_ring_fwd_bwd_thd(order, dtype):
    cp = 4
    lens = [8, 64, 200, 16, 1000, 8, 248]      # short sub-sequences: tiles span several
    cu = cu_from_lengths(lens)
    T = int(cu[-1])
    H, Hkv = 4, 2
    d = 64 if dtype == torch.float32 else 128
    p, q, k, v, do = _ring_case(1, T, H, Hkv, d, cp, dtype, order, seed=9, cu=cu)
    idx, _ = api.partition_indices(p)
    qd, kd, vd, dod = (_to_order(p, x.to(DEV), idx) for x in (q, k, v, do))
    o, l = api.ring_attn_fwd(p, qd, kd, vd)
    dq, dk, dv = api.ring_attn_bwd(p, qd, kd, vd, o, l, dod)
    assert api.device_error() == 0
    o, dq, dk, dv = (_from_order(p, x, idx) for x in (o, dq, dk, dv))
    l = _lse_to_original(p, l, idx)
    torch.cuda.synchronize()
    seq, pos = A.token_meta_from_cu(cu)
    ro, rl = A.attention_forward(f64(q), f64(k), f64(v), seq, pos)
    tol_o = TOL_F32 if dtype == torch.float32 else TOL_O_BF16
    assert max_abs(f64(o), ro) <= tol_o
    tol_l = TOL_F32 if dtype == torch.float32 else TOL_LSE_BF16
    assert max_abs(f64(l), rl) <= tol_l
    rq, rk, rv = A.attention_backward(f64(q), f64(k), f64(v), f64(do), seq, pos)
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        scale = np.max(np.abs(ref))
        tol = TOL_F32 * max(1.0, scale) if dtype == torch.float32 else TOL_GRAD_REL * scale
        assert max_abs(f64(got), ref) <= tol


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_ring_fwd_bwd_thd_with_empty_sub_sequences(dtype):
    """A packed batch whose sub-sequences include empty ones (first, middle
    and last): they own no token, no chunk and no edge, and the others are
    computed as if they were alone."""
    cp = 4
    lens = [0, 16, 0, 0, 296, 8, 0]
    cu = cu_from_lengths(lens)
    T = int(cu[-1])
    d = 64 if dtype == torch.float32 else 128
    p, q, k, v, do = _ring_case(1, T, 2, 2, d, cp, dtype, api.CP_ORDER_ORIGINAL, seed=41, cu=cu)
    qd, kd, vd, dod = (x.to(DEV) for x in (q, k, v, do))
    o, l = api.ring_attn_fwd(p, qd, kd, vd)
    dq, dk, dv = api.ring_attn_bwd(p, qd, kd, vd, o, l, dod)
    assert api.device_error() == 0
    torch.cuda.synchronize()
    seq, pos = A.token_meta_from_cu(cu)
    ro, rl = A.attention_forward(f64(q), f64(k), f64(v), seq, pos)
    assert max_abs(f64(o), ro) <= (TOL_F32 if dtype == torch.float32 else TOL_O_BF16)
    assert max_abs(f64(l), rl) <= (TOL_F32 if dtype == torch.float32 else TOL_LSE_BF16)
    rq, rk, rv = A.attention_backward(f64(q), f64(k), f64(v), f64(do), seq, pos)
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        scale = np.max(np.abs(ref))
        tol = TOL_F32 * max(1.0, scale) if dtype == torch.float32 else TOL_GRAD_REL * scale
        assert max_abs(f64(got), ref) <= tol


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_ring_fwd_bwd_empty_problem(dtype):
    """No tokens at all (BSHD seqlen 0, and a packed batch of empty
    sub-sequences): both calls succeed, launch nothing that fails and leave
    the device error word clear."""
    d = 64 if dtype == torch.float32 else 128
    for cu in (None, [0, 0, 0]):
        p = _prob(batch=1, heads_q=2, heads_kv=2, head_dim=d, cp=2, seqlen=0, dtype=dtype, cu_seqlens=cu)
        shape = (0, 2, d) if cu is not None else (1, 0, 2, d)
        q = torch.zeros(shape, dtype=dtype, device=DEV)
        o, l = api.ring_attn_fwd(p, q, q, q)
        dq, dk, dv = api.ring_attn_bwd(p, q, q, q, o, l, q)
        assert o.numel() == 0 and l.numel() == 0 and dq.numel() == 0
        assert api.device_error() == 0


STRIPED_RING = [
    # b, s, H, Hkv, d, cp, dtype (s / cp rows per rank: ragged tiles included)
    (1, 256, 2, 1, 64, 4, torch.float32),
    (1, 96, 2, 2, 64, 3, torch.float32),
    (2, 1000, 4, 2, 128, 8, torch.bfloat16),
    (1, 2304, 4, 4, 128, 3, torch.bfloat16),
    (2, 2048, 4, 2, 128, 8, torch.bfloat16),
    (1, 512, 2, 2, 128, 1, torch.bfloat16),
]


def _ring_check(p, q, k, v, do, o, l, dq, dk, dv, dtype, ref_f, ref_b):
    tol_o = TOL_F32 if dtype == torch.float32 else TOL_O_BF16
    tol_l = TOL_F32 if dtype == torch.float32 else TOL_LSE_BF16
    ro, rl = ref_f
    assert max_abs(f64(o), ro) <= tol_o
    assert max_abs(f64(l), rl) <= tol_l
    for got, ref in zip((dq, dk, dv), ref_b):
        # a gradient that is exactly zero (a band of one key: dS = P (dP - D)
        # = 0) is held to the float32 rounding of dP - D, under 1e-3 x 3e-2
        scale = max(float(np.max(np.abs(ref))), 1e-3)
        tol = TOL_F32 * max(1.0, scale) if dtype == torch.float32 else TOL_GRAD_REL * scale
        assert max_abs(f64(got), ref) <= tol


@pytest.mark.parametrize("case", STRIPED_RING)
def test_ring_fwd_bwd_striped_bshd(case):
    """Striped split ("Sequence Parallelism + Ring Attention" §5): rank-local
    tensors in, exact causal attention by original position out."""
    b, s, H, Hkv, d, cp, dtype = case
    q, k, v, do = make_inputs(b, s, H, Hkv, d, 11, dtype, with_do=True)
    p = _prob(batch=b, heads_q=H, heads_kv=Hkv, head_dim=d, cp=cp, seqlen=s, dtype=dtype, **STRIPED)
    idx, _ = api.partition_indices(p)
    qd, kd, vd, dod = (api.permute_tokens(p, idx, x.to(DEV)) for x in (q, k, v, do))
    o, l = api.ring_attn_fwd(p, qd, kd, vd)
    dq, dk, dv = api.ring_attn_bwd(p, qd, kd, vd, o, l, dod)
    assert api.device_error() == 0
    o, dq, dk, dv = (api.permute_tokens(p, idx, x, inverse=True) for x in (o, dq, dk, dv))
    l = _lse_to_original(p, l, idx)
    torch.cuda.synchronize()
    for bi in range(b):
        sl = slice(bi, bi + 1)
        ref_f = [x[0] for x in A.attention_forward_bshd(f64(q[sl]), f64(k[sl]), f64(v[sl]))]
        ref_b = [x[0] for x in A.attention_backward_bshd(f64(q[sl]), f64(k[sl]), f64(v[sl]), f64(do[sl]))]
        _ring_check(p, q, k, v, do, o[bi], l[bi], dq[bi], dk[bi], dv[bi], dtype, ref_f, ref_b)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_ring_fwd_bwd_striped_thd(dtype):
    cp = 4
    lens = [12, 4, 200, 36, 1000, 8, 252, 0, 4]   # multiples of cp, not all of 2cp
    cu = cu_from_lengths(lens)
    T = int(cu[-1])
    H, Hkv = 4, 2
    d = 64 if dtype == torch.float32 else 128
    q, k, v, do = make_inputs(1, T, H, Hkv, d, 13, dtype, with_do=True, thd=True)
    p = _prob(batch=1, heads_q=H, heads_kv=Hkv, head_dim=d, cp=cp, seqlen=T, dtype=dtype, cu_seqlens=cu,
              **STRIPED)
    idx, _ = api.partition_indices(p)
    qd, kd, vd, dod = (api.permute_tokens(p, idx, x.to(DEV)) for x in (q, k, v, do))
    o, l = api.ring_attn_fwd(p, qd, kd, vd)
    dq, dk, dv = api.ring_attn_bwd(p, qd, kd, vd, o, l, dod)
    assert api.device_error() == 0
    o, dq, dk, dv = (api.permute_tokens(p, idx, x, inverse=True) for x in (o, dq, dk, dv))
    l = _lse_to_original(p, l, idx)
    torch.cuda.synchronize()
    seq, pos = A.token_meta_from_cu(cu)
    ref_f = A.attention_forward(f64(q), f64(k), f64(v), seq, pos)
    ref_b = A.attention_backward(f64(q), f64(k), f64(v), f64(do), seq, pos)
    _ring_check(p, q, k, v, do, o, l, dq, dk, dv, dtype, ref_f, ref_b)


WINDOW_RING = [
    # b, s, H, Hkv, d, cp, dtype, window, partition
    (1, 512, 2, 1, 64, 2, torch.float32, 100, api.CP_PARTITION_ZIGZAG),
    (2, 2048, 4, 2, 128, 4, torch.bfloat16, 300, api.CP_PARTITION_ZIGZAG),
    (1, 2048, 2, 2, 128, 8, torch.bfloat16, 128, api.CP_PARTITION_ZIGZAG),
    (1, 1024, 2, 2, 128, 2, torch.bfloat16, 1, api.CP_PARTITION_ZIGZAG),
    (1, 2048, 4, 2, 128, 4, torch.bfloat16, 2048, api.CP_PARTITION_ZIGZAG),   # band = whole sequence
    (1, 1000, 2, 1, 64, 8, torch.float32, 77, api.CP_PARTITION_STRIPED),
    (2, 2048, 4, 2, 128, 8, torch.bfloat16, 500, api.CP_PARTITION_STRIPED),
    (1, 768, 2, 2, 128, 3, torch.bfloat16, 5, api.CP_PARTITION_STRIPED),
]


@pytest.mark.parametrize("case", WINDOW_RING)
def test_ring_fwd_bwd_window_bshd(case):
    """Sliding window ("Context Parallelism (CP)" §2.1: a sparser edge set):
    exact banded causal attention and gradients, rank-local tensors."""
    b, s, H, Hkv, d, cp, dtype, w, part = case
    q, k, v, do = make_inputs(b, s, H, Hkv, d, 21, dtype, with_do=True)
    p = _prob(batch=b, heads_q=H, heads_kv=Hkv, head_dim=d, cp=cp, seqlen=s, dtype=dtype,
              order=api.CP_ORDER_RANK_LOCAL, partition=part, window=w)
    idx, _ = api.partition_indices(p)
    qd, kd, vd, dod = (api.permute_tokens(p, idx, x.to(DEV)) for x in (q, k, v, do))
    o, l = api.ring_attn_fwd(p, qd, kd, vd)
    dq, dk, dv = api.ring_attn_bwd(p, qd, kd, vd, o, l, dod)
    assert api.device_error() == 0
    o, dq, dk, dv = (api.permute_tokens(p, idx, x, inverse=True) for x in (o, dq, dk, dv))
    l = _lse_to_original(p, l, idx)
    torch.cuda.synchronize()
    for bi in range(b):
        sl = slice(bi, bi + 1)
        ref_f = [x[0] for x in A.attention_forward_bshd(f64(q[sl]), f64(k[sl]), f64(v[sl]), window=w)]
        ref_b = [x[0] for x in A.attention_backward_bshd(f64(q[sl]), f64(k[sl]), f64(v[sl]), f64(do[sl]),
                                                         window=w)]
        _ring_check(p, q, k, v, do, o[bi], l[bi], dq[bi], dk[bi], dv[bi], dtype, ref_f, ref_b)


@pytest.mark.parametrize("dtype,order", [(torch.float32, api.CP_ORDER_ORIGINAL),
                                         (torch.bfloat16, api.CP_ORDER_RANK_LOCAL)])
def test_ring_fwd_bwd_window_thd(dtype, order):
    cp, w = 4, 150
    lens = [8, 64, 200, 16, 1000, 8, 248]
    cu = cu_from_lengths(lens)
    T = int(cu[-1])
    H, Hkv = 4, 2
    d = 64 if dtype == torch.float32 else 128
    p, q, k, v, do = _ring_case(1, T, H, Hkv, d, cp, dtype, order, seed=22, cu=cu)
    p = _prob(batch=1, heads_q=H, heads_kv=Hkv, head_dim=d, cp=cp, seqlen=T, dtype=dtype, cu_seqlens=cu,
              order=order, window=w)
    idx, _ = api.partition_indices(p)
    qd, kd, vd, dod = (_to_order(p, x.to(DEV), idx) for x in (q, k, v, do))
    o, l = api.ring_attn_fwd(p, qd, kd, vd)
    dq, dk, dv = api.ring_attn_bwd(p, qd, kd, vd, o, l, dod)
    assert api.device_error() == 0
    o, dq, dk, dv = (_from_order(p, x, idx) for x in (o, dq, dk, dv))
    l = _lse_to_original(p, l, idx)
    torch.cuda.synchronize()
    seq, pos = A.token_meta_from_cu(cu)
    ref_f = A.attention_forward(f64(q), f64(k), f64(v), seq, pos, window=w)
    ref_b = A.attention_backward(f64(q), f64(k), f64(v), f64(do), seq, pos, window=w)
    _ring_check(p, q, k, v, do, o, l, dq, dk, dv, dtype, ref_f, ref_b)


# --------------------------------------------------------------- hybrid CP --
def _hybrid_rounds(lens, world, cap):
    """Rounds of the library's schedule: (sub-stream cu, cp per sequence, rank0, original rows)."""
    rnd, cp, r0, n = api.hybrid_schedule(lens, world, cap)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    out = []
    for r in range(n):
        ks = [i for i in range(len(lens)) if rnd[i] == r]
        sub_cu = cu_from_lengths([lens[i] for i in ks])
        rows = np.concatenate([np.arange(cu[i], cu[i + 1]) for i in ks]) if ks else np.zeros(0, np.int64)
        out.append((sub_cu, cp[ks], r0[ks], rows))
    return out


@pytest.mark.parametrize("seed,world,cap", [(0, 8, 2048), (1, 4, 4096), (2, 16, 512)])
def test_partition_hybrid_bitexact(seed, world, cap):
    """Each round of a hybrid schedule ("04 · Megatron-LM 实现" §7): slot table
    and index, bit-exact against the oracle's layout."""
    rng = np.random.default_rng(seed)
    raw = np.exp(rng.normal(np.log(cap) - 0.5, 1.3, 40))
    lens = [int(min(world * cap, max(2 * world, x)) // (2 * world) * (2 * world)) for x in raw]
    for sub_cu, gcp, g0, _ in _hybrid_rounds(lens, world, cap):
        T = int(sub_cu[-1])
        p = _prob(batch=1, heads_q=1, heads_kv=1, head_dim=64, cp=world, seqlen=T, cu_seqlens=sub_cu,
                  seq_cp=gcp, seq_rank0=g0, order=api.CP_ORDER_RANK_LOCAL)
        idx, lcu = api.partition_indices(p)
        torch.cuda.synchronize()
        ridx, rlcu = HY.hybrid_layout(sub_cu, gcp, g0, world)
        assert np.array_equal(idx.cpu().numpy(), ridx)
        assert np.array_equal(lcu.cpu().numpy(), rlcu)


@pytest.mark.parametrize("dtype,order", [(torch.bfloat16, api.CP_ORDER_RANK_LOCAL),
                                         (torch.bfloat16, api.CP_ORDER_ORIGINAL),
                                         (torch.float32, api.CP_ORDER_RANK_LOCAL)])
def test_ring_fwd_bwd_hybrid_round(dtype, order):
    """One hybrid round: sequences of CP size 1 .. world on their own groups,
    ranks of different lengths; exact attention and gradients."""
    world = 4
    lens = [512, 64, 256, 8, 128, 0, 40, 384]
    seq_cp, seq_r0 = [4, 1, 2, 1, 1, 1, 2, 2], [0, 3, 2, 2, 0, 1, 0, 2]
    cu = cu_from_lengths(lens)
    T, H, Hkv = int(cu[-1]), 4, 2
    d = 64 if dtype == torch.float32 else 128
    q, k, v, do = make_inputs(1, T, H, Hkv, d, 31, dtype, with_do=True, thd=True)
    p = _prob(batch=1, heads_q=H, heads_kv=Hkv, head_dim=d, cp=world, seqlen=T, dtype=dtype, cu_seqlens=cu,
              order=order, seq_cp=seq_cp, seq_rank0=seq_r0)
    idx, _ = api.partition_indices(p)
    qd, kd, vd, dod = (_to_order(p, x.to(DEV), idx) for x in (q, k, v, do))
    o, l = api.ring_attn_fwd(p, qd, kd, vd)
    dq, dk, dv = api.ring_attn_bwd(p, qd, kd, vd, o, l, dod)
    assert api.device_error() == 0
    o, dq, dk, dv = (_from_order(p, x, idx) for x in (o, dq, dk, dv))
    l = _lse_to_original(p, l, idx)
    torch.cuda.synchronize()
    seq, pos = A.token_meta_from_cu(cu)
    ref_f = A.attention_forward(f64(q), f64(k), f64(v), seq, pos)
    ref_b = A.attention_backward(f64(q), f64(k), f64(v), f64(do), seq, pos)
    _ring_check(p, q, k, v, do, o, l, dq, dk, dv, dtype, ref_f, ref_b)


def test_ring_hybrid_schedule_rounds_bf16():
    """Every round of a scheduled long-tail batch through the ring, against
    the oracle on the round's own packed stream."""
    world, cap = 8, 1024
    rng = np.random.default_rng(7)
    raw = np.exp(rng.normal(np.log(cap) - 0.7, 1.2, 24))
    lens = [int(min(world * cap, max(2 * world, x)) // (2 * world) * (2 * world)) for x in raw]
    H, Hkv, d = 2, 1, 128
    for sub_cu, gcp, g0, _ in _hybrid_rounds(lens, world, cap):
        T = int(sub_cu[-1])
        q, k, v, do = make_inputs(1, T, H, Hkv, d, 41, torch.bfloat16, with_do=True, thd=True)
        p = _prob(batch=1, heads_q=H, heads_kv=Hkv, head_dim=d, cp=world, seqlen=T, cu_seqlens=sub_cu,
                  order=api.CP_ORDER_RANK_LOCAL, seq_cp=gcp, seq_rank0=g0)
        idx, _ = api.partition_indices(p)
        qd, kd, vd, dod = (api.permute_tokens(p, idx, x.to(DEV)) for x in (q, k, v, do))
        o, l = api.ring_attn_fwd(p, qd, kd, vd)
        dq, dk, dv = api.ring_attn_bwd(p, qd, kd, vd, o, l, dod)
        assert api.device_error() == 0
        o, dq, dk, dv = (api.permute_tokens(p, idx, x, inverse=True) for x in (o, dq, dk, dv))
        l = _lse_to_original(p, l, idx)
        torch.cuda.synchronize()
        seq, pos = A.token_meta_from_cu(sub_cu)
        ref_f = A.attention_forward(f64(q), f64(k), f64(v), seq, pos)
        ref_b = A.attention_backward(f64(q), f64(k), f64(v), f64(do), seq, pos)
        _ring_check(p, q, k, v, do, o, l, dq, dk, dv, torch.bfloat16, ref_f, ref_b)


def test_ring_partials_match_oracle_edges():
    """The ring forward's merged result equals the oracle's ring walk, and the
    single-edge entry point reproduces one of the oracle's partial states."""
    cp, s, H, d = 2, 256, 1, 64
    q, k, v = make_inputs(1, s, H, H, d, seed=3, dtype=torch.float32)
    cu = [0, s]
    ro, rl, parts = R.ring_forward(f64(q[0]), f64(k[0]), f64(v[0]), cu, cp, return_partials=True)
    # rank 1 at ring step 1 holds the K/V of rank 0: chunks 0 and 3 (64 tokens each)
    # for its query chunk 1 (positions 64..127) only chunk 0 is visible
    p = _prob(batch=1, heads_q=H, heads_kv=H, head_dim=d, cp=cp, seqlen=s, dtype=torch.float32)
    o, l = api.tile_attn_fwd(p, q.to(DEV), k.to(DEV), v.to(DEV), 64, 64, 64, 0, 0, 64)
    torch.cuda.synchronize()
    o_r1_t1, l_r1_t1 = parts[1][0][1], parts[1][1][1]    # rank 1, step 1, rank-local rows
    assert max_abs(f64(o[0]), o_r1_t1[:64]) <= TOL_F32
    assert max_abs(f64(l[0]), l_r1_t1[:64]) <= TOL_F32


def test_invalid_arguments_rejected_on_host():
    p = _prob(batch=1, heads_q=2, heads_kv=2, head_dim=128, cp=2, seqlen=256)
    q = torch.zeros(1, 256, 2, 128, dtype=torch.bfloat16, device=DEV)
    ws = api.workspace(p)
    small = ws[: ws.numel() // 2]
    with pytest.raises(api.CpError) as e:
        api.ring_attn_fwd(p, q, q, q, ws=small)
    assert e.value.code == -4
    with pytest.raises(api.CpError) as e:
        api.tile_attn_fwd(p, q, q, q, 200, 200, 100, 0, 0, 10)   # q range leaves the tensor
    assert e.value.code == -1
    assert api.device_error() == 0
