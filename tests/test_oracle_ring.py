"""Pins for the oracle's ring pipeline: sharded results equal the plain
definition ("Context Parallelism (CP)" §2.2: the merge of every edge's partial
state is exact attention; "上下文并行" 01-05: sharded replay with gradients
returned to their owner equals the full reference)."""

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import ring as R


@pytest.mark.parametrize("cu,cp,H,Hkv", [
    ([0, 64], 2, 2, 2),
    ([0, 96], 3, 2, 1),
    ([0, 16, 48, 64, 128], 2, 4, 2),
    ([0, 8, 40], 4, 1, 1),
])
def test_ring_forward_equals_full(cu, cp, H, Hkv):
    rng = np.random.default_rng(0)
    T, d = cu[-1], 8
    q = rng.standard_normal((T, H, d))
    k = rng.standard_normal((T, Hkv, d))
    v = rng.standard_normal((T, Hkv, d))
    seq, pos = A.token_meta_from_cu(cu)
    ref_o, ref_l = A.attention_forward(q, k, v, seq, pos, True)
    o, l, parts = R.ring_forward(q, k, v, cu, cp, return_partials=True)
    assert np.max(np.abs(o - ref_o)) < 1e-12
    assert np.max(np.abs(l - ref_l)) < 1e-12
    assert len(parts) == cp and all(len(p[0]) == cp for p in parts)


@pytest.mark.parametrize("cu,cp", [([0, 64], 2), ([0, 16, 48, 64, 128], 2), ([0, 96], 3)])
def test_ring_backward_equals_full(cu, cp):
    rng = np.random.default_rng(1)
    T, H, Hkv, d = cu[-1], 2, 1, 8
    q = rng.standard_normal((T, H, d))
    k = rng.standard_normal((T, Hkv, d))
    v = rng.standard_normal((T, Hkv, d))
    do = rng.standard_normal((T, H, d))
    seq, pos = A.token_meta_from_cu(cu)
    ref = A.attention_backward(q, k, v, do, seq, pos, True)
    got = R.ring_backward(q, k, v, do, cu, cp)
    for a, b in zip(got, ref):
        assert np.max(np.abs(a - b)) < 1e-11


def test_two_owner_uneven_lab_setup():
    """Five positions, 2-D vectors, owners {0,1} and {2,3,4}, upstream G/5
    (global mean), binary64: sharded forward, replay and gradient return give
    the full autograd reference.  The page's printed values were lost in
    extraction; this pins the setup by the equality it asserts."""
    rng = np.random.default_rng(2026)
    n, d = 5, 2
    q = rng.standard_normal((n, 1, d))
    k = rng.standard_normal((n, 1, d))
    v = rng.standard_normal((n, 1, d))
    G = rng.standard_normal((n, 1, d))
    owners = [np.array([0, 1]), np.array([2, 3, 4])]
    seq, pos = np.zeros(n, int), np.arange(n)
    # forward: each rank keeps its queries and absorbs both owners' blocks
    out = np.zeros((n, 1, d))
    lse = np.zeros((n, 1))
    for r, qi in enumerate(owners):
        parts = []
        for t in range(2):
            kj = owners[(r - t) % 2]
            vis = A.visibility(seq[qi], pos[qi], seq[kj], pos[kj], True)
            parts.append(A.masked_attention(q[qi], k[kj], v[kj], vis))
        o_r, l_r = A.lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
        out[qi], lse[qi] = o_r, l_r
    # the block (rank 0 queries, rank 1 keys) is entirely masked: an empty block
    vis01 = A.visibility(seq[owners[0]], pos[owners[0]], seq[owners[1]], pos[owners[1]], True)
    assert not vis01.any()
    # backward with upstream G/5, replayed per block, dK/dV returned to owners
    do = G / 5
    delta = np.einsum("nhd,nhd->nh", do, out)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for qi in owners:
        for kj in owners:
            vis = A.visibility(seq[qi], pos[qi], seq[kj], pos[kj], True)
            a, b, c = A.block_backward(q[qi], k[kj], v[kj], do[qi], lse[qi], delta[qi], vis)
            dq[qi] += a
            dk[kj] += b
            dv[kj] += c
    tq, tk, tv = (torch.tensor(x[:, 0], requires_grad=True) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq[None], tk[None], tv[None], is_causal=True)[0]
    loss = (ref * torch.from_numpy(G[:, 0])).sum() / 5   # global mean over the 5 queries
    loss.backward()
    assert np.max(np.abs(out[:, 0] - ref.detach().numpy())) < 1e-14
    assert np.max(np.abs(dq[:, 0] - tq.grad.numpy())) < 1e-13
    assert np.max(np.abs(dk[:, 0] - tk.grad.numpy())) < 1e-13
    assert np.max(np.abs(dv[:, 0] - tv.grad.numpy())) < 1e-13


@pytest.mark.parametrize("cu,cp", [([0, 64], 4), ([0, 12, 36, 36, 60], 3), ([0, 40], 8)])
def test_striped_ring_equals_full(cu, cp):
    """The ring walk over the striped split ("Sequence Parallelism + Ring
    Attention" §5) gives exact attention and gradients as well."""
    rng = np.random.default_rng(7)
    T, H, Hkv, d = cu[-1], 2, 1, 8
    q = rng.standard_normal((T, H, d))
    k = rng.standard_normal((T, Hkv, d))
    v = rng.standard_normal((T, Hkv, d))
    do = rng.standard_normal((T, H, d))
    seq, pos = A.token_meta_from_cu(cu)
    ref_o, ref_l = A.attention_forward(q, k, v, seq, pos, True)
    o, l = R.ring_forward(q, k, v, cu, cp, partition="striped")
    assert np.max(np.abs(o - ref_o)) < 1e-12
    assert np.max(np.abs(l - ref_l)) < 1e-12
    ref = A.attention_backward(q, k, v, do, seq, pos, True)
    got = R.ring_backward(q, k, v, do, cu, cp, partition="striped")
    for a, b in zip(got, ref):
        assert np.max(np.abs(a - b)) < 1e-11


@pytest.mark.parametrize("cu,cp,W,partition", [
    ([0, 64], 2, 9, "zigzag"), ([0, 16, 48, 64, 128], 2, 5, "zigzag"),
    ([0, 64], 4, 7, "striped"), ([0, 12, 36, 36, 60], 3, 4, "striped"), ([0, 40], 8, 3, "striped"),
])
def test_window_ring_equals_full(cu, cp, W, partition):
    """The ring walk under a sliding window: whole edges drop out of the task
    graph, the merged result and the returned gradients stay exact."""
    rng = np.random.default_rng(8)
    T, H, Hkv, d = cu[-1], 2, 1, 8
    q = rng.standard_normal((T, H, d))
    k = rng.standard_normal((T, Hkv, d))
    v = rng.standard_normal((T, Hkv, d))
    do = rng.standard_normal((T, H, d))
    seq, pos = A.token_meta_from_cu(cu)
    ref_o, ref_l = A.attention_forward(q, k, v, seq, pos, True, window=W)
    o, l = R.ring_forward(q, k, v, cu, cp, partition=partition, window=W)
    assert np.max(np.abs(o - ref_o)) < 1e-12
    assert np.max(np.abs(l - ref_l)) < 1e-12
    ref = A.attention_backward(q, k, v, do, seq, pos, True, window=W)
    got = R.ring_backward(q, k, v, do, cu, cp, partition=partition, window=W)
    for a, b in zip(got, ref):
        assert np.max(np.abs(a - b)) < 1e-11
