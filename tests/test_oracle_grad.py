"""Pins for the oracle's backward pass: finite differences, invariants that
follow from the softmax, and torch autograd in float64."""

import numpy as np
import pytest
import torch

from oracle import attention as A


def _loss(q, k, v, g, seq, pos, causal):
    out, _ = A.attention_forward(q, k, v, seq, pos, causal)
    return float((out * g).sum())


@pytest.mark.parametrize("causal,H,Hkv", [(True, 2, 1), (False, 2, 2)])
def test_central_finite_differences(causal, H, Hkv):
    rng = np.random.default_rng(0)
    n, d = 6, 3
    q = rng.standard_normal((n, H, d))
    k = rng.standard_normal((n, Hkv, d))
    v = rng.standard_normal((n, Hkv, d))
    g = rng.standard_normal((n, H, d))
    seq, pos = np.zeros(n, int), np.arange(n)
    dq, dk, dv = A.attention_backward(q, k, v, g, seq, pos, causal)
    h = 1e-6
    for x, dx in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + h
            fp = _loss(q, k, v, g, seq, pos, causal)
            x[idx] = old - h
            fm = _loss(q, k, v, g, seq, pos, causal)
            x[idx] = old
            num[idx] = (fp - fm) / (2 * h)
        assert np.max(np.abs(num - dx)) < 1e-7


def test_gradient_invariants():
    """sum_j dK_j = 0 (each dS row sums to zero) and sum_j dV_j = sum_i dO_i
    (each P row sums to one)."""
    rng = np.random.default_rng(1)
    n, H, Hkv, d = 64, 4, 2, 8
    q = rng.standard_normal((n, H, d))
    k = rng.standard_normal((n, Hkv, d))
    v = rng.standard_normal((n, Hkv, d))
    do = rng.standard_normal((n, H, d))
    seq, pos = np.zeros(n, int), np.arange(n)
    dq, dk, dv = A.attention_backward(q, k, v, do, seq, pos, True)
    assert np.max(np.abs(dk.sum(0))) < 1e-11
    grp = H // Hkv
    do_sum = do.sum(0).reshape(Hkv, grp, d).sum(1)
    assert np.max(np.abs(dv.sum(0) - do_sum)) < 1e-11


def test_matches_torch_autograd_float64_packed_gqa():
    rng = np.random.default_rng(2)
    lens = [16, 40, 8]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, H, Hkv, d = cu[-1], 4, 2, 32
    q = rng.standard_normal((T, H, d))
    k = rng.standard_normal((T, Hkv, d))
    v = rng.standard_normal((T, Hkv, d))
    do = rng.standard_normal((T, H, d))
    seq, pos = A.token_meta_from_cu(cu)
    dq, dk, dv = A.attention_backward(q, k, v, do, seq, pos, True)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    outs = []
    for a, b in zip(cu[:-1], cu[1:]):
        qq = tq[a:b].permute(1, 0, 2)
        kk = tk[a:b].repeat_interleave(H // Hkv, dim=1).permute(1, 0, 2)
        vv = tv[a:b].repeat_interleave(H // Hkv, dim=1).permute(1, 0, 2)
        outs.append(torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, is_causal=True)
                    .permute(1, 0, 2))
    out = torch.cat(outs)
    (out * torch.from_numpy(do)).sum().backward()
    assert np.max(np.abs(tq.grad.numpy() - dq)) < 1e-11
    assert np.max(np.abs(tk.grad.numpy() - dk)) < 1e-11
    assert np.max(np.abs(tv.grad.numpy() - dv)) < 1e-11


def test_window_central_finite_differences():
    """The backward under a sliding window (band of 3) by central differences."""
    rng = np.random.default_rng(5)
    n, H, Hkv, d, W = 7, 2, 1, 3, 3
    q = rng.standard_normal((n, H, d))
    k = rng.standard_normal((n, Hkv, d))
    v = rng.standard_normal((n, Hkv, d))
    g = rng.standard_normal((n, H, d))
    seq, pos = np.zeros(n, int), np.arange(n)
    dq, dk, dv = A.attention_backward(q, k, v, g, seq, pos, True, window=W)

    def loss():
        out, _ = A.attention_forward(q, k, v, seq, pos, True, window=W)
        return float((out * g).sum())

    h = 1e-6
    for x, dx in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + h
            fp = loss()
            x[idx] = old - h
            fm = loss()
            x[idx] = old
            num[idx] = (fp - fm) / (2 * h)
        assert np.max(np.abs(num - dx)) < 1e-7
