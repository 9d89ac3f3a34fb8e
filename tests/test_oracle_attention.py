"""Pins for the oracle's masked attention (TileAttention) against facts fixed
outside the oracle: the pages' worked example, closed forms, brute force and an
independent library routine."""

import math
import os

import numpy as np
import pytest
import torch

from oracle import attention as A

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "p5_attention_softmax.txt")


def _read_golden():
    blocks, cur = {}, None
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line in ("scores", "probabilities"):
                cur = line
                blocks[cur] = []
                continue
            blocks[cur].append([float(x) for x in line.split()])
    return np.array(blocks["scores"]), np.array(blocks["probabilities"])


def test_worked_example_softmax_rows():
    """The 4-token example: attention weights = the printed softmax rows.

    Queries and keys are chosen so the scaled scores equal the printed logits
    (k = identity, q = scores / scale); with V = identity the output rows are
    the attention weights themselves.
    """
    scores, probs = _read_golden()
    d = 4
    scale = A.default_scale(d)
    q = (scores / scale)[:, None, :]
    k = np.eye(4)[:, None, :]
    v = np.eye(4)[:, None, :]
    vis = np.ones((4, 4), dtype=bool)
    out, lse = A.masked_attention(q, k, v, vis, scale)
    # printed to 3 decimals from 3-decimal logits: 1e-3 covers both roundings
    assert np.max(np.abs(out[:, 0, :] - probs)) <= 1e-3
    # the LSE makes the weights sum to one: exp(s - L) summed over keys = 1
    assert np.allclose(np.exp(scores - lse[:, 0:1]).sum(1), 1.0, atol=1e-12)
    # the sharpest row, Q(The) -> K(cat), is the one the page points at
    assert int(np.argmax(out[0, 0])) == 1


def test_zero_query_gives_prefix_mean():
    """Q = 0: every visible key has score 0, so O_i = mean_{j<=i} V_j and
    L_i = ln(i + 1) under the causal mask."""
    rng = np.random.default_rng(0)
    n, d = 9, 8
    q = np.zeros((n, 1, d))
    k = rng.standard_normal((n, 1, d))
    v = rng.standard_normal((n, 1, d))
    seq, pos = np.zeros(n, int), np.arange(n)
    out, lse = A.attention_forward(q, k, v, seq, pos, causal=True)
    for i in range(n):
        assert np.allclose(out[i, 0], v[: i + 1, 0].mean(0), atol=1e-14)
        assert abs(lse[i, 0] - math.log(i + 1)) < 1e-14


def test_single_key_and_first_row():
    rng = np.random.default_rng(1)
    d = 16
    q = rng.standard_normal((5, 2, d))
    k = rng.standard_normal((5, 1, d))
    v = rng.standard_normal((5, 1, d))
    seq, pos = np.zeros(5, int), np.arange(5)
    out, lse = A.attention_forward(q, k, v, seq, pos, causal=True)
    scale = 1 / math.sqrt(d)
    for h in range(2):
        # row 0 sees only key 0: O = v_0, L = s_00
        assert np.allclose(out[0, h], v[0, 0], atol=1e-14)
        assert abs(lse[0, h] - scale * q[0, h] @ k[0, 0]) < 1e-13


def test_empty_row_is_neg_inf_and_zero():
    q = np.ones((3, 1, 4))
    k = np.ones((2, 1, 4))
    v = np.ones((2, 1, 4))
    vis = np.array([[True, False], [False, False], [True, True]])
    out, lse = A.masked_attention(q, k, v, vis)
    assert lse[1, 0] == -np.inf and np.all(out[1] == 0)
    assert np.isfinite(lse[[0, 2], 0]).all()
    assert not np.isnan(out).any()


def test_brute_force_scalar_loops():
    """Tiny causal GQA case against a scalar loop written from the definition."""
    rng = np.random.default_rng(2)
    n, H, Hkv, d = 7, 4, 2, 3
    q = rng.standard_normal((n, H, d))
    k = rng.standard_normal((n, Hkv, d))
    v = rng.standard_normal((n, Hkv, d))
    seq, pos = np.zeros(n, int), np.arange(n)
    out, lse = A.attention_forward(q, k, v, seq, pos, causal=True)
    scale = 1 / math.sqrt(d)
    for h in range(H):
        g = h // (H // Hkv)
        for i in range(n):
            w = [math.exp(scale * sum(q[i, h, t] * k[j, g, t] for t in range(d))) for j in range(i + 1)]
            z = sum(w)
            assert abs(lse[i, h] - math.log(z)) < 1e-12
            for t in range(d):
                ref = sum(w[j] * v[j, g, t] for j in range(i + 1)) / z
                assert abs(out[i, h, t] - ref) < 1e-12


@pytest.mark.parametrize("causal", [True, False])
def test_matches_torch_sdpa_float64(causal):
    """Independent library cross-check: torch's CPU scaled_dot_product_attention
    in float64, and torch.logsumexp of the masked scaled scores."""
    rng = np.random.default_rng(3)
    s, H, d = 200, 3, 64
    q = rng.standard_normal((s, H, d))
    k = rng.standard_normal((s, H, d))
    v = rng.standard_normal((s, H, d))
    seq, pos = np.zeros(s, int), np.arange(s)
    out, lse = A.attention_forward(q, k, v, seq, pos, causal=causal)
    tq, tk, tv = (torch.from_numpy(x).permute(1, 0, 2) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal)
    assert np.max(np.abs(out - ref.permute(1, 0, 2).numpy())) < 1e-12
    sc = (tq @ tk.transpose(1, 2)) / math.sqrt(d)
    if causal:
        sc = sc.masked_fill(torch.ones(s, s, dtype=torch.bool).triu(1), float("-inf"))
    ref_lse = torch.logsumexp(sc, dim=-1).permute(1, 0).numpy()
    assert np.max(np.abs(lse - ref_lse)) < 1e-12


def test_packed_block_diagonal_equals_per_sequence():
    """Packed stream = each sub-sequence attended on its own (torch SDPA)."""
    rng = np.random.default_rng(4)
    lens = [5, 12, 1, 30]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, H, Hkv, d = cu[-1], 4, 1, 16
    q = rng.standard_normal((T, H, d))
    k = rng.standard_normal((T, Hkv, d))
    v = rng.standard_normal((T, Hkv, d))
    seq, pos = A.token_meta_from_cu(cu)
    out, _ = A.attention_forward(q, k, v, seq, pos, causal=True)
    for a, b in zip(cu[:-1], cu[1:]):
        tq = torch.from_numpy(q[a:b]).permute(1, 0, 2)
        tk = torch.from_numpy(np.repeat(k[a:b], H, axis=1)).permute(1, 0, 2)
        tv = torch.from_numpy(np.repeat(v[a:b], H, axis=1)).permute(1, 0, 2)
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
        assert np.max(np.abs(out[a:b] - ref.permute(1, 0, 2).numpy())) < 1e-12


def test_rows_subset_equals_full():
    rng = np.random.default_rng(5)
    s, H, d = 300, 2, 8
    q = rng.standard_normal((s, H, d))
    k = rng.standard_normal((s, 1, d))
    v = rng.standard_normal((s, 1, d))
    seq, pos = np.zeros(s, int), np.arange(s)
    out, lse = A.attention_forward(q, k, v, seq, pos)
    rows = np.array([0, 7, 150, 299])
    o2, l2 = A.attention_forward_rows(rows, q, k, v, seq, pos)
    assert np.array_equal(o2, out[rows]) or np.max(np.abs(o2 - out[rows])) < 1e-14
    assert np.max(np.abs(l2 - lse[rows])) < 1e-14


# ------------------------------------------------------------ sliding window --
def test_window_brute_force_scalar_loops():
    """Causal band of width W: query i averages keys max(0, i-W+1) .. i
    (scalar loop written from that definition)."""
    rng = np.random.default_rng(12)
    n, H, Hkv, d, W = 9, 2, 1, 3, 3
    q = rng.standard_normal((n, H, d))
    k = rng.standard_normal((n, Hkv, d))
    v = rng.standard_normal((n, Hkv, d))
    seq, pos = np.zeros(n, int), np.arange(n)
    out, lse = A.attention_forward(q, k, v, seq, pos, causal=True, window=W)
    scale = 1 / math.sqrt(d)
    for h in range(H):
        g = h // (H // Hkv)
        for i in range(n):
            keys = range(max(0, i - W + 1), i + 1)
            w = {j: math.exp(scale * sum(q[i, h, t] * k[j, g, t] for t in range(d))) for j in keys}
            z = sum(w.values())
            assert abs(lse[i, h] - math.log(z)) < 1e-12
            for t in range(d):
                assert abs(out[i, h, t] - sum(w[j] * v[j, g, t] for j in keys) / z) < 1e-12


def test_window_special_cases():
    rng = np.random.default_rng(13)
    n, H, d = 40, 2, 8
    q = rng.standard_normal((n, H, d))
    k = rng.standard_normal((n, H, d))
    v = rng.standard_normal((n, H, d))
    seq, pos = np.zeros(n, int), np.arange(n)
    # W = 1: every query sees only its own key: O_i = V_i, L_i = q_i . k_i / sqrt(d)
    out, lse = A.attention_forward(q, k, v, seq, pos, window=1)
    assert np.max(np.abs(out - v)) < 1e-14
    assert np.max(np.abs(lse - np.einsum("nhd,nhd->nh", q, k) / math.sqrt(d))) < 1e-12
    # W >= n: the plain causal mask
    o1, l1 = A.attention_forward(q, k, v, seq, pos, window=n)
    o2, l2 = A.attention_forward(q, k, v, seq, pos)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    with pytest.raises(ValueError):
        A.visibility(seq, pos, seq, pos, causal=False, window=4)


@pytest.mark.parametrize("n,W", [(10, 3), (64, 16), (33, 40), (5, 1)])
def test_window_pair_count_closed_form(n, W):
    """sum_i min(i + 1, W) = W (W + 1) / 2 + (n - W) W for W < n."""
    seq, pos = np.zeros(n, int), np.arange(n)
    got = int(A.visibility(seq, pos, seq, pos, True, W).sum())
    want = n * (n + 1) // 2 if W >= n else W * (W + 1) // 2 + (n - W) * W
    assert got == want
