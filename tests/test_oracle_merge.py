"""Pins for the oracle's LSE merge and online recurrence ("Context Parallelism
(CP)" §2.2; "上下文并行" 02 ONE ROW)."""

import numpy as np
import pytest

from oracle import attention as A


def _problem(seed, n=40, m=97, H=2, d=8):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((n, H, d)) * 2.0
    k = rng.standard_normal((m, H, d))
    v = rng.standard_normal((m, H, d))
    vis = rng.random((n, m)) < 0.7
    vis[:, 0] = True            # every row sees at least one key
    vis[0, 1:] = False          # row 0 sees key 0 only: empty partials elsewhere
    return q, k, v, vis


def _partials(q, k, v, vis, groups):
    o_parts, l_parts = [], []
    for g in groups:
        o, l = A.masked_attention(q, k[g], v[g], vis[:, g])
        o_parts.append(o)
        l_parts.append(l)
    return np.stack(o_parts), np.stack(l_parts)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_merge_of_any_key_partition_equals_full(seed):
    q, k, v, vis = _problem(seed)
    full_o, full_l = A.masked_attention(q, k, v, vis)
    rng = np.random.default_rng(100 + seed)
    perm = rng.permutation(k.shape[0])
    cuts = np.sort(rng.choice(np.arange(1, k.shape[0]), size=5, replace=False))
    groups = np.split(perm, cuts)
    o_parts, l_parts = _partials(q, k, v, vis, groups)
    # some partials are empty for some rows (L = -inf): weight 0
    assert np.isinf(l_parts).any()
    o, l = A.lse_merge(o_parts, l_parts)
    assert np.max(np.abs(o - full_o)) < 1e-12
    assert np.max(np.abs(l - full_l)) < 1e-12


def test_merge_associative_and_commutative():
    q, k, v, vis = _problem(7)
    groups = np.array_split(np.arange(k.shape[0]), 6)
    o_parts, l_parts = _partials(q, k, v, vis, groups)
    flat_o, flat_l = A.lse_merge(o_parts, l_parts)
    rng = np.random.default_rng(8)
    for _ in range(5):
        order = rng.permutation(6)
        # ((p0 + p1) + (p2 + p3 + p4)) + p5 in a shuffled order
        a = A.lse_merge(o_parts[order[:2]], l_parts[order[:2]])
        b = A.lse_merge(o_parts[order[2:5]], l_parts[order[2:5]])
        ab = A.lse_merge(np.stack([a[0], b[0]]), np.stack([a[1], b[1]]))
        tot = A.lse_merge(np.stack([ab[0], o_parts[order[5]]]), np.stack([ab[1], l_parts[order[5]]]))
        assert np.max(np.abs(tot[0] - flat_o)) < 1e-12
        assert np.max(np.abs(tot[1] - flat_l)) < 1e-12


def test_equal_weight_average_is_wrong():
    """Averaging per-block softmax outputs with equal weights is not attention
    ("上下文并行" 02: block weights come from each block's exponential mass)."""
    q, k, v, vis = _problem(9)
    vis[:] = True
    full_o, _ = A.masked_attention(q, k, v, vis)
    groups = np.array_split(np.arange(k.shape[0]), 3)
    o_parts, l_parts = _partials(q, k, v, vis, groups)
    naive = o_parts.mean(axis=0)
    assert np.max(np.abs(naive - full_o)) > 1e-2
    merged, _ = A.lse_merge(o_parts, l_parts)
    assert np.max(np.abs(merged - full_o)) < 1e-12


def test_merge_all_empty_row():
    o = np.zeros((3, 2, 1, 4))
    l = np.full((3, 2, 1), -np.inf)
    l[1, 0, 0] = 0.5
    o[1, 0, 0] = 1.0
    mo, ml = A.lse_merge(o, l)
    assert ml[1, 0] == -np.inf and np.all(mo[1] == 0)
    assert abs(ml[0, 0] - 0.5) < 1e-15 and np.allclose(mo[0, 0], 1.0)


def test_merge_single_partial_identity_and_two_equal():
    rng = np.random.default_rng(11)
    o = rng.standard_normal((1, 5, 3, 4))
    l = rng.standard_normal((1, 5, 3))
    mo, ml = A.lse_merge(o, l)
    assert np.allclose(mo, o[0], atol=1e-15) and np.allclose(ml, l[0], atol=1e-15)
    # two identical partials: same output, LSE + ln 2
    mo2, ml2 = A.lse_merge(np.concatenate([o, o]), np.concatenate([l, l]))
    assert np.allclose(mo2, o[0], atol=1e-14) and np.allclose(ml2, l[0] + np.log(2), atol=1e-14)


def test_merge_large_lse_no_overflow():
    o = np.ones((2, 1, 1, 2))
    l = np.array([[[1000.0]], [[1000.0]]])
    mo, ml = A.lse_merge(o, l)
    assert abs(ml[0, 0] - (1000 + np.log(2))) < 1e-12 and np.allclose(mo, 1.0)


@pytest.mark.parametrize("seed", [0, 1])
def test_online_recurrence_equals_two_pass(seed):
    rng = np.random.default_rng(seed)
    m, d = 50, 6
    s = rng.standard_normal(m) * 5
    v = rng.standard_normal((m, d))
    s[[3, 17]] = -np.inf        # masked keys
    blocks = [slice(0, 7), slice(7, 8), slice(8, 30), slice(30, 50)]
    o, lam = A.online_softmax_row([s[b] for b in blocks], [v[b] for b in blocks])
    w = np.exp(s - s.max())
    ref = (w / w.sum()) @ v
    assert np.max(np.abs(o - ref)) < 1e-12
    assert abs(lam - (s.max() + np.log(w.sum()))) < 1e-12
