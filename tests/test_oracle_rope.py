"""Pins of the rotary-embedding oracle (oracle/rope.py) against properties the
mathematics fixes, and the pages' rule that the RoPE positions follow the
same zigzag split as the tokens ("04 · Megatron-LM 实现" §5 and §9 item 1)."""
import math

import numpy as np
import pytest

from oracle import attention as A
from oracle import partition as P
from oracle import rope as R
from tile_attention_lse_gb300.synthetic import cu_from_lengths, packed_lengths

pytestmark = pytest.mark.filterwarnings("ignore")


def _x(T=16, H=3, d=8, seed=0):
    return np.random.default_rng(seed).standard_normal((T, H, d))


def test_position_zero_is_identity():
    x = _x()
    assert np.array_equal(R.rotate(x, np.zeros(x.shape[0], dtype=np.int64)), x)


def test_rotation_preserves_each_pair_norm():
    x = _x(d=16)
    y = R.rotate(x, np.arange(x.shape[0]) * 37 + 5, base=500.0)
    h = x.shape[-1] // 2
    nx = x[..., :h] ** 2 + x[..., h:] ** 2
    ny = y[..., :h] ** 2 + y[..., h:] ** 2
    assert np.allclose(nx, ny, rtol=1e-13, atol=1e-13)


def test_rotations_compose_and_invert():
    x = _x(d=8)
    p1 = np.arange(x.shape[0]) * 3
    p2 = np.arange(x.shape[0])[::-1] * 11 + 2
    assert np.allclose(R.rotate(R.rotate(x, p1), p2), R.rotate(x, p1 + p2), atol=1e-12)
    assert np.allclose(R.rotate(R.rotate(x, p1), p1, inverse=True), x, atol=1e-12)


def test_scores_depend_only_on_relative_position():
    # the defining property of the rotary embedding: <R(m) q, R(n) k> is a
    # function of m - n
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal((1, 1, 64)), rng.standard_normal((1, 1, 64))
    for m, n, c in [(5, 2, 7), (1000, 3, 91), (0, 40, 1234)]:
        a = np.sum(R.rotate(q, [m]) * R.rotate(k, [n]))
        b = np.sum(R.rotate(q, [m + c]) * R.rotate(k, [n + c]))
        assert abs(a - b) < 1e-10 * max(1.0, abs(a))
    # and it does change with m - n
    assert abs(np.sum(R.rotate(q, [5]) * R.rotate(k, [2])) - np.sum(R.rotate(q, [6]) * R.rotate(k, [2]))) > 1e-6


def test_closed_form_two_dimensional_rotations():
    # d = 2: one pair, frequency 1 -> rotation of (1, 0) by pos radians
    for pos in (1, 2, 3):
        y = R.rotate(np.array([[[1.0, 0.0]]]), [pos])
        assert y[0, 0, 0] == pytest.approx(math.cos(pos), abs=1e-15)
        assert y[0, 0, 1] == pytest.approx(math.sin(pos), abs=1e-15)
    # d = 4, base 100: pairs (x0, x2) at frequency 1 and (x1, x3) at 100**-0.5
    y = R.rotate(np.array([[[0.0, 1.0, 0.0, 0.0]]]), [5], base=100.0)
    assert np.allclose(y[0, 0], [0.0, math.cos(0.5), 0.0, math.sin(0.5)], atol=1e-15)


def test_positions_follow_the_token_split_thd():
    # roping in original order and then gathering equals gathering with each
    # token's own position; contiguous positions in rank-local order would not
    lens = packed_lengths(1024, 4, seed=1, mu=5.0, sigma=1.0, lo=8, hi=512)
    cu = cu_from_lengths(lens)
    T = int(cu[-1])
    _, pos = A.token_meta_from_cu(cu)
    idx = P.thd_partition_indices(cu, 4).ravel()
    assert np.array_equal(idx, P.thd_rope_segments(cu, 4).ravel())
    x = np.random.default_rng(5).standard_normal((2, T, 2, 16))
    expect = R.rotate(x, pos)[:, idx]
    got = R.permute_rope(x, idx, pos)
    assert np.allclose(got, expect, atol=1e-12)
    wrong = R.rotate(x[:, idx], np.arange(T))  # positions not split with the tokens
    assert not np.allclose(wrong, expect, atol=1e-3)
    # the inverse gather undoes it
    assert np.allclose(R.permute_rope(got, idx, pos, inverse=True), x, atol=1e-12)
