"""Pins for the oracle's partition rules ("04 · Megatron-LM 实现" §1.1, §1.2,
§5; "Context Parallelism (CP)" §4)."""

import numpy as np
import pytest

from oracle import attention as A
from oracle import partition as P


def test_cp2_example_chunks():
    """cp = 2: four chunks, (chunk0, chunk3) -> rank 0 and (chunk1, chunk2) -> rank 1."""
    idx = P.zigzag_indices(8, 2)
    assert idx.tolist() == [[0, 1, 6, 7], [2, 3, 4, 5]]


def test_alignment_rule():
    with pytest.raises(P.PartitionError):
        P.zigzag_indices(12, 4)          # 12 % 8 != 0
    with pytest.raises(P.PartitionError):
        P.thd_partition_indices([0, 8, 18], 2)   # 10 % 4 != 0


@pytest.mark.parametrize("s,cp", [(256, 2), (64, 8), (96, 3), (8, 1)])
def test_zigzag_is_permutation_and_chunked(s, cp):
    idx = P.zigzag_indices(s, cp)
    assert sorted(idx.ravel().tolist()) == list(range(s))
    c = s // (2 * cp)
    for r in range(cp):
        assert idx[r, 0] == r * c and idx[r, c] == (2 * cp - 1 - r) * c
        assert np.all(np.diff(idx[r, :c]) == 1) and np.all(np.diff(idx[r, c:]) == 1)


@pytest.mark.parametrize("s,cp", [(256, 2), (128, 4), (96, 3), (512, 8)])
def test_zigzag_balance_closed_form(s, cp):
    """Every rank sees exactly c(2 cp c + 1) unmasked causal pairs; with the
    plain contiguous split the counts differ."""
    c = s // (2 * cp)
    idx = P.zigzag_indices(s, cp)
    seq, pos = np.zeros(s, int), np.arange(s)
    vis = A.visibility(seq, pos, seq, pos, True)
    counts = [int(vis[idx[r]].sum()) for r in range(cp)]
    assert counts == [c * (2 * cp * c + 1)] * cp
    assert sum(counts) == s * (s + 1) // 2
    if cp > 1:
        contiguous = [int(vis[r * (s // cp):(r + 1) * (s // cp)].sum()) for r in range(cp)]
        assert len(set(contiguous)) == cp


@pytest.mark.parametrize("cp", [2, 4, 8])
def test_zigzag_chunk_edge_counts(cp):
    """Per rank: 2cp-1 full chunk pairs plus 2 diagonal ones."""
    s = 2 * cp * 4
    c = 4
    idx = P.zigzag_indices(s, cp)
    for r in range(cp):
        q_chunks = [int(idx[r, 0]) // c, int(idx[r, c]) // c]
        full = diag = 0
        for a in q_chunks:
            for b in range(2 * cp):
                if b < a:
                    full += 1
                elif b == a:
                    diag += 1
        assert (full, diag) == (2 * cp - 1, 2)


def test_thd_matches_rope_rule_and_single_sequence():
    cu = [0, 16, 24, 64, 72]
    for cp in (1, 2, 4):
        idx = P.thd_partition_indices(cu, cp)
        assert np.array_equal(idx, P.thd_rope_segments(cu, cp))
        assert sorted(idx.ravel().tolist()) == list(range(72))
    # one sub-sequence: identical to the plain zigzag split
    assert np.array_equal(P.thd_partition_indices([0, 64], 4), P.zigzag_indices(64, 4))


def test_thd_per_subsequence_balance():
    cu = [0, 16, 48, 64, 128]
    cp = 2
    idx = P.thd_partition_indices(cu, cp)
    seq, pos = A.token_meta_from_cu(cu)
    vis = A.visibility(seq, pos, seq, pos, True)
    counts = [int(vis[idx[r]].sum()) for r in range(cp)]
    lens = np.diff(cu)
    cks = lens // (2 * cp)
    assert counts == [int(sum(ck * (2 * cp * ck + 1) for ck in cks))] * cp
    # each rank holds len/cp tokens of every sub-sequence
    for r in range(cp):
        assert np.bincount(seq[idx[r]], minlength=len(lens)).tolist() == (lens // cp).tolist()
    assert P.local_cu_seqlens(cu, cp).tolist() == [0, 8, 24, 32, 64]


def test_thd_sub_sequence_of_exactly_2cp():
    idx = P.thd_partition_indices([0, 8], 4)
    assert idx.tolist() == [[0, 7], [1, 6], [2, 5], [3, 4]]


# ----------------------------------------------------------------- striped --
def test_striped_page_example():
    """"Sequence Parallelism + Ring Attention" §5: four cards take the
    interleaved blocks [0, 4, 8, ...] and [1, 5, 9, ...] (and so on)."""
    idx = P.striped_indices(12, 4)
    assert idx.tolist() == [[0, 4, 8], [1, 5, 9], [2, 6, 10], [3, 7, 11]]


def test_striped_alignment_rule():
    with pytest.raises(P.PartitionError):
        P.striped_indices(10, 4)
    with pytest.raises(P.PartitionError):
        P.thd_striped_indices([0, 8, 14], 4)   # 6 % 4 != 0
    P.striped_indices(12, 4)                   # a multiple of cp, not of 2cp, is fine


@pytest.mark.parametrize("s,cp", [(256, 2), (64, 8), (96, 3), (8, 1), (12, 4)])
def test_striped_is_permutation_and_strided(s, cp):
    idx = P.striped_indices(s, cp)
    assert sorted(idx.ravel().tolist()) == list(range(s))
    for r in range(cp):
        assert idx[r, 0] == r and np.all(np.diff(idx[r]) == cp)
        assert np.all(idx[r] % cp == r)


@pytest.mark.parametrize("s,cp", [(256, 2), (128, 4), (96, 3), (512, 8)])
def test_striped_balance_closed_form(s, cp):
    """Rank r holds tokens r + cp u (u < n = s / cp); token i sees i + 1 keys,
    so the rank's causal pairs are n (r + 1) + cp n (n - 1) / 2: ranks differ
    by n per step of r, against n^2 per step for the contiguous split."""
    n = s // cp
    idx = P.striped_indices(s, cp)
    seq, pos = np.zeros(s, int), np.arange(s)
    vis = A.visibility(seq, pos, seq, pos, True)
    counts = [int(vis[idx[r]].sum()) for r in range(cp)]
    assert counts == [n * (r + 1) + cp * n * (n - 1) // 2 for r in range(cp)]
    assert sum(counts) == s * (s + 1) // 2
    assert max(counts) - min(counts) == (cp - 1) * n


def test_thd_striped_per_subsequence():
    cu = [0, 16, 48, 48, 64, 128]
    cp = 4
    idx = P.thd_striped_indices(cu, cp)
    assert sorted(idx.ravel().tolist()) == list(range(128))
    seq, pos = A.token_meta_from_cu(cu)
    lens = np.diff(cu)
    for r in range(cp):
        # every rank holds len/cp tokens of every sub-sequence, in sub-sequence order,
        # at in-sequence positions r, r + cp, ...
        assert np.bincount(seq[idx[r]], minlength=len(lens)).tolist() == (lens // cp).tolist()
        assert np.all(np.diff(seq[idx[r]]) >= 0)
        assert np.all(pos[idx[r]] % cp == r)
    # one sub-sequence: the plain striped split
    assert np.array_equal(P.thd_striped_indices([0, 64], 4), P.striped_indices(64, 4))


@pytest.mark.parametrize("cp", [1, 2, 3, 5, 8])
def test_striped_virtual_position_relation(cp):
    """Causality between two striped ranks in their own slot numbers: key u of
    rank s is visible to query w of rank r (s + cp u <= r + cp w) exactly when
    u + [s > r] <= w, the rule the tile kernels apply with rank s's keys
    placed at virtual position [s > r]."""
    n = 5
    for r in range(cp):
        for s_ in range(cp):
            for u in range(n):
                for w in range(n):
                    assert (s_ + cp * u <= r + cp * w) == (u + (1 if s_ > r else 0) <= w)


@pytest.mark.parametrize("cp,W", [(1, 3), (2, 1), (3, 4), (4, 2), (5, 11), (8, 3)])
def test_striped_window_virtual_band(cp, W):
    """A sliding window between two striped ranks in their slot numbers: with
    rank s's keys at virtual position u + d (d = [s > r]), the token distance
    (r + cp w) - (s + cp u) is below W exactly when w - (u + d) < M - d,
    M = ceil((W + s - r) / cp); no pair of the two ranks is in the band when
    M - d <= 0.  This is the per-edge band the planner gives the kernels."""
    n = 6
    for r in range(cp):
        for s_ in range(cp):
            d = 1 if s_ > r else 0
            x = W + s_ - r
            band = (-(-x // cp) - d) if x > 0 else 0
            for w in range(n):
                for u in range(n):
                    i, j = r + cp * w, s_ + cp * u
                    true_vis = j <= i and i - j < W
                    virt_vis = band > 0 and u + d <= w and w - (u + d) < band
                    assert true_vis == virt_vis
