"""Pins for the oracle's hybrid CP schedule and layout ("04 · Megatron-LM 实现"
§7.1 balanced scheduler, §2.3 aligned power-of-two groups, §1.1 zigzag split
over a sequence's group)."""

import math

import numpy as np
import pytest

from oracle import attention as A
from oracle import hybrid as HY
from oracle import partition as P
from oracle import ring as R


@pytest.mark.parametrize("length,cap", [(1, 8), (8, 8), (9, 8), (16, 8), (17, 8), (1000, 7), (65536, 4096),
                                        (65537, 4096), (3, 1)])
def test_gpus_needed_printed_formula(length, cap):
    """max(1, 2^ceil(log2(seq_len / max_seqlen_per_rank))), the page's formula."""
    want = max(1, 2 ** math.ceil(math.log2(length / cap)))
    assert HY.gpus_needed(length, cap) == want


def test_workload_is_square_over_cp():
    assert HY.workload(64, 1) == 4096 and HY.workload(64, 4) == 1024 and HY.workload(0, 2) == 0


def _check_valid(lens, world, cap, rnd, cp, rank0, n_rounds):
    """Every sequence in exactly one round, on an aligned power-of-two group
    at least as large as it needs, within capacity; groups of one round are
    disjoint (sequences of one group share it exactly)."""
    assert rnd.min() == 0 and rnd.max() == n_rounds - 1
    for k, x in enumerate(lens):
        g, r0 = int(cp[k]), int(rank0[k])
        assert g & (g - 1) == 0 and g >= HY.gpus_needed(x, cap) and g <= world
        assert r0 % g == 0 and r0 + g <= world
        assert x % (2 * g) == 0
    for r in range(n_rounds):
        ks = np.nonzero(rnd == r)[0]
        blocks = {(int(rank0[k]), int(cp[k])) for k in ks}
        owner = [None] * world
        for r0, g in blocks:
            for q in range(r0, r0 + g):
                assert owner[q] is None       # groups do not overlap
                owner[q] = (r0, g)
            tokens = sum(lens[k] // g for k in ks if (int(rank0[k]), int(cp[k])) == (r0, g))
            assert tokens <= cap or len([k for k in ks if (int(rank0[k]), int(cp[k])) == (r0, g)]) == 1


def test_single_long_sequence_spans_its_group():
    lens = [64 * 16]
    rnd, cp, rank0, n = HY.schedule(lens, 8, 256)
    assert n == 1 and cp[0] == 4 and rank0[0] == 0 and rnd[0] == 0 or cp[0] == 8
    # the idle half of the ranks is merged into the group
    assert cp[0] == 8 and rank0[0] == 0


def test_equal_short_sequences_one_per_rank():
    """world short sequences that each fit one rank: one per rank, one round,
    perfectly balanced."""
    world = 4
    lens = [64] * world
    rnd, cp, rank0, n = HY.schedule(lens, world, 64)
    assert n == 1
    assert sorted(int(x) for x in rank0) == list(range(world)) and set(cp.tolist()) == {1}
    loads = HY.rank_loads(lens, cp, rank0, world)
    assert loads.tolist() == [64 * 64] * world


def test_hand_worked_round():
    """world 4, capacity 64: lengths 128, 64, 64, 32, 32 (multiples of 8).
    need = 2, 1, 1, 1, 1; cost 8192, 4096, 4096, 1024, 1024 (total 18432);
    two buckets, target 9216, closed past 10137.6: {128} | {64, 64, 32, 32}.
    Round 0: 128 opens ranks 0-1; at the bucket step ranks 2-3 are idle (no
    stop); 64 opens rank 2; the next 64 does not fit rank 2 (128 tokens >
    64) and opens rank 3; neither 32 fits a rank holding 64 tokens and no
    rank is idle: both wait.  Trim: the 64 on rank 3 sits on a less loaded
    group than ranks 0-1: nothing shed.  No buddy block idle.
    Round 1: 32 opens rank 0, the other 32 joins it (64 tokens fit); slack
    0, nothing trimmed; rank 0's group doubles over idle rank 1, then over
    idle ranks 2-3: both sequences on a group of 4."""
    lens = [128, 64, 64, 32, 32]
    rnd, cp, rank0, n = HY.schedule(lens, 4, 64)
    assert n == 2
    assert rnd.tolist() == [0, 0, 0, 1, 1]
    assert cp.tolist() == [2, 1, 1, 4, 4]
    assert rank0.tolist() == [0, 2, 3, 0, 0]


def test_trim_and_merge_steps():
    """world 2, capacity 128: 64, 16, 16 (need 1 each) all fit rank 0 (96
    tokens); rank 1 stays idle, busy slack 0: nothing trimmed; merge: rank
    0's group doubles over rank 1."""
    rnd, cp, rank0, n = HY.schedule([64, 16, 16], 2, 128)
    assert n == 1 and cp.tolist() == [2, 2, 2] and rank0.tolist() == [0, 0, 0]
    # capacity 64: 64 opens rank 0, 16 does not fit it and opens rank 1, the
    # second 16 joins rank 1; dropping it would widen the slack (4096 - 512
    # -> 4096 - 256): kept, one round
    rnd, cp, rank0, n = HY.schedule([64, 16, 16], 2, 64)
    assert n == 1 and cp.tolist() == [1, 1, 1] and rank0.tolist() == [0, 1, 1]
    # the last placed sequence sits on a less loaded group: never shed
    rnd, cp, rank0, n = HY.schedule([32, 32, 16], 2, 64)
    assert n == 1 and cp.tolist() == [1, 1, 1] and rank0.tolist() == [0, 0, 1]
    # capacity 72: 40 opens rank 0 (1600), 36 does not fit it and opens rank 1
    # (1296), 32 fits both and joins the less loaded rank 1 (2320): slack 720;
    # shedding it leaves 1600 - 1296 = 304 < 720: it waits.  36 is then on
    # the less loaded group: stop.  Round 1: 32 alone, doubled over both ranks.
    rnd, cp, rank0, n = HY.schedule([40, 36, 32], 2, 72)
    assert n == 2 and rnd.tolist() == [0, 0, 1]
    assert cp.tolist() == [1, 1, 2] and rank0.tolist() == [0, 1, 0]


def test_early_stop_at_bucket_step():
    """world 2, capacity 64: 64, 64, 8, 8 all need one rank: one bucket, no
    step, no early stop.  64 -> rank 0, 64 -> rank 1, the 8s cannot join a
    full rank and wait; round 1: both 8s on rank 0, doubled over rank 1."""
    rnd, cp, rank0, n = HY.schedule([64, 64, 8, 8], 2, 64)
    assert n == 2 and rnd.tolist() == [0, 0, 1, 1]
    assert cp.tolist() == [1, 1, 2, 2] and rank0.tolist() == [0, 1, 0, 0]
    # two needs: 128 (need 2, cost 8192) then 8, 8 (need 1, cost 64): buckets
    # {128} | {8, 8}; at the step every rank is busy with equal loads: stop,
    # the 8s go to round 1
    rnd, cp, rank0, n = HY.schedule([128, 8, 8], 2, 64)
    assert n == 2 and rnd.tolist() == [0, 1, 1]
    assert cp.tolist() == [2, 2, 2]


@pytest.mark.parametrize("seed,world,cap", [(0, 8, 4096), (1, 8, 2048), (2, 4, 8192), (3, 16, 1024),
                                            (4, 2, 4096)])
def test_schedule_valid_on_long_tail_streams(seed, world, cap):
    rng = np.random.default_rng(seed)
    raw = np.exp(rng.normal(7.0, 1.2, 60))
    lens = [int(max(1, min(world * cap, x)) // (2 * world) * (2 * world)) or 2 * world for x in raw]
    rnd, cp, rank0, n = HY.schedule(lens, world, cap)
    _check_valid(lens, world, cap, rnd, cp, rank0, n)


def test_schedule_rejects():
    with pytest.raises(HY.ScheduleError):
        HY.schedule([64], 3, 64)               # world not a power of two
    with pytest.raises(HY.ScheduleError):
        HY.schedule([60], 4, 64)               # 60 % 8
    with pytest.raises(HY.ScheduleError):
        HY.schedule([1024], 4, 64)             # needs 16 ranks


def test_layout_per_group_zigzag():
    """A sequence alone on all ranks is the plain zigzag split; the layout is
    a permutation, rank by rank, and local_cu marks each part."""
    cu = [0, 64]
    idx, lcu = HY.hybrid_layout(cu, [4], [0], 4)
    assert np.array_equal(idx.reshape(4, 16), P.zigzag_indices(64, 4))
    cu = [0, 16, 48, 64, 128]
    seq_cp, seq_r0 = [2, 1, 2, 4], [0, 3, 2, 0]
    idx, lcu = HY.hybrid_layout(cu, seq_cp, seq_r0, 4)
    assert sorted(idx.tolist()) == list(range(128))
    # rank 3 holds sequence 1 whole (cp 1: chunk 0 then chunk 1 = in order),
    # sequence 2's chunk 1 and 2 of 4 (rank 3 is member 1 of group 2-3), and
    # sequence 3's chunks 3 and 4 of 8
    r3 = idx[lcu[3, 0]:lcu[3, 4]].tolist()
    assert r3 == list(range(16, 48)) + list(range(52, 60)) + list(range(88, 104))
    assert lcu[0, 0] == 0 and lcu[3, 4] == 128
    for r in range(4):
        assert lcu[r, 4] == (lcu[r + 1, 0] if r < 3 else 128)


@pytest.mark.parametrize("seed", [0, 1])
def test_hybrid_ring_equals_full(seed):
    """The ring walk over one round's rank streams (ranks of different
    lengths, sequences confined to their groups) is exact attention."""
    rng = np.random.default_rng(seed)
    world = 4
    lens = [16, 8, 64, 40, 8, 24]
    cu = np.concatenate([[0], np.cumsum(lens)])
    rnd, cp, rank0, n = HY.schedule(lens, world, 32)
    T, H, d = int(cu[-1]), 2, 8
    q = rng.standard_normal((T, H, d))
    k = rng.standard_normal((T, 1, d))
    v = rng.standard_normal((T, 1, d))
    do = rng.standard_normal((T, H, d))
    seq, pos = A.token_meta_from_cu(cu)
    for r in range(n):
        # the round's sequences form their own packed stream
        ks = [i for i in range(len(lens)) if rnd[i] == r]
        sub_cu = np.concatenate([[0], np.cumsum([lens[i] for i in ks])])
        rows = np.concatenate([np.arange(cu[i], cu[i + 1]) for i in ks])
        idx, lcu = HY.hybrid_layout(sub_cu, cp[ks], rank0[ks], world)
        ranks = [idx[lcu[w, 0]:lcu[w, -1]] for w in range(world)]
        s2, p2 = A.token_meta_from_cu(sub_cu)
        o, l = R.ring_forward(q[rows], k[rows], v[rows], sub_cu, world, ranks=ranks)
        ro, rl = A.attention_forward(q[rows], k[rows], v[rows], s2, p2)
        assert np.max(np.abs(o - ro)) < 1e-12 and np.max(np.abs(l - rl)) < 1e-12
        got = R.ring_backward(q[rows], k[rows], v[rows], do[rows], sub_cu, world, ranks=ranks)
        ref = A.attention_backward(q[rows], k[rows], v[rows], do[rows], s2, p2)
        for a, b in zip(got, ref):
            assert np.max(np.abs(a - b)) < 1e-11
