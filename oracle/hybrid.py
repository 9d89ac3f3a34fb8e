"""Hybrid context parallelism: the per-sub-sequence CP schedule and the token
layout it implies, as plain Python loops.

Test infrastructure only (see ``oracle/attention.py``).

Sources:

* "04 · Megatron-LM 实现" (llm-infra-atlas, 04_cp/04_megatron_cp_integration)
  §7.1, the balanced scheduler, function by function: the cost of a sequence
  is seq_len^2 / cp_size (a proxy, not a FLOP count); the ranks a sequence
  needs are max(1, 2^ceil(log2(seq_len / max_seqlen_per_rank))); sequences
  are bucketed, one bucket per distinct rank count, each bucket aiming at
  total work / buckets and closed once it passes 1.1x that target; the round
  loop puts a sequence into an existing group of its size (the least loaded
  one) and opens a new group only when it does not fit, charges the
  sequence to every rank of the group, stops early when the CP size steps
  down and the rank loads are within 5% (max - min <= 5% of max), then
  trims recently placed sequences to cut slack and merges idle ranks into
  a neighbouring group (ranks stay contiguous); the outer loop sorts by
  length, longest first, and repeats rounds until every sequence is placed.
* same page §2.3: the groups are contiguous power-of-two blocks of ranks,
  aligned to their size (ranks[i : i + size] for i a multiple of size).
* same page §1 and §1.1: a sequence with local CP size g is split over its
  group by the zigzag rule with cp = g.

Readings taken where the page is silent (the page itself calls the scheduler
a heuristic and leaves its capacity test and repair steps open):

* lengths are multiples of 2 * world, so every power-of-two group size up to
  world splits every sequence evenly; the cost seq_len^2 / cp is then an
  exact integer;
* a sequence fits a group of size g when the group's tokens per rank plus
  seq_len / g stay within max_seqlen_per_rank; a new group takes the lowest
  aligned block of g idle ranks; a sequence that fits nowhere waits for the
  next round;
* "the CP size steps down" is the step from one bucket to the next; the
  early stop needs every rank busy;
* trimming ("trim_overload") sheds the last placed sequence while it sits
  on a most loaded group and dropping it strictly lowers the slack, max -
  min of the loads of the busy ranks (idle ranks are the merge step's
  business); merging doubles the most loaded group whose aligned buddy
  block is idle, until none is;
* ties go to the lower rank / earlier sequence.
"""

from __future__ import annotations

import numpy as np


class ScheduleError(ValueError):
    pass


def gpus_needed(length: int, capacity: int) -> int:
    """Smallest power of two g >= 1 with length <= g * capacity."""
    g = 1
    while g * capacity < length:
        g *= 2
    return g


def workload(length: int, cp: int) -> int:
    """The page's cost proxy seq_len^2 / cp_size (exact for the lengths allowed)."""
    return length * length // cp


class _Group:
    def __init__(self, rank0, size):
        self.rank0, self.size = rank0, size
        self.members = []

    def load(self, lens):
        return sum(workload(lens[k], self.size) for k in self.members)

    def tokens(self, lens):
        return sum(lens[k] // self.size for k in self.members)


def _rank_loads(groups, world, lens):
    loads = [0] * world
    for g in groups:
        x = g.load(lens)
        for r in range(g.rank0, g.rank0 + g.size):
            loads[r] = x
    return loads


def _slack(groups, lens):
    """max - min of the loads of the busy ranks (every rank of a group
    carries the group's load)."""
    busy = [g.load(lens) for g in groups if g.members]
    return max(busy) - min(busy) if busy else 0


def _one_round(pending, lens, need, world, capacity):
    """Place what fits of `pending` (longest first) into one round.

    Returns ({sequence: (cp, rank0)}, sequences left for later rounds)."""
    # buckets: one per distinct rank count, closed past 1.1 x the equal share
    nb = len({need[k] for k in pending})
    total = sum(workload(lens[k], need[k]) for k in pending)
    bucket, b, acc = [], 0, 0
    for k in pending:
        w = workload(lens[k], need[k])
        if acc > 0 and b < nb - 1 and 10 * nb * (acc + w) > 11 * total:
            b, acc = b + 1, 0
        bucket.append(b)
        acc += w

    groups, owner_of = [], [None] * world
    placed, left = [], []
    for pos, k in enumerate(pending):
        if pos > 0 and bucket[pos] != bucket[pos - 1]:
            loads = _rank_loads(groups, world, lens)
            if all(o is not None for o in owner_of) and 20 * (max(loads) - min(loads)) <= max(loads):
                left.extend(pending[pos:])
                break
        g = need[k]
        fits = [G for G in groups if G.size == g and G.tokens(lens) + lens[k] // g <= capacity]
        if fits:
            G = min(fits, key=lambda G: (G.load(lens), G.rank0))
        else:
            G = None
            for r0 in range(0, world, g):
                if all(owner_of[r] is None for r in range(r0, r0 + g)):
                    G = _Group(r0, g)
                    groups.append(G)
                    for r in range(r0, r0 + g):
                        owner_of[r] = G
                    break
            if G is None:
                left.append(k)
                continue
        G.members.append(k)
        placed.append(k)

    # trim: an overloaded group sheds its last placed sequence while that
    # strictly cuts the slack
    while len(placed) > 1:
        k = placed[-1]
        before = _slack(groups, lens)
        G = next(G for G in groups if k in G.members)
        if G.load(lens) < max(x.load(lens) for x in groups if x.members):
            break
        G.members.remove(k)
        if _slack(groups, lens) < before:
            placed.pop()
            left.append(k)
            if not G.members:
                groups.remove(G)
                for r in range(G.rank0, G.rank0 + G.size):
                    owner_of[r] = None
        else:
            G.members.append(k)
            break

    # merge idle ranks: double the most loaded group whose buddy block is idle
    while True:
        grown = False
        for G in sorted(groups, key=lambda G: (-G.load(lens), G.rank0)):
            if 2 * G.size > world:
                continue
            buddy = G.rank0 ^ G.size
            if all(owner_of[r] is None for r in range(buddy, buddy + G.size)):
                G.rank0 = min(G.rank0, buddy)
                G.size *= 2
                for r in range(G.rank0, G.rank0 + G.size):
                    owner_of[r] = G
                grown = True
                break
        if not grown:
            break

    out = {k: (G.size, G.rank0) for G in groups for k in G.members}
    return out, left


def schedule(lens, world: int, capacity: int):
    """Rounds of the hybrid schedule.

    Returns int arrays (round, cp, rank0) per sequence and the round count."""
    lens = [int(x) for x in lens]
    if world < 1 or world & (world - 1):
        raise ScheduleError("world must be a power of two")
    if capacity < 1:
        raise ScheduleError("capacity must be >= 1")
    for x in lens:
        if x < 0 or x % (2 * world):
            raise ScheduleError(f"length {x} is not a non-negative multiple of 2*world")
    need = [gpus_needed(x, capacity) for x in lens]
    if any(g > world for g in need):
        raise ScheduleError("a sequence needs more ranks than world")
    n = len(lens)
    rnd, cp, rank0 = np.full(n, -1), np.zeros(n, dtype=np.int64), np.zeros(n, dtype=np.int64)
    pending = sorted(range(n), key=lambda k: (-lens[k], k))
    r = 0
    while pending:
        placed, left = _one_round(pending, lens, need, world, capacity)
        if not placed:
            raise ScheduleError("no progress")
        for k, (g, r0) in placed.items():
            rnd[k], cp[k], rank0[k] = r, g, r0
        pending = sorted(left, key=lambda k: (-lens[k], k))
        r += 1
    return rnd, cp, rank0, r


def rank_loads(lens, cp, rank0, world: int):
    """Cost per rank of one round's assignment (sum of seq_len^2 / cp)."""
    loads = np.zeros(world, dtype=np.int64)
    for x, g, r0 in zip(lens, cp, rank0):
        loads[int(r0):int(r0) + int(g)] += workload(int(x), int(g))
    return loads


def hybrid_layout(cu_seqlens, seq_cp, seq_rank0, world: int):
    """Rank-local token order of one round: rank 0's stream, then rank 1's, ...

    Rank r's stream holds, for every sub-sequence k whose group contains r (in
    sub-sequence order), its zigzag chunk o = r - rank0_k then chunk
    2 cp_k - 1 - o (chunk length len_k / (2 cp_k)).  Returns the original
    token index of every slot (int64 [T]) and local_cu [world][n + 1]: the
    slot where k's part of rank r starts (k = n: where rank r's stream ends).
    """
    cu = [int(x) for x in cu_seqlens]
    n = len(cu) - 1
    idx, local_cu = [], np.zeros((world, n + 1), dtype=np.int64)
    for r in range(world):
        for k in range(n):
            local_cu[r, k] = len(idx)
            g, r0 = int(seq_cp[k]), int(seq_rank0[k])
            if not r0 <= r < r0 + g:
                continue
            length = cu[k + 1] - cu[k]
            if length % (2 * g):
                raise ScheduleError(f"sub-sequence {k} length {length} not a multiple of 2*cp_k")
            c, o = length // (2 * g), r - r0
            for chunk in (o, 2 * g - 1 - o):
                idx.extend(cu[k] + chunk * c + t for t in range(c))
        local_cu[r, n] = len(idx)
    return np.array(idx, dtype=np.int64), local_cu
