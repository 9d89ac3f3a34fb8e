"""Partition rules of the context-parallel split, as plain integer loops.

Test infrastructure only (see ``oracle/attention.py``).

* Zigzag split, "04 · Megatron-LM 实现" (llm-infra-atlas, 04_cp/
  04_megatron_cp_integration) §1.1 and "Context Parallelism (CP)" §4: the
  sequence is viewed as 2*cp chunks of equal length and rank r keeps chunk r
  followed by chunk 2*cp-1-r; the length must be a multiple of 2*cp.
* Packed (THD) split, same page §1.2 and §5: the balancing is done inside
  each sub-sequence ("per-sub-sequence zigzag"); on the RoPE side rank r takes
  the front segment [r*seg, (r+1)*seg) and the mirrored back segment
  [full-(r+1)*seg, full-r*seg) of every sub-sequence and concatenates them.
  Reading: sub-sequence major, front then back, seg = len / (2*cp), every
  sub-sequence length a multiple of 2*cp.
* Striped split, "Sequence Parallelism + Ring Attention" §5 (the interleaved
  assignment [0, 4, 8, ...], [1, 5, 9, ...] for four cards): token i goes to
  rank i mod cp, in increasing order.  Reading: the unit is one token, and
  for a packed stream the rule is applied inside every sub-sequence (token
  start_k + r + cp*u at slot u of sub-sequence k on rank r), each length a
  multiple of cp.
"""

from __future__ import annotations

import numpy as np


class PartitionError(ValueError):
    pass


def zigzag_indices(seqlen: int, cp: int) -> np.ndarray:
    """Original token index held at each rank-local slot: int64 [cp, seqlen // cp]."""
    if cp < 1 or seqlen % (2 * cp) != 0:
        raise PartitionError(f"seqlen {seqlen} is not a multiple of 2*cp = {2 * cp}")
    c = seqlen // (2 * cp)
    out = np.empty((cp, 2 * c), dtype=np.int64)
    for r in range(cp):
        front, back = r, 2 * cp - 1 - r
        for t in range(c):
            out[r, t] = front * c + t
            out[r, c + t] = back * c + t
    return out


def thd_partition_indices(cu_seqlens, cp: int) -> np.ndarray:
    """Rank-local token indices of a packed stream: int64 [cp, T // cp].

    For every sub-sequence k (in order), rank r takes its chunk r and its
    chunk 2*cp-1-r, each of length len_k / (2*cp).
    """
    cu = [int(x) for x in cu_seqlens]
    if cp < 1:
        raise PartitionError("cp must be >= 1")
    total = cu[-1]
    if cu[0] != 0:
        raise PartitionError("cu_seqlens must start at 0")
    per_rank = [[] for _ in range(cp)]
    for k in range(len(cu) - 1):
        start, length = cu[k], cu[k + 1] - cu[k]
        if length < 0:
            raise PartitionError("cu_seqlens must be non-decreasing")
        if length % (2 * cp) != 0:
            raise PartitionError(f"sub-sequence {k} length {length} not a multiple of 2*cp")
        c = length // (2 * cp)
        for r in range(cp):
            for chunk in (r, 2 * cp - 1 - r):
                for t in range(c):
                    per_rank[r].append(start + chunk * c + t)
    if total % cp != 0:
        raise PartitionError("total tokens not a multiple of cp")
    return np.array(per_rank, dtype=np.int64).reshape(cp, total // cp)


def thd_rope_segments(cu_seqlens, cp: int) -> np.ndarray:
    """The same split as produced on the RoPE side ("04 · Megatron-LM 实现" §5).

    Per sub-sequence of length `full` with seg = full / (2*cp): rank r takes
    positions [r*seg, (r+1)*seg) then [full-(r+1)*seg, full-r*seg).
    Returned as original token indices, int64 [cp, T // cp].
    """
    cu = [int(x) for x in cu_seqlens]
    per_rank = [[] for _ in range(cp)]
    for k in range(len(cu) - 1):
        full = cu[k + 1] - cu[k]
        seg = full // (2 * cp)
        for r in range(cp):
            front = list(range(r * seg, (r + 1) * seg))
            back = list(range(full - (r + 1) * seg, full - r * seg))
            per_rank[r].extend(cu[k] + p for p in front + back)
    return np.array(per_rank, dtype=np.int64).reshape(cp, cu[-1] // cp)


def striped_indices(seqlen: int, cp: int) -> np.ndarray:
    """Striped split of one sequence: rank r holds tokens r, r + cp, r + 2cp, ...

    int64 [cp, seqlen // cp]; seqlen must be a multiple of cp.
    """
    if cp < 1 or seqlen % cp != 0:
        raise PartitionError(f"seqlen {seqlen} is not a multiple of cp = {cp}")
    n = seqlen // cp
    out = np.empty((cp, n), dtype=np.int64)
    for r in range(cp):
        for u in range(n):
            out[r, u] = r + cp * u
    return out


def thd_striped_indices(cu_seqlens, cp: int) -> np.ndarray:
    """Striped split of a packed stream: int64 [cp, T // cp].

    For every sub-sequence k (in order) rank r takes its tokens r, r + cp, ...
    (len_k / cp of them), so the rank-local stream is sub-sequence major.
    """
    cu = [int(x) for x in cu_seqlens]
    if cp < 1:
        raise PartitionError("cp must be >= 1")
    if cu[0] != 0:
        raise PartitionError("cu_seqlens must start at 0")
    per_rank = [[] for _ in range(cp)]
    for k in range(len(cu) - 1):
        start, length = cu[k], cu[k + 1] - cu[k]
        if length < 0:
            raise PartitionError("cu_seqlens must be non-decreasing")
        if length % cp != 0:
            raise PartitionError(f"sub-sequence {k} length {length} not a multiple of cp")
        for r in range(cp):
            per_rank[r].extend(start + r + cp * u for u in range(length // cp))
    return np.array(per_rank, dtype=np.int64).reshape(cp, cu[-1] // cp)


def local_cu_seqlens(cu_seqlens, cp: int) -> np.ndarray:
    """Sub-sequence boundaries inside one rank's local stream (each holds len/cp)."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    return cu // cp
