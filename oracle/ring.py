"""The context-parallel pipeline in oracle form: ring walk, partial states, merge.

Test infrastructure only (see ``oracle/attention.py``).

* "Context Parallelism (CP)" §2.1/§2.3 (strategy 1, Q stays and K/V moves):
  rank r keeps its queries; at ring step t it receives the K/V of owner
  s = (r - t) mod cp ("Sequence Parallelism + Ring Attention" §2: the block
  arrives from the previous card; step 0 is the local block).  Each (rank,
  step) pair is one TileAttention edge that yields a partial state.
* same page §2.2: the partial states of a row are merged with the LSE merge.
* "上下文并行" 01 and 02: backward replays each block from the merged row LSE
  and the output, keeps dQ at the query owner and returns the dK/dV
  contributions to the key owner, where they are summed.

Ranks are logical here: everything runs in one process, in ring order.
"""

from __future__ import annotations

import numpy as np

from . import attention as A
from . import partition as P


def rank_indices(cu_seqlens, cp: int, partition: str = "zigzag") -> np.ndarray:
    """Rank-local token order: zigzag (per sub-sequence for THD) or striped."""
    if partition == "zigzag":
        return P.thd_partition_indices(cu_seqlens, cp)
    if partition == "striped":
        return P.thd_striped_indices(cu_seqlens, cp)
    raise ValueError(f"unknown partition {partition!r}")


def ring_forward(q, k, v, cu_seqlens, cp: int, causal: bool = True, scale=None,
                 return_partials: bool = False, partition: str = "zigzag", window: int | None = None,
                 ranks=None):
    """Context-parallel forward over one packed stream.

    q: [T, H, d]; k, v: [T, Hkv, d] in original token order.  Returns O [T, H, d]
    and L [T, H] in original order (plus, if asked, the per-rank list of the
    cp partial states in ring-step order, each in rank-local order).  `ranks`,
    if given, is the list of every rank's token indices (ranks of different
    lengths, e.g. a hybrid round) and replaces the partition rule.
    """
    seq, pos = A.token_meta_from_cu(cu_seqlens)
    idx = rank_indices(cu_seqlens, cp, partition) if ranks is None else [np.asarray(x) for x in ranks]
    cp = len(idx)
    T, H, d = np.shape(q)
    out = np.zeros((T, H, d))
    lse = np.full((T, H), A.NEG_INF)
    partials = []
    for r in range(cp):
        qi = idx[r]
        o_parts, l_parts = [], []
        for t in range(cp):
            s = (r - t) % cp
            kj = idx[s]
            vis = A.visibility(seq[qi], pos[qi], seq[kj], pos[kj], causal, window)
            o_rs, l_rs = A.masked_attention(np.asarray(q)[qi], np.asarray(k)[kj],
                                            np.asarray(v)[kj], vis, scale)
            o_parts.append(o_rs)
            l_parts.append(l_rs)
        o_r, l_r = A.lse_merge(np.stack(o_parts), np.stack(l_parts))
        out[qi] = o_r
        lse[qi] = l_r
        partials.append((o_parts, l_parts))
    if return_partials:
        return out, lse, partials
    return out, lse


def ring_backward(q, k, v, do, cu_seqlens, cp: int, causal: bool = True, scale=None,
                  out=None, lse=None, partition: str = "zigzag", window: int | None = None, ranks=None):
    """Context-parallel backward: replay per (query rank, key owner) block.

    dQ stays with the query rank; each block's dK/dV contribution is returned
    to the key owner and summed there.  Inputs in original token order.
    """
    seq, pos = A.token_meta_from_cu(cu_seqlens)
    if out is None or lse is None:
        out, lse = ring_forward(q, k, v, cu_seqlens, cp, causal, scale, partition=partition, window=window,
                                ranks=ranks)
    q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
    delta = np.einsum("nhd,nhd->nh", do, np.asarray(out, dtype=np.float64))
    idx = rank_indices(cu_seqlens, cp, partition) if ranks is None else [np.asarray(x) for x in ranks]
    cp = len(idx)
    dq = np.zeros(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    for r in range(cp):
        qi = idx[r]
        for t in range(cp):
            s = (r - t) % cp
            kj = idx[s]
            vis = A.visibility(seq[qi], pos[qi], seq[kj], pos[kj], causal, window)
            dq_c, dk_c, dv_c = A.block_backward(q[qi], k[kj], v[kj], do[qi],
                                                np.asarray(lse)[qi], delta[qi], vis, scale)
            dq[qi] += dq_c
            dk[kj] += dk_c          # returned to owner s and summed there
            dv[kj] += dv_c
    return dq, dk, dv
