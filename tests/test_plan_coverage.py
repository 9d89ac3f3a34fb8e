"""The planner's task graph, pair by pair: every (query, key) pair that the
oracle's mask makes visible is covered exactly once by the planner's tables
under the kernels' mask rule (key position <= query position when causal,
query - key < band when a band is set), and no invisible pair is covered.
Checked for all four tables (forward 128-row and 256-row items, backward
key-tile items, dQ items) on the zigzag, packed, striped, sliding-window and
hybrid-CP graphs, in both token orders ("Context Parallelism (CP)" §2.1: the
edge set of the Q-KV graph; host only, no GPU)."""

import numpy as np
import pytest

from oracle import attention as A
from oracle import hybrid as HY
from oracle import partition as P
from tile_attention_lse_gb300 import api
from tile_attention_lse_gb300.synthetic import cu_from_lengths

TABLES = ("fwd", "fwd_wide", "bwd", "dq")


def _token_of_row(p, cu):
    """Original token index held at each row of the token tensors."""
    T = int(cu[-1])
    if p.order == api.CP_ORDER_ORIGINAL:
        return np.arange(T)
    if p.seq_cp is not None:
        return HY.hybrid_layout(cu, p.seq_cp, p.seq_rank0, p.cp)[0]
    if p.partition == api.CP_PARTITION_STRIPED:
        return P.thd_striped_indices(cu, p.cp).reshape(-1)
    return P.thd_partition_indices(cu, p.cp).reshape(-1)


def _coverage(p, cu, which):
    T = int(cu[-1])
    tok = _token_of_row(p, cu)
    items, segs = api.plan_tables(p, which)
    cover = np.zeros((T, T), dtype=np.int32)           # [query token, key token]
    stationary_is_query = which in ("fwd", "fwd_wide", "dq")
    for row0, pos0, ln, sb, sc, _, _, _ in items:
        assert 0 <= row0 and row0 + ln <= T
        srow = np.arange(ln)
        for s_row0, s_pos0, s_len, win in segs[sb:sb + sc]:
            assert 0 <= s_row0 and s_row0 + s_len <= T and s_len > 0
            orow = np.arange(s_len)
            if stationary_is_query:
                qr, kr = row0 + srow[:, None], s_row0 + orow[None, :]
                qp, kp = pos0 + srow[:, None], s_pos0 + orow[None, :]
            else:
                kr, qr = row0 + srow[:, None], s_row0 + orow[None, :]
                kp, qp = pos0 + srow[:, None], s_pos0 + orow[None, :]
            vis = np.ones(np.broadcast(qr, kr).shape, dtype=bool)
            if p.causal:
                vis &= kp <= qp
            if win > 0:
                vis &= qp - kp < win
            qt = np.broadcast_to(tok[qr], vis.shape)[vis]
            kt = np.broadcast_to(tok[kr], vis.shape)[vis]
            np.add.at(cover, (qt, kt), 1)
    return cover


def _check(p, cu):
    seq, pos = A.token_meta_from_cu(cu)
    ref = A.visibility(seq, pos, seq, pos, p.causal, p.window or None).astype(np.int32)
    for which in TABLES:
        got = _coverage(p, cu, which)
        assert np.array_equal(got, ref), which


def _p(**kw):
    base = dict(batch=1, heads_q=4, heads_kv=2, head_dim=128, cp=4, device="cpu")
    base.update(kw)
    return api.Problem(**base)


@pytest.mark.parametrize("order", [api.CP_ORDER_RANK_LOCAL, api.CP_ORDER_ORIGINAL])
@pytest.mark.parametrize("s,cp,causal", [(512, 4, True), (768, 3, True), (256, 2, False), (2048, 8, True)])
def test_zigzag_bshd(order, s, cp, causal):
    _check(_p(seqlen=s, cp=cp, order=order, causal=causal), cu_from_lengths([s]))


@pytest.mark.parametrize("order", [api.CP_ORDER_RANK_LOCAL, api.CP_ORDER_ORIGINAL])
def test_zigzag_thd(order):
    cu = cu_from_lengths([8, 64, 200, 16, 1000, 0, 8, 248])
    _check(_p(seqlen=int(cu[-1]), cu_seqlens=cu, order=order), cu)


@pytest.mark.parametrize("lens,cp", [([1000], 8), ([12, 4, 200, 36, 1000, 8, 252, 0, 4], 4), ([96], 3)])
def test_striped(lens, cp):
    cu = cu_from_lengths(lens)
    kw = dict(cu_seqlens=cu) if len(lens) > 1 else {}
    _check(_p(seqlen=int(cu[-1]), cp=cp, partition=api.CP_PARTITION_STRIPED,
              order=api.CP_ORDER_RANK_LOCAL, **kw), cu)


@pytest.mark.parametrize("lens,cp,w,part", [
    ([2048], 4, 300, api.CP_PARTITION_ZIGZAG), ([2048], 8, 128, api.CP_PARTITION_ZIGZAG),
    ([1024], 2, 1, api.CP_PARTITION_ZIGZAG), ([1000], 8, 77, api.CP_PARTITION_STRIPED),
    ([768], 3, 5, api.CP_PARTITION_STRIPED), ([8, 64, 200, 16, 1000, 8, 248], 4, 150, api.CP_PARTITION_ZIGZAG),
    ([12, 4, 200, 36, 1000, 8, 252, 0, 4], 4, 60, api.CP_PARTITION_STRIPED),
])
def test_sliding_window(lens, cp, w, part):
    cu = cu_from_lengths(lens)
    kw = dict(cu_seqlens=cu) if len(lens) > 1 else {}
    _check(_p(seqlen=int(cu[-1]), cp=cp, window=w, partition=part, order=api.CP_ORDER_RANK_LOCAL, **kw), cu)


@pytest.mark.parametrize("order,w", [(api.CP_ORDER_RANK_LOCAL, 0), (api.CP_ORDER_ORIGINAL, 0),
                                     (api.CP_ORDER_RANK_LOCAL, 100)])
def test_hybrid_round(order, w):
    lens = [512, 64, 256, 8, 128, 0, 40, 384]
    cu = cu_from_lengths(lens)
    _check(_p(seqlen=int(cu[-1]), cu_seqlens=cu, order=order, window=w,
              seq_cp=[4, 1, 2, 1, 1, 1, 2, 2], seq_rank0=[0, 3, 2, 2, 0, 1, 0, 2]), cu)


def test_hybrid_scheduled_rounds():
    world, cap = 8, 256
    rng = np.random.default_rng(3)
    raw = np.exp(rng.normal(np.log(cap) - 0.5, 1.2, 20))
    lens = [int(min(world * cap, max(2 * world, x)) // (2 * world) * (2 * world)) for x in raw]
    rnd, cp, r0, n = api.hybrid_schedule(lens, world, cap)
    for r in range(n):
        ks = [i for i in range(len(lens)) if rnd[i] == r]
        cu = cu_from_lengths([lens[i] for i in ks])
        _check(_p(seqlen=int(cu[-1]), cp=world, cu_seqlens=cu, order=api.CP_ORDER_RANK_LOCAL,
                  seq_cp=cp[ks], seq_rank0=r0[ks]), cu)


def _first_tile_contract(p, cu):
    """The tensor-core forward streams a 256-row item's key tiles segment by
    segment and lets its first Q tile (rows 0..127) stop after the tiles its
    last row can see when those form a prefix of the stream (else it walks
    the whole stream).  Every pair that the first Q tile sees must lie in
    the tiles it walks."""
    items, segs = api.plan_tables(p, "fwd_wide")
    for row0, pos0, ln, sb, sc, _, _, _ in items:
        rows0 = min(ln, 128)
        qlast, qlast0 = pos0 + ln - 1, pos0 + rows0 - 1

        def vis(s_pos0, s_len, last):
            e = s_len
            if p.causal:
                e = min(e, last - s_pos0 + 1)
            return max(e, 0)

        n, n0, cut, prefix = 0, 0, False, True
        walked = []   # (segment, first key offset, last key offset + 1) of every streamed tile
        for si, (s_row0, s_pos0, s_len, win) in enumerate(segs[sb:sb + sc]):
            nt = -(-vis(s_pos0, s_len, qlast) // 128)
            nt0 = -(-vis(s_pos0, s_len, qlast0) // 128)
            if cut and nt0 > 0:
                prefix = False
            if nt0 < nt:
                cut = True
            for t in range(nt):
                walked.append((si, t * 128, min(s_len, t * 128 + 128)))
            n += nt
            n0 += nt0
        nq0 = n0 if prefix else n
        seen = set()
        for si, a, b in walked[:nq0]:
            seen.update((si, j) for j in range(a, b))
        for si, (s_row0, s_pos0, s_len, win) in enumerate(segs[sb:sb + sc]):
            for j in range(s_len):
                kp = s_pos0 + j
                for i in range(rows0):
                    qp = pos0 + i
                    if (not p.causal or kp <= qp) and (win == 0 or qp - kp < win):
                        assert (si, j) in seen
                        break


@pytest.mark.parametrize("kw", [
    dict(seqlen=2048, cp=4),
    dict(seqlen=1000, cp=8, partition=api.CP_PARTITION_STRIPED),
    dict(seqlen=2048, cp=4, window=300),
    dict(seqlen=1000, cp=8, window=77, partition=api.CP_PARTITION_STRIPED),
])
def test_first_q_tile_walks_every_tile_it_sees(kw):
    p = _p(order=api.CP_ORDER_RANK_LOCAL, **kw)
    _first_tile_contract(p, cu_from_lengths([kw["seqlen"]]))


@pytest.mark.parametrize("kw", [
    dict(seqlen=2048, cp=4), dict(seqlen=768, cp=3, order=api.CP_ORDER_ORIGINAL),
    dict(seqlen=1000, cp=8, partition=api.CP_PARTITION_STRIPED), dict(seqlen=2048, cp=8, window=128),
    dict(seqlen=32768, cp=8),
])
def test_partial_rows_written_once_and_merged_to_their_query_row(kw):
    """Forward bookkeeping: every query row is produced exactly once, either
    merged from the partial-state rows that items computed for it (chunks of
    two or more streaming parts: every partial row written by exactly one
    item of each item table) or written directly, final, by exactly one item
    of each table (out_row0 = -1: the chunk's only part)."""
    p = _p(**{"order": api.CP_ORDER_RANK_LOCAL, **kw})
    T = kw["seqlen"]
    merge, _ = api.plan_tables(p, "merge")
    part_of = {}                          # partial row -> query row the merge expects
    for out0, ln, part0, n_parts, stride, _, _, _ in merge:
        assert n_parts >= 2
        for e in range(n_parts):
            for i in range(ln):
                pr = part0 + e * stride + i
                assert pr not in part_of
                part_of[pr] = out0 + i
    merged_rows = set(part_of.values())
    for which in ("fwd", "fwd_wide"):
        items, _ = api.plan_tables(p, which)
        written, direct = {}, set()
        for row0, _, ln, _, _, out0, _, _ in items:
            for i in range(ln):
                if out0 < 0:
                    assert row0 + i not in direct
                    direct.add(row0 + i)
                else:
                    assert out0 + i not in written
                    written[out0 + i] = row0 + i
        assert written == part_of, which
        assert not (direct & merged_rows), which
        assert sorted(direct | merged_rows) == list(range(T)), which    # every query row once
