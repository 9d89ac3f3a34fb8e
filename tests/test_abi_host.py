"""CPU-only checks of the C ABI: the library loads, exports every declared
symbol, validates descriptors and plans the task graph (no GPU calls)."""

import os
import re

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import partition as P
from tile_attention_lse_gb300 import api
from tile_attention_lse_gb300.synthetic import cu_from_lengths, packed_lengths

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "cpattn.h")).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(cp_\w+)\s*\(", src, re.M)))


def test_library_exports_every_declared_symbol():
    L = api.lib()
    declared = _declared()
    assert set(declared) == set(api.EXPORTS), declared
    for name in declared:
        assert hasattr(L, name), name


def test_status_strings():
    for code, name in api.STATUS.items():
        assert api.status_string(code) == name


def _p(**kw):
    base = dict(batch=1, heads_q=4, heads_kv=4, head_dim=128, cp=2, seqlen=256, device="cpu")
    base.update(kw)
    return api.Problem(**base)


def test_validation_codes():
    assert api.validate(_p()) == 0
    assert api.validate(_p(seqlen=250)) == -2                       # not a multiple of 2cp
    assert api.validate(_p(head_dim=96)) == -3
    assert api.validate(_p(heads_q=6, heads_kv=4)) == -3
    assert api.validate(_p(batch=4, seqlen=(1 << 29) + (1 << 20))) == -3  # 2^31 rows: 32-bit row index
    assert api.validate(_p(cp=0)) == -1
    assert api.validate(_p(seqlen=48, cu_seqlens=[0, 16, 48])) == 0
    assert api.validate(_p(seqlen=48, cu_seqlens=[0, 18, 48])) == -2  # 18 % 4
    assert api.validate(_p(seqlen=48, cu_seqlens=[0, 32, 16, 48])) == -1  # decreasing
    assert api.validate(_p(seqlen=48, cu_seqlens=[0, 16, 40])) == -1  # total mismatch
    assert api.validate(_p(batch=2, seqlen=48, cu_seqlens=[0, 48])) == -1
    assert api.validate(_p(seqlen=0)) == 0


def _parts_per_chunk(a, cp, c, part_tiles=128):
    """Streaming parts of causal Q chunk a (BSHD): its edges in ring order
    (owner s = (r - t) mod cp; chunks s, 2cp-1-s visible when <= a), consecutive
    edges grouped until a part holds its share of about part_tiles key tiles
    (128, the planner's part size)."""
    r = a if a < cp else 2 * cp - 1 - a
    tiles = -(-c // 128)
    edge_tiles = []
    for t in range(cp):
        s_ = (r - t) % cp
        n = sum(1 for b in (s_, 2 * cp - 1 - s_) if b <= a)
        if n:
            edge_tiles.append(n * tiles)
    total = sum(edge_tiles)
    want = max(1, min(len(edge_tiles), -(-total // part_tiles)))
    parts, acc, filled = 1, 0, False
    for x in edge_tiles:
        if filled and parts < want and acc * want >= total * parts:
            parts += 1
        filled = True
        acc += x
    return parts, len(edge_tiles)


@pytest.mark.parametrize("s,cp", [(256, 2), (16384, 8), (131072, 16), (32768, 8), (64, 1)])
def test_plan_counts_bshd(s, cp):
    st = api.plan_stats(_p(seqlen=s, cp=cp))
    c = s // (2 * cp)
    assert st["pairs"] == s * (s + 1) // 2
    # edges per rank: (r + 1) for the front chunk, cp for the back chunk
    n_edges = sum(r + 1 + cp for r in range(cp))
    assert sum(_parts_per_chunk(a, cp, c)[1] for a in range(2 * cp)) == n_edges
    per_chunk = [_parts_per_chunk(a, cp, c)[0] for a in range(2 * cp)]
    parts = sum(per_chunk)
    q_tiles = -(-c // 128)
    assert st["fwd_items"] == parts * q_tiles
    # partial states only for chunks walked in two or more parts; a chunk of
    # one part is written to the outputs by its items
    multi = [x for x in per_chunk if x > 1]
    assert st["partial_rows"] == sum(multi) * c <= n_edges * c == s * (3 * cp + 1) // 4
    assert st["merge_segments"] == len(multi)
    assert st["bwd_items"] == 2 * cp * q_tiles
    # key-tile visits do not depend on how edges are grouped: every visible
    # chunk once per Q tile
    vis_chunks = sum(a + 1 for a in range(2 * cp))
    assert st["fwd_key_tiles"] == vis_chunks * q_tiles * q_tiles - (2 * cp) * (q_tiles * (q_tiles - 1) // 2)


def test_plan_parts_bench_shape():
    # b2 h32 s32768 cp8 (c = 2048 = 16 key tiles per chunk): one part per front
    # chunk (written to the outputs directly), two per back chunk (two partial
    # states each, merged): one partial row per query row on average instead
    # of one per edge (6.25), and merges for half of the rows
    st = api.plan_stats(_p(seqlen=32768, cp=8))
    assert st["partial_rows"] == 8 * 2 * 2048
    assert st["merge_segments"] == 8


def test_plan_pairs_thd_match_oracle():
    lens = packed_lengths(4096, 4, seed=0, mu=5.0, sigma=1.0, lo=8, hi=2048)
    cu = cu_from_lengths(lens)
    st = api.plan_stats(_p(seqlen=int(cu[-1]), cp=4, cu_seqlens=cu))
    seq, pos = A.token_meta_from_cu(cu)
    vis = A.visibility(seq, pos, seq, pos, True)
    assert st["pairs"] == int(vis.sum())
    # chunks of at most 256 tokens see at most 16 key tiles: one part each,
    # written directly, so nothing is merged
    assert st["merge_segments"] == 0 and st["partial_rows"] == 0


def test_workspace_sizes():
    p = _p(seqlen=32768, cp=8, heads_q=32, heads_kv=32, batch=2)
    st = api.plan_stats(p)
    fwd = api.workspace_bytes(p, False)
    bwd = api.workspace_bytes(p, True)
    assert fwd >= 2 * st["partial_rows"] * 32 * (128 * 4 + 4)
    assert bwd >= 2 * 32768 * 32 * 8          # D and log2-scaled LSE per (row, head)
    assert api.workspace_bytes(_p(seqlen=250), False) == 0


def test_workspace_zero_for_unbuilt_attention_shapes():
    # bf16 attention is built for head_dim 128 only: no workspace (the entry
    # points return CP_ERR_UNSUPPORTED instead of running another kernel class)
    assert api.workspace_bytes(_p(head_dim=64)) == 0
    assert api.workspace_bytes(_p(head_dim=64), True) == 0
    assert api.workspace_bytes(_p(head_dim=64, dtype=torch.float32)) > 0
    assert api.workspace_bytes(_p()) > 0
    assert api.validate(_p(head_dim=64)) == 0      # the partition and gathers still take it


def test_wait_limit_host_checks():
    L = api.lib()
    assert L.cp_debug_set_wait_limit(10 ** 12) == -1   # above the default budget
    assert L.cp_debug_set_wait_limit(1000) == 0
    assert L.cp_debug_set_wait_limit(0) == 0           # back to the default
    assert L.cp_debug_set_wait_limit(-3) == 0


def test_synthetic_packed_lengths_recipe():
    for seed in range(4):
        lens = packed_lengths(65536, 4, seed)
        assert sum(lens) == 65536
        assert all(x % 8 == 0 and x >= 128 for x in lens)
        assert max(lens) <= 16384
    # the partition oracle accepts the stream
    P.thd_partition_indices(cu_from_lengths(packed_lengths(65536, 4, 0)), 4)


def test_bwd_schedule_covers_every_work_index_once_and_balances():
    """The tensor-core backward's per-CTA work lists: every (batch, kv-head,
    item) index exactly once, each CTA's list in increasing (head-major)
    order, and planned CTA loads within one item of each other (the greedy
    least-loaded assignment)."""
    import numpy as np
    cases = [dict(batch=2, heads_q=32, heads_kv=32, seqlen=32768, cp=8),
             dict(batch=3, heads_q=8, heads_kv=2, seqlen=4096, cp=4),
             dict(batch=1, heads_q=4, heads_kv=4, seqlen=256, cp=2)]
    for kw in cases:
        p = _p(**kw)
        st = api.plan_stats(p)
        sc = api.bwd_schedule(p)
        total = kw["batch"] * kw["heads_kv"] * st["bwd_items"]
        assert 0 < sc["grid"] <= total
        assert sc["cta"][0] == 0 and sc["cta"][-1] == total and np.all(np.diff(sc["cta"]) >= 0)
        assert np.array_equal(np.sort(sc["work"]), np.arange(total))
        for c in range(sc["grid"]):
            w = sc["work"][sc["cta"][c]:sc["cta"][c + 1]]
            assert np.all(np.diff(w) > 0)
        group = kw["heads_q"] // kw["heads_kv"]
        max_item = (kw["seqlen"] // 128 + 1) * group + 1  # query tiles one key tile can see
        assert int(sc["load"].max() - sc["load"].min()) <= max_item
        assert int(sc["load"].sum()) >= 2 * total  # every item: at least one query tile + 1


def test_validation_striped():
    S, L = api.CP_PARTITION_STRIPED, api.CP_ORDER_RANK_LOCAL
    assert api.validate(_p(seqlen=12, cp=4, partition=S, order=L)) == 0      # a multiple of cp suffices
    assert api.validate(_p(seqlen=12, cp=4, order=L)) == -2                  # zigzag wants 2cp
    assert api.validate(_p(seqlen=10, cp=4, partition=S, order=L)) == -2
    assert api.validate(_p(seqlen=12, cp=4, partition=S)) == -3              # original order: strided ranks
    assert api.validate(_p(seqlen=48, cp=4, partition=S, order=L, cu_seqlens=[0, 12, 48])) == 0
    assert api.validate(_p(seqlen=48, cp=4, partition=S, order=L, cu_seqlens=[0, 14, 48])) == -2
    assert api.validate(_p(seqlen=12, cp=4, partition=2, order=L)) == -1


@pytest.mark.parametrize("s,cp", [(256, 2), (32768, 8), (12, 4), (3000, 8), (64, 1)])
def test_plan_counts_striped(s, cp):
    """Striped split ("Sequence Parallelism + Ring Attention" §5): one Q chunk
    per rank (n = s / cp rows at virtual positions 0 .. n-1), every owner's
    stream visible from virtual position [owner > rank]."""
    p = _p(seqlen=s, cp=cp, partition=api.CP_PARTITION_STRIPED, order=api.CP_ORDER_RANK_LOCAL)
    st = api.plan_stats(p)
    n = s // cp
    assert st["pairs"] == s * (s + 1) // 2
    # a rank's chunk streams every owner's visible keys (n - [owner > rank] of
    # them for its last row) in parts of about 128 key tiles; only chunks of
    # two or more parts get partial rows and a merge segment
    parts = []
    for r in range(cp):
        tiles = [-(-(n - (1 if s_ > r else 0)) // 128) for s_ in range(cp)]
        tiles = [t for t in tiles if t > 0]
        parts.append(max(1, min(len(tiles), -(-sum(tiles) // 128))))
    assert st["merge_segments"] == sum(1 for x in parts if x > 1)
    assert st["partial_rows"] == sum(x for x in parts if x > 1) * n
    q_tiles = -(-n // 128)
    assert st["bwd_items"] == cp * q_tiles
    key_tiles = 0
    for r in range(cp):
        for j in range(q_tiles):
            qlast = min(n, 128 * (j + 1)) - 1
            for s_ in range(cp):
                vis = max(0, min(n, qlast - (1 if s_ > r else 0) + 1))
                key_tiles += -(-vis // 128)
    assert st["fwd_key_tiles"] == key_tiles


def test_validation_window():
    assert api.validate(_p(window=100)) == 0
    assert api.validate(_p(window=-1)) == -1
    assert api.validate(_p(window=1 << 30)) == -1
    assert api.validate(_p(window=100, causal=False)) == -3      # a causal band only


@pytest.mark.parametrize("kw", [
    dict(seqlen=4096, cp=4, window=300),
    dict(seqlen=32768, cp=8, window=4096),
    dict(seqlen=3000, cp=8, window=77, partition=api.CP_PARTITION_STRIPED, order=api.CP_ORDER_RANK_LOCAL),
    dict(seqlen=4096, cp=4, window=1),
])
def test_plan_window_pairs_and_tiles(kw):
    """Under a sliding window the plan covers exactly the band's pairs (the
    oracle's visibility count) and streams fewer key tiles than without it;
    a band as wide as the sequence plans the plain causal graph."""
    st = api.plan_stats(_p(**kw))
    s, w = kw["seqlen"], kw["window"]
    if s <= 4096:
        seq, pos = np.zeros(s, int), np.arange(s)
        assert st["pairs"] == int(A.visibility(seq, pos, seq, pos, True, w).sum())
    else:  # the band's closed form (pinned against the oracle's mask on small cases)
        assert st["pairs"] == w * (w + 1) // 2 + (s - w) * w
    full = api.plan_stats(_p(**{**kw, "window": 0}))
    assert st["fwd_key_tiles"] < full["fwd_key_tiles"]
    assert st["fwd_key_tiles"] * 128 * 128 >= st["pairs"]
    assert api.plan_stats(_p(**{**kw, "window": s})) == full


def test_plan_window_thd_pairs():
    lens = packed_lengths(4096, 4, seed=1, mu=5.0, sigma=1.0, lo=8, hi=2048)
    cu = cu_from_lengths(lens)
    st = api.plan_stats(_p(seqlen=int(cu[-1]), cp=4, cu_seqlens=cu, window=100))
    seq, pos = A.token_meta_from_cu(cu)
    assert st["pairs"] == int(A.visibility(seq, pos, seq, pos, True, 100).sum())


# ---------------------------------------------------------------- hybrid CP --
def _long_tail(seed, n, world, cap):
    rng = np.random.default_rng(seed)
    raw = np.exp(rng.normal(np.log(cap) - 0.5, 1.3, n))
    return [int(min(world * cap, max(2 * world, x)) // (2 * world) * (2 * world)) for x in raw]


@pytest.mark.parametrize("seed,n,world,cap", [(0, 40, 8, 4096), (1, 60, 8, 2048), (2, 25, 4, 8192),
                                              (3, 80, 16, 1024), (4, 10, 2, 4096), (5, 1, 8, 512),
                                              (6, 200, 8, 8192), (7, 30, 1, 65536)])
def test_hybrid_schedule_matches_oracle(seed, n, world, cap):
    """The library's scheduler and the oracle's, written apart from the same
    reading of the page, agree on every round, CP size and group."""
    from oracle import hybrid as HY
    lens = _long_tail(seed, n, world, cap)
    rnd, cp, r0, nr = api.hybrid_schedule(lens, world, cap)
    ornd, ocp, or0, onr = HY.schedule(lens, world, cap)
    assert nr == onr
    assert rnd.tolist() == ornd.tolist() and cp.tolist() == ocp.tolist() and r0.tolist() == or0.tolist()


def test_hybrid_schedule_hand_case_and_errors():
    rnd, cp, r0, nr = api.hybrid_schedule([128, 64, 64, 32, 32], 4, 64)
    assert nr == 2 and rnd.tolist() == [0, 0, 0, 1, 1]
    assert cp.tolist() == [2, 1, 1, 4, 4] and r0.tolist() == [0, 2, 3, 0, 0]
    assert api.hybrid_schedule([], 4, 64)[3] == 0
    for args, code in ((([64], 3, 64), -1), (([60], 4, 64), -2), (([1024], 4, 64), -3), (([64], 4, 0), -1),
                       (([-8], 4, 64), -1)):
        with pytest.raises(api.CpError) as e:
            api.hybrid_schedule(*args)
        assert e.value.code == code


def test_validation_hybrid():
    cu = [0, 16, 48, 64, 128]
    ok = dict(seqlen=128, cp=4, cu_seqlens=cu, seq_cp=[2, 1, 2, 4], seq_rank0=[0, 3, 2, 0])
    assert api.validate(_p(**ok)) == 0
    assert api.validate(_p(**{**ok, "seq_cp": [2, 1, 2, 3]})) == -1       # not a power of two
    assert api.validate(_p(**{**ok, "seq_rank0": [1, 3, 2, 0]})) == -1    # group not aligned
    assert api.validate(_p(**{**ok, "seq_rank0": [0, 3, 2, 2]})) == -1    # past the last rank
    assert api.validate(_p(**{**ok, "seq_cp": [2, 1, 2, 8]})) == -1       # larger than cp
    assert api.validate(_p(seqlen=44, cp=4, cu_seqlens=[0, 12, 44], seq_cp=[4, 1], seq_rank0=[0, 0])) == -2  # 12 % 8
    assert api.validate(_p(seqlen=44, cp=4, cu_seqlens=[0, 12, 44], seq_cp=[2, 1], seq_rank0=[0, 0])) == 0
    assert api.validate(_p(**{**ok, "partition": api.CP_PARTITION_STRIPED,
                              "order": api.CP_ORDER_RANK_LOCAL})) == -1
    assert api.validate(_p(seqlen=128, cp=4, seq_cp=[4], seq_rank0=[0])) == -1   # BSHD


def test_plan_hybrid_counts():
    """Each sub-sequence on its group: 2 cp_k chunks (each streamed in one part
    here: at most 16 key tiles, so written directly and never merged), the band
    of causal pairs unchanged, backward items per chunk tile of its own split."""
    cu = [0, 16, 48, 64, 128, 128, 384]
    seq_cp, seq_r0 = [2, 1, 2, 4, 1, 8], [0, 3, 2, 0, 5, 0]
    st = api.plan_stats(_p(seqlen=384, cp=8, cu_seqlens=cu, seq_cp=seq_cp, seq_rank0=seq_r0,
                           order=api.CP_ORDER_RANK_LOCAL))
    lens = np.diff(cu)
    assert st["pairs"] == int(sum(x * (x + 1) // 2 for x in lens))
    assert st["merge_segments"] == 0 and st["partial_rows"] == 0
    assert st["fwd_items"] == sum(2 * g * -(-(x // (2 * g)) // 128) for x, g in zip(lens, seq_cp) if x > 0)
    assert st["bwd_items"] == sum(2 * g * -(-(x // (2 * g)) // 128) for x, g in zip(lens, seq_cp) if x > 0)


def test_header_is_plain_c():
    """include/cpattn.h is a C header (the boundary is a C ABI): it parses as
    C99 and as C++17 without warnings."""
    import shutil
    import subprocess
    hdr = os.path.join(ROOT, "include", "cpattn.h")
    for cc, std, lang in (("gcc", "c99", "c"), ("g++", "c++17", "c++")):
        if shutil.which(cc) is None:
            pytest.skip(f"{cc} not installed")
        res = subprocess.run([cc, "-fsyntax-only", f"-std={std}", "-Wall", "-Wextra", "-Werror", "-x", lang, hdr],
                             capture_output=True, text=True)
        assert res.returncode == 0, res.stderr
