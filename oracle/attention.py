"""Float64 CPU oracle for context-parallel causal attention (test infrastructure).

This module is the checker, not the product: only the test suite, the smoke
check in ``__graft_entry__`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may import it.  It shares no code with the CUDA library
and never imports it.

Everything is computed in numpy float64 from the plain definitions on the
pages.  Matrix products (``@``) are the only library primitive; every other
step is written out.  Work is batched over query rows only to bound memory:
each row is still computed exactly as its definition says (the rows of an
attention matrix are independent).

Sources (page title, section, equation):

* "Context Parallelism (CP)" (llm-infra-atlas, parallel/04_cp), §2.1: the
  Q-KV task graph and the partial state A_ij = (O_ij, L_ij) =
  TileAttention(Q_i, K_j, V_j, M_ij), where L_ij is the row log-sum-exp of the
  masked Q_i K_j^T / sqrt(d) and O_ij is normalised inside the segment only.
* same page, §2.2: the merge  L_i = log sum_j exp L_ij,
  O_i = sum_j exp(L_ij - L_i) O_ij, associative and commutative.
* "上下文并行：一条序列跨卡，仍算同一个目标" (glenzli.com, context-parallel),
  02 ONE ROW: the online recurrence (m, l, a) -> O = a / l,
  lambda = m + log l; 01 BACKWARD/REPLAY and GRADIENT/RETURN with the
  second aligned equations of 02: block gradients replayed from the full-row
  LSE, dK/dV contributions summed at the key owner.  01 OWNERSHIP: the causal
  rule uses global positions (j <= i), local indices are storage only.
* "Sequence Parallelism + Ring Attention" (naphjohn LLM-blog,
  sys2-ring-attention), §2: Q stays, K/V blocks arrive in ring order,
  scale 1/sqrt(d).

Reading taken where the pages are silent: natural log for every LSE; a row
with no visible key has L = -inf and O = 0 (never NaN); grouped-query heads map
q-head h to kv-head h // (H / Hkv).

Sliding window ("Context Parallelism (CP)" §2.1 names it as a sparser edge set
of the same graph and gives no formula): reading taken, a causal band of
width W, the query at position i sees the keys at positions i-W+1 .. i of its
sequence (W = 0 or None: no band).
"""

from __future__ import annotations

import math

import numpy as np

NEG_INF = -np.inf

# Rows per block when a query block is materialised against all keys: bounds
# the float64 score block to about 32 MB.
_BLOCK_ELEMS = 1 << 22


def _as_f64(x):
    return np.asarray(x, dtype=np.float64)


def default_scale(head_dim: int) -> float:
    """1/sqrt(d): "Context Parallelism (CP)" §2.1 (Q_i K_j^T / sqrt(d))."""
    return 1.0 / math.sqrt(head_dim)


def token_meta_from_cu(cu_seqlens) -> tuple[np.ndarray, np.ndarray]:
    """Per-token (sequence id, position inside its sequence) of a packed stream.

    "Context Parallelism (CP)" §5: in the packed (THD) layout every document
    restarts its positions at 0 and attention never crosses documents.
    """
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    total = int(cu[-1])
    seq = np.empty(total, dtype=np.int64)
    pos = np.empty(total, dtype=np.int64)
    for k in range(len(cu) - 1):
        a, b = int(cu[k]), int(cu[k + 1])
        seq[a:b] = k
        pos[a:b] = np.arange(b - a)
    return seq, pos


def visibility(q_seq, q_pos, k_seq, k_pos, causal: bool = True, window: int | None = None) -> np.ndarray:
    """M[i, j] = True iff key j is visible to query i.

    Same sequence (block-diagonal mask of the packed layout) and, if causal,
    key position <= query position measured in GLOBAL positions ("上下文并行"
    01 OWNERSHIP; "04 · Megatron-LM 实现" checklist on masking by real
    position after the zigzag split); with a window W > 0 (causal only) also
    query position - key position < W.
    """
    q_seq = np.asarray(q_seq)[:, None]
    k_seq = np.asarray(k_seq)[None, :]
    vis = q_seq == k_seq
    if causal:
        vis = vis & (np.asarray(k_pos)[None, :] <= np.asarray(q_pos)[:, None])
    if window:
        if not causal:
            raise ValueError("a sliding window is a causal band")
        vis = vis & (np.asarray(q_pos)[:, None] - np.asarray(k_pos)[None, :] < window)
    return vis


def masked_attention(q, k, v, vis, scale: float | None = None):
    """TileAttention(Q_i, K_j, V_j, M_ij) -> (O_ij, L_ij).

    "Context Parallelism (CP)" §2.1, equation for A_ij: L is the row
    log-sum-exp of the masked scaled scores, O the output normalised over the
    visible keys of this key set only.  Called with every key of the sequence
    it is plain full attention.

    q: [n, H, d]; k, v: [m, Hkv, d]; vis: bool [n, m].
    Returns O [n, H, d] and L [n, H] (natural log); rows with no visible key
    get O = 0 and L = -inf.
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    n, H, d = q.shape
    m, Hkv, _ = k.shape
    assert H % Hkv == 0
    group = H // Hkv
    if scale is None:
        scale = default_scale(d)
    vis = np.asarray(vis, dtype=bool)
    out = np.zeros((n, H, d))
    lse = np.full((n, H), NEG_INF)
    if n == 0 or m == 0:
        return out, lse
    rows = max(1, _BLOCK_ELEMS // m)
    for r0 in range(0, n, rows):
        r1 = min(n, r0 + rows)
        blk_vis = vis[r0:r1]
        any_vis = blk_vis.any(axis=1)
        for h in range(H):
            g = h // group
            s = scale * (q[r0:r1, h, :] @ k[:, g, :].T)
            s = np.where(blk_vis, s, NEG_INF)
            mx = np.max(s, axis=1)
            mx_safe = np.where(any_vis, mx, 0.0)
            e = np.exp(s - mx_safe[:, None])          # exp(-inf) = 0 for masked keys
            den = e.sum(axis=1)
            with np.errstate(divide="ignore"):
                row_lse = np.where(any_vis, mx_safe + np.log(den), NEG_INF)
            p = np.where(any_vis[:, None], e / np.where(any_vis, den, 1.0)[:, None], 0.0)
            out[r0:r1, h, :] = p @ v[:, g, :]
            lse[r0:r1, h] = row_lse
    return out, lse


def attention_forward(q, k, v, seq_id, pos, causal: bool = True, scale: float | None = None,
                      window: int | None = None):
    """Full masked attention over one token stream (self-attention).

    The plain definition that the whole context-parallel pipeline must
    reproduce ("Context Parallelism (CP)" §2.2: the merge of all partial
    states equals attention over every visible key).
    q: [T, H, d], k/v: [T, Hkv, d]; seq_id/pos: [T].
    """
    vis = visibility(seq_id, pos, seq_id, pos, causal, window)
    return masked_attention(q, k, v, vis, scale)


def attention_forward_rows(rows, q, k, v, seq_id, pos, causal: bool = True,
                           scale: float | None = None, window: int | None = None):
    """Full attention evaluated only for the query rows listed in ``rows``.

    Each output row depends on its own query and on the keys it sees, so a
    subset of rows is computed exactly as in :func:`attention_forward`.
    """
    rows = np.asarray(rows, dtype=np.int64)
    seq_id, pos = np.asarray(seq_id), np.asarray(pos)
    vis = visibility(seq_id[rows], pos[rows], seq_id, pos, causal, window)
    return masked_attention(np.asarray(q)[rows], k, v, vis, scale)


def lse_merge(o_parts, l_parts):
    """The merge  A_i = (+)_j A_ij  of partial states.

    "Context Parallelism (CP)" §2.2: L_i = log sum_j exp(L_ij) and
    O_i = sum_j exp(L_ij - L_i) O_ij.  The log-sum-exp is evaluated with the
    usual max shift; partials with L = -inf carry weight 0, and a row whose
    partials are all -inf merges to L = -inf, O = 0.

    o_parts: [P, n, H, d]; l_parts: [P, n, H].
    """
    o_parts, l_parts = _as_f64(o_parts), _as_f64(l_parts)
    mx = np.max(l_parts, axis=0)                       # [n, H]
    alive = np.isfinite(mx)
    mx_safe = np.where(alive, mx, 0.0)
    w_un = np.exp(l_parts - mx_safe[None])             # exp(-inf) = 0
    tot = w_un.sum(axis=0)
    with np.errstate(divide="ignore"):
        lse = np.where(alive, mx_safe + np.log(np.where(alive, tot, 1.0)), NEG_INF)
    w = np.where(alive[None], np.exp(l_parts - np.where(alive, lse, 0.0)[None]), 0.0)
    out = np.einsum("pnh,pnhd->nhd", w, o_parts)
    return out, lse


def online_softmax_row(score_blocks, value_blocks):
    """One query row absorbed block by block with the running state (m, l, a).

    "上下文并行" 02 ONE ROW: m' = max(m, max_B S), c = e^(m - m'),
    l' = c l + sum_B e^(S - m'), a' = c a + sum_B e^(S - m') V, and at the end
    O = a / l, lambda = m + log l.  Masked scores are -inf.
    score_blocks: list of [b] arrays; value_blocks: list of [b, d] arrays.
    """
    d = value_blocks[0].shape[1]
    m, ell, acc = NEG_INF, 0.0, np.zeros(d)
    for s, vb in zip(score_blocks, value_blocks):
        s = _as_f64(s)
        vb = _as_f64(vb)
        m_new = max(m, float(np.max(s))) if s.size else m
        if m_new == NEG_INF:
            continue
        c = math.exp(m - m_new) if m != NEG_INF else 0.0
        e = np.exp(s - m_new)
        ell = c * ell + float(e.sum())
        acc = c * acc + e @ vb
        m = m_new
    if ell == 0.0:
        return np.zeros(d), NEG_INF
    return acc / ell, m + math.log(ell)


def block_backward(q, k, v, do, lse, delta, vis, scale: float | None = None):
    """Replay of one (query block, key block) pair of the backward pass.

    "上下文并行" 01 BACKWARD/REPLAY: the local probabilities are rebuilt from the
    full-row LSE, P_ij = exp(S_ij - L_i); with the output-gradient dot product
    D_i = <dO_i, O_i> the block gives
      dV_j += sum_i P_ij dO_i,   dP_ij = <dO_i, V_j>,   dS_ij = P_ij (dP_ij - D_i),
      dQ_i += scale sum_j dS_ij K_j,   dK_j += scale sum_i dS_ij Q_i,
    the textbook softmax-attention gradient that 02's second aligned equations
    state for dK and dV.  Grouped heads sum into their kv-head.

    q, do: [n, H, d]; k, v: [m, Hkv, d]; lse, delta: [n, H]; vis: bool [n, m].
    Returns (dq [n,H,d], dk [m,Hkv,d], dv [m,Hkv,d]) contributions.
    """
    q, k, v, do = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(do)
    lse, delta = _as_f64(lse), _as_f64(delta)
    n, H, d = q.shape
    m, Hkv, _ = k.shape
    group = H // Hkv
    if scale is None:
        scale = default_scale(d)
    vis = np.asarray(vis, dtype=bool)
    dq = np.zeros((n, H, d))
    dk = np.zeros((m, Hkv, d))
    dv = np.zeros((m, Hkv, d))
    if n == 0 or m == 0:
        return dq, dk, dv
    rows = max(1, _BLOCK_ELEMS // m)
    for r0 in range(0, n, rows):
        r1 = min(n, r0 + rows)
        blk_vis = vis[r0:r1]
        for h in range(H):
            g = h // group
            row_l = lse[r0:r1, h]
            ok = np.isfinite(row_l)
            s = scale * (q[r0:r1, h, :] @ k[:, g, :].T)
            p = np.where(blk_vis & ok[:, None],
                         np.exp(s - np.where(ok, row_l, 0.0)[:, None]), 0.0)
            dv[:, g, :] += p.T @ do[r0:r1, h, :]
            dp = do[r0:r1, h, :] @ v[:, g, :].T
            ds = p * (dp - delta[r0:r1, h][:, None])
            dq[r0:r1, h, :] += scale * (ds @ k[:, g, :])
            dk[:, g, :] += scale * (ds.T @ q[r0:r1, h, :])
    return dq, dk, dv


def attention_backward(q, k, v, do, seq_id, pos, causal: bool = True,
                       scale: float | None = None, out=None, lse=None, window: int | None = None):
    """Gradients (dQ, dK, dV) of full masked attention for upstream dO.

    O and LSE come from :func:`attention_forward` unless given; D_i is the
    dot product of dO_i with the forward output O_i ("上下文并行" 01
    BACKWARD/REPLAY: the replay uses the full-row LSE and the output).
    """
    if out is None or lse is None:
        out, lse = attention_forward(q, k, v, seq_id, pos, causal, scale, window)
    delta = np.einsum("nhd,nhd->nh", _as_f64(do), _as_f64(out))
    vis = visibility(seq_id, pos, seq_id, pos, causal, window)
    return block_backward(q, k, v, do, lse, delta, vis, scale)


# ---------------------------------------------------------------------------
# Batched (BSHD) conveniences: every batch entry is an independent sequence.
# ---------------------------------------------------------------------------

def attention_forward_bshd(q, k, v, causal: bool = True, scale: float | None = None,
                           window: int | None = None):
    """q: [b, s, H, d]; k/v: [b, s, Hkv, d] -> O [b, s, H, d], L [b, s, H]."""
    b, s = q.shape[:2]
    seq = np.zeros(s, dtype=np.int64)
    pos = np.arange(s)
    outs, lses = [], []
    for i in range(b):
        o, l = attention_forward(q[i], k[i], v[i], seq, pos, causal, scale, window)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


def attention_backward_bshd(q, k, v, do, causal: bool = True, scale: float | None = None,
                            window: int | None = None):
    b, s = q.shape[:2]
    seq = np.zeros(s, dtype=np.int64)
    pos = np.arange(s)
    res = [attention_backward(q[i], k[i], v[i], do[i], seq, pos, causal, scale, window=window)
           for i in range(b)]
    return tuple(np.stack([r[j] for r in res]) for j in range(3))
