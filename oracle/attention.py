"""Oracle: block-sparse multi-head attention forward, final and partial outputs.

Test infrastructure only. All arithmetic in fp64 (numpy).

What is computed (the plain definition the method reaches by skipping blocks):
* 6D attention notes §2.1 (ring-attention pseudocode, step 2): per chunk of KV the
  local attention returns the unnormalised output O, the row maximum m and the row
  sum l of the softmax numerators; the final answer (last line of the loop) is O/l.
* db-SP blog, scenario 2, first bullet: a query attends to the keys of a KV-block
  only where the head's block mask marks that (Q-block, KV-block) pair dense.
* 6D attention notes §2.3: under a causal mask a position attends only to
  positions at or before it.

Readings where the pages are silent: the softmax scale is 1/sqrt(d) unless given;
m, l and the log-sum-exp are in natural-log units of the scaled score; a row with
no admissible key returns O = 0, LSE = -inf (partials: O = 0, m = -inf, l = 0);
causal positions are global (q_pos >= k_pos with S_q = S_kv).

Rows of a query block are independent, so the drivers below evaluate the
definition one query block (or one head) at a time; nothing is fused or reordered
inside a row.
"""

import numpy as np


def allowed_keys(mask_row, block, qb, S, causal):
    """Boolean [block, S]: which keys each query row of Q-block ``qb`` may see.

    mask_row: [nK] entries of the head's block mask for row ``qb``.
    """
    dense_cols = np.repeat(np.asarray(mask_row) != 0, block)  # [S]
    allowed = np.broadcast_to(dense_cols, (block, S)).copy()
    if causal:
        q_pos = qb * block + np.arange(block)
        k_pos = np.arange(S)
        allowed &= k_pos[None, :] <= q_pos[:, None]
    return allowed


def softmax_rows(q_rows, k, v, allowed, scale):
    """Masked softmax attention for a set of query rows, fp64.

    q_rows [R, d], k and v [S, d], allowed [R, S] bool.
    Returns dict with o (normalised) [R, d], lse [R], o_unnorm [R, d], m [R], l [R].
    """
    q_rows = np.asarray(q_rows, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    s = (q_rows @ k.T) * scale
    s = np.where(allowed, s, -np.inf)
    m = s.max(axis=1) if s.shape[1] else np.full(s.shape[0], -np.inf)
    nonempty = np.isfinite(m)
    shift = np.where(nonempty, m, 0.0)
    p = np.exp(s - shift[:, None])  # exp(-inf) = 0 where masked
    l = p.sum(axis=1)
    o_unnorm = p @ v
    safe_l = np.where(nonempty, l, 1.0)
    o = np.where(nonempty[:, None], o_unnorm / safe_l[:, None], 0.0)
    lse = np.where(nonempty, m + np.log(safe_l), -np.inf)
    m_out = np.where(nonempty, m, -np.inf)
    l_out = np.where(nonempty, l, 0.0)
    o_unnorm = np.where(nonempty[:, None], o_unnorm, 0.0)
    return {"o": o, "lse": lse, "o_unnorm": o_unnorm, "m": m_out, "l": l_out}


def default_scale(d):
    return 1.0 / np.sqrt(d)


def attention_item(q, k, v, mask, b, h, qb, block, causal, scale=None):
    """One item (b, h, qb): the ``block`` query rows of Q-block qb of head (b, h).

    q, k, v: arrays [B, H, S, d] (any float dtype; upcast to fp64).
    mask: [B, H, nQ, nK]. Returns the dict of ``softmax_rows``.
    """
    S, d = q.shape[2], q.shape[3]
    if scale is None:
        scale = default_scale(d)
    rows = slice(qb * block, (qb + 1) * block)
    allowed = allowed_keys(mask[b, h, qb], block, qb, S, causal)
    return softmax_rows(q[b, h, rows], k[b, h], v[b, h], allowed, scale)


def admissible_key_positions(mask_row, block, qb, causal):
    """Key positions of the dense KV-blocks of one mask row, ascending, cut at the last
    query position of Q-block ``qb`` when causal (later keys are admissible to no row
    of the block)."""
    cols = np.flatnonzero(np.asarray(mask_row) != 0)
    pos = (cols[:, None] * block + np.arange(block)[None, :]).reshape(-1)
    if causal:
        pos = pos[pos <= (qb + 1) * block - 1]
    return pos


def attention_item_keys(q_rows, k_head, v_head, mask_row, block, qb, causal, scale=None):
    """One item (the ``block`` query rows of Q-block qb), evaluated over its admissible
    keys only: the same masked softmax as ``attention_item``, whose excluded keys carry
    weight exp(-inf) = 0, written as a sum over the admissible set itself. Used where
    the sequence is long and the row sparse.

    q_rows [block, d]; k_head, v_head [S, d] of the item's head; mask_row [nK].
    Returns the dict of ``softmax_rows``.
    """
    d = q_rows.shape[-1]
    if scale is None:
        scale = default_scale(d)
    pos = admissible_key_positions(mask_row, block, qb, causal)
    allowed = np.ones((block, pos.size), dtype=bool)
    if causal:
        q_pos = qb * block + np.arange(block)
        allowed &= pos[None, :] <= q_pos[:, None]
    return softmax_rows(q_rows, np.asarray(k_head)[pos], np.asarray(v_head)[pos], allowed, scale)


def attention_head(q, k, v, mask, b, h, block, causal, scale=None):
    """All query rows of head (b, h), one Q-block at a time.

    Returns dict of arrays over the head's S rows (o [S,d], lse [S], o_unnorm,
    m, l).
    """
    S, d = q.shape[2], q.shape[3]
    nQ = S // block
    kh = np.asarray(k[b, h], dtype=np.float64)
    vh = np.asarray(v[b, h], dtype=np.float64)
    out = {"o": np.zeros((S, d)), "lse": np.zeros(S), "o_unnorm": np.zeros((S, d)),
           "m": np.zeros(S), "l": np.zeros(S)}
    if scale is None:
        scale = default_scale(d)
    for qb in range(nQ):
        rows = slice(qb * block, (qb + 1) * block)
        allowed = allowed_keys(mask[b, h, qb], block, qb, S, causal)
        r = softmax_rows(q[b, h, rows], kh, vh, allowed, scale)
        for key in out:
            out[key][rows] = r[key]
    return out


def attention(q, k, v, mask, block, causal, scale=None):
    """Whole [B, H, S, d] problem. Returns (o [B,H,S,d], lse [B,H,S]) in fp64."""
    B, H, S, d = q.shape
    o = np.zeros((B, H, S, d))
    lse = np.zeros((B, H, S))
    for b in range(B):
        for h in range(H):
            r = attention_head(q, k, v, mask, b, h, block, causal, scale)
            o[b, h], lse[b, h] = r["o"], r["lse"]
    return o, lse


def attention_partials(q, k, v, mask, block, causal, scale=None):
    """Unnormalised partial triple over the whole problem, for one KV shard.

    The shard is expressed by ``mask`` already restricted to the shard's KV-block
    columns (global positions kept). Returns (o_unnorm [B,H,S,d], m [B,H,S],
    l [B,H,S]) in fp64.
    """
    B, H, S, d = q.shape
    o = np.zeros((B, H, S, d))
    m = np.zeros((B, H, S))
    l = np.zeros((B, H, S))
    for b in range(B):
        for h in range(H):
            r = attention_head(q, k, v, mask, b, h, block, causal, scale)
            o[b, h], m[b, h], l[b, h] = r["o_unnorm"], r["m"], r["l"]
    return o, m, l
