"""Oracle: dense-block loads of a block-sparse attention mask (test infrastructure only).

db-SP blog, scenario 2, first bullet: the mask of one head is a 2-D matrix whose
row index is the Q-block and whose column index is the KV-block; an entry that is
non-zero marks a dense block. The work of a Q-block is the number of dense blocks
in its row, the work of a KV-block the number of dense blocks in its column.
db-SP blog, scenario 1: the work of a whole head (the item that head-level
balancing moves between machines) is the number of dense blocks of the head.

db-SP blog, scenario 2: when the KV sequence is split into shards that every head
shares, the load a KV-block brings to its shard is its column count summed over all
heads (``kv_block_loads``).

Two versions are kept: ``block_mask_loads_loops`` walks every entry with Python
loops (tiny masks only) and ``block_mask_loads`` uses numpy sums over ``mask != 0``.
The tests cross-check them on mid-sized masks.

``dense_block_lists`` lists each row's dense blocks themselves (the blocks a row's load
counts), in ascending KV-block order; causal attention computes only those on or below
the diagonal (6D notes, §2.3), so the causal lists stop there.
"""

import numpy as np


def block_mask_loads_loops(mask):
    """Row, column and head loads by explicit loops over every mask entry.

    mask: integer array [B, H, nQ, nK]; any non-zero entry is a dense block.
    Returns (row [B,H,nQ], col [B,H,nK], head [B,H]) as int64 arrays.
    """
    mask = np.asarray(mask)
    B, H, nQ, nK = mask.shape
    row = np.zeros((B, H, nQ), dtype=np.int64)
    col = np.zeros((B, H, nK), dtype=np.int64)
    head = np.zeros((B, H), dtype=np.int64)
    for b in range(B):
        for h in range(H):
            for i in range(nQ):
                for j in range(nK):
                    if mask[b, h, i, j] != 0:
                        row[b, h, i] += 1
                        col[b, h, j] += 1
                        head[b, h] += 1
    return row, col, head


def block_mask_loads(mask):
    """Row, column and head loads with numpy sums of ``mask != 0`` (int64).

    mask: integer array [B, H, nQ, nK]. Returns (row, col, head) like
    ``block_mask_loads_loops``.
    """
    dense = np.asarray(mask) != 0
    row = dense.sum(axis=3, dtype=np.int64)
    col = dense.sum(axis=2, dtype=np.int64)
    head = dense.sum(axis=(2, 3), dtype=np.int64)
    return row, col, head


def kv_block_loads(mask):
    """Column loads summed over (b, h): int64 [nK], by explicit loops over heads."""
    _, col, _ = block_mask_loads(mask)
    B, H, nK = col.shape
    out = np.zeros(nK, dtype=np.int64)
    for b in range(B):
        for h in range(H):
            out += col[b, h]
    return out


def dense_block_lists_loops(mask, causal=False):
    """Each row's dense KV-block indices, ascending, by explicit loops (tiny masks only).

    mask: integer array [B, H, nQ, nK]; rows r = (b*H + h)*nQ + qb. With ``causal`` only
    the blocks j <= qb. Returns a list of int64 arrays, one per row.
    """
    mask = np.asarray(mask)
    B, H, nQ, nK = mask.shape
    rows = mask.reshape(-1, nK)
    out = []
    for r in range(rows.shape[0]):
        limit = min(nK, r % nQ + 1) if causal else nK
        out.append(np.array([j for j in range(limit) if rows[r, j] != 0], dtype=np.int64))
    return out


def dense_block_lists(mask, causal=False):
    """Same as ``dense_block_lists_loops``, with numpy's flatnonzero per row."""
    mask = np.asarray(mask)
    B, H, nQ, nK = mask.shape
    rows = mask.reshape(-1, nK)
    out = []
    for r in range(rows.shape[0]):
        limit = min(nK, r % nQ + 1) if causal else nK
        out.append(np.flatnonzero(rows[r, :limit]).astype(np.int64))
    return out
