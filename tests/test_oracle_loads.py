"""Pins for oracle.loads: the page's definition on a hand-made 4x4 mask, closed forms
on structured masks, the page's causal shard count, and loop/numpy agreement."""

import numpy as np
import pytest

from oracle import loads as L
from load_balancing_gb300 import workloads as W
from conftest import load_golden


def test_4x4_definition_example():
    g = load_golden("loads_4x4.json")
    mask = np.array(g["mask"], dtype=np.uint8)[None, None]
    for fn in (L.block_mask_loads, L.block_mask_loads_loops):
        row, col, head = fn(mask)
        assert row[0, 0].tolist() == g["row_loads"]
        assert col[0, 0].tolist() == g["col_loads"]
        assert int(head[0, 0]) == g["head_load"]


def test_loops_match_numpy_on_random_masks():
    rng = np.random.default_rng(7)
    for shape in [(1, 1, 1, 1), (2, 3, 5, 7), (1, 2, 16, 9), (2, 2, 13, 13)]:
        mask = (rng.random(shape) < 0.4).astype(np.uint8) * rng.integers(1, 255, shape).astype(np.uint8)
        a = L.block_mask_loads(mask)
        b = L.block_mask_loads_loops(mask)
        for x, y in zip(a, b):
            np.testing.assert_array_equal(x, y)


def test_row_and_column_totals_agree():
    rng = np.random.default_rng(1)
    mask = (rng.random((2, 4, 33, 47)) < 0.3).astype(np.uint8)
    row, col, head = L.block_mask_loads(mask)
    np.testing.assert_array_equal(row.sum(-1), col.sum(-1))
    np.testing.assert_array_equal(row.sum(-1), head)


def test_llm_local_heads_closed_form():
    """Window of 4 blocks (diagonal included) plus the block-0 sink, causal.

    Row i keeps {max(0,i-3)..i} and block 0: rows 0..3 see 1,2,3,4 blocks and every
    later row sees 4 + 1 = 5. Column 0 is seen by every row (64); column j >= 1 by
    rows j..j+3 that exist: 4 for j <= 60, then 3, 2, 1. Both total 310 per head.
    """
    w = W.WORKLOADS["llm"]
    mask = W.make_mask(w)
    row, col, head = L.block_mask_loads(mask)
    nQ = w.nQ
    exp_row = np.array([min(i + 1, 4) if i < 4 else 5 for i in range(nQ)])
    exp_col = np.array([nQ] + [min(4, nQ - j) for j in range(1, nQ)])
    for h in range(16, 32):
        np.testing.assert_array_equal(row[0, h], exp_row)
        np.testing.assert_array_equal(col[0, h], exp_col)
        assert head[0, h] == 310
    # global heads: diagonal forced and nothing above it
    assert (row[0, :16] >= 1).all()
    assert (np.triu(mask[0, :16], 1) == 0).all()


def test_full_causal_closed_form_and_shard_sums():
    """Full lower-triangular 256x256 mask: r_i = i+1, c_j = 256-j, total 32896.

    Contiguous shard s owns columns 32s..32s+31, so its column-load sum is
    sum_{j} (256 - j) = 7696 - 1024 s; striped shard s owns j = 8t + s, whose sum
    is 4224 - 32 s.
    """
    w = W.WORKLOADS["sharded"]
    mask = W.make_mask(w)[:, :2]  # two heads are enough; all heads are identical
    row, col, head = L.block_mask_loads(mask)
    n = w.nQ
    np.testing.assert_array_equal(row[0, 0], np.arange(1, n + 1))
    np.testing.assert_array_equal(col[0, 0], n - np.arange(n))
    assert head[0, 0] == n * (n + 1) // 2 == 32896
    for layout, expect in [("contiguous", [7696 - 1024 * s for s in range(8)]),
                           ("striped", [4224 - 32 * s for s in range(8)])]:
        sums = [int(col[0, 0][cols].sum()) for cols in W.shard_columns(n, 8, layout)]
        assert sums == expect
        assert sum(sums) == 32896
        # the same through per-shard masks
        sm = W.shard_masks(mask, 8, layout)
        per = [int(L.block_mask_loads(sm[s])[2][0, 0]) for s in range(8)]
        assert per == expect


@pytest.mark.parametrize("n_shards", [4, 8])
def test_causal_ring_nonempty_pairs(n_shards):
    """6D attention notes §2.3: CP=4 contiguous causal shards leave 10 of 16
    (Q-shard, KV-shard) pairs with work; in general n(n+1)/2 of n^2."""
    g = load_golden("causal_ring_pairs.json")
    nQ = 64
    mask = np.tril(np.ones((nQ, nQ), dtype=np.uint8))[None, None]
    shards = W.shard_columns(nQ, n_shards, "contiguous")
    row_shards = W.shard_columns(nQ, n_shards, "contiguous")
    nonempty = 0
    for qs in row_shards:
        sub = W.shard_masks(mask[:, :, qs, :], n_shards, "contiguous")
        for s in range(n_shards):
            if L.block_mask_loads(sub[s])[2][0, 0] > 0:
                nonempty += 1
    assert nonempty == n_shards * (n_shards + 1) // 2
    if n_shards == g["n_shards"]:
        assert nonempty == g["nonempty_pairs"]
        assert n_shards * n_shards == g["total_pairs"]
    assert len(shards) == n_shards


def test_kv_block_loads_closed_form_and_total():
    """Full causal mask on every head: column j of each head has nQ - j dense blocks,
    so the KV-block load over B*H heads is B*H*(nQ - j); the loads sum to the total."""
    w = W.WORKLOADS["sharded"]
    mask = W.make_mask(w)[:, :3]
    kv = L.kv_block_loads(mask)
    np.testing.assert_array_equal(kv, 3 * (w.nQ - np.arange(w.nK)))
    rng = np.random.default_rng(5)
    m2 = (rng.random((2, 3, 9, 11)) < 0.4).astype(np.uint8)
    kv2 = L.kv_block_loads(m2)
    assert kv2.sum() == (m2 != 0).sum()
    np.testing.assert_array_equal(kv2, (m2 != 0).sum(axis=(0, 1, 2)))


def test_dense_block_lists_pins():
    """The lists: their lengths are the row loads (the independent sums above), every
    entry is a non-zero block in ascending order within the causal limit, the loop and
    numpy versions agree, and the full causal mask lists exactly 0..qb in row qb."""
    g = load_golden("loads_4x4.json")
    mask = np.array(g["mask"], dtype=np.uint8)[None, None]
    lists = L.dense_block_lists(mask)
    assert [len(x) for x in lists] == g["row_loads"]
    for i, x in enumerate(lists):
        assert [j for j in range(4) if g["mask"][i][j] != 0] == x.tolist()
    rng = np.random.default_rng(3)
    for shape in [(1, 1, 1, 1), (2, 3, 7, 7), (1, 2, 16, 16), (1, 1, 9, 20)]:
        m = (rng.random(shape) < 0.4).astype(np.uint8) * rng.integers(1, 255, shape).astype(np.uint8)
        row, _, _ = L.block_mask_loads(m)
        for causal in ([False, True] if shape[2] == shape[3] else [False]):
            a = L.dense_block_lists(m, causal)
            b = L.dense_block_lists_loops(m, causal)
            nQ = shape[2]
            for r, (x, y) in enumerate(zip(a, b)):
                np.testing.assert_array_equal(x, y)
                assert np.all(np.diff(x) > 0)
                assert np.all(m.reshape(-1, shape[3])[r, x] != 0)
                if causal:
                    assert np.all(x <= r % nQ)
            if not causal:
                assert [len(x) for x in a] == row.reshape(-1).tolist()
    full = np.ones((1, 1, 12, 12), dtype=np.uint8)
    for qb, x in enumerate(L.dense_block_lists(full, causal=True)):
        assert x.tolist() == list(range(qb + 1))
